// cbq_budget.h -- host-side glue of the expert-budget kernel (cbq_budget.cu)
// for the C entry point in cbq_api.cu.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace cbq {

// At most this many experts (one shared-memory word per expert) and at most
// this many choices per token (the routing cbq_grouped_gemm takes has at most 8).
constexpr int kMaxBudgetExperts = 4096;
constexpr int kMaxBudgetK = 8;

int launch_budget(const float* logits, int T, int E, int k, int B, int32_t* budget, int32_t* topk,
                  cudaStream_t stream);

}  // namespace cbq
