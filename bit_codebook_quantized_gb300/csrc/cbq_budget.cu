// cbq_budget.cu -- the shared expert budget of one verify round.
//
// "Hibana: Fast Agentic Inference on Unified-Memory Devices", section
// "Adaptive speculation / Expert sharing": checking a round of drafted tokens
// has to read every expert chosen by at least one of them; limiting the whole
// round to one common set of experts cuts the bytes read, and a token whose
// choice falls outside the set takes its best expert inside it instead.  The
// page illustrates this on a small example only; the rule (every decision a
// comparison or an integer sum, so it is reproducible exactly):
//  1. each token ranks the experts by its router logit (higher first, equal
//     logits -> lower id) and takes its own top-k;
//  2. expert e scores sum over tokens of (k - r), r its 0-based rank in that
//     token's own top-k;
//  3. the budget is the B highest-scoring experts (ties -> lower id);
//  4. each token takes its top-k among the budget experts, in rank order.
// The result (topk_idx, [T][k]) is what cbq_grouped_gemm reads.
//
// One CTA of 8 warps (a round has at most a few dozen tokens): a warp copies a
// token's logits into its own shared-memory row once, then finds each next
// choice as the best (logit, id) that ranks after the previous one, so no
// per-token state beyond the previous pick is kept; expert scores are
// shared-memory integers.
#include <cuda_runtime.h>

#include <cstdint>

#include "cbq_budget.h"
#include "cbq_internal.h"

namespace cbq {
namespace {

constexpr int kBudgetWarps = 8;
constexpr int kBudgetThreads = kBudgetWarps * 32;

// (v, e) ranks before (w, f): larger value first, equal values -> lower id.
template <typename V>
__device__ __forceinline__ bool ranks_before(V v, int e, V w, int f) {
  return v > w || (v == w && e < f);
}

// Keep (ov, oe) in (bv, be) if it ranks before it (id -1 = nothing yet).
template <typename V>
__device__ __forceinline__ void keep_better(V& bv, int& be, V ov, int oe) {
  if (oe >= 0 && (be < 0 || ranks_before(ov, oe, bv, be))) {
    bv = ov;
    be = oe;
  }
}

template <typename V>
__device__ __forceinline__ void warp_best(V& bv, int& be) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const V ov = __shfl_xor_sync(0xffffffffu, bv, off);
    const int oe = __shfl_xor_sync(0xffffffffu, be, off);
    keep_better(bv, be, ov, oe);
  }
}

// A token's next choice: the best (logit, id) of its row that ranks after
// (pv, pe) (pe < 0: the first choice), among the experts `allowed` marks (all
// if null).  Every lane of the warp returns it.
__device__ __forceinline__ int next_choice(const float* row, int E, float pv, int pe, const uint8_t* allowed,
                                           float& bv) {   // row: the warp's shared-memory copy
  const int lane = threadIdx.x & 31;
  int be = -1;
  bv = 0.f;
  for (int e = lane; e < E; e += 32) {
    if (allowed && !allowed[e]) continue;
    const float v = row[e];
    if (pe >= 0 && !ranks_before(pv, pe, v, e)) continue;
    keep_better(bv, be, v, e);
  }
  warp_best(bv, be);
  return be;
}

__global__ void __launch_bounds__(kBudgetThreads) budget_kernel(const float* __restrict__ logits, int T, int E,
                                                                 int k, int B, int32_t* __restrict__ budget_out,
                                                                 int32_t* __restrict__ topk_out) {
  __shared__ int score[kMaxBudgetExperts];
  __shared__ uint8_t in_budget[kMaxBudgetExperts];
  __shared__ int red_s[kBudgetWarps], red_e[kBudgetWarps];
  __shared__ int pick;
  extern __shared__ float rows[];                       // [kBudgetWarps][E]: one token row per warp
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* my_row = rows + static_cast<size_t>(warp) * E;
  auto stage_row = [&](int t) {                         // the token's logits, coalesced, once
    __syncwarp();
    const float* g = logits + static_cast<size_t>(t) * E;
    for (int e = lane; e < E; e += 32) my_row[e] = g[e];
    __syncwarp();
  };
  for (int e = tid; e < E; e += kBudgetThreads) {
    score[e] = 0;
    in_budget[e] = 0;
  }
  __syncthreads();
  // 1, 2: own top-k of every token, scores
  for (int t = warp; t < T; t += kBudgetWarps) {
    stage_row(t);
    float pv = 0.f;
    int pe = -1;
    for (int r = 0; r < k; ++r) {
      float bv;
      const int be = next_choice(my_row, E, pv, pe, nullptr, bv);
      if (lane == 0) atomicAdd(&score[be], k - r);
      pv = bv;
      pe = be;
    }
  }
  __syncthreads();
  // 3: the budget, one expert per pass: the best (score, id) after the last pick
  int ps = 0, pid = -1;
  for (int j = 0; j < B; ++j) {
    int bs = 0, be = -1;
    for (int e = tid; e < E; e += kBudgetThreads) {
      const int s = score[e];
      if (pid >= 0 && !ranks_before(ps, pid, s, e)) continue;
      keep_better(bs, be, s, e);
    }
    warp_best(bs, be);
    if (lane == 0) {
      red_s[warp] = bs;
      red_e[warp] = be;
    }
    __syncthreads();
    if (warp == 0) {
      bs = lane < kBudgetWarps ? red_s[lane] : 0;
      be = lane < kBudgetWarps ? red_e[lane] : -1;
      warp_best(bs, be);
      if (lane == 0) {
        pick = be;
        in_budget[be] = 1;
      }
    }
    __syncthreads();
    pid = pick;
    ps = score[pid];
  }
  __syncthreads();
  // the budget in ascending expert order
  if (warp == 0) {
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const bool f = e < E && in_budget[e];
      const unsigned m = __ballot_sync(0xffffffffu, f);
      if (f) budget_out[base + __popc(m & ((1u << lane) - 1u))] = e;
      base += __popc(m);
    }
  }
  // 4: every token's top-k inside the budget
  for (int t = warp; t < T; t += kBudgetWarps) {
    stage_row(t);
    float pv = 0.f;
    int pe = -1;
    for (int r = 0; r < k; ++r) {
      float bv;
      const int be = next_choice(my_row, E, pv, pe, in_budget, bv);
      if (lane == 0) topk_out[static_cast<size_t>(t) * k + r] = be;
      pv = bv;
      pe = be;
    }
  }
}

}  // namespace

int launch_budget(const float* logits, int T, int E, int k, int B, int32_t* budget, int32_t* topk,
                  cudaStream_t stream) {
  const int smem = kBudgetWarps * E * static_cast<int>(sizeof(float));
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(budget_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return CBQ_ECUDA;
  budget_kernel<<<1, kBudgetThreads, smem, stream>>>(logits, T, E, k, B, budget, topk);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? CBQ_OK : CBQ_ECUDA;
}

}  // namespace cbq
