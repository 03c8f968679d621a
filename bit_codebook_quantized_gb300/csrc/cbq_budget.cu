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
// Logits are compared through a 32-bit key that orders floats as numbers
// (-0 and +0 equal) and puts NaN below every other value, so the kernel is
// total: any input gives k valid, distinct expert ids per token.
//
// One CTA of 32 warps.  A (key, id) pair is one 64-bit word, key in the high
// half and (2^32 - 1 - id) in the low half, so "ranks before" is plain
// unsigned ">".  Steps 1 and 4: one warp per token; every lane keeps the
// best 8 words of its experts (a branch-free insertion chain, taken only when
// a word beats the lane's 8th), then k rounds of a warp-wide maximum merge the
// 32 lists.  Step 2: shared-memory atomic adds of (k - r) into the high half
// of each expert's word.  Step 3: one bitonic sort of those words.
#include <cuda_runtime.h>

#include <cstdint>

#include "cbq_budget.h"
#include "cbq_internal.h"

namespace cbq {
namespace {

constexpr int kBudgetWarps = 32;
constexpr int kBudgetThreads = kBudgetWarps * 32;
constexpr int kListLen = kMaxBudgetK;                  // per-lane candidate list

// Order-preserving key of a logit: larger logit -> larger key; -0 == +0;
// NaN -> 0, below every other value (no other float maps to 0).
__device__ __forceinline__ uint32_t logit_key(float v) {
  if (v != v) return 0u;
  if (v == 0.f) v = 0.f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t rank_word(uint32_t key, int e) {
  return (static_cast<uint64_t>(key) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e));
}
__device__ __forceinline__ int word_id(uint64_t w) { return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(w)); }

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, v, off);
    v = o > v ? o : v;
  }
  return v;
}

// Insert w into the lane's descending list (only called when w beats its last).
__device__ __forceinline__ void insert(uint64_t (&list)[kListLen], uint64_t w) {
#pragma unroll
  for (int i = 0; i < kListLen; ++i) {
    const uint64_t hi = list[i] > w ? list[i] : w;
    w = list[i] > w ? w : list[i];
    list[i] = hi;
  }
}

// The token's top-k among `count` experts (expert of candidate j: ids ? ids[j]
// : j), merged over the warp; calls emit(r, e) on lane 0 for rank r = 0..k-1.
template <typename Emit>
__device__ __forceinline__ void token_topk(const float* __restrict__ row, const int16_t* ids, int count, int k,
                                           Emit emit) {
  const int lane = threadIdx.x & 31;
  uint64_t list[kListLen];
#pragma unroll
  for (int i = 0; i < kListLen; ++i) list[i] = 0;     // below every real word
  for (int j = lane; j < count; j += 32) {
    const int e = ids ? ids[j] : j;
    const uint64_t w = rank_word(logit_key(__ldg(row + e)), e);
    if (w > list[kListLen - 1]) insert(list, w);
  }
  for (int r = 0; r < k; ++r) {
    const uint64_t m = warp_max_u64(list[0]);
    if (list[0] == m) {                                // the one lane that held it pops it
#pragma unroll
      for (int i = 0; i + 1 < kListLen; ++i) list[i] = list[i + 1];
      list[kListLen - 1] = 0;
    }
    if (lane == 0) emit(r, word_id(m));
  }
}

__global__ void __launch_bounds__(kBudgetThreads) budget_kernel(const float* __restrict__ logits, int T, int E,
                                                                 int k, int B, int32_t* __restrict__ budget_out,
                                                                 int32_t* __restrict__ topk_out) {
  __shared__ unsigned long long words[kMaxBudgetExperts];   // (score, id) of every expert
  __shared__ uint8_t in_budget[kMaxBudgetExperts];
  __shared__ int16_t blist[kMaxBudgetExperts];              // budget ids, ascending
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int P = 32;                                               // sort width: power of two >= E
  while (P < E) P <<= 1;
  for (int e = tid; e < P; e += kBudgetThreads) {
    words[e] = e < E ? rank_word(0u, e) : 0ull;             // padding sorts last
    in_budget[e] = 0;
  }
  __syncthreads();
  // 1, 2: own top-k of every token; score (k - r) into the expert's high half
  for (int t = warp; t < T; t += kBudgetWarps)
    token_topk(logits + static_cast<size_t>(t) * E, nullptr, E, k, [&](int r, int e) {
      atomicAdd(&words[e], static_cast<unsigned long long>(k - r) << 32);
    });
  __syncthreads();
  // 3: bitonic sort, descending: words[0..B) are the budget
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P / 2; i += kBudgetThreads) {
        const int lo = 2 * i - (i & (stride - 1));          // first of the pair
        const int hi = lo + stride;
        const bool desc = (lo & size) == 0;
        const unsigned long long a = words[lo], b = words[hi];
        if ((a < b) == desc) {
          words[lo] = b;
          words[hi] = a;
        }
      }
      __syncthreads();
    }
  }
  for (int j = tid; j < B; j += kBudgetThreads) in_budget[word_id(words[j])] = 1;
  __syncthreads();
  // the budget in ascending expert order
  if (warp == 0) {
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const bool f = e < E && in_budget[e];
      const unsigned m = __ballot_sync(0xffffffffu, f);
      if (f) {
        const int at = base + __popc(m & ((1u << lane) - 1u));
        budget_out[at] = e;
        blist[at] = static_cast<int16_t>(e);
      }
      base += __popc(m);
    }
  }
  __syncthreads();
  // 4: every token's top-k inside the budget
  for (int t = warp; t < T; t += kBudgetWarps)
    token_topk(logits + static_cast<size_t>(t) * E, blist, B, k,
               [&](int r, int e) { topk_out[static_cast<size_t>(t) * k + r] = e; });
}

}  // namespace

int launch_budget(const float* logits, int T, int E, int k, int B, int32_t* budget, int32_t* topk,
                  cudaStream_t stream) {
  budget_kernel<<<1, kBudgetThreads, 0, stream>>>(logits, T, E, k, B, budget, topk);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? CBQ_OK : CBQ_ECUDA;
}

}  // namespace cbq
