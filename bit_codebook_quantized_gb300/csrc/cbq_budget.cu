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
// A (key, id) pair is one 64-bit word, key in the high
// half and (2^32 - 1 - id) in the low half, so "ranks before" is plain
// unsigned ">".  Three kernels, each launched to overlap the previous one's
// tail (programmatic dependent launch): step 1 with one warp per token over
// ceil(T / 8) CTAs, steps 2-3 in one CTA of 32 warps, step 4 with one warp
// per token again.  Steps 1 and 4: one warp per
// token; every lane keeps the best 8 words of its experts (a branch-free
// insertion chain, taken only when a word beats the lane's 8th; 8 loads in
// flight per lane), then k rounds of a warp-wide maximum merge the 32 lists.
// Step 2: shared-memory atomic adds of (k - r) into the high half of each
// expert's word.  Step 3: up to 256 experts, each expert's place among those
// words (all distinct) by counting the larger ones (E^2/32 broadcast loads);
// beyond, one bitonic sort of the words (fewer steps than that); places
// 0..B-1 are the budget.
#include <cuda_runtime.h>

#include <cstdint>

#include "cbq_budget.h"
#include "cbq_device.cuh"
#include "cbq_internal.h"

namespace cbq {
namespace {

constexpr int kBudgetWarps = 32;
constexpr int kBudgetThreads = kBudgetWarps * 32;
constexpr int kListLen = kMaxBudgetK;                  // per-lane candidate list
constexpr int kLoadBatch = 8;                         // loads in flight per lane and batch

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
// `row` is in shared or global memory.
template <typename Emit>
__device__ __forceinline__ void token_topk(const float* row, const int16_t* ids, int count, int k, Emit emit) {
  const int lane = threadIdx.x & 31;
  uint64_t list[kListLen];
#pragma unroll
  for (int i = 0; i < kListLen; ++i) list[i] = 0;     // below every real word
  for (int j0 = lane; j0 < count; j0 += 32 * kLoadBatch) {
    int ee[kLoadBatch];
    float v[kLoadBatch];
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int j = j0 + 32 * u;
      ee[u] = j < count ? (ids ? ids[j] : j) : -1;
    }
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) v[u] = ee[u] >= 0 ? row[ee[u]] : 0.f;
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u)
      if (ee[u] >= 0) {
        const uint64_t w = rank_word(logit_key(v[u]), ee[u]);
        if (w > list[kListLen - 1]) insert(list, w);
      }
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

constexpr int kOwnWarps = 8;                          // tokens per CTA of the first kernel

// Steps 1 (first kernel, one warp per token over ceil(T / 8) CTAs): every
// token's own top-k, written to topk_out, which holds it until the second
// kernel has read it.
__global__ void __launch_bounds__(kOwnWarps * 32) budget_own_kernel(const float* __restrict__ logits, int T, int E,
                                                                     int k, int32_t* __restrict__ topk_out) {
  grid_launch_dependents();                                 // the second kernel may start its prologue
  grid_dependency_wait();                                   // the logits of an earlier kernel
  const int t = blockIdx.x * kOwnWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  token_topk(logits + static_cast<size_t>(t) * E, nullptr, E, k,
             [&](int r, int e) { topk_out[static_cast<size_t>(t) * k + r] = e; });
}

// How many of words[0..n) are larger than w (eight loads in flight).
__device__ __forceinline__ unsigned count_larger(const unsigned long long* words, unsigned n, unsigned long long w) {
  unsigned c = 0;
  for (unsigned j0 = 0; j0 < n; j0 += 8) {
    unsigned long long x[8];
#pragma unroll
    for (unsigned u = 0; u < 8; ++u) x[u] = words[min(j0 + u, n - 1u)];
#pragma unroll
    for (unsigned u = 0; u < 8; ++u) c += (j0 + u < n && x[u] > w) ? 1u : 0u;
  }
  return c;
}

constexpr int kCountMaxExperts = 256;                 // place by counting up to here, else sort

// Steps 2-3 (second kernel, one CTA of 32 warps): scores from all the own
// top-k lists, then the B best words (the words are distinct: the id is in
// the low half), written in ascending expert order.
__global__ void __launch_bounds__(kBudgetThreads) budget_sort_kernel(int T, int E, int k, int B,
                                                                      const int32_t* __restrict__ own,
                                                                      int32_t* __restrict__ budget_out) {
  __shared__ unsigned long long words[kMaxBudgetExperts];   // (score, id) of every expert
  __shared__ uint8_t in_budget[kMaxBudgetExperts];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  grid_launch_dependents();
  int P = 32;                                               // sort width: power of two >= E
  while (P < E) P <<= 1;
  for (int e = tid; e < P; e += kBudgetThreads) {
    words[e] = e < E ? rank_word(0u, e) : 0ull;             // padding sorts last
    in_budget[e] = 0;
  }
  grid_dependency_wait();                                   // the own top-k lists
  __syncthreads();
  // 2: score (k - r) into the high half of the word of each token's rank-r expert
  const int tk = T * k;
  for (int i = tid; i < tk; i += kBudgetThreads)
    atomicAdd(&words[own[i]], static_cast<unsigned long long>(k - i % k) << 32);
  __syncthreads();
  if (E <= kCountMaxExperts) {
    // 3: the B experts whose words no more than B - 1 others beat
    for (int e = tid; e < E; e += kBudgetThreads)
      in_budget[e] = count_larger(words, static_cast<unsigned>(E), words[e]) < static_cast<unsigned>(B) ? 1 : 0;
  } else {
    // 3: bitonic sort, descending: words[0..B) are the budget
    for (int size = 2; size <= P; size <<= 1) {
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
        for (int i = tid; i < P / 2; i += kBudgetThreads) {
          const int lo = 2 * i - (i & (stride - 1));        // first of the pair
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
  }
  __syncthreads();
  if (warp == 0) {                                          // ascending expert order
    int base = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const bool f = e < E && in_budget[e];
      const unsigned m = __ballot_sync(0xffffffffu, f);
      if (f) budget_out[base + __popc(m & ((1u << lane) - 1u))] = e;
      base += __popc(m);
    }
  }
}

// Step 4 (third kernel, one warp per token over ceil(T / 8) CTAs): the
// token's top-k among the budget experts (their logits only), over its own
// list (read by the second kernel, which has finished).
__global__ void __launch_bounds__(kOwnWarps * 32) budget_pick_kernel(const float* __restrict__ logits, int T, int E,
                                                                      int k, int B,
                                                                      const int32_t* __restrict__ budget,
                                                                      int32_t* __restrict__ topk_out) {
  __shared__ int16_t blist[kMaxBudgetExperts];
  grid_dependency_wait();                                   // the budget
  for (int j = threadIdx.x; j < B; j += kOwnWarps * 32) blist[j] = static_cast<int16_t>(budget[j]);
  __syncthreads();
  const int t = blockIdx.x * kOwnWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  token_topk(logits + static_cast<size_t>(t) * E, blist, B, k,
             [&](int r, int e) { topk_out[static_cast<size_t>(t) * k + r] = e; });
}

}  // namespace

// Launch with programmatic stream serialisation: the kernel may start while
// the previous one runs and waits for it with griddepcontrol.wait.
template <typename... Args>
cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args...);
  note_launch();
  return e;
}

int launch_budget(const float* logits, int T, int E, int k, int B, int32_t* budget, int32_t* topk,
                  cudaStream_t stream) {
  const dim3 tok_grid((T + kOwnWarps - 1) / kOwnWarps), tok_block(kOwnWarps * 32);
  // topk_idx holds every token's own top-k until the second kernel has read it
  if (launch_pdl(budget_own_kernel, tok_grid, tok_block, stream, logits, T, E, k, topk) != cudaSuccess ||
      launch_pdl(budget_sort_kernel, dim3(1), dim3(kBudgetThreads), stream, T, E, k, B,
                 static_cast<const int32_t*>(topk), budget) != cudaSuccess ||
      launch_pdl(budget_pick_kernel, tok_grid, tok_block, stream, logits, T, E, k, B,
                 static_cast<const int32_t*>(budget), topk) != cudaSuccess)
    return CBQ_ECUDA;
  return CBQ_OK;
}

}  // namespace cbq
