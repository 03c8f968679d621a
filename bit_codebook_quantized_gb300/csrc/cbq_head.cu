// cbq_head.cu -- the two-bit draft head's shortlist and FP8 rescoring.
//
// "Hibana: Fast Agentic Inference on Unified-Memory Devices", section "Model
// surgery / Two-bit draft head": the drafter's vocabulary head scores every
// token from a 2-bit copy of its weights (the stream-K kernel with 2-bit
// codes writes the scores), keeps the 16 best and rescores only those with
// the FP8 head.  Here:
//  * head_topk_chunk_kernel: grid (row chunks, tokens); the 16 best (score,
//    row) pairs of each chunk -- per lane a sorted list of 16, merged over the
//    warp by 16 rounds of a warp-wide maximum, then over the CTA's warps;
//  * head_select_kernel: one CTA per token; the 16 best of all chunks' lists
//    (the shortlist: descending score, equal scores -> lower row), then each
//    shortlisted row's FP8 logit a_scale * row_scale * sum_k a w8 (products
//    exact in fp32, sums in fp32), and the pick: the highest logit, equal
//    logits -> the earlier row of the shortlist.
// A (score, row) pair is one 64-bit word: an order-preserving key of the fp32
// score (-0 equals +0, NaN below every number) in the high half and
// 2^32 - 1 - row in the low half, so "ranks before" is unsigned ">".
#include <cuda_runtime.h>

#include <cuda_fp8.h>

#include <cstdint>

#include "cbq_device.cuh"
#include "cbq_internal.h"

namespace cbq {
namespace {

constexpr int kList = kHeadShortlist;                  // 16
constexpr int kChunkWarps = 8;
constexpr int kSelectWarps = 4;

__device__ __forceinline__ uint32_t score_key(float v) {
  if (v != v) return 0u;
  if (v == 0.f) v = 0.f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint64_t pair_word(float v, int row) {
  return (static_cast<uint64_t>(score_key(v)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(row));
}
__device__ __forceinline__ int word_row(uint64_t w) { return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(w)); }

__device__ __forceinline__ uint64_t warp_max64(uint64_t v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, v, off);
    v = o > v ? o : v;
  }
  return v;
}

// Insert w into a descending list (called when it beats the last entry).
__device__ __forceinline__ void insert16(uint64_t (&list)[kList], uint64_t w) {
#pragma unroll
  for (int i = 0; i < kList; ++i) {
    const uint64_t hi = list[i] > w ? list[i] : w;
    w = list[i] > w ? w : list[i];
    list[i] = hi;
  }
}

// The warp's 16 best words from every lane's descending list; lane 0 gets
// them in order in out[0..15] (shared memory).
__device__ __forceinline__ void warp_merge16(uint64_t (&list)[kList], uint64_t* out) {
  const int lane = threadIdx.x & 31;
  for (int r = 0; r < kList; ++r) {
    const uint64_t m = warp_max64(list[0]);
    if (list[0] == m && m != 0ull) {                   // the one lane that held it pops it
#pragma unroll
      for (int i = 0; i + 1 < kList; ++i) list[i] = list[i + 1];
      list[kList - 1] = 0ull;
    }
    if (lane == 0) out[r] = m;
  }
}

__global__ void __launch_bounds__(kChunkWarps * 32) head_topk_chunk_kernel(const float* __restrict__ scores, int N,
                                                                           int chunk, uint64_t* __restrict__ cand) {
  __shared__ uint64_t warp_best[kChunkWarps][kList];
  __shared__ uint64_t best[kList];
  grid_dependency_wait();                              // the scores of the matmul kernel
  const int m = blockIdx.y, nchunks = gridDim.x;
  const int lo = blockIdx.x * chunk, hi = min(N, lo + chunk);
  const float* s = scores + static_cast<size_t>(m) * N;
  uint64_t list[kList];
#pragma unroll
  for (int i = 0; i < kList; ++i) list[i] = 0ull;      // below every real word
  for (int n = lo + threadIdx.x; n < hi; n += kChunkWarps * 32) {
    const uint64_t w = pair_word(__ldg(s + n), n);
    if (w > list[kList - 1]) insert16(list, w);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  warp_merge16(list, warp_best[warp]);
  __syncthreads();
  if (warp == 0) {
    // the CTA's 16 best of the warps' 8 x 16 words
    uint64_t l2[kList];
#pragma unroll
    for (int i = 0; i < kList; ++i) l2[i] = 0ull;
    for (int i = lane; i < kChunkWarps * kList; i += 32) {
      const uint64_t w = warp_best[i / kList][i % kList];
      if (w > l2[kList - 1]) insert16(l2, w);
    }
    uint64_t* dst = cand + (static_cast<size_t>(m) * nchunks + blockIdx.x) * kList;
    warp_merge16(l2, best);
    __syncwarp();
    if (lane < kList) dst[lane] = best[lane];
  }
}

__global__ void __launch_bounds__(kSelectWarps * 32) head_select_kernel(
    const uint64_t* __restrict__ cand, int nchunks, const uint8_t* __restrict__ a, const float* __restrict__ a_scale,
    const uint8_t* __restrict__ head8, const float* __restrict__ row_scale, int N, int K,
    int32_t* __restrict__ rows_out, float* __restrict__ logits_out, int32_t* __restrict__ pick_out) {
  __shared__ uint64_t best[kList];
  __shared__ float logit_s[kList];
  grid_dependency_wait();                              // the chunks' lists
  const int m = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    uint64_t list[kList];
#pragma unroll
    for (int i = 0; i < kList; ++i) list[i] = 0ull;
    const uint64_t* c = cand + static_cast<size_t>(m) * nchunks * kList;
    for (int i = lane; i < nchunks * kList; i += 32) {
      const uint64_t w = c[i];
      if (w > list[kList - 1]) insert16(list, w);
    }
    warp_merge16(list, best);
    __syncwarp();
    if (lane < kList) rows_out[static_cast<size_t>(m) * kList + lane] = word_row(best[lane]);
  }
  __syncthreads();
  // FP8 rescoring: warp w takes shortlisted rows w, w + 4, ...; a lane takes
  // 16 consecutive k per step
  const uint8_t* am = a + static_cast<size_t>(m) * K;
  for (int i = warp; i < kList; i += kSelectWarps) {
    const int n = word_row(best[i]);
    const uint8_t* wn = head8 + static_cast<size_t>(n) * K;
    float acc = 0.f;
    for (int k = 16 * lane; k < K; k += 16 * 32) {
      const uint4 av = __ldg(reinterpret_cast<const uint4*>(am + k));
      const uint4 wv = __ldg(reinterpret_cast<const uint4*>(wn + k));
      const uint32_t aw[4] = {av.x, av.y, av.z, av.w}, ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const __half2 ah(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(aw[q] >> (16 * h)), __NV_E4M3));
          const __half2 wh(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(ww[q] >> (16 * h)), __NV_E4M3));
          const float2 af = __half22float2(ah), wf = __half22float2(wh);
          acc += af.x * wf.x;                          // products of two E4M3 values are exact in fp32
          acc += af.y * wf.y;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
      const float lg = acc * (__ldg(a_scale + m) * __ldg(row_scale + n));
      logit_s[i] = lg;
      logits_out[static_cast<size_t>(m) * kList + i] = lg;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int bi = 0;
    for (int i = 1; i < kList; ++i)
      if (logit_s[i] > logit_s[bi]) bi = i;            // equal logits: the earlier row of the shortlist
    pick_out[m] = word_row(best[bi]);
  }
}

// Launch with programmatic stream serialisation (waits on the kernel before).
template <typename... Args>
cudaError_t launch_pdl_head(void (*kern)(Args...), dim3 grid, dim3 block, cudaStream_t stream, Args... args) {
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

}  // namespace

int head_chunking(int N, int* chunk) {
  // at most kHeadMaxChunks chunks of at least 4096 rows
  int c = 4096;
  while ((N + c - 1) / c > kHeadMaxChunks) c *= 2;
  *chunk = c;
  return (N + c - 1) / c;
}

int launch_head_select(const float* scores, int M, int N, int K, const uint8_t* a, const float* a_scale,
                       const uint8_t* head8, const float* row_scale, uint64_t* cand, int32_t* rows, float* logits,
                       int32_t* pick, cudaStream_t stream) {
  int chunk = 0;
  const int nchunks = head_chunking(N, &chunk);
  if (launch_pdl_head(head_topk_chunk_kernel, dim3(nchunks, M), dim3(kChunkWarps * 32), stream, scores, N, chunk,
                      cand) != cudaSuccess ||
      launch_pdl_head(head_select_kernel, dim3(M), dim3(kSelectWarps * 32), stream,
                      static_cast<const uint64_t*>(cand), nchunks, a, a_scale, head8, row_scale, N, K, rows, logits,
                      pick) != cudaSuccess)
    return CBQ_ECUDA;
  return CBQ_OK;
}

}  // namespace cbq
