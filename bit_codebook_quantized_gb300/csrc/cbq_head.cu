// cbq_head.cu -- the two-bit draft head's shortlist and FP8 rescoring.
//
// "Hibana: Fast Agentic Inference on Unified-Memory Devices", section "Model
// surgery / Two-bit draft head": the drafter's vocabulary head scores every
// token from a 2-bit copy of its weights (the stream-K kernel with 2-bit
// codes writes the scores), keeps the 16 best and rescores only those with
// the FP8 head.  Here:
//  * head_topk_chunk_kernel: grid (1024-row chunks, tokens), 256 threads, four
//    rows a thread; the 16 best (score, row) pairs of each chunk.  Every warp
//    sorts its 32 lane maxima (a bitonic network over shuffles); a tree of
//    bitonic merges of the warps' 16 largest gives the 16 largest lane maxima
//    of the chunk, and the 16th, T, is reached by exactly the 16 lanes that
//    hold them.  Their pairs >= T (at most 64) go to shared memory and each
//    finds its place among them by counting the larger ones; places 0..15
//    are the chunk's list.
//  * head_select_kernel: one CTA of 16 warps per token.  The same sort and
//    merge tree over the chunks' first entries gives the 16 leading chunks
//    and T, their 16th first entry; only their entries >= T (at most 16 x 16)
//    can be in the shortlist, and they are ranked by counting as above (the
//    shortlist: descending score, equal scores -> lower row).  Warp i then the
//    FP8 logit of shortlisted row i, a_scale * row_scale * sum_k a w8
//    (products exact in fp32, sums in fp32; all of a lane's loads in flight
//    at once), and the pick: the highest logit, equal logits -> the earlier
//    row of the shortlist.
// A (score, row) pair is one 64-bit word: an order-preserving key of the fp32
// score (-0 equals +0, NaN below every number) in the high half and
// 2^32 - 1 - row in the low half, so "ranks before" is unsigned ">", no two
// rows' words are equal and no word is 0 (0 marks an empty list entry).
#include <cuda_runtime.h>

#include <cuda_fp8.h>

#include <cstdint>

#include "cbq_device.cuh"
#include "cbq_internal.h"

namespace cbq {
namespace {

constexpr int kList = kHeadShortlist;                  // 16
constexpr int kChunkWarps = 8;
constexpr int kPerThread = kHeadChunkRows / (kChunkWarps * 32);   // 4
constexpr int kSelectWarps = kList;                    // one warp per shortlisted row
constexpr int kSelectCand = kList * kList;             // entries of the 16 leading chunks
constexpr int kChunkCand = kList * kPerThread;         // words of the 16 leading lanes

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

// The warp's 32 words sorted descending over the lanes (lane 0 the largest):
// a bitonic network, one compare-exchange with lane ^ j per step.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
      const bool take_max = ((lane & j) == 0) == ((lane & k) == 0);
      v = take_max == (o > v) ? o : v;
    }
  }
  return v;
}

// Lanes 0..15 hold one descending list, lanes 16..31 another in ascending
// order (a bitonic sequence); afterwards the 32 words are descending.
__device__ __forceinline__ uint64_t warp_merge_desc(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const uint64_t o = __shfl_xor_sync(0xffffffffu, v, j);
    v = ((lane & j) == 0) == (o > v) ? o : v;
  }
  return v;
}

// lists[16 i .. 16 i + 15], i < nl (a power of two, nl <= 2 x warps): nl
// descending lists in shared memory.  Afterwards lists[0..15] holds the 16
// largest words of all, descending: a tree of pairwise bitonic merges, warp w
// merging lists 2 s w and 2 s w + s at step s.  Every thread of the block
// calls it.
__device__ __forceinline__ void merge_tree16(uint64_t* lists, int nl) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int st = 1; st < nl; st <<= 1) {
    const int a = 2 * st * warp, b = a + st;
    uint64_t v = 0ull;
    if (b < nl) v = warp_merge_desc(lane < kList ? lists[a * kList + lane] : lists[b * kList + 31 - lane]);
    __syncthreads();
    if (b < nl && lane < kList) lists[a * kList + lane] = v;
    __syncthreads();
  }
}

// Append w to list[] (shared memory, count *n) for every lane whose flag is
// set: one atomic per warp.
__device__ __forceinline__ void warp_append(bool flag, uint64_t w, uint64_t* list, unsigned* n) {
  const unsigned ballot = __ballot_sync(0xffffffffu, flag);
  if (ballot == 0u) return;
  const int lane = threadIdx.x & 31;
  unsigned base = 0;
  if (lane == 0) base = atomicAdd(n, static_cast<unsigned>(__popc(ballot)));
  base = __shfl_sync(0xffffffffu, base, 0);
  if (flag) list[base + __popc(ballot & ((1u << lane) - 1u))] = w;
}

// How many of list[0..n) are larger than w (eight loads in flight).
__device__ __forceinline__ unsigned count_larger(const uint64_t* list, unsigned n, uint64_t w) {
  unsigned c = 0;
  for (unsigned j0 = 0; j0 < n; j0 += 8) {
    uint64_t x[8];
#pragma unroll
    for (unsigned u = 0; u < 8; ++u) x[u] = list[min(j0 + u, n - 1u)];
#pragma unroll
    for (unsigned u = 0; u < 8; ++u) c += (j0 + u < n && x[u] > w) ? 1u : 0u;
  }
  return c;
}

// Each of the n distinct words of list[] finds its place among them by
// counting the larger ones; the words of places 0..15 go to out[place].
__device__ __forceinline__ void rank_places(const uint64_t* list, unsigned n, uint64_t* out, int nthreads) {
  for (unsigned i = threadIdx.x; i < n; i += nthreads) {
    const uint64_t w = list[i];
    const unsigned place = count_larger(list, n, w);
    if (place < static_cast<unsigned>(kList)) out[place] = w;
  }
}

__global__ void __launch_bounds__(kChunkWarps * 32) head_topk_chunk_kernel(const float* __restrict__ scores, int N,
                                                                           uint64_t* __restrict__ cand) {
  __shared__ uint64_t tops[kChunkWarps * kList];
  __shared__ uint64_t pool[kChunkCand];
  __shared__ unsigned npool;
  grid_launch_dependents();                            // the select kernel may start (it waits for this grid)
  grid_dependency_wait();                              // the scores of the matmul kernel
  const int m = blockIdx.y, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lo = blockIdx.x * kHeadChunkRows;
  const float* s = scores + static_cast<size_t>(m) * N;
  uint64_t w[kPerThread], mx = 0ull;
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int n = lo + threadIdx.x + j * kChunkWarps * 32;
    w[j] = n < N ? pair_word(__ldg(s + n), n) : 0ull;   // 0: no row
    mx = w[j] > mx ? w[j] : mx;
  }
  const uint64_t srt = warp_sort_desc(mx);
  if (lane < kList) tops[warp * kList + lane] = srt;
  if (threadIdx.x == 0) npool = 0;
  __syncthreads();
  merge_tree16(tops, kChunkWarps);                     // the chunk's 16 largest lane maxima
  // T is reached by the 16 lanes whose maxima are tops[0..15] (T = 0: fewer
  // than 16 lanes hold a row, and those hold every word)
  const uint64_t T = tops[kList - 1];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) warp_append(w[j] != 0ull && w[j] >= T, w[j], pool, &npool);
  __syncthreads();
  const unsigned n = npool;
  uint64_t* dst = cand + (static_cast<size_t>(m) * gridDim.x + blockIdx.x) * kList;
  rank_places(pool, n, dst, kChunkWarps * 32);
  if (threadIdx.x < kList && threadIdx.x >= n) dst[threadIdx.x] = 0ull;   // fewer than 16 rows
}

__global__ void __launch_bounds__(kSelectWarps * 32) head_select_kernel(
    const uint64_t* __restrict__ cand, int nchunks, const uint8_t* __restrict__ a, const float* __restrict__ a_scale,
    const uint8_t* __restrict__ head8, const float* __restrict__ row_scale, int N, int K,
    int32_t* __restrict__ rows_out, float* __restrict__ logits_out, int32_t* __restrict__ pick_out) {
  __shared__ uint64_t tops[kSelectWarps * kList];
  __shared__ uint64_t pool[kSelectCand];
  __shared__ uint64_t best[kList];
  __shared__ float logit_s[kList];
  __shared__ unsigned npool;
  // the next kernel may start: it waits for this grid before it writes
  // anything this one reads (the next matmul's scores and workspace)
  grid_launch_dependents();
  grid_dependency_wait();                              // the chunks' lists
  const int m = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t* c = cand + static_cast<size_t>(m) * nchunks * kList;
  {
    // thread i: the first entry of chunk i (nchunks <= 256 < threads)
    const int i = threadIdx.x;
    const uint64_t srt = warp_sort_desc(i < nchunks ? c[static_cast<size_t>(i) * kList] : 0ull);
    if (lane < kList) tops[warp * kList + lane] = srt;
  }
  if (threadIdx.x == 0) npool = 0;
  __syncthreads();
  merge_tree16(tops, kSelectWarps);                    // the 16 largest first entries (distinct)
  // every entry >= T lies in one of the leading chunks; fewer than 16 chunks:
  // T = 0, every entry
  const uint64_t T = nchunks >= kList ? tops[kList - 1] : 0ull;
  {
    const int q = threadIdx.x / kList, e = threadIdx.x % kList;   // entry e of leading chunk q
    const uint64_t lead = q < kList ? tops[q] : 0ull;
    const uint64_t w = lead != 0ull ? c[static_cast<size_t>(word_row(lead) / kHeadChunkRows) * kList + e] : 0ull;
    warp_append(w != 0ull && w >= T, w, pool, &npool);
  }
  __syncthreads();
  rank_places(pool, npool, best, kSelectWarps * 32);
  __syncthreads();
  if (threadIdx.x < kList) rows_out[static_cast<size_t>(m) * kList + threadIdx.x] = word_row(best[threadIdx.x]);
  // FP8 rescoring: warp i takes shortlisted row i; a lane takes 16
  // consecutive k per step, four steps' loads in flight together
  const uint8_t* am = a + static_cast<size_t>(m) * K;
  const int n = word_row(best[warp]);
  const uint8_t* wn = head8 + static_cast<size_t>(n) * K;
  float acc = 0.f;
  for (int k0 = 16 * lane; k0 < K; k0 += 4 * 16 * 32) {
    uint4 av[4], wv[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int k = k0 + u * 16 * 32;
      if (k < K) {
        av[u] = __ldg(reinterpret_cast<const uint4*>(am + k));
        wv[u] = __ldg(reinterpret_cast<const uint4*>(wn + k));
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (k0 + u * 16 * 32 >= K) continue;
      const uint32_t aw[4] = {av[u].x, av[u].y, av[u].z, av[u].w}, ww[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
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
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    const float lg = acc * (__ldg(a_scale + m) * __ldg(row_scale + n));
    logit_s[warp] = lg;
    logits_out[static_cast<size_t>(m) * kList + warp] = lg;
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

int head_chunks(int N) { return (N + kHeadChunkRows - 1) / kHeadChunkRows; }

int launch_head_select(const float* scores, int M, int N, int K, const uint8_t* a, const float* a_scale,
                       const uint8_t* head8, const float* row_scale, uint64_t* cand, int32_t* rows, float* logits,
                       int32_t* pick, cudaStream_t stream) {
  const int nchunks = head_chunks(N);
  if (nchunks > kHeadMaxChunks) return CBQ_EINVAL;
  if (launch_pdl_head(head_topk_chunk_kernel, dim3(nchunks, M), dim3(kChunkWarps * 32), stream, scores, N,
                      cand) != cudaSuccess ||
      launch_pdl_head(head_select_kernel, dim3(M), dim3(kSelectWarps * 32), stream,
                      static_cast<const uint64_t*>(cand), nchunks, a, a_scale, head8, row_scale, N, K, rows, logits,
                      pick) != cudaSuccess)
    return CBQ_ECUDA;
  return CBQ_OK;
}

}  // namespace cbq
