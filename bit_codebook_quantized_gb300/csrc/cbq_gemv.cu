// cbq_gemv.cu -- small-M kernel of the codebook-quantised matmul, plus the
// unpack (decode-to-fp32) kernel.
//
// "Hibana: Fast Agentic Inference on Unified-Memory Devices", section "Model
// surgery / Three-bit weights": decode is bound by memory bandwidth, so the
// kernel streams only the packed bytes (3 bits per weight + 8 bits per group
// of 32), turns each code into its value in the row's 8-entry E4M3 codebook
// on the fly and multiplies on FP8 tensor cores.  Section "Adaptive speculation / Expert sharing": the grouped
// variant reads only the experts that the round's tokens route to.
//
// Design (GB300):
//  * work unit = 16 weight rows ("slab") x the whole K; units are handed out
//    round-robin to a persistent grid;
//  * one producer warp streams the slab's code bytes with 1-D bulk copies of
//    [16 rows][48 B] (48 B = 4 groups = 128 k; contiguous in the tile-ordered
//    code stream), 8 copies per pipeline stage, into a 4-stage mbarrier ring;
//  * 8 consumer warps take one box each per stage (an 8-way split of K inside
//    the CTA; 8 warps hide the latency of the decode-MMA-FFMA chain better
//    than 4 with twice the stages: -4 % per call on the decode workload,
//    -16 % on a 2048 x 2048 matrix).  A lane reads its 24-bit quarter of a group with two 32-bit
//    shared loads (row pitch 48 B: conflict-free), spreads the 8 codes to
//    nibbles and turns them into E4M3 bytes with two byte-permutes through
//    the codebook held in two registers;
//  * the 16x32 decoded tile is multiplied with 8 tokens' activations by one
//    m16n8k32 E4M3 MMA (fp32 accumulate), and the group's E8M0 scale is
//    applied to the MMA result with one FFMA per output element;
//  * the 8 K-split partials are summed in shared memory (in warp order) and
//    a_scale is applied on the store.  No atomics and no global scratch.
//  Inside one MMA the K order is permuted (lane t of a quad owns codes
//  8t..8t+7 of the group); the activation fragment uses the same permutation,
//  so the dot product is unchanged.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "cbq_device.cuh"
#include "cbq_internal.h"

namespace cbq {

static __device__ unsigned g_status_gemv = 0;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kSlabRows = 16;
constexpr int kBoxBytes = kSlabRows * 48;            // one [16][48 B] TMA box
constexpr int kStageBytes = kConsumerWarps * kBoxBytes;
constexpr int kStages = 4;
constexpr int kMaxExperts = 4096;
constexpr int kMaxRouting = 64 * 8;

constexpr long long kDrainLimitNs = 10000000000LL;   // copies always land; 10 s is a backstop

__device__ __forceinline__ void raise(unsigned bits) { atomicOr(&g_status_gemv, bits); }

// Wait for an mbarrier phase, suspended in the barrier between polls.  Gives
// up (returns false) at once when the CTA's abort flag is up, or after
// `limit_ns`, raising the flag and the library's timeout status.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             long long limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = global_ns();
  // suspended polls (20 us hint) for the normal limit; under a limit below
  // that, non-blocking tests, so that a wait not already satisfied does give
  // up (try_wait may block until the phase completes)
  const bool poll = limit_ns < 20000;
  for (;;) {
    if (poll ? mbar_test_wait(bar, parity) : mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      raise(kErrTimeout);
      return false;
    }
  }
}

// Wait for bulk copies this CTA issued itself, whatever the abort flag says.
__device__ __forceinline__ void wait_drain(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  const long long t0 = global_ns();
  while (!mbar_try_wait_suspend(bar, parity, 20000u)) {
    if (global_ns() - t0 > kDrainLimitNs) {
      raise(kErrTimeout);
      return;
    }
  }
}

struct SmemLayout {
  static constexpr int stages_off = 0;
  static constexpr int red_off = kStages * kStageBytes;
  template <int TOKC>
  __host__ __device__ static constexpr int red_bytes() { return kConsumerWarps * kSlabRows * 8 * TOKC * 4; }
  template <int TOKC>
  __host__ __device__ static constexpr int bar_off() { return red_off + red_bytes<TOKC>(); }
  template <int TOKC>
  __host__ __device__ static constexpr int route_off() { return bar_off<TOKC>() + 2 * kStages * 8 + 16; }
  // routing area (grouped only): topk copy, token list, used-expert list
  template <int TOKC, bool GROUPED>
  __host__ __device__ static constexpr int total() {
    return route_off<TOKC>() +
           (GROUPED ? (kMaxRouting * 4 + 64 * 4 + kMaxExperts * 2 + kMaxExperts + 16) : 0);
  }
};

// ---------------------------------------------------------------------------
template <int TOKC, bool GROUPED>
__global__ void __launch_bounds__(kThreads)
gemv_kernel(const __grid_constant__ GemvParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stage_buf = smem + SmemLayout::stages_off;
  float* red = reinterpret_cast<float*>(smem + SmemLayout::red_off);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + SmemLayout::bar_off<TOKC>());
  uint64_t* empty_bar = full_bar + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty_bar + kStages);
  const long long wait_ns = p.wait_ns;
  uint8_t* route = smem + SmemLayout::route_off<TOKC>();
  int32_t* topk_s = reinterpret_cast<int32_t*>(route);
  int32_t* list_tok = reinterpret_cast<int32_t*>(route + kMaxRouting * 4);  // token | slot<<8
  uint16_t* used_list = reinterpret_cast<uint16_t*>(route + kMaxRouting * 4 + 64 * 4);
  uint8_t* used_flag = route + kMaxRouting * 4 + 64 * 4 + kMaxExperts * 2;
  int* n_used_s = reinterpret_cast<int*>(used_flag + kMaxExperts);
  int* list_n_s = n_used_s + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nchunks = p.K / 128;
  const int nstages_unit = (nchunks + kConsumerWarps - 1) / kConsumerWarps;
  const int slabs = (p.N + kSlabRows - 1) / kSlabRows;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }

  int n_units;
  if constexpr (GROUPED) {
    // Which experts does this round read?  Every CTA derives the same
    // ascending list from topk_idx, so no extra launch is needed.
    const int nr = p.M * p.topk;
    for (int e = threadIdx.x; e < p.E; e += kThreads) used_flag[e] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < nr; i += kThreads) {
      int e = p.topk_idx[i];
      topk_s[i] = e;
      if (e >= 0 && e < p.E) used_flag[e] = 1;
      else raise(kErrRouting);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < nr; i += kThreads) {   // distinct experts per token
      const int row0 = (i / p.topk) * p.topk;
      for (int j = row0; j < i; ++j)
        if (topk_s[j] == topk_s[i]) raise(kErrRouting);
    }
    if (warp == 0) {
      int base = 0;
      for (int e0 = 0; e0 < p.E; e0 += 32) {
        int e = e0 + lane;
        bool u = (e < p.E) && used_flag[e];
        unsigned m = __ballot_sync(0xffffffffu, u);
        if (u) used_list[base + __popc(m & ((1u << lane) - 1u))] = static_cast<uint16_t>(e);
        base += __popc(m);
      }
      if (lane == 0) *n_used_s = base;
    }
    __syncthreads();
    n_units = *n_used_s * slabs;
  } else {
    __syncthreads();
    n_units = slabs;
  }

  // ------------------------------------------------------------ producer --
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      uint32_t it = 0;
      bool stop = false;
      const uint64_t pol = l2_evict_first_policy();
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        // the slab's rows inside its 128-row tile; each k-tile piece of the
        // slab is contiguous (rows x 48 B) in the tile-ordered code stream
        const uint8_t* mat = p.codes;
        int slab_row0;
        if constexpr (GROUPED) {
          const int e = used_list[u / slabs];
          mat += static_cast<long long>(e) * (3LL * p.K / 8) * p.N;
          slab_row0 = (u % slabs) * kSlabRows;
        } else {
          slab_row0 = u * kSlabRows;
        }
        const int t = slab_row0 / 128, i0 = slab_row0 % 128;
        const int rows_t = tile_rows(t, p.N);
        const uint32_t piece = static_cast<uint32_t>(min(kSlabRows, rows_t - i0)) * 48;
        const uint8_t* tile = mat + tile_base(t, p.K) + static_cast<long long>(i0) * 48;
        for (int st = 0; st < nstages_unit; ++st, ++it) {
          const int slot = it % kStages;
          const uint32_t ph = (it / kStages) & 1u;
          if (it >= static_cast<uint32_t>(kStages)) {
            // the slot's previous stage must be consumed, and its copies
            // landed (always so after a normal release; checked so that no
            // give-up elsewhere can re-arm a barrier with copies in flight)
            if (!wait_bounded(&empty_bar[slot], ph ^ 1u, abort_flag, wait_ns)) {
              stop = true;
              break;
            }
            wait_drain(&full_bar[slot], ph ^ 1u);
          }
          const int c0 = st * kConsumerWarps;
          const int nvalid = min(kConsumerWarps, nchunks - c0);
          mbar_arrive_expect_tx(&full_bar[slot], nvalid * piece);
          for (int c = 0; c < nvalid; ++c)
            bulk_g2s(stage_buf + slot * kStageBytes + c * kBoxBytes,
                     tile + static_cast<long long>(c0 + c) * rows_t * 48, piece, &full_bar[slot], pol);
        }
      }
      // every copy this CTA issued has landed before the thread (and so the
      // CTA) can end
      for (uint32_t j = it > static_cast<uint32_t>(kStages) ? it - kStages : 0u; j < it; ++j)
        wait_drain(&full_bar[j % kStages], (j / kStages) & 1u);
    }
    return;
  }

  // ------------------------------------------------------------ consumers --
  const int g = lane >> 2;       // fragment row group
  const int t = lane & 3;        // quarter of the group this lane decodes
  const uint32_t lo_off = 4u * ((3u * t) >> 2);
  const uint32_t hi_off = (t == 3) ? lo_off : lo_off + 4u;
  const uint32_t sh = (3u * t & 3u) * 8u;
  const int ktiles_stride = p.K / 32;   // scale bytes per row
  uint32_t it = 0;

  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    int row_base, row_end, slab_row0;
    int ntok;
    if constexpr (GROUPED) {
      const int e = used_list[u / slabs];
      slab_row0 = (u % slabs) * kSlabRows;
      row_base = e * p.N + slab_row0;
      row_end = e * p.N + p.N;
      // token list of this expert: (token, slot) pairs in routing order
      if (warp == 0) {
        const int nr = p.M * p.topk;
        int base = 0;
        for (int i0 = 0; i0 < nr; i0 += 32) {
          int i = i0 + lane;
          bool hit = (i < nr) && topk_s[i] == e;
          unsigned m = __ballot_sync(0xffffffffu, hit);
          int pos = base + __popc(m & ((1u << lane) - 1u));
          if (hit && pos < 64) list_tok[pos] = (i / p.topk) | ((i % p.topk) << 8);
          base += __popc(m);
        }
        if (lane == 0) {
          if (base > p.M) raise(kErrRouting);
          *list_n_s = min(base, 64);
        }
      }
      named_bar_sync(1, kConsumerWarps * 32);
      ntok = *list_n_s;
    } else {
      slab_row0 = u * kSlabRows;
      row_base = slab_row0;
      row_end = p.N;
      ntok = p.M;
    }
    const int rA = row_base + g, rB = row_base + g + 8;
    const bool okA = rA < row_end, okB = rB < row_end;

    // codebooks of the lane's two rows: entries 0-3 and 4-7 in two registers
    uint2 cbA = okA ? *reinterpret_cast<const uint2*>(p.codebooks + size_t(rA) * 8) : make_uint2(0, 0);
    uint2 cbB = okB ? *reinterpret_cast<const uint2*>(p.codebooks + size_t(rB) * 8) : make_uint2(0, 0);
    const uint8_t* scA = p.scales + size_t(okA ? rA : 0) * ktiles_stride;
    const uint8_t* scB = p.scales + size_t(okB ? rB : 0) * ktiles_stride;

    // activation row pointers of the lane's token in each 8-token chunk
    const uint8_t* arow[TOKC];
#pragma unroll
    for (int tc = 0; tc < TOKC; ++tc) {
      int i = tc * 8 + g;
      int tok = -1;
      if (i < ntok) {
        if constexpr (GROUPED) tok = list_tok[i] & 0xff;
        else tok = i;
      }
      arow[tc] = tok >= 0 ? p.a + size_t(tok) * p.K + 8 * t : nullptr;
    }

    float acc[TOKC][4];
#pragma unroll
    for (int tc = 0; tc < TOKC; ++tc)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[tc][i] = 0.f;

    for (int st = 0; st < nstages_unit; ++st, ++it) {
      const int slot = it % kStages;
      const uint32_t ph = (it / kStages) & 1u;
      const int chunk = st * kConsumerWarps + warp;
      // loads that do not depend on the TMA stage go first
      uint32_t sA = 0, sB = 0;
      uint2 av[TOKC][4];
      if (chunk < nchunks) {
        sA = okA ? *reinterpret_cast<const uint32_t*>(scA + chunk * 4) : 0u;
        sB = okB ? *reinterpret_cast<const uint32_t*>(scB + chunk * 4) : 0u;
#pragma unroll
        for (int tc = 0; tc < TOKC; ++tc)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            av[tc][q] = arow[tc] ? __ldg(reinterpret_cast<const uint2*>(arow[tc] + chunk * 128 + q * 32))
                                 : make_uint2(0, 0);
      }
      wait_bounded(&full_bar[slot], ph, abort_flag, wait_ns);
      if (chunk < nchunks) {
        const uint32_t box = smem_u32(stage_buf + slot * kStageBytes + warp * kBoxBytes);
        const uint32_t rowA = box + g * 48, rowB = box + (g + 8) * 48;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t fA = __funnelshift_r(lds32(rowA + 12 * q + lo_off), lds32(rowA + 12 * q + hi_off), sh);
          uint32_t fB = __funnelshift_r(lds32(rowB + 12 * q + lo_off), lds32(rowB + 12 * q + hi_off), sh);
          uint32_t selA = spread_codes8(fA), selB = spread_codes8(fB);
          uint32_t a0 = lookup4(cbA.x, cbA.y, selA);
          uint32_t a2 = lookup4(cbA.x, cbA.y, upper_half(selA));
          uint32_t a1 = lookup4(cbB.x, cbB.y, selB);
          uint32_t a3 = lookup4(cbB.x, cbB.y, upper_half(selB));
          const float fsA = e8m0_word_byte_to_f32(sA, q);
          const float fsB = e8m0_word_byte_to_f32(sB, q);
#pragma unroll
          for (int tc = 0; tc < TOKC; ++tc) {
            if (tc * 8 < ntok) {
              float d[4];
              mma_e4m3_16832(d, a0, a1, a2, a3, av[tc][q].x, av[tc][q].y);
              acc[tc][0] = fmaf(d[0], fsA, acc[tc][0]);
              acc[tc][1] = fmaf(d[1], fsA, acc[tc][1]);
              acc[tc][2] = fmaf(d[2], fsB, acc[tc][2]);
              acc[tc][3] = fmaf(d[3], fsB, acc[tc][3]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[slot]);
    }

    // ---- sum the 4 K-split partials, apply a_scale, store ----
    constexpr int TW = 8 * TOKC;
#pragma unroll
    for (int tc = 0; tc < TOKC; ++tc) {
      const int c0 = tc * 8 + 2 * t;
      red[(warp * kSlabRows + g) * TW + c0] = acc[tc][0];
      red[(warp * kSlabRows + g) * TW + c0 + 1] = acc[tc][1];
      red[(warp * kSlabRows + g + 8) * TW + c0] = acc[tc][2];
      red[(warp * kSlabRows + g + 8) * TW + c0 + 1] = acc[tc][3];
    }
    named_bar_sync(1, kConsumerWarps * 32);
    for (int idx = threadIdx.x; idx < kSlabRows * ntok; idx += kConsumerWarps * 32) {
      const int i = idx / kSlabRows, r = idx % kSlabRows;
      const int row = row_base + r;
      if (row >= row_end) continue;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) s += red[(w * kSlabRows + r) * TW + i];   // in warp order
      if constexpr (GROUPED) {
        const int tok = list_tok[i] & 0xff, slot = list_tok[i] >> 8;
        p.y[(size_t(tok) * p.topk + slot) * p.N + slab_row0 + r] = s * p.a_scale[tok];
      } else {
        p.y[size_t(i) * p.N + row] = s * p.a_scale[i];
      }
    }
    named_bar_sync(1, kConsumerWarps * 32);
  }
}

// ---------------------------------------------------------------------------
// Unpack: one thread per group of 32 weights -> 32 exact fp32 values.
__global__ void unpack_kernel(const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales,
                              const uint8_t* __restrict__ codebooks, int N, int K,
                              float* __restrict__ W) {
  const int groups_row = K / 32;
  const long long ngroups = static_cast<long long>(N) * groups_row;
  for (long long gi = blockIdx.x * (long long)blockDim.x + threadIdx.x; gi < ngroups;
       gi += (long long)gridDim.x * blockDim.x) {
    const long long n = gi / groups_row;
    const int g = static_cast<int>(gi % groups_row);
    const int t = static_cast<int>(n / 128);
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(
        codes + tile_base(t, K) + static_cast<long long>(g / 4) * tile_rows(t, N) * 48 + (n % 128) * 48 +
        (g % 4) * 12);
    const uint32_t w0 = wp[0], w1 = wp[1], w2 = wp[2];
    const uint2 cb = *reinterpret_cast<const uint2*>(codebooks + n * 8);
    const float sc = e8m0_to_f32(scales[gi]);
    float4* out = reinterpret_cast<float4*>(W + gi * 32);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t sel = spread_codes8(group_field(w0, w1, w2, q));
      const uint32_t b_lo = lookup4(cb.x, cb.y, sel), b_hi = lookup4(cb.x, cb.y, upper_half(sel));
      float v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[i] = __half2float(__half(__nv_cvt_fp8_to_halfraw(
                   static_cast<__nv_fp8_storage_t>((b_lo >> (8 * i)) & 0xff), __NV_E4M3))) * sc;
        v[4 + i] = __half2float(__half(__nv_cvt_fp8_to_halfraw(
                       static_cast<__nv_fp8_storage_t>((b_hi >> (8 * i)) & 0xff), __NV_E4M3))) * sc;
      }
      out[2 * q] = make_float4(v[0], v[1], v[2], v[3]);
      out[2 * q + 1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

template <int TOKC, bool GROUPED>
int launch_gemv_t(const GemvParams& p, int units_upper, cudaStream_t stream) {
  const int smem = SmemLayout::total<TOKC, GROUPED>();
  // the shared-memory attribute and the occupancy, once per device and
  // template instance (the attribute is a per-device setting)
  static std::atomic<int> occupancy_of[64] = {};
  auto kern = gemv_kernel<TOKC, GROUPED>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CBQ_EDEVICE;
  int occupancy = occupancy_of[dev].load(std::memory_order_acquire);
  if (occupancy == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return CBQ_ECUDA;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem) != cudaSuccess)
      return CBQ_ECUDA;
    occupancy = occ > 0 ? occ : 1;
    occupancy_of[dev].store(occupancy, std::memory_order_release);
  }
  const int grid = std::max(1, std::min(units_upper, device_sm_count() * occupancy));
  kern<<<grid, kThreads, smem, stream>>>(p);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? CBQ_OK : CBQ_ECUDA;
}

}  // namespace

int launch_gemv(const GemvParams& p, bool grouped, cudaStream_t stream) {
  const int slabs = (p.N + kSlabRows - 1) / kSlabRows;
  const int tokens = grouped ? std::min(p.M, 64) : p.M;
  const int tokc = (tokens + 7) / 8;
  int units = slabs;
  if (grouped) units = std::min(p.E, p.M * p.topk) * slabs;
  if (grouped) {
    if (tokc <= 1) return launch_gemv_t<1, true>(p, units, stream);
    if (tokc <= 2) return launch_gemv_t<2, true>(p, units, stream);
    if (tokc <= 4) return launch_gemv_t<4, true>(p, units, stream);
    return launch_gemv_t<8, true>(p, units, stream);
  }
  if (tokc <= 1) return launch_gemv_t<1, false>(p, units, stream);
  if (tokc <= 2) return launch_gemv_t<2, false>(p, units, stream);
  if (tokc <= 4) return launch_gemv_t<4, false>(p, units, stream);
  return launch_gemv_t<8, false>(p, units, stream);
}

int launch_unpack(const uint8_t* codes, const uint8_t* scales, const uint8_t* codebooks, int N,
                  int K, float* W, cudaStream_t stream) {
  const long long ngroups = static_cast<long long>(N) * (K / 32);
  const int threads = 256;
  const long long want = (ngroups + threads - 1) / threads;
  const int grid = static_cast<int>(std::min<long long>(want, device_sm_count() * 16LL));
  unpack_kernel<<<std::max(grid, 1), threads, 0, stream>>>(codes, scales, codebooks, N, K, W);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? CBQ_OK : CBQ_ECUDA;
}

unsigned take_status_gemv(cudaStream_t stream) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_status_gemv, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return kErrTimeout;
  cudaMemcpyToSymbolAsync(g_status_gemv, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  cudaStreamSynchronize(stream);
  return v;
}

}  // namespace cbq
