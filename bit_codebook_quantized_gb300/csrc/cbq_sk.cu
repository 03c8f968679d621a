// cbq_sk.cu -- stream-K kernel of the codebook-quantised matmul for dense
// calls: every SM streams an equal, contiguous share of the packed weights,
// decodes the 3-bit codes to E4M3 straight into tensor memory and multiplies
// them with the block-scaled FP8 tensor cores (tcgen05), fp32 accumulators in
// TMEM.
//
// "Hibana: Fast Agentic Inference on Unified-Memory Devices", section "Model
// surgery / Three-bit weights": codes look up an 8-entry FP8 codebook per
// row, one 8-bit power-of-two scale per 32 weights, FP8 tensor-core matmul;
// section "Adaptive speculation": a decode step multiplies one token row (a
// verify round up to 64) by the same weights, so the matmul is a stream over
// the weights and the work is split over the weights, not over the tokens.
//
// Work split (stream-K): a unit is 128 weight rows x 128 k (a tile's k-tile,
// 6 KB of codes); units are numbered tile-major, k-tile-minor, which is also
// their order in the tile-ordered code stream, so CTA b's share
// [b U / G, (b + 1) U / G) is ONE contiguous byte range of the codes.  A
// tile whose k-tiles are shared by several CTAs is finished by whichever of
// them arrives last on the tile's counter: each writes its fp32 partial tile
// to scratch, the last one sums the parts in part order (deterministic) and
// writes y.
//
// Roles (one CTA per SM, 704 threads):
//  * warp 0 (one lane): 1-D bulk copies of 4 consecutive units (24 KB, one
//    contiguous piece of the stream) into a ring of shared-memory stages;
//  * warps 2..17: four decoder warpgroups, group g takes unit g of every
//    stage; thread = weight row = TMEM lane.  A thread loads its row's 48
//    code bytes (three 128-bit loads at a conflict-free 48-byte pitch),
//    releases the stage, spreads the codes to nibbles and turns them into
//    E4M3 bytes with byte-permutes through the row's codebook (two
//    registers), writes the 128 bytes into its TMEM lane as the MMA's A
//    operand (32 columns) and its 4 E8M0 group scales as the A scale factors;
//  * warp 1 (one lane): 4 tcgen05.mma kind::mxf8f6f4.block_scale (K = 32)
//    per unit, A from TMEM, B (the activations, resident in shared memory
//    for the CTA's k-tiles) from a K-major descriptor; the E8M0 group scale
//    is the MX block scale of its 32-wide K block;
//  * warps 18..21: epilogue -- tcgen05.ld the accumulator (two alternate, one
//    per tile segment), then either y = a_scale * acc or the partial-tile
//    protocol above.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "cbq_device.cuh"
#include "cbq_internal.h"

namespace cbq {

static __device__ unsigned g_status_sk = 0;

namespace {

constexpr int kRows = 128;                            // MMA M: weight rows per tile
constexpr int kUnitsPerStage = 4;
constexpr int kStageBytes = kUnitsPerStage * kRows * 48;   // 24 KB
constexpr int kMaxStages = 8;
constexpr int kASlots = 8;                            // decoded units in TMEM
constexpr int kDecGroups = 4;
constexpr int kDecWarps = 4 * kDecGroups;
constexpr int kEpiWarp0 = 2 + kDecWarps;
constexpr int kThreads = (kEpiWarp0 + 4) * 32;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 64;                          // accumulator i at column 64 i
constexpr int kSfaCol = 128;                          // + 4 * A slot (4-column aligned)
constexpr int kSfbCol = 192;                          // 8 columns of 2^0
constexpr int kACol = 256;                            // + 32 * A slot
constexpr int kMaxSmem = 232448;
constexpr int kMinSmem = 120 * 1024;                  // one CTA per SM: it owns all of TMEM
constexpr int kNumBars = 2 * kMaxStages + 2 * kASlots + 4;
constexpr int kBarBytes = (kNumBars * 8 + 16 + 127) / 128 * 128;
static_assert(kACol + 32 * kASlots <= kTmemCols, "A slots exceed the allocation");
static_assert(kSfaCol + 4 * kASlots <= kSfbCol && kSfbCol + 8 <= kACol, "TMEM areas overlap");
static_assert(2 * kAccCols <= kSfaCol, "accumulators overlap the scale factors");

__device__ __forceinline__ void raise(unsigned bits) { atomicOr(&g_status_sk, bits); }
__device__ __forceinline__ bool status_set() {
  return *reinterpret_cast<volatile unsigned*>(&g_status_sk) != 0u;
}

// Spin on an mbarrier phase.  After ~0.5 ms give up at once if another wait
// already timed out; after kWaitLimitCycles raise kErrTimeout and give up.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 63u) == 0) {
      const long long dt = clock64() - t0;
      if (dt > (1LL << 20)) {
        if (status_set()) return false;
        if (dt > kWaitLimitCycles) {
          raise(kErrTimeout);
          return false;
        }
      }
    }
  }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Unit geometry of an N x K weight in the tile-ordered code stream.  Unit
// u = t * KT + c is k-tile c of 128-row tile t; positions inside the loops
// advance incrementally (no division per unit).
struct Geo {
  int N, K, KT;                       // KT = k-tiles per row
  long long U, G;                     // units, CTAs
  __device__ __forceinline__ int rows(int t) const { return min(kRows, N - kRows * t); }
  // byte offset of unit (t, c): tile t at 48 K t, k-tile block c at c * rows * 48
  __device__ __forceinline__ long long off(int t, int c) const {
    return 48LL * K * t + static_cast<long long>(c) * rows(t) * 48;
  }
  __device__ __forceinline__ void advance(int& t, int& c, int n) const {
    c += n;
    while (c >= KT) {
      c -= KT;
      ++t;
    }
  }
  __device__ __forceinline__ long long first_unit(long long b) const { return b * U / G; }
  // the CTA whose share holds unit u
  __device__ __forceinline__ long long owner(long long u) const { return ((u + 1) * G + U - 1) / U - 1; }
};

template <int NTOK>
__global__ void __launch_bounds__(kThreads, 1) sk_kernel(const __grid_constant__ SkParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int NS = p.stages;
  uint8_t* codes_s = smem;
  uint8_t* b_s = smem + NS * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(b_s + p.b_ktiles * NTOK * 128);
  uint64_t* full = bars;
  uint64_t* empty = full + kMaxStages;
  uint64_t* a_full = empty + kMaxStages;
  uint64_t* a_empty = a_full + kASlots;
  uint64_t* acc_full = a_empty + kASlots;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  Geo geo;
  geo.N = p.N;
  geo.K = p.K;
  geo.KT = p.K / 128;
  geo.U = static_cast<long long>((p.N + kRows - 1) / kRows) * geo.KT;
  geo.G = gridDim.x;
  const int KT = geo.KT;
  const long long u0 = geo.first_unit(blockIdx.x), u1 = geo.first_unit(blockIdx.x + 1LL);
  const int n_units = static_cast<int>(u1 - u0);
  const int n_stages = (n_units + kUnitsPerStage - 1) / kUnitsPerStage;
  const int t_first = static_cast<int>(u0 / KT), c_first = static_cast<int>(u0 % KT);

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kDecWarps);                 // every decoder warp, once per stage
    }
    for (int i = 0; i < kASlots; ++i) {
      mbar_init(&a_full[i], 4);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    fence_barrier_init();
  }
  __syncthreads();

  uint32_t tbase = 0;
  if (warp == 0) {
    // -------------------------------------------------------- bulk producer --
    if (lane == 0) {
      int ta = t_first, ca = c_first;                 // first unit of stage j
      for (int j = 0; j < n_stages; ++j) {
        const int slot = j % NS;
        const int nu = min(kUnitsPerStage, n_units - j * kUnitsPerStage);
        int tl = ta, cl = ca;
        geo.advance(tl, cl, nu - 1);                   // last unit of the stage
        const long long oa = geo.off(ta, ca);
        const uint32_t bytes = static_cast<uint32_t>(geo.off(tl, cl) + geo.rows(tl) * 48LL - oa);
        geo.advance(ta, ca, kUnitsPerStage);
        wait_bounded(&empty[slot], ((j / NS) & 1u) ^ 1u);
        mbar_arrive_expect_tx(&full[slot], bytes);
        bulk_g2s(codes_s + slot * kStageBytes, p.codes + oa, bytes, &full[slot]);
      }
      // every copy has landed before the CTA can leave
      for (int j = max(0, n_stages - NS); j < n_stages; ++j) wait_bounded(&full[j % NS], (j / NS) & 1u);
    }
    __syncwarp();
  } else {
    if (warp == 1) {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
    // Resident activations: k-tile c of this CTA's share sits in slot
    // (c - c_first) mod KT, K-major core-matrix layout inside a slot: chunk
    // (16 k) cc at cc * NTOK * 16, token group at * 128, token % 8 at * 16.
    {
      const int nb = min(KT, n_units);
      const int total = nb * 8 * NTOK;
      for (int i = tid - 32; i < total; i += kThreads - 32) {
        const int tok = i % NTOK, ch = i / NTOK;        // ch = slot * 8 + chunk
        int c = c_first + (ch >> 3);
        if (c >= KT) c -= KT;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (tok < p.M)
          v = __ldg(reinterpret_cast<const uint4*>(p.a + static_cast<size_t>(tok) * p.K + c * 128 + (ch & 7) * 16));
        *reinterpret_cast<uint4*>(b_s + ch * NTOK * 16 + (tok >> 3) * 128 + (tok & 7) * 16) = v;
      }
      fence_proxy_async_smem();
    }
    tc_fence_before();
    named_bar_sync(1, kThreads - 32);                  // everyone but the producer
    tc_fence_after();
    tbase = *tmem_slot;
    if (warp >= kEpiWarp0) {                            // B scale factors: 2^0
      const uint32_t q = warp & 3;
      for (int c = 0; c < 8; c += 4)
        tmem_st_x4(tbase + ((32 * q) << 16) + kSfbCol + c, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_st_wait();
    }
    tc_fence_before();
    named_bar_sync(1, kThreads - 32);
    tc_fence_after();

    if (warp == 1) {
      // --------------------------------------------------------- MMA issuer --
      if (lane == 0) {
        const uint32_t b_base = smem_u32(b_s);
        const uint32_t idesc = umma_idesc_mxf8(NTOK, 0, 0);
        int seg = 0, c = c_first;
        for (int i = 0; i < n_units; ++i, c = (c + 1 == KT) ? 0 : c + 1) {
          const bool seg_first = (i == 0) || (c == 0);
          const int abuf = seg & 1;
          if (seg_first) {
            wait_bounded(&acc_empty[abuf], ((seg >> 1) & 1u) ^ 1u);
            tc_fence_after();
          }
          const int as = i % kASlots;
          wait_bounded(&a_full[as], (i / kASlots) & 1u);
          tc_fence_after();
          int bsl = c - c_first;
          if (bsl < 0) bsl += KT;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t bd = umma_desc_kmajor(b_base + (bsl * 8 + 2 * j) * NTOK * 16, NTOK * 16, 128);
            umma_mxf8_ts(tbase + abuf * kAccCols, tbase + kACol + as * 32 + j * 8, bd, idesc | (uint32_t(j) << 29),
                         tbase + kSfaCol + as * 4, tbase + kSfbCol, (seg_first && j == 0) ? 0u : 1u);
          }
          umma_commit(&a_empty[as]);
          if (c == KT - 1 || i == n_units - 1) {
            umma_commit(&acc_full[abuf]);
            ++seg;
          }
        }
      }
      __syncwarp();
    } else if (warp < kEpiWarp0) {
      // ------------------------------------------------------------ decoders --
      const int g = (warp - 2) >> 2, q = warp & 3;
      const int r = 32 * q + lane;                      // row inside the tile == TMEM lane
      const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
      const uint32_t codes_base = smem_u32(codes_s);
      const int gk = p.K / 32;
      // scale word and codebook of this row for unit (t, c) (loaded one of
      // this group's units ahead)
      auto unit_inputs = [&](bool valid, int t, int c, uint32_t& sw, uint2& cb) {
        sw = 0x7F7F7F7Fu;
        cb = make_uint2(0, 0);
        const int n = t * kRows + r;
        if (valid && n < p.N) {
          sw = __ldg(reinterpret_cast<const uint32_t*>(p.scales + static_cast<size_t>(n) * gk + 4 * c));
          cb = __ldg(reinterpret_cast<const uint2*>(p.codebooks + static_cast<size_t>(n) * 8));
        }
      };
      int tu = t_first, cu = c_first;                   // this group's unit in the current stage
      geo.advance(tu, cu, g);
      int tn = tu, cn = cu;                             // and in the next stage
      geo.advance(tn, cn, kDecGroups);
      uint32_t sw_next;
      uint2 cb_next;
      unit_inputs(g < n_units, tu, cu, sw_next, cb_next);
      for (int j = 0; j < n_stages; ++j) {
        const int i = j * kUnitsPerStage + g;
        const int slot = j % NS;
        const uint32_t sw = sw_next;
        const uint2 cb = cb_next;
        unit_inputs(i + kDecGroups < n_units, tn, cn, sw_next, cb_next);
        // every decoder warp waits for every stage before releasing it, so an
        // early release can never count towards an older phase
        wait_bounded(&full[slot], (j / NS) & 1u);
        const bool has = i < n_units;
        uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0, c2 = c0;
        if (has && r < geo.rows(tu)) {
          // units before this one in the stage: g of them, each rows * 48 bytes
          int tb = tu, cb0 = cu, rel = 0;
          for (int k = 0; k < g; ++k) {
            if (cb0 == 0) {
              --tb;
              cb0 = KT;
            }
            --cb0;
            rel += geo.rows(tb) * 48;
          }
          const uint32_t at = codes_base + slot * kStageBytes + rel + r * 48;
          c0 = lds128(at);
          c1 = lds128(at + 16);
          c2 = lds128(at + 32);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        tu = tn;
        cu = cn;
        geo.advance(tn, cn, kDecGroups);
        if (has) {
          uint32_t v[32];
          decode_group(c0.x, c0.y, c0.z, cb.x, cb.y, v);
          decode_group(c0.w, c1.x, c1.y, cb.x, cb.y, v + 8);
          decode_group(c1.z, c1.w, c2.x, cb.x, cb.y, v + 16);
          decode_group(c2.y, c2.z, c2.w, cb.x, cb.y, v + 24);
          const int as = i % kASlots;
          wait_bounded(&a_empty[as], ((i / kASlots) & 1u) ^ 1u);
          tc_fence_after();
          tmem_st_x32(tbase + lane_addr + kACol + as * 32, v);
          // A scale of row m: TMEM lane m, column base + m / 32, byte = a_sf_id
          tmem_st_x1(tbase + lane_addr + kSfaCol + as * 4 + q, sw);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[as]);
        }
      }
    } else {
      // ------------------------------------------------------------ epilogue --
      const int q = warp & 3;
      const int r = 32 * q + lane;
      const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
      const bool leader = tid == kEpiWarp0 * 32;
      int seg = 0, t = t_first, c = c_first, seg_c = c_first;   // seg_c: k-tile the segment starts at
      for (int i = 0; i < n_units; ++i, geo.advance(t, c, 1)) {
        if (c != KT - 1 && i != n_units - 1) continue;
        const bool complete = seg_c == 0 && c == KT - 1;
        const int n = t * kRows + r;
        const bool ok = n < p.N;
        const int abuf = seg & 1;
        wait_bounded(&acc_full[abuf], (seg >> 1) & 1u);
        tc_fence_after();
        float* part = p.partial + (static_cast<size_t>(2 * blockIdx.x + (seg > 0 ? 1 : 0)) * kRows + r) * NTOK;
#pragma unroll 1
        for (int c0 = 0; c0 < NTOK; c0 += 16) {
          uint32_t tv[16];
          tmem_ld_x16(tbase + lane_addr + abuf * kAccCols + c0, tv);
          tmem_ld_wait();
          if (complete) {
            if (ok) {
#pragma unroll
              for (int k = 0; k < 16; ++k)
                if (c0 + k < p.M)
                  p.y[static_cast<size_t>(c0 + k) * p.N + n] = __uint_as_float(tv[k]) * __ldg(p.a_scale + c0 + k);
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(part + c0);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              dst[k] = make_float4(__uint_as_float(tv[4 * k]), __uint_as_float(tv[4 * k + 1]),
                                   __uint_as_float(tv[4 * k + 2]), __uint_as_float(tv[4 * k + 3]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[abuf]);
        if (!complete) {
          // partial tile: publish, count, and the last part sums them all
          const long long tu = static_cast<long long>(t) * KT;
          const long long b_first = geo.owner(tu);
          const int nparts = static_cast<int>(geo.owner(tu + KT - 1) - b_first + 1);
          __threadfence();
          named_bar_sync(2, 128);
          if (leader) *last_flag = atomicAdd(p.counters + t, 1u) == static_cast<unsigned>(nparts - 1);
          named_bar_sync(2, 128);
          if (*last_flag) {
            __threadfence();
#pragma unroll 1
            for (int c0 = 0; c0 < NTOK; c0 += 16) {
              float acc[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) acc[k] = 0.f;
#pragma unroll 1
              for (int pi = 0; pi < nparts; ++pi) {
                // part 0's CTA reaches this tile as its last segment if its
                // share started in an earlier tile; every later part as its first
                const long long b = b_first + pi;
                const int pslot = 2 * static_cast<int>(b) + ((pi == 0 && geo.first_unit(b) < tu) ? 1 : 0);
                const float4* src =
                    reinterpret_cast<const float4*>(p.partial + (static_cast<size_t>(pslot) * kRows + r) * NTOK + c0);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  const float4 f = __ldcg(src + k);
                  acc[4 * k] += f.x;
                  acc[4 * k + 1] += f.y;
                  acc[4 * k + 2] += f.z;
                  acc[4 * k + 3] += f.w;
                }
              }
              if (ok) {
#pragma unroll
                for (int k = 0; k < 16; ++k)
                  if (c0 + k < p.M) p.y[static_cast<size_t>(c0 + k) * p.N + n] = acc[k] * __ldg(p.a_scale + c0 + k);
              }
            }
            if (leader) p.counters[t] = 0u;              // ready for the next call
          }
          named_bar_sync(2, 128);
        }
        seg_c = c + 1 == KT ? 0 : c + 1;
        ++seg;
      }
    }
  }

  // ---- teardown: the epilogue waited on the last commit, so every tcgen05
  // op has completed; the producer saw its last copies land.
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

int ntok_for(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

struct Plan {
  int ntok = 0, grid = 0, stages = 0, b_ktiles = 0, smem = 0, tiles = 0;
};

bool plan_for(int M, int N, int K, Plan& pl) {
  if (M < 1 || M > 64 || N < 1 || K < 128 || K % 128 != 0) return false;
  const int KT = K / 128;
  const long long tiles = (N + kRows - 1) / kRows;
  const long long U = tiles * KT;
  const long long G = std::min<long long>(U, device_sm_count());
  const long long per = (U + G - 1) / G;               // most units of any CTA
  pl.ntok = ntok_for(M);
  pl.b_ktiles = static_cast<int>(std::min<long long>(KT, per));
  const int b_bytes = pl.b_ktiles * pl.ntok * 128;
  const int room = kMaxSmem - b_bytes - kBarBytes;
  pl.stages = std::min(kMaxStages, room / kStageBytes);
  if (pl.stages < 3) return false;
  pl.smem = std::max(pl.stages * kStageBytes + b_bytes + kBarBytes, kMinSmem);
  pl.grid = static_cast<int>(G);
  pl.tiles = static_cast<int>(tiles);
  return true;
}

// Per (device, stream) scratch: partial tiles (two slots of 128 x 64 fp32 per
// CTA) and one arrival counter per tile (all zero between calls).
struct Scratch {
  float* partial = nullptr;
  size_t partial_floats = 0;
  unsigned* counters = nullptr;
  size_t n_counters = 0;
};
std::mutex g_scratch_mu;
std::map<std::pair<int, cudaStream_t>, Scratch> g_scratch;

int scratch_for(cudaStream_t s, size_t partial_floats, size_t n_counters, Scratch& out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CBQ_ECUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  Scratch& sc = g_scratch[std::make_pair(dev, s)];
  if (sc.partial_floats < partial_floats || sc.n_counters < n_counters) {
    // Growing never frees the old buffers: a kernel in flight, or a graph
    // captured earlier, may still use them.  cudaMalloc is allowed while the
    // calling thread captures a graph (relaxed mode); the zeroing of new
    // counters is ordered on the call's stream.
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    cudaError_t e = cudaSuccess;
    if (sc.partial_floats < partial_floats) {
      const size_t want = std::max(partial_floats, size_t(2) * device_sm_count() * kRows * 64);
      float* ptr = nullptr;
      e = cudaMalloc(&ptr, want * sizeof(float));
      if (e == cudaSuccess) {
        sc.partial = ptr;
        sc.partial_floats = want;
      }
    }
    if (e == cudaSuccess && sc.n_counters < n_counters) {
      const size_t want = std::max<size_t>(n_counters, 1 << 16);
      unsigned* ptr = nullptr;
      e = cudaMalloc(&ptr, want * sizeof(unsigned));
      if (e == cudaSuccess) e = cudaMemsetAsync(ptr, 0, want * sizeof(unsigned), s);
      if (e == cudaSuccess) {
        sc.counters = ptr;
        sc.n_counters = want;
      }
    }
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return CBQ_ECUDA;
    }
  }
  out = sc;
  return CBQ_OK;
}

template <int NTOK>
int launch_t(const SkParams& p, const Plan& pl, cudaStream_t stream) {
  auto kern = sk_kernel<NTOK>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem) != cudaSuccess)
    return CBQ_ECUDA;
  kern<<<pl.grid, kThreads, pl.smem, stream>>>(p);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? CBQ_OK : CBQ_ECUDA;
}

}  // namespace

bool sk_applicable(int M, int N, int K) {
  Plan pl;
  return plan_for(M, N, K, pl);
}

int launch_sk(const SkParams& p_in, cudaStream_t stream) {
  Plan pl;
  if (!plan_for(p_in.M, p_in.N, p_in.K, pl)) return CBQ_EINVAL;
  Scratch sc;
  const int st = scratch_for(stream, size_t(2) * pl.grid * kRows * pl.ntok, size_t(pl.tiles), sc);
  if (st != CBQ_OK) return st;
  SkParams p = p_in;
  p.partial = sc.partial;
  p.counters = sc.counters;
  p.stages = pl.stages;
  p.b_ktiles = pl.b_ktiles;
  if (pl.ntok == 16) return launch_t<16>(p, pl, stream);
  if (pl.ntok == 32) return launch_t<32>(p, pl, stream);
  return launch_t<64>(p, pl, stream);
}

unsigned take_status_sk(cudaStream_t stream) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_status_sk, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return kErrTimeout;
  cudaMemcpyToSymbolAsync(g_status_sk, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  cudaStreamSynchronize(stream);
  if (v != 0) {
    // a kernel gave up part-way: tile counters may be left non-zero
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    for (auto& kv : g_scratch)
      if (kv.second.counters) cudaMemset(kv.second.counters, 0, kv.second.n_counters * sizeof(unsigned));
  }
  return v;
}

}  // namespace cbq
