// cbq_sk.cu -- stream-K kernel of the codebook-quantised matmul for dense
// calls: every SM streams an equal, contiguous share of the packed weights,
// decodes the 3-bit codes to E4M3 in shared memory and multiplies them with
// the block-scaled FP8 tensor cores (tcgen05), fp32 accumulators in TMEM.
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
// Roles (one CTA per SM, 768 threads; a warp's sub-partition is warp % 4):
//  * warp 5: 1-D bulk copies of 4 consecutive units (24 KB, one contiguous
//    piece of the stream) into a ring of shared-memory stages;
//  * 12 decoder warps, all on sub-partitions 0, 2, 3 (so the MMA issuer on
//    sub-partition 1 has its issue slots to itself), in 3 groups of 4: group
//    g decodes the units i = g mod 3, one warp per 32 rows; a thread (one
//    row) loads its 48 code bytes, releases the stage,
//    spreads the codes to nibbles and turns them into E4M3 bytes with
//    byte-permutes through the row's codebook (two registers), and stores
//    the 128 bytes into the unit's A slot in shared memory (K-major
//    core-matrix layout, conflict-free 16-byte stores) with the row's 4 E8M0
//    group scales beside them;
//  * warp 1 (one lane): per unit one tcgen05.cp of the scales into TMEM and
//    4 tcgen05.mma kind::mxf8f6f4.block_scale (K = 32) with A and B (the
//    activations, resident in shared memory for the CTA's k-tiles, landed by
//    TMA) from shared-memory descriptors; the E8M0 group scale is the MX
//    block scale of its 32-wide K block;
//  * warps 16..19: epilogue -- tcgen05.ld the accumulator (two alternate, one
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
constexpr int kMaxASlots = 8;
constexpr int kASlotA = kRows * 128;                  // decoded E4M3 A of one unit
constexpr int kASlotBytes = kASlotA + kRows * 16;     // + one 16-byte scale row per weight row
constexpr int kTasksPerUnit = 4;                      // 32 rows each
constexpr int kDecGroups = 3;                         // unit i goes to group i % 3
static_assert(kDecGroups * kTasksPerUnit == 12, "12 decoder warps");
constexpr int kMmaWarp = 1;
constexpr int kProdWarp = 5;
constexpr int kEpiWarp0 = 16;                         // warps 16..19: quadrants 0..3
constexpr int kNumWarps = 24;
constexpr int kThreads = kNumWarps * 32;
constexpr int kTmemCols = 256;
constexpr int kMaxSmem = 232448;
constexpr int kMinSmem = 120 * 1024;                  // one CTA per SM
constexpr int kNumBars = 2 * kMaxStages + 2 * kMaxASlots + 5;
constexpr int kBarBytes = (kNumBars * 8 + 16 + 127) / 128 * 128;

// Decoder index of a warp (0..11), or -1: warps 0..15 off sub-partition 1
// (sub-partition 1 belongs to the MMA issuer).  Warps 9, 13, 20..23 idle.
__device__ __forceinline__ int decoder_index(int warp) {
  if (warp >= 16) return -1;
  const int q = warp & 3;
  return q == 1 ? -1 : (warp >> 2) * 3 + (q == 0 ? 0 : q - 1);
}

// Tensor-memory columns for NTOK token columns: two fp32 accumulators (32-column
// aligned), 8 columns of B scale factors (2^0), then 4 scale-factor columns per
// A slot (4-column aligned).
template <int NTOK>
struct TmemMap {
  static constexpr int kAccStride = NTOK < 32 ? 32 : NTOK;
  static constexpr int kAcc = 0;                              // + kAccStride * buffer
  static constexpr int kSfb = 2 * kAccStride;
  static constexpr int kSfa = kSfb + 8;                       // + 4 * slot
  static_assert(kSfa + 4 * kMaxASlots <= kTmemCols, "TMEM map exceeds the allocation");
};

__device__ __forceinline__ void raise(unsigned bits) { atomicOr(&g_status_sk, bits); }
__device__ __forceinline__ bool status_set() {
  return *reinterpret_cast<volatile unsigned*>(&g_status_sk) != 0u;
}

// Wait for an mbarrier phase, suspended in the barrier rather than spinning
// (spinning warps would steal issue slots from the warps that work).  After
// ~0.5 ms give up at once if another wait already timed out; after
// kWaitLimitNs raise kErrTimeout and give up.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = global_ns();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    const long long dt = global_ns() - t0;
    if (dt > 500000LL) {
      if (status_set()) return false;
      if (dt > kWaitLimitNs) {
        raise(kErrTimeout);
        return false;
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

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
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
  using TM = TmemMap<NTOK>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int NS = p.stages, S = p.a_slots;
  uint8_t* codes_s = smem;
  uint8_t* b_s = smem + NS * kStageBytes;
  uint8_t* a_s = b_s + p.b_ktiles * NTOK * 128;
  uint64_t* bars = reinterpret_cast<uint64_t*>(a_s + S * kASlotBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + kMaxStages;
  uint64_t* a_full = empty + kMaxStages;
  uint64_t* a_empty = a_full + kMaxASlots;
  uint64_t* acc_full = a_empty + kMaxASlots;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* b_full = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(b_full + 1);
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
      mbar_init(&empty[i], kUnitsPerStage * kTasksPerUnit);   // every task of the stage, once
    }
    for (int i = 0; i < S; ++i) {
      mbar_init(&a_full[i], kTasksPerUnit);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);
    }
    mbar_init(b_full, 1);
    fence_barrier_init();
  }
  __syncthreads();
  // The next kernel on the stream may start its prologue (and, if it is this
  // one, its weight stream) as soon as SMs free up; whatever this grid reads
  // from or writes for earlier kernels waits on grid_dependency_wait below.
  grid_launch_dependents();

  uint32_t tbase = 0;
  if (warp == kProdWarp) {
    // -------------------------------------------------------- bulk producer --
    if (lane == 0) {
      int ta = t_first, ca = c_first;                 // first unit of stage j
      const uint64_t pol = l2_evict_first_policy();
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
        bulk_g2s(codes_s + slot * kStageBytes, p.codes + oa, bytes, &full[slot], pol);
      }
      // every copy has landed before the CTA can leave
      for (int j = max(0, n_stages - NS); j < n_stages; ++j) wait_bounded(&full[j % NS], (j / NS) & 1u);
    }
    __syncwarp();
  } else {
    if (warp == kMmaWarp) {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    named_bar_sync(1, kThreads - 32);                  // everyone but the producer
    tc_fence_after();
    tbase = *tmem_slot;

    const int dec = decoder_index(warp);
    if (warp == kMmaWarp) {
      // --------------------------------------------------------- MMA issuer --
      named_bar_sync(3, 160);                          // B scale factors are in TMEM
      tc_fence_after();
      if (lane == 0) {
        // Resident activations (written by an earlier kernel, so after the
        // grid dependency): k-tile c of this CTA's share lands in slot
        // (c - c_first) mod KT as ntok rows of 128 bytes in the 128-byte
        // swizzled K-major layout (one TMA box); token rows >= M are outside
        // the tensor and arrive as zeros.
        grid_dependency_wait();
        const int nb = min(KT, n_units);
        mbar_arrive_expect_tx(b_full, static_cast<uint32_t>(nb * NTOK * 128));
        for (int sl = 0; sl < nb; ++sl) {
          int c = c_first + sl;
          if (c >= KT) c -= KT;
          uint8_t* dst = b_s + sl * NTOK * 128;
          if (p.b_layout == 0) tma_load_2d(dst, &p.a_map, b_full, c * 128, 0);
          else tma_load_3d(dst, &p.a_map, b_full, 0, 0, 8 * c);
        }
        // Descriptors advance by adding offsets in their 16-byte address
        // units (every shared address here is below 256 KB, so the 14-bit
        // address field never carries): A slot as at as * kASlotBytes, its
        // K chunk pair j at 2 j * 2048; B slot at bsl * NTOK * 128, its MMA j
        // at 32 j (swizzled) or 2 j * NTOK * 16 bytes (core matrices).
        const uint32_t a_base = smem_u32(a_s);
        const uint64_t ad0 = umma_desc_kmajor(a_base, kRows * 16, 128);
        const uint64_t sd0 = umma_desc_kmajor(a_base + kASlotA, 128, 128);
        const uint64_t bd0 = p.b_layout == 0 ? umma_desc_kmajor_sw128(smem_u32(b_s))
                                             : umma_desc_kmajor(smem_u32(b_s), NTOK * 16, 128);
        const uint32_t b_step_j = p.b_layout == 0 ? 2u : 2u * NTOK;
        const uint32_t idesc = umma_idesc_mxf8(NTOK, 0, 0);
        const uint32_t sfa0 = tbase + TM::kSfa, sfb = tbase + TM::kSfb;
        wait_bounded(b_full, 0);
        int seg = 0, c = c_first, as = 0, bsl = 0;
        uint32_t a_phase = 0;
        for (int i = 0; i < n_units; ++i) {
          const bool seg_first = (i == 0) || (c == 0);
          const int abuf = seg & 1;
          if (seg_first) {
            wait_bounded(&acc_empty[abuf], ((seg >> 1) & 1u) ^ 1u);
            tc_fence_after();
          }
          wait_bounded(&a_full[as], a_phase);
          tc_fence_after();
          const uint64_t a_off = static_cast<uint64_t>(as * (kASlotBytes >> 4));
          // the unit's scale rows -> 4 TMEM columns (row r's scale word sits
          // in every 32-bit word of its 16-byte row, whichever column the MMA
          // reads for it)
          tmem_cp_128x128b(sfa0 + 4 * as, sd0 + a_off);
          const uint64_t adu = ad0 + a_off;
          const uint64_t bdu = bd0 + static_cast<uint64_t>(bsl * NTOK * 8);
          const uint32_t d_col = tbase + TM::kAcc + abuf * TM::kAccStride;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            umma_mxf8(d_col, adu + static_cast<uint64_t>(j * 256), bdu + static_cast<uint64_t>(j * b_step_j),
                      idesc | (uint32_t(j) << 29), sfa0 + 4 * as, sfb, (seg_first && j == 0) ? 0u : 1u);
          umma_commit(&a_empty[as]);
          if (++as == S) {
            as = 0;
            a_phase ^= 1u;
          }
          if (c == KT - 1 || i == n_units - 1) {
            umma_commit(&acc_full[abuf]);
            ++seg;
          }
          c = (c + 1 == KT) ? 0 : c + 1;
          bsl = (bsl + 1 == KT) ? 0 : bsl + 1;        // (c - c_first) mod KT
        }
      }
      __syncwarp();
    } else if (dec >= 0) {
      // ------------------------------------------------------------ decoders --
      // Decoder d = 4 g + q takes rows 32 q .. 32 q + 31 of the units
      // i = g, g + 3, ... (group g = i % 3).  A group walks its units in
      // order and the A-slot count is a multiple of 3, so a slot always goes
      // back to the same group: the slot's parity wait can never be a phase
      // (two uses) early.  Row r's 128 bytes go to the A slot as 8 chunks of
      // 16 (chunk x at x * 2048 + r * 16: core matrices of 8 rows x 16 bytes,
      // 128 bytes apart along M, 2048 apart along K), its scale word to the
      // slot's scale row r (4 copies).
      const uint32_t codes_base = smem_u32(codes_s);
      const uint32_t a_base = smem_u32(a_s);
      const int gk = p.K / 32;
      const int grp = dec / kTasksPerUnit, q = dec % kTasksPerUnit;
      const int r = 32 * q + lane;                      // row inside the tile
      // scale word and codebook of row r for the unit at (t, c)
      auto load_sc = [&](int t, int c, bool valid, uint32_t& sw, uint2& cb) {
        sw = 0x7F7F7F7Fu;
        cb = make_uint2(0, 0);
        const int n = t * kRows + r;
        if (valid && n < p.N) {
          sw = __ldg(reinterpret_cast<const uint32_t*>(p.scales + static_cast<size_t>(n) * gk + 4 * c));
          cb = __ldg(reinterpret_cast<const uint2*>(p.codebooks + static_cast<size_t>(n) * 8));
        }
      };
      // Stage slot / phase and A slot / phase of the current unit, advanced
      // incrementally (no division by the runtime ring sizes per unit).
      int st_j = 0, st_slot = 0, a_slot = 0;
      uint32_t st_phase = 0, a_phase = 0;
      auto seek = [&](int i) {                          // i only grows, by 3 at most 1 stage
        const int j = i / kUnitsPerStage;
        while (st_j < j) {
          ++st_j;
          if (++st_slot == NS) {
            st_slot = 0;
            st_phase ^= 1u;
          }
        }
      };
      auto process = [&](int i, int tu, int cu, uint32_t sw, uint2 cb) {
        const int k = i % kUnitsPerStage;
        seek(i);
        const int slot = st_slot;
        // every task waits for its stage before releasing it, so an early
        // release can never count towards an older phase
        wait_bounded(&full[slot], st_phase);
        uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0, c2 = c0;
        const int rows_u = geo.rows(tu);
        if (r < rows_u) {
          // units before this one in the stage: k of them, min(k, cu) in tile
          // tu (rows_u rows each; tu may be the ragged last tile) and the
          // rest in full tiles before it
          const int kin = min(k, cu);
          const uint32_t at = codes_base + slot * kStageBytes + (kin * rows_u + (k - kin) * kRows + r) * 48;
          c0 = lds128(at);
          c1 = lds128(at + 16);
          c2 = lds128(at + 32);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        uint32_t v[32];
        decode_group(c0.x, c0.y, c0.z, cb.x, cb.y, v);
        decode_group(c0.w, c1.x, c1.y, cb.x, cb.y, v + 8);
        decode_group(c1.z, c1.w, c2.x, cb.x, cb.y, v + 16);
        decode_group(c2.y, c2.z, c2.w, cb.x, cb.y, v + 24);
        const int as = a_slot;
        wait_bounded(&a_empty[as], a_phase ^ 1u);
        const uint32_t slot_addr = a_base + as * kASlotBytes;
#pragma unroll
        for (int x = 0; x < 8; ++x)
          sts128(slot_addr + x * (kRows * 16) + r * 16, v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
        sts128(slot_addr + kASlotA + r * 16, sw, sw, sw, sw);
        fence_proxy_async_smem();                       // visible to the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[as]);
        a_slot += kDecGroups;                           // this group's next slot
        if (a_slot >= S) {
          a_slot -= S;
          a_phase ^= 1u;
        }
      };
      // Two register sets for the scale word and codebook, so the loads for
      // the group's next unit are in flight during the current one (unrolled
      // by two: no register copy has to wait for a load).
      int ta = t_first, ca = c_first;                   // unit i (set A)
      geo.advance(ta, ca, grp);
      a_slot = grp;                                     // unit grp's A slot (S is a multiple of 3)
      uint32_t swA, swB;
      uint2 cbA, cbB;
      load_sc(ta, ca, grp < n_units, swA, cbA);
      for (int i = grp; i < n_units; i += 2 * kDecGroups) {
        int tb = ta, cbb = ca;                          // unit i + 3 (set B)
        geo.advance(tb, cbb, kDecGroups);
        load_sc(tb, cbb, i + kDecGroups < n_units, swB, cbB);
        process(i, ta, ca, swA, cbA);
        if (i + kDecGroups >= n_units) break;
        ta = tb;                                        // unit i + 6 (set A)
        ca = cbb;
        geo.advance(ta, ca, kDecGroups);
        load_sc(ta, ca, i + 2 * kDecGroups < n_units, swA, cbA);
        process(i + kDecGroups, tb, cbb, swB, cbB);
      }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
      const int q = warp & 3;
      const int r = 32 * q + lane;
      const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
      const bool leader = tid == kEpiWarp0 * 32;
      // scale factors of B: 2^0 in every byte of 8 columns, all 128 lanes
      for (int cc = 0; cc < 8; cc += 4)
        tmem_st_x4(tbase + lane_addr + TM::kSfb + cc, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_st_wait();
      tc_fence_before();
      named_bar_sync(3, 160);
      grid_dependency_wait();                           // y and the scratch may still be in use
      int seg = 0, t = t_first, c = c_first, seg_c = c_first;   // seg_c: k-tile the segment starts at
      for (int i = 0; i < n_units; ++i, geo.advance(t, c, 1)) {
        if (c != KT - 1 && i != n_units - 1) continue;
        const bool complete = seg_c == 0 && c == KT - 1;
        const int n = t * kRows + r;
        const bool ok = n < p.N;
        const int abuf = seg & 1;
        const uint32_t acc_addr = tbase + lane_addr + TM::kAcc + abuf * TM::kAccStride;
        wait_bounded(&acc_full[abuf], (seg >> 1) & 1u);
        tc_fence_after();
        if (complete) {
#pragma unroll 1
          for (int c0 = 0; c0 < NTOK; c0 += 16) {
            uint32_t tv[16];
            tmem_ld_x16(acc_addr + c0, tv);
            tmem_ld_wait();
            if (ok) {
#pragma unroll
              for (int k = 0; k < 16; ++k)
                if (c0 + k < p.M)
                  p.y[static_cast<size_t>(c0 + k) * p.N + n] = __uint_as_float(tv[k]) * __ldg(p.a_scale + c0 + k);
            }
          }
        } else {
          // Partial tile.  Each part's fp32 tile goes to its scratch slot and
          // bumps the tile's counter; the part that finds every other part
          // published sums all parts in part order and writes y.  A CTA's
          // last segment usually arrives after the other parts (first segments
          // of later CTAs, finished early), so it first just reads the counter.
          const long long tu = static_cast<long long>(t) * KT;
          const long long b_first = geo.owner(tu);
          const int nparts = static_cast<int>(geo.owner(tu + KT - 1) - b_first + 1);
          const int pme = static_cast<int>(blockIdx.x - b_first);
          bool own_published = false, last = false;
          if (i == n_units - 1) {                         // this CTA's last segment
            if (leader) *last_flag = ld_acquire_gpu(p.counters + t) == static_cast<unsigned>(nparts - 1);
            named_bar_sync(2, 128);
            last = *last_flag;
            named_bar_sync(2, 128);
          }
          if (!last) {
            float* part = p.partial + (static_cast<size_t>(2 * blockIdx.x + (seg > 0 ? 1 : 0)) * kRows + r) * NTOK;
#pragma unroll 1
            for (int c0 = 0; c0 < NTOK; c0 += 16) {
              uint32_t tv[16];
              tmem_ld_x16(acc_addr + c0, tv);
              tmem_ld_wait();
              float4* dst = reinterpret_cast<float4*>(part + c0);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                dst[k] = make_float4(__uint_as_float(tv[4 * k]), __uint_as_float(tv[4 * k + 1]),
                                     __uint_as_float(tv[4 * k + 2]), __uint_as_float(tv[4 * k + 3]));
            }
            own_published = true;
            __threadfence();
            named_bar_sync(2, 128);
            if (leader) *last_flag = atomicAdd(p.counters + t, 1u) == static_cast<unsigned>(nparts - 1);
            named_bar_sync(2, 128);
            last = *last_flag;
          }
          if (last) {
            __threadfence();
#pragma unroll 1
            for (int c0 = 0; c0 < NTOK; c0 += 16) {
              uint32_t tv[16];
              if (!own_published) {
                tmem_ld_x16(acc_addr + c0, tv);
                tmem_ld_wait();
              }
              float acc[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) acc[k] = 0.f;
#pragma unroll 1
              for (int pi = 0; pi < nparts; ++pi) {
                if (pi == pme && !own_published) {
#pragma unroll
                  for (int k = 0; k < 16; ++k) acc[k] += __uint_as_float(tv[k]);
                  continue;
                }
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
          named_bar_sync(2, 128);                        // last_flag is reused by the next segment
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[abuf]);
        seg_c = c + 1 == KT ? 0 : c + 1;
        ++seg;
      }
    }
  }

  // ---- teardown: the epilogue waited on the last commit, so every tcgen05
  // op has completed; the producer saw its last copies land.
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

int ntok_for(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

struct Plan {
  int ntok = 0, grid = 0, stages = 0, a_slots = 0, b_ktiles = 0, smem = 0, tiles = 0;
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
  // A slots first (6 or 3: a multiple of the decoder groups), then as many
  // code stages as fit (3..8)
  const int room = kMaxSmem - b_bytes - kBarBytes;
  pl.a_slots = room - 6 * kASlotBytes >= 3 * kStageBytes ? 6 : 3;
  pl.stages = std::min(kMaxStages, (room - pl.a_slots * kASlotBytes) / kStageBytes);
  if (pl.stages < 3) return false;
  pl.smem = std::max(pl.stages * kStageBytes + b_bytes + pl.a_slots * kASlotBytes + kBarBytes, kMinSmem);
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
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(pl.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = pl.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  note_launch();
  return e == cudaSuccess ? CBQ_OK : CBQ_ECUDA;
}

// Activations a[M][K] as a TMA tensor whose box is one k-tile of `ntok`
// token rows: a 2-D view with a (128 B, ntok) box and the 128-byte swizzle;
// rows past M read as zeros.  If the driver refuses it, a 3-D view (16 bytes,
// M rows of stride K, K/16 chunks of stride 16) with a (16, ntok, 8) box that
// lands in the unswizzled core-matrix layout.
int encode_a_map(SkParams& p, int ntok) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return CBQ_ECUDA;
  void* base = const_cast<uint8_t*>(p.a);
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(p.M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.K)};
    const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(ntok)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&p.a_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      p.b_layout = 0;
      return CBQ_OK;
    }
  }
  const cuuint64_t dims[3] = {16, static_cast<cuuint64_t>(p.M), static_cast<cuuint64_t>(p.K / 16)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.K), 16};
  const cuuint32_t box[3] = {16, static_cast<cuuint32_t>(ntok), 8};
  const cuuint32_t estr[3] = {1, 1, 1};
  if (enc(&p.a_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CBQ_ECUDA;
  p.b_layout = 1;
  return CBQ_OK;
}

}  // namespace

bool sk_applicable(int M, int N, int K) {
  Plan pl;
  return plan_for(M, N, K, pl);
}

namespace {

int launch_planned(const SkParams& p_in, const Plan& pl, float* partial, unsigned* counters, cudaStream_t stream) {
  SkParams p = p_in;
  p.partial = partial;
  p.counters = counters;
  p.stages = pl.stages;
  p.a_slots = pl.a_slots;
  p.b_ktiles = pl.b_ktiles;
  const int em = encode_a_map(p, pl.ntok);
  if (em != CBQ_OK) return em;
  if (pl.ntok == 16) return launch_t<16>(p, pl, stream);
  if (pl.ntok == 32) return launch_t<32>(p, pl, stream);
  return launch_t<64>(p, pl, stream);
}

// Static scratch of the allocation-free entry point: partial tiles for up to
// kStaticCtas CTAs at 64 token columns, and counters for kStaticTiles tiles.
// Zero at module load; each kernel returns the counters it used to zero.
constexpr int kStaticCtas = 160;
constexpr int kStaticTiles = 1 << 16;
__device__ __align__(256) float g_static_partial[2 * kStaticCtas * kRows * 64];
__device__ __align__(256) unsigned g_static_counters[kStaticTiles];

}  // namespace

int launch_sk(const SkParams& p_in, cudaStream_t stream) {
  Plan pl;
  if (!plan_for(p_in.M, p_in.N, p_in.K, pl)) return CBQ_EINVAL;
  Scratch sc;
  const int st = scratch_for(stream, size_t(2) * pl.grid * kRows * pl.ntok, size_t(pl.tiles), sc);
  if (st != CBQ_OK) return st;
  return launch_planned(p_in, pl, sc.partial, sc.counters, stream);
}

int launch_sk_static(const SkParams& p_in, cudaStream_t stream) {
  Plan pl;
  if (!plan_for(p_in.M, p_in.N, p_in.K, pl)) return CBQ_EINVAL;
  if (pl.grid > kStaticCtas || pl.tiles > kStaticTiles) return CBQ_EINVAL;
  // the static buffers' addresses on the current device
  static std::mutex mu;
  static void* partial_at[64] = {};
  static void* counters_at[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CBQ_EDEVICE;
  void *partial = nullptr, *counters = nullptr;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!partial_at[dev] || !counters_at[dev]) {
      void *a = nullptr, *b = nullptr;
      if (cudaGetSymbolAddress(&a, g_static_partial) != cudaSuccess ||
          cudaGetSymbolAddress(&b, g_static_counters) != cudaSuccess) {
        cudaGetLastError();
        return CBQ_ECUDA;
      }
      partial_at[dev] = a;
      counters_at[dev] = b;
    }
    partial = partial_at[dev];
    counters = counters_at[dev];
  }
  // the counters of the tiles this call uses start at zero even if an
  // earlier call gave up part-way
  if (cudaMemsetAsync(counters, 0, sizeof(unsigned) * pl.tiles, stream) != cudaSuccess) return CBQ_ECUDA;
  return launch_planned(p_in, pl, static_cast<float*>(partial), static_cast<unsigned*>(counters), stream);
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
