// cbq_umma.cu -- verify-round kernel of the codebook-quantised matmul:
// TMA-staged packed codes, register decode to E4M3 straight into tensor
// memory, block-scaled FP8 MMA on the 5th-generation tensor cores (tcgen05)
// with fp32 accumulators in TMEM.
//
// "Hibana: Fast Agentic Inference on Unified-Memory Devices", section "Model
// surgery / Three-bit weights": each 3-bit code becomes its value in the
// row's 8-entry FP8 codebook on the fly, and the products run on the FP8
// tensor cores; section "Adaptive
// speculation": a verify round multiplies the drafted tokens of all requests
// (up to 64 rows) by the same weights, and with "Expert sharing" reads only
// the experts the round's tokens route to.
//
// Mapping to sm_103a (swap-AB: weight rows are the MMA's M = 128, token rows
// its N = 16, 32 or 64):
//  * warp 0 (one lane) streams the tile's code bytes with 1-D bulk copies of
//    4 k-tiles (24 KB, contiguous in the tile-ordered stream) into a ring of
//    up to 6 stages, starting right after barrier set-up;
//  * warps 2..17 are four decoder groups of 4 warps taking k-tiles round
//    robin; thread = weight row = TMEM lane.  A thread reads its row's 48
//    code bytes (three 128-bit shared loads at a conflict-free 48-byte
//    pitch), spreads the codes to nibbles and turns them into E4M3 bytes with
//    byte-permutes through the row's codebook (two registers), then writes the
//    128 bytes into its TMEM lane (tcgen05.st, 32 columns) as the MMA's A
//    operand, and its 4 E8M0 group-scale bytes into TMEM as the A scale
//    factors.  Each group owns two A slots; while one warp waits for its
//    TMEM stores the other groups' warps decode (deferring that wait past the
//    warp's next decode measured no different); scale bytes are pulled into
//    L1 16 k-tiles ahead and the next tile's codebook is loaded during the
//    current one;
//  * warp 1 (one lane) issues 4 tcgen05.mma kind::mxf8f6f4.block_scale
//    (K = 32 each) per k-tile with A from TMEM and B (the E4M3 activations,
//    resident in shared memory for the CTA's K range: one TMA box of ntok
//    rows x 128 B per k-tile with the 128-byte swizzle, issued by an epilogue
//    thread while the decoders start) from a K-major swizzled shared-memory
//    descriptor; B scale factors are 2^0.  The E8M0 group scale is exactly the
//    MX block scale of a 32-wide K block, so the tensor core applies it;
//  * warps 18..21 are the epilogue: tcgen05.ld the accumulator (two
//    accumulators alternate between tiles so the MMA never waits for the
//    stores), multiply by a_scale, store fp32 y;
//  * narrow problems split K over a thread-block cluster; partial tiles are
//    summed in the leader CTA's shared memory through DSMEM stores;
//  * grouped calls (one MoE verify round): every CTA derives the ascending
//    list of the experts the round routes to from topk_idx, and takes a
//    contiguous block of (expert, tile) units; all tokens stay resident, the
//    MMAs run over every token column, and the epilogue stores the columns of
//    the tokens routed to the unit's expert into their y slots.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include "cbq_device.cuh"
#include "cbq_internal.h"

namespace cbq {

static __device__ unsigned g_status_umma = 0;

namespace {

constexpr int kRows = 128;                    // MMA M (weight rows per tile)
constexpr int kKtPerStage = 4;                // k-tiles per code stage (one bulk copy)
constexpr int kCodeStage = kKtPerStage * kRows * 48;   // 24 KB
constexpr int kMaxCodeStages = 6;
constexpr int kAStages = 8;                   // decoded k-tiles in TMEM
constexpr int kDecGroups = 4;
constexpr int kDecWarps = 4 * kDecGroups;
static_assert(kAStages == 2 * kDecGroups, "each decoder group owns two A slots");
constexpr int kEpiWarp0 = 2 + kDecWarps;      // first epilogue warp
constexpr int kThreads = (kEpiWarp0 + 4) * 32;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 64;                  // accumulator i at column 64 * i
constexpr int kSfaCol = 128;                  // + 4 * A stage (4-column aligned)
constexpr int kSfbCol = 192;                  // 8 columns of 2^0
constexpr int kACol = 256;                    // + 32 * A stage
constexpr int kMaxExperts = 4096;
constexpr int kMaxRouting = 64 * 8;
constexpr int kMaxSmem = 232448;
constexpr int kMinSmem = 120 * 1024;          // > half an SM: one CTA per SM owns all of TMEM

constexpr long long kDrainLimitNs = 10000000000LL;   // copies and MMAs always finish; 10 s is a backstop

__device__ __forceinline__ void raise(unsigned bits) { atomicOr(&g_status_umma, bits); }

// Wait for an mbarrier phase, suspended in the barrier between polls (a
// polling warp takes issue slots from the warps it waits for).  Gives up
// (returns false) at once when the CTA's abort flag is up, or after
// `limit_ns`, raising the flag and the library's timeout status.
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                             long long limit_ns) {
  if (CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_test_wait(bar, parity)) return true;
  const long long t0 = global_ns();
  // suspended polls (20 us hint) for the normal limit; under a limit below
  // that, non-blocking tests (cluster-scope waits: plain polls), so that a
  // wait not already satisfied does give up (try_wait may block until the
  // phase completes)
  const bool poll = limit_ns < 20000;
  for (;;) {
    const bool done = poll ? (CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_test_wait(bar, parity))
                           : (CLUSTER ? mbar_try_wait_cluster_suspend(bar, parity, 20000u)
                                      : mbar_try_wait_suspend(bar, parity, 20000u));
    if (done) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      raise(kErrTimeout);
      return false;
    }
  }
}

// Wait for asynchronous work this CTA issued itself (bulk copies, TMA loads,
// tensor-core work), whatever the abort flag says: it always completes.
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

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// mbarriers (codes full/empty, A full/empty, 2 accumulators full/empty,
// B, split-K full/free, MMA drain), then the TMEM base slot and four ints.
constexpr int kNumBars = 2 * kMaxCodeStages + 2 * kAStages + 4 + 4;
constexpr int kBarBytes = (kNumBars * 8 + 24 + 127) / 128 * 128;
static_assert(kNumBars * 8 + 24 <= kBarBytes, "barrier area too small");

// Shared-memory carve-up (byte offsets), identical on host and device.
struct Layout {
  int codes, b, red, bars, route, total;
  __host__ __device__ Layout(int code_stages, int b_bytes, int red_bytes, bool grouped) {
    codes = 0;
    b = codes + code_stages * kCodeStage;
    red = b + b_bytes;
    bars = red + red_bytes;
    route = bars + kBarBytes;
    total = route + (grouped ? (kMaxRouting * 4 + 64 * 4 + 16 + kMaxExperts * 2 + kMaxExperts) : 0);
  }
};

template <int NTOK, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1) umma_kernel(const __grid_constant__ UmmaParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const Layout L(p.code_stages, p.b_bytes, p.red_bytes, GROUPED);
  const int NS = p.code_stages;
  uint8_t* codes_s = smem + L.codes;
  uint8_t* b_s = smem + L.b;
  float* red_s = reinterpret_cast<float*>(smem + L.red);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
  uint64_t* codes_full = bars;
  uint64_t* codes_empty = codes_full + kMaxCodeStages;
  uint64_t* a_full = codes_empty + kMaxCodeStages;
  uint64_t* a_empty = a_full + kAStages;
  uint64_t* acc_full = a_empty + kAStages;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* b_full = acc_empty + 2;                      // resident activations landed
  uint64_t* red_full = b_full + 1;
  uint64_t* red_free = red_full + 1;
  uint64_t* drain = red_free + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* misc = reinterpret_cast<int*>(tmem_slot + 2);     // [1] experts used (grouped)
  volatile int* abort_flag = misc + 2;
  const long long wait_ns = p.wait_ns;
  int32_t* topk_s = reinterpret_cast<int32_t*>(smem + L.route);
  int32_t* slot_of = topk_s + kMaxRouting;               // grouped: y slot of each token for the current expert, or -1
  uint16_t* used_list = reinterpret_cast<uint16_t*>(slot_of + 64 + 4);
  uint8_t* used_flag = reinterpret_cast<uint8_t*>(used_list + kMaxExperts);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cs = p.ksplit;
  const int rank = cs > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int cluster_id = blockIdx.x / cs, n_clusters = gridDim.x / cs;
  const int nkt = p.K / 128;
  const int kt0 = rank * nkt / cs, kt1 = (rank + 1) * nkt / cs;
  const int tiles = (p.N + kRows - 1) / kRows;
  const int gk = p.K / 32;                                // scale bytes per row
  const int n_stages_u = (kt1 - kt0 + kKtPerStage - 1) / kKtPerStage;   // code stages per unit

  if (warp == 0) {                                        // barriers initialised by the lanes side by side
    for (int i = lane; i < NS; i += 32) {
      mbar_init(&codes_full[i], 1);
      mbar_init(&codes_empty[i], kDecWarps);            // every decoder warp, once per stage
    }
    for (int i = lane; i < kAStages; i += 32) {
      mbar_init(&a_full[i], 4);
      mbar_init(&a_empty[i], 1);
    }
    if (lane < 2) {
      mbar_init(&acc_full[lane], 1);
      mbar_init(&acc_empty[lane], 4);
    }
    if (lane == 2) mbar_init(b_full, 1);
    if (lane == 3) mbar_init(red_full, (cs > 1 ? cs - 1 : 1) * 128);
    if (lane == 4) mbar_init(red_free, 128);
    if (lane == 5) mbar_init(drain, 1);
    if (lane == 0) *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Cluster peers' barriers must exist before any remote arrive; arrive now,
  // wait right before the first DSMEM access (epilogue) or at the end.
  if (cs > 1) cluster_arrive();

  // ---- which units does this CTA own? ----
  int n_units, u_begin, u_step;
  if constexpr (GROUPED) {
    const int nr = p.M * p.topk;                       // <= kThreads (64 x 8)
    const int e_mine = tid < nr ? p.topk_idx[tid] : 0; // load issued before the flags are cleared
    for (int e = tid; e < p.E; e += kThreads) used_flag[e] = 0;
    __syncthreads();
    for (int i = tid; i < nr; i += kThreads) {
      const int e = i == tid ? e_mine : p.topk_idx[i];
      topk_s[i] = e;
      if (e >= 0 && e < p.E) used_flag[e] = 1;
      else raise(kErrRouting);
    }
    __syncthreads();
    for (int i = tid; i < nr; i += kThreads) {
      const int row0 = (i / p.topk) * p.topk;
      for (int j = row0; j < i; ++j)
        if (topk_s[j] == topk_s[i]) raise(kErrRouting);
    }
    if (warp == 0) {
      int base = 0;
      for (int e0 = 0; e0 < p.E; e0 += 32) {
        const int e = e0 + lane;
        const bool u = (e < p.E) && used_flag[e];
        const unsigned m = __ballot_sync(0xffffffffu, u);
        if (u) used_list[base + __popc(m & ((1u << lane) - 1u))] = static_cast<uint16_t>(e);
        base += __popc(m);
      }
      if (lane == 0) misc[1] = base;
    }
    __syncthreads();
    // contiguous blocks of (expert, tile) units so consecutive units share an expert
    // floor(b total / G) = b q + floor(b r / G) with total = q G + r, in
    // 32-bit arithmetic (b r < G^2)
    const uint32_t total = static_cast<uint32_t>(misc[1] * tiles), G = gridDim.x;
    const uint32_t q = total / G, rem = total - q * G, b = blockIdx.x;
    u_begin = static_cast<int>(b * q + (b * rem) / G);
    n_units = static_cast<int>((b + 1) * q + ((b + 1) * rem) / G) - u_begin;
    u_step = 1;
  } else {
    u_begin = cluster_id;
    n_units = cluster_id < tiles ? (tiles - 1 - cluster_id) / n_clusters + 1 : 0;
    u_step = n_clusters;
  }

  // rows of a unit (global row index for scales / codebooks) and where its
  // 128-row tile starts in the tile-ordered code stream
  auto unit_rows = [&](int ui, int& row0, int& row_end, int& e) {
    const int u = u_begin + ui * u_step;
    if constexpr (GROUPED) {
      e = used_list[u / tiles];
      row0 = e * p.N + (u % tiles) * kRows;
      row_end = e * p.N + p.N;
    } else {
      e = 0;
      row0 = u * kRows;
      row_end = p.N;
    }
  };
  auto unit_tile = [&](int ui, int& rows_t) -> const uint8_t* {
    const int u = u_begin + ui * u_step;
    int t = u;
    const uint8_t* mat = p.codes;
    if constexpr (GROUPED) {
      t = u % tiles;
      mat += static_cast<long long>(used_list[u / tiles]) * (3LL * p.K / 8) * p.N;
    }
    rows_t = tile_rows(t, p.N);
    return mat + tile_base(t, p.K);
  };

  uint32_t tbase = 0;
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    // Starts streaming at once; the rest of the CTA sets up TMEM and the
    // resident activations meanwhile.  One bulk copy per stage: up to 4
    // consecutive k-tiles of the tile, contiguous in the code stream.
    if (lane == 0) {
      uint32_t sg = 0;
      bool stop = false;
      const uint64_t pol = l2_evict_first_policy();
      for (int ui = 0; ui < n_units && !stop; ++ui) {
        int rows_t;
        const uint8_t* tile = unit_tile(ui, rows_t);
        for (int st = 0; st < n_stages_u; ++st, ++sg) {
          const int slot = sg % NS;
          const int kb = kt0 + st * kKtPerStage, nk = min(kKtPerStage, kt1 - kb);
          const uint32_t bytes = static_cast<uint32_t>(nk * rows_t * 48);
          if (sg >= static_cast<uint32_t>(NS)) {
            // the slot's previous stage must be released, and its copy
            // landed (always so after a normal release; checked so that no
            // give-up elsewhere can re-arm a barrier with a copy in flight)
            if (!wait_bounded(&codes_empty[slot], ((sg / NS) & 1u) ^ 1u, abort_flag, wait_ns)) {
              stop = true;
              break;
            }
            wait_drain(&codes_full[slot], ((sg / NS) & 1u) ^ 1u);
          }
          mbar_arrive_expect_tx(&codes_full[slot], bytes);
          bulk_g2s(codes_s + slot * kCodeStage, tile + static_cast<long long>(kb) * rows_t * 48, bytes,
                   &codes_full[slot], pol);
        }
      }
      // every copy this CTA issued has landed before it can leave
      for (uint32_t j = sg > static_cast<uint32_t>(NS) ? sg - NS : 0u; j < sg; ++j)
        wait_drain(&codes_full[j % NS], (j / NS) & 1u);
    }
    __syncwarp();
    if (cs > 1) cluster_wait();
  } else {
    if (warp == 1) {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    named_bar_sync(3, kThreads - 32);                     // everyone but the producer
    tc_fence_after();
    tbase = *tmem_slot;
    // scale factors of B: 2^0 in every byte of 8 columns, all 128 lanes
    if (warp >= kEpiWarp0) {
      const uint32_t q = warp & 3;
      for (int c = 0; c < 8; c += 4)
        tmem_st_x4(tbase + ((32 * q) << 16) + kSfbCol + c, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_st_wait();
    }
    tc_fence_before();
    named_bar_sync(3, kThreads - 32);
    tc_fence_after();

    if (warp == 1) {
      if (cs > 1) cluster_wait();
      // --------------------------------------------------------- MMA issuer --
      if (lane == 0) {
        // k-tile i (from kt0) of a unit belongs to decoder group i % kDecGroups,
        // which owns A slots g and g + kDecGroups and uses them alternately:
        // use n of group g -> slot (n & 1) * kDecGroups + g, phase n >> 1,
        // with n = (its uses in earlier units) + i / kDecGroups.  The loop is
        // unrolled over the groups so each group's use count is a register,
        // and descriptors advance by adding offsets: this thread shares its
        // sub-partition with decoder warps, so every instruction here counts.
        const int nk = kt1 - kt0;
        const uint64_t bd0 = umma_desc_kmajor_sw128(smem_u32(b_s));
        const uint32_t idesc = umma_idesc_mxf8(NTOK, 0, 0);
        const uint32_t a_col = tbase + kACol, sfa_col = tbase + kSfaCol, sfb_col = tbase + kSfbCol;
        uint32_t nbase[kDecGroups];
#pragma unroll
        for (int g = 0; g < kDecGroups; ++g) nbase[g] = 0;
        wait_bounded(b_full, 0, abort_flag, wait_ns);   // resident activations landed
        tc_fence_after();
        for (int ui = 0; ui < n_units; ++ui) {
          const int abuf = ui & 1;
          wait_bounded(&acc_empty[abuf], ((ui >> 1) & 1) ^ 1, abort_flag, wait_ns);
          tc_fence_after();
          const uint32_t d_col = tbase + abuf * kAccCols;
          for (int i0 = 0; i0 < nk; i0 += kDecGroups) {
#pragma unroll
            for (int g = 0; g < kDecGroups; ++g) {
              const int i = i0 + g;
              if (i < nk) {
                const uint32_t n = nbase[g] + static_cast<uint32_t>(i0 / kDecGroups);
                const uint32_t slot = (n & 1u) * kDecGroups + g;
                wait_bounded(&a_full[slot], (n >> 1) & 1u, abort_flag, wait_ns);
                tc_fence_after();
                // B of k-tile i: NTOK swizzled rows of 128 bytes at i * NTOK * 128,
                // i.e. i * NTOK * 8 in the descriptor's 16-byte address units;
                // MMA j reads K bytes [32 j, 32 j + 32) of the rows (+2 j)
                const uint64_t bdi = bd0 + static_cast<uint64_t>(i * NTOK * 8);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  umma_mxf8_ts(d_col, a_col + slot * 32 + j * 8, bdi + static_cast<uint64_t>(2 * j),
                               idesc | (uint32_t(j) << 29), sfa_col + slot * 4, sfb_col, (i | j) != 0);
                umma_commit(&a_empty[slot]);
              }
            }
          }
#pragma unroll
          for (int g = 0; g < kDecGroups; ++g) nbase[g] += static_cast<uint32_t>((nk + kDecGroups - 1 - g) / kDecGroups);
          umma_commit(&acc_full[abuf]);
        }
        // all tensor-core work and the activation loads are done before TMEM
        // is freed and the CTA ends
        umma_commit(drain);
        wait_drain(drain, 0);
        wait_drain(b_full, 0);
      }
      __syncwarp();
    } else if (warp < kEpiWarp0) {
      if (cs > 1) cluster_wait();
      // ------------------------------------------------------------ decoders --
      const int dw = warp - 2, dg = dw >> 2, q = warp & 3;
      const int r = 32 * q + lane;                      // row inside the tile == TMEM lane
      const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
      const uint32_t codes_base = smem_u32(codes_s);
      // Stage bookkeeping: a unit's k-tiles come in stages of kKtPerStage;
      // each decoder warp releases every stage of the unit exactly once,
      // after its last read from it.
      uint32_t sg_unit = 0;                             // global index of the unit's first stage
      int released = 0, rows_t = kRows;
      // Every release is preceded by a wait for that stage, so an early
      // release can never count towards an older phase of its slot.
      auto release_until = [&](int s_end) {
        for (; released < s_end; ++released) {
          const uint32_t sg = sg_unit + released;
          wait_bounded(&codes_full[sg % NS], (sg / NS) & 1u, abort_flag, wait_ns);
          __syncwarp();
          if (lane == 0) mbar_arrive(&codes_empty[sg % NS]);
        }
      };
      // Load a k-tile's code row from shared memory and decode it into 32
      // TMEM columns worth of E4M3 bytes.
      auto load_decode = [&](int kt, uint2 cb, uint32_t (&v)[32]) {
        const int s = (kt - kt0) / kKtPerStage, j = (kt - kt0) % kKtPerStage;
        release_until(s);
        const uint32_t sgi = sg_unit + s;
        wait_bounded(&codes_full[sgi % NS], (sgi / NS) & 1u, abort_flag, wait_ns);
        const uint32_t crow = codes_base + (sgi % NS) * kCodeStage + (j * rows_t + r) * 48;
        const uint4 c0 = lds128(crow), c1 = lds128(crow + 16), c2 = lds128(crow + 32);
        decode_group(c0.x, c0.y, c0.z, cb.x, cb.y, v);
        decode_group(c0.w, c1.x, c1.y, cb.x, cb.y, v + 8);
        decode_group(c1.z, c1.w, c2.x, cb.x, cb.y, v + 16);
        decode_group(c2.y, c2.z, c2.w, cb.x, cb.y, v + 24);
      };
      // Issue the TMEM stores of a decoded k-tile (A operand and its scale
      // factors); publish() waits for them and hands the slot to the MMA.
      // This group's A slots are dg and dg + kDecGroups, used alternately in
      // the group's own k-tile order (so a slot's parity wait cannot be two
      // uses early): use n -> slot (n & 1) * kDecGroups + dg, phase n >> 1.
      uint32_t uses = 0;
      auto store = [&](uint32_t n, uint32_t sw, const uint32_t (&v)[32]) {
        const int aslot = static_cast<int>(n & 1u) * kDecGroups + dg;
        wait_bounded(&a_empty[aslot], ((n >> 1) & 1u) ^ 1u, abort_flag, wait_ns);
        tc_fence_after();
        tmem_st_x32(tbase + lane_addr + kACol + aslot * 32, v);
        // A scale of row m is read from TMEM lane m, column (base + m / 32),
        // byte = the MMA's a_sf_id: quadrant q writes column base + q
        tmem_st_x1(tbase + lane_addr + kSfaCol + aslot * 4 + q, sw);
      };
      auto publish = [&](uint32_t n) {
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[static_cast<int>(n & 1u) * kDecGroups + dg]);
      };
      int row0n, row_endn, en;
      if (n_units > 0) unit_rows(0, row0n, row_endn, en);
      uint2 cb_next = (n_units > 0 && row0n + r < row_endn)
                          ? __ldg(reinterpret_cast<const uint2*>(p.codebooks + size_t(row0n + r) * 8))
                          : make_uint2(0, 0);
      for (int ui = 0; ui < n_units; ++ui) {
        int row0, row_end, e;
        unit_rows(ui, row0, row_end, e);
        unit_tile(ui, rows_t);
        sg_unit = static_cast<uint32_t>(ui) * n_stages_u;
        released = 0;
        const bool ok = row0 + r < row_end;
        const uint2 cb = cb_next;
        if (ui + 1 < n_units) {                         // next unit's codebook, in flight meanwhile
          unit_rows(ui + 1, row0n, row_endn, en);
          cb_next = row0n + r < row_endn
                        ? __ldg(reinterpret_cast<const uint2*>(p.codebooks + size_t(row0n + r) * 8))
                        : make_uint2(0, 0);
        }
        const uint32_t* srow = reinterpret_cast<const uint32_t*>(p.scales + size_t(ok ? row0 + r : 0) * gk);
        // warm L1 with this row's scale bytes: 8 k-tiles per 32-byte sector
        if (ok)
          for (int kt = kt0; kt < kt1 && kt < kt0 + 16; kt += 8) prefetch_l1(srow + kt);
        // this group's k-tiles are kt0 + dg, kt0 + dg + G, ...; the other
        // groups' warps fill the issue slots while this one waits on TMEM
        for (int kt = kt0 + dg; kt < kt1; kt += kDecGroups) {
          const uint32_t it = uses++;
          if (ok && kt + 16 < kt1 && ((kt + 16) & 7) < kDecGroups) prefetch_l1(srow + kt + 16);
          const uint32_t sw = ok ? __ldg(srow + kt) : 0x7F7F7F7Fu;
          uint32_t v[32];
          load_decode(kt, cb, v);
          store(it, sw, v);
          publish(it);
        }
        release_until(n_stages_u);
      }
    } else {
      // ------------------------------------------------------------ epilogue --
      if (tid == kEpiWarp0 * 32) {
        // Resident activations for this CTA's K range, issued by one thread
        // of the epilogue (nothing else to do before the first accumulator;
        // the decoders start at once): one TMA box per k-tile, NTOK token
        // rows of 128 bytes in the 128-byte swizzled K-major layout at
        // (kt - kt0) * NTOK * 128; token rows >= M are outside the tensor and
        // arrive as zeros.  A grouped call keeps every token resident: the
        // MMAs run over all token columns and the epilogue keeps the columns
        // of the tokens routed to the unit's expert.
        mbar_arrive_expect_tx(b_full, static_cast<uint32_t>((kt1 - kt0) * NTOK * 128));
        for (int c = kt0; c < kt1; ++c) tma_load_2d(b_s + (c - kt0) * NTOK * 128, &p.a_map, b_full, c * 128, 0);
      }
      if (cs > 1) cluster_wait();
      const int q = warp & 3;
      const int r = 32 * q + lane;
      const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
      int prev_e = -1;
      for (int ui = 0; ui < n_units; ++ui) {
        int row0, row_end, e;
        unit_rows(ui, row0, row_end, e);
        if constexpr (GROUPED) {
          if (e != prev_e) {
            // y slot of every token routed to expert e (a token lists an
            // expert at most once; the routing check above raised otherwise)
            named_bar_sync(2, 128);
            for (int t = tid - kEpiWarp0 * 32; t < 64; t += 128) slot_of[t] = -1;
            named_bar_sync(2, 128);
            const int nr = p.M * p.topk;
            for (int i = tid - kEpiWarp0 * 32; i < nr; i += 128)
              if (topk_s[i] == e) slot_of[i / p.topk] = i % p.topk;
            named_bar_sync(2, 128);
            prev_e = e;
          }
        }

        const int grow = row0 + r;
        const bool ok = grow < row_end;
        const int abuf = ui & 1;
        wait_bounded(&acc_full[abuf], (ui >> 1) & 1, abort_flag, wait_ns);
        tc_fence_after();
        const bool split = !GROUPED && cs > 1;
        if (split && rank != 0) wait_bounded<true>(red_free, (ui & 1) ^ 1, abort_flag, wait_ns);
        if (split && rank == 0) wait_bounded<true>(red_full, ui & 1, abort_flag, wait_ns);
        // 16 accumulator columns (token rows) at a time: load, reduce, store
#pragma unroll 1
        for (int c0 = 0; c0 < NTOK; c0 += 16) {
          uint32_t t[16];
          tmem_ld_x16(tbase + lane_addr + abuf * kAccCols + c0, t);
          tmem_ld_wait();
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(t[i]);
          if (split) {
            if (rank != 0) {
              // split K: partial tiles meet in the leader CTA's shared memory
              const uint32_t dst = mapa_shared(
                  smem_u32(red_s) + ((rank - 1) * kRows * NTOK + r * NTOK + c0) * 4, 0);
#pragma unroll
              for (int i = 0; i < 16; i += 4) st_cluster_v4(dst + i * 4, v[i], v[i + 1], v[i + 2], v[i + 3]);
              continue;
            }
            for (int sidx = 0; sidx < cs - 1; ++sidx) {
              const float4* src = reinterpret_cast<const float4*>(red_s + sidx * kRows * NTOK + r * NTOK + c0);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float4 f = src[i];
                v[4 * i] += f.x;
                v[4 * i + 1] += f.y;
                v[4 * i + 2] += f.z;
                v[4 * i + 3] += f.w;
              }
            }
          }
          if (ok) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int c = c0 + i;
              if (c < p.M) {
                if constexpr (GROUPED) {
                  const int slot = slot_of[c];
                  if (slot >= 0) p.y[(size_t(c) * p.topk + slot) * p.N + (grow - e * p.N)] = v[i] * __ldg(p.a_scale + c);
                } else {
                  p.y[size_t(c) * p.N + grow] = v[i] * __ldg(p.a_scale + c);
                }
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[abuf]);
        if (split) {
          if (rank != 0) {
            mbar_arrive_remote(mapa_shared(smem_u32(red_full), 0));
          } else {
            // tell every other CTA of the cluster that its slot may be reused
            for (int sidx = 1; sidx < cs; ++sidx) mbar_arrive_remote(mapa_shared(smem_u32(red_free), sidx));
          }
        }
      }
    }
  }

  // ---- teardown: every tcgen05 op has completed (the epilogue waited on
  // the last commit); cluster peers may still touch our barriers until all
  // of them get here.
  tc_fence_before();
  __syncthreads();
  if (cs > 1) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

// The kernel's attributes (largest dynamic shared memory, non-portable
// cluster sizes), set once per device and template instance.
template <int NTOK, bool GROUPED>
cudaError_t configure(int smem, int cs) {
  (void)smem;
  (void)cs;
  static std::atomic<int> done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return e != cudaSuccess ? e : cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  auto kern = umma_kernel<NTOK, GROUPED>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
  return e;
}

template <int NTOK, bool GROUPED>
int max_clusters_t(int cs, int smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, int, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_tuple(dev, cs, smem);
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int n = 0;
  if (configure<NTOK, GROUPED>(smem, cs) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cs * 64);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, umma_kernel<NTOK, GROUPED>, &cfg) != cudaSuccess) n = 0;
  }
  cudaGetLastError();
  cache[key] = n;
  return n;
}

int max_clusters(int ntok, int cs, int smem) {
  if (ntok <= 16) return max_clusters_t<16, false>(cs, smem);
  if (ntok <= 32) return max_clusters_t<32, false>(cs, smem);
  return max_clusters_t<64, false>(cs, smem);
}

template <int NTOK, bool GROUPED>
int launch_t(const UmmaParams& p, int grid, int cs, int smem, cudaStream_t stream) {
  auto kern = umma_kernel<NTOK, GROUPED>;
  if (configure<NTOK, GROUPED>(smem, cs) != cudaSuccess) return CBQ_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (cs > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  note_launch();
  return e == cudaSuccess ? CBQ_OK : CBQ_ECUDA;
}

template <bool GROUPED>
int dispatch(const UmmaParams& p, int ntok, int grid, int cs, int smem, cudaStream_t s) {
  if (ntok <= 16) return launch_t<16, GROUPED>(p, grid, cs, smem, s);
  if (ntok <= 32) return launch_t<32, GROUPED>(p, grid, cs, smem, s);
  return launch_t<64, GROUPED>(p, grid, cs, smem, s);
}

// Deepest code-stage ring that fits next to the other shared-memory areas.
int code_stages_for(int b_bytes, int red_bytes, bool grouped) {
  for (int st = kMaxCodeStages; st >= 2; --st)
    if (Layout(st, b_bytes, red_bytes, grouped).total <= kMaxSmem) return st;
  return 0;
}

// Token columns of the MMA (its N): 16, 32 or 64.
int ntok_for(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

// Activations a[M][K] as a TMA tensor whose box is one k-tile (128 bytes) of
// ntok token rows, landed with the 128-byte swizzle; rows past M read as zeros.
int encode_a_map(UmmaParams& p, int ntok) { return encode_activation_map(&p.a_map, p.a, p.M, p.K, ntok); }

}  // namespace

int launch_umma(const UmmaParams& p_in, bool grouped, cudaStream_t stream) {
  UmmaParams p = p_in;
  const int sms = device_sm_count();
  const int ntok = ntok_for(p.M);
  if (const int em = encode_a_map(p, ntok); em != CBQ_OK) return em;
  const int nkt = p.K / 128;
  const int tiles = (p.N + kRows - 1) / kRows;
  if (grouped) {
    p.ksplit = 1;
    p.b_bytes = ntok * p.K;
    p.red_bytes = 0;
    p.code_stages = code_stages_for(p.b_bytes, 0, true);
    if (p.code_stages < 2) return CBQ_EINVAL;    // K too long for a resident B tile
    const Layout L(p.code_stages, p.b_bytes, 0, true);
    const int units = std::min(p.E, p.M * p.topk) * tiles;
    const int grid = std::max(1, std::min(units, sms));
    return dispatch<true>(p, ntok, grid, 1, std::max(L.total, kMinSmem), stream);
  }
  // Split K over a cluster when there are too few tiles to fill the GPU:
  // minimise (rounds of tiles over the resident clusters) x (k-tiles per CTA).
  int best_cs = 0, best_clusters = 0;
  long long best_cost = 0;
  for (int cs = 1; cs <= 8 && cs <= nkt; ++cs) {
    const int per = (nkt + cs - 1) / cs;
    const int b_bytes = ntok * per * 128, red_bytes = cs > 1 ? (cs - 1) * kRows * ntok * 4 : 0;
    const int stages = code_stages_for(b_bytes, red_bytes, false);
    if (stages < 2) continue;
    const Layout L(stages, b_bytes, red_bytes, false);
    const int smem = std::max(L.total, kMinSmem);
    const int clusters = cs == 1 ? sms : max_clusters(ntok, cs, smem);
    if (clusters <= 0) continue;
    const long long rounds = (tiles + clusters - 1) / clusters;
    const long long cost = rounds * per * 16 + (cs > 1 ? 8 : 0);
    if (best_cs == 0 || cost < best_cost) {
      best_cs = cs;
      best_cost = cost;
      best_clusters = clusters;
    }
  }
  if (best_cs == 0) return CBQ_EINVAL;
  const int cs = best_cs;
  p.ksplit = cs;
  p.b_bytes = ntok * ((nkt + cs - 1) / cs) * 128;
  p.red_bytes = cs > 1 ? (cs - 1) * kRows * ntok * 4 : 0;
  p.code_stages = code_stages_for(p.b_bytes, p.red_bytes, false);
  const Layout L(p.code_stages, p.b_bytes, p.red_bytes, false);
  const int grid = std::min(tiles, best_clusters) * cs;
  return dispatch<false>(p, ntok, grid, cs, std::max(L.total, kMinSmem), stream);
}

unsigned take_status_umma(cudaStream_t stream) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_status_umma, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return kErrTimeout;
  cudaMemcpyToSymbolAsync(g_status_umma, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  cudaStreamSynchronize(stream);
  return v;
}

}  // namespace cbq
