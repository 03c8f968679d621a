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
// them arrives last on the tile's counter in the caller's workspace: each
// writes its fp32 partial tile there, the last one sums the parts in part
// order (deterministic) and writes y.
//
// Roles (one CTA per SM, 20 warps; a warp's sub-partition is warp % 4, and
// a warp reaches only TMEM lane quarter warp % 4):
//  * warp 0: 1-D bulk copies of 4 consecutive units (24 KB, one contiguous
//    piece of the stream) into a ring of shared-memory stages;
//  * warps 4..15: decoders in 3 groups of 4, warp 4 + 4 g + q decoding rows
//    32 q .. 32 q + 31 of group g's units (i = g mod 3): a thread (one row)
//    loads its 48 code bytes, spreads the codes to nibbles, turns them into
//    E4M3 bytes with byte permutes through the row's codebook (two
//    registers) and stores the 128 bytes straight into one of the group's A
//    slots in TMEM (tcgen05.st, 32 columns of its lane), its 4 E8M0 group
//    scales into the slot's scale-factor columns;
//  * warps 1..3, one per group: the group's MMAs -- per unit 4 tcgen05.mma
//    kind::mxf8f6f4.block_scale (K = 32) with A and its scale factors from
//    TMEM and B (the activations, resident for the CTA's k-tiles) from
//    shared memory, into the group's own accumulator; the E8M0 group scale is
//    exactly the MX block scale of its 32-wide K block.  A thread issues MMAs
//    at about half the tensor core's rate when its sub-partition also runs
//    decode arithmetic (measured: 48 -> ~100 cycles per K = 32 MMA), so the
//    three groups issue side by side;
//  * warps 16..19: epilogue -- the leader loads the activations by TMA once
//    the grid dependency resolves; tcgen05.ld the groups' accumulators (two
//    per group alternate between tile segments) and sum them in group order,
//    then either y = a_scale * acc or the partial-tile protocol above.
//
// Fused gate-up epilogue (GATE_UP): the weight's 128-row tile t holds, for the
// R/2 features 64 t .., their gate rows followed by their up rows (R = the
// tile's rows).  The CTA that finishes a tile pairs gate row r with up row
// r + R/2 through shared memory, writes h = SiLU(a_scale g) * (a_scale u) to
// the workspace as fp32 and raises the token's running max |h| with an atomic
// max.  Up to kFusedQuant products, the CTA that finishes last (a
// release-acquire count of finished CTAs in the workspace) then turns every
// product into E4M3 with its token's scale max/448, with all its threads, and
// returns the maxima and the count to zero; beyond that (one SM would read
// too many products) the last CTA writes the scales and returns the maxima
// and the count to zero, and gate_up_quant_kernel quantises the products in
// chunks of 2048 (a CTA per chunk and token).
//
// Bounded waits: every mbarrier wait gives up after the call's wait limit and
// raises the CTA's abort flag; later waits of the CTA then give up at once.
// Giving up never leaves asynchronous work behind: the producer re-arms a
// stage only after the copy it held has landed and, before the CTA ends,
// waits for every copy it issued; each MMA thread waits for all its
// tensor-core work before TMEM is freed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda_fp8.h>

#include "cbq_device.cuh"
#include "cbq_internal.h"

namespace cbq {

static __device__ unsigned g_status_sk = 0;

namespace {

constexpr int kRows = 128;                            // MMA M: weight rows per tile
constexpr int kUnitBytes = kRows * 48;                // codes of one full unit
constexpr int kUnitsPerStage = 4;
constexpr int kStageBytes = kUnitsPerStage * kUnitBytes;   // 24 KB
constexpr int kMaxStages = 8;
constexpr int kGroups = 3;                            // decoder groups: unit i -> group i % 3
// the decoders step a group's stage position by kGroups units with one wrap,
// and start it at its group number without one
static_assert(kUnitsPerStage >= kGroups, "a group's next unit lies in this stage or the next");
constexpr int kMaxSlots = 2;                          // decoded units in TMEM per group (at most)
constexpr int kProdWarp = 0;                          // code stream
constexpr int kAllocWarp = 1;                         // TMEM allocation (also group 0's MMA warp)
constexpr int kMmaWarp0 = 1;                          // warps 1..3: group g's MMAs
constexpr int kDecWarp0 = 4;                          // warps 4..15: group (w - 4) / 4, quarter w % 4
constexpr int kEpiWarp0 = 16;                         // warps 16..19: quarter w % 4 (warp 16 also loads B)
constexpr int kNumWarps = 20;
constexpr int kThreads = kNumWarps * 32;
constexpr int kTmemCols = 512;
constexpr int kSfbCol = 504;                          // 8 columns of B scale factors (2^0)
static_assert(kDecWarp0 % 4 == 0 && kEpiWarp0 % 4 == 0, "a warp's TMEM lane quarter is warp % 4");
constexpr int kMaxSmem = 232448;
constexpr int kMinSmem = 120 * 1024;                  // one CTA per SM: it owns all of TMEM
// k-tiles of resident activations, each with its own barrier (a CTA's share
// of at most this many k-tiles of one row, or all K / 128 of them)
constexpr int kMaxBSlots = 128;
// barriers: code stages full/empty, A slots full/empty, per (group, buffer)
// accumulator full/empty, per group MMA drain, per B slot full
constexpr int kNumBars = 2 * kMaxStages + 2 * kGroups * kMaxSlots + 2 * kGroups * 2 + kGroups + kMaxBSlots;
constexpr int kXchgStride = 17;                       // floats per exchanged row (conflict-free)
constexpr int kXchgBytes = (64 * kXchgStride * 4 + 127) / 128 * 128;
constexpr int kBarBytes = (kNumBars * 8 + 16 + 127) / 128 * 128;
constexpr long long kDrainLimitNs = 10000000000LL;    // copies and MMAs always finish; 10 s is a backstop

// Tensor-memory columns: accumulator (group g, buffer b) at (2 g + b) *
// kStride (two per group alternate between tile segments), then the groups'
// A slots (kSlots each, 32 columns: 128 E4M3 bytes of a row per lane), then
// each slot's 4 scale-factor columns, B's scale factors at kSfbCol.
template <int NTOK>
struct TmemMap {
  static constexpr int kStride = NTOK < 32 ? 32 : NTOK;
  static constexpr int kSlots = NTOK > 32 ? 1 : 2;
  static constexpr int kACol = 2 * kGroups * kStride;
  static constexpr int kSfaCol = kACol + 32 * kGroups * kSlots;
  static_assert(kSlots <= kMaxSlots, "A slots");
  static_assert(kSfaCol + 4 * kGroups * kSlots <= kSfbCol, "A scale factors overlap B's");
  static __device__ __forceinline__ uint32_t acc(int g, int b) { return (2 * g + b) * kStride; }
};

__device__ __forceinline__ void raise(unsigned bits) { atomicOr(&g_status_sk, bits); }

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

// Wait for asynchronous work this CTA issued itself (a bulk copy, a TMA load,
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
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Unit geometry of an N x K weight in the tile-ordered code stream.  Unit
// u = T * KT + c is k-tile c of tile T; positions inside the loops advance
// incrementally (no division per unit).  Grouped calls number the tiles of
// the experts the routing uses one after the other (T = i * tiles + t: tile
// t of the i-th used expert, used[i]); a dense call is one expert.
//
// Division by the tile count is by multiplication (Granlund and Montgomery,
// "Division by invariant integers using multiplication", 1994): with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1, n / d equals
// (mulhi(n, m) + n) >> l for every n < 2^31.
struct FastDiv {
  uint32_t d, m, l;
  __device__ __forceinline__ void init(uint32_t dd) {
    d = dd;
    l = 0;
    while ((1ull << l) < dd) ++l;
    m = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - dd)) / dd + 1);
  }
  __device__ __forceinline__ int div(int n) const {
    return static_cast<int>((__umulhi(static_cast<uint32_t>(n), m) + static_cast<uint32_t>(n)) >> l);
  }
};

template <bool GROUPED, int BITS>
struct GeoT {
  static constexpr int RB = BITS * 16;                // code bytes of one row of a unit (128 codes)
  int N, K, KT;                       // KT = k-tiles per row
  int tiles;                          // 128-row tiles per expert
  long long U, G;                     // units (< 2^31), CTAs
  uint32_t uq, ur;                    // U = uq G + ur
  const uint16_t* used;               // grouped: the used experts, ascending
  long long eb;                       // grouped: code bytes per expert, 3 K N / 8
  FastDiv by_tiles;                   // grouped: division by tiles
  __device__ __forceinline__ int local_tile(int T) const { return GROUPED ? T - by_tiles.div(T) * tiles : T; }
  __device__ __forceinline__ int expert(int T) const { return GROUPED ? used[by_tiles.div(T)] : 0; }
  __device__ __forceinline__ int rows(int T) const { return min(kRows, N - kRows * local_tile(T)); }
  // weight row (of the stacked experts) of row r of tile T
  __device__ __forceinline__ long long row_of(int T, int r) const {
    return GROUPED ? static_cast<long long>(expert(T)) * N + kRows * local_tile(T) + r
                   : static_cast<long long>(kRows) * T + r;
  }
  // byte offset of unit (T, c) in the code stream: the expert's codes, tile
  // t at 48 K t, k-tile block c at c * rows * 48
  __device__ __forceinline__ long long off(int T, int c) const {
    const long long base = GROUPED ? expert(T) * eb : 0;
    return base + static_cast<long long>(RB) * K * local_tile(T) + static_cast<long long>(c) * rows(T) * RB;
  }
  __device__ __forceinline__ void advance(int& t, int& c, int n) const {
    c += n;
    while (c >= KT) {
      c -= KT;
      ++t;
    }
  }
  // floor(b U / G) = b uq + floor(b ur / G), in 32-bit arithmetic (b ur < G^2)
  __device__ __forceinline__ long long first_unit(long long b) const {
    const uint32_t b32 = static_cast<uint32_t>(b);
    return static_cast<long long>(b32 * uq + (b32 * ur) / static_cast<uint32_t>(G));
  }
  // the CTA whose share holds unit u
  __device__ __forceinline__ long long owner(long long u) const { return ((u + 1) * G + U - 1) / U - 1; }
};

// Routing of a grouped call in shared memory: used-expert bit mask, the used
// experts (ascending), a copy of topk_idx, their count.
constexpr int kMaxRouted = 512;                       // M x topk <= 64 x 8
constexpr int kRouteBytes = 128 * 4 + kMaxRouted * 2 + kMaxRouted * 4 + 128;

template <int NTOK, bool GATE_UP, bool GROUPED, int BITS>
__global__ void __launch_bounds__(kThreads, 1) sk_kernel(const __grid_constant__ SkParams p) {
  static_assert(!(GATE_UP && GROUPED), "one epilogue");
  static_assert(BITS == 3 || (BITS == 2 && !GATE_UP && !GROUPED), "two-bit codes: dense calls only");
  constexpr int RB = BITS * 16;                         // code bytes of one row of a unit
  using TM = TmemMap<NTOK>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int NS = p.stages;                             // code stages
  uint8_t* codes_s = smem;
  uint8_t* b_s = smem + NS * kStageBytes;
  float* xchg = reinterpret_cast<float*>(b_s + p.b_ktiles * NTOK * 128);   // GATE_UP: up rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xchg) + (GATE_UP ? kXchgBytes : 0));
  uint64_t* full = bars;
  uint64_t* empty = full + kMaxStages;
  uint64_t* a_full = empty + kMaxStages;               // [group][slot]
  uint64_t* a_empty = a_full + kGroups * kMaxSlots;    // [group][slot]
  uint64_t* acc_full = a_empty + kGroups * kMaxSlots;  // [group][2]
  uint64_t* acc_empty = acc_full + 2 * kGroups;        // [group][2]
  uint64_t* drain = acc_empty + 2 * kGroups;           // [group]
  uint64_t* b_full = drain + kGroups;                  // [B slot]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(b_full + kMaxBSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;
  uint8_t* route_s = reinterpret_cast<uint8_t*>(bars) + kBarBytes;   // GROUPED: routing
  uint32_t* umask = reinterpret_cast<uint32_t*>(route_s);
  uint16_t* used_s = reinterpret_cast<uint16_t*>(umask + 128);
  int32_t* topk_s = reinterpret_cast<int32_t*>(used_s + kMaxRouted);
  volatile int* n_used_s = reinterpret_cast<volatile int*>(topk_s + kMaxRouted);
  const long long wait_ns = p.wait_ns;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // The CTA's share of the units.  A dense call knows it before anything
  // else, so the producer issues its first copy while the block sets up; a
  // grouped call knows it after the routing scan.
  GeoT<GROUPED, BITS> geo;
  struct Share {
    long long u0;
    int n_units, n_stages, t_first, c_first;
  };
  auto make_share = [&](int n_used_) {
    geo.N = p.N;
    geo.K = p.K;
    geo.KT = p.K / 128;
    geo.tiles = (p.N + kRows - 1) / kRows;
    if constexpr (GROUPED) geo.by_tiles.init(static_cast<uint32_t>(geo.tiles));
    geo.U = static_cast<long long>(n_used_) * geo.tiles * geo.KT;
    // shares over at most U CTAs, so that every sharing CTA has a unit (a
    // grouped call is planned for the most experts its routing can name;
    // with fewer, the CTAs from G on have no share)
    geo.G = geo.U < static_cast<long long>(gridDim.x) ? (geo.U > 0 ? geo.U : 1) : static_cast<long long>(gridDim.x);
    geo.uq = static_cast<uint32_t>(geo.U) / static_cast<uint32_t>(geo.G);
    geo.ur = static_cast<uint32_t>(geo.U) - geo.uq * static_cast<uint32_t>(geo.G);
    geo.used = used_s;
    geo.eb = static_cast<long long>(BITS) * p.K * p.N / 8;
    const long long b0 = blockIdx.x, b1 = blockIdx.x + 1LL;
    Share r;
    r.u0 = geo.first_unit(b0 < geo.G ? b0 : geo.G);
    r.n_units = static_cast<int>(geo.first_unit(b1 < geo.G ? b1 : geo.G) - r.u0);
    if constexpr (GROUPED) {
      // whole tiles per CTA (no partial-tile fix-up) when the used experts'
      // T tiles spread over the G CTAs with at most 10 % over the mean and a
      // CTA's activation slots hold every k-tile of a row (MoE round: 288
      // tiles on 152 CTAs, 31.9 -> 27.5 us)
      const long long T = geo.U / geo.KT, G = geo.G;
      if (geo.KT <= p.b_ktiles && T >= G && ((T + G - 1) / G) * G * 10 <= 11 * T) {
        const long long tb0 = (b0 < G ? b0 : G) * T / G, tb1 = (b1 < G ? b1 : G) * T / G;
        r.u0 = tb0 * geo.KT;
        r.n_units = static_cast<int>((tb1 - tb0) * geo.KT);
      }
    }
    r.n_stages = (r.n_units + kUnitsPerStage - 1) / kUnitsPerStage;
    r.t_first = static_cast<int>(static_cast<uint32_t>(r.u0) / static_cast<uint32_t>(geo.KT));
    r.c_first = static_cast<int>(r.u0) - r.t_first * geo.KT;
    return r;
  };
  Share sh{0, 0, 0, 0, 0};
  if constexpr (!GROUPED) sh = make_share(1);
  // Dense: stage j's copy, one contiguous piece of the stream (units from
  // (ts, cs) on, nu of them) into code slot `slot`.
  auto issue_dense_stage = [&](int ts, int cs, int nu, int slot, uint64_t pol) {
    int tl = ts, cl = cs;
    geo.advance(tl, cl, nu - 1);                       // last unit of the stage
    const long long oa = geo.off(ts, cs);
    const uint32_t bytes = static_cast<uint32_t>(geo.off(tl, cl) + geo.rows(tl) * static_cast<long long>(RB) - oa);
    mbar_arrive_expect_tx(&full[slot], bytes);
    bulk_g2s(codes_s + slot * kStageBytes, p.codes + oa, bytes, &full[slot], pol);
  };

  if (warp == 0) {                                     // barriers initialised by the lanes side by side
    for (int i = lane; i < NS; i += 32) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4 * kUnitsPerStage);       // four row blocks of each unit of a full stage
    }
    for (int sl = lane; sl < kGroups * kMaxSlots; sl += 32) {
      mbar_init(&a_full[sl], 4);                      // the group's four decoder warps
      mbar_init(&a_empty[sl], 1);                     // the group's MMAs read the slot
    }
    if (lane < kGroups) {
      const int g = lane;
      mbar_init(&acc_full[2 * g], 1);
      mbar_init(&acc_full[2 * g + 1], 1);
      mbar_init(&acc_empty[2 * g], 4);                // the four epilogue warps
      mbar_init(&acc_empty[2 * g + 1], 4);
      mbar_init(&drain[g], 1);
    }
    if (lane == 0) *abort_flag = 0;
    fence_barrier_init();
    if constexpr (!GROUPED) {
      // this lane initialised full[0]: stage 0's copy goes out now
      if (lane == 0 && sh.n_stages > 0)
        issue_dense_stage(sh.t_first, sh.c_first, min(kUnitsPerStage, sh.n_units), 0, l2_evict_first_policy());
    }
  } else if (warp == 1) {                              // the B slots' barriers, one per lane
    for (int sl = lane; sl < p.b_ktiles; sl += 32) mbar_init(&b_full[sl], 1);
    fence_barrier_init();
  }
  __syncthreads();

  // ---- grouped: the experts the routing uses (every CTA reads the routing)
  int n_used = 1;
  if constexpr (GROUPED) {
    const int nw = (p.E + 31) >> 5, nr = p.M * p.topk;
    for (int w = tid; w < nw; w += kThreads) umask[w] = 0;
    grid_dependency_wait();                            // the routing, written by an earlier kernel
    __syncthreads();
    for (int i = tid; i < nr; i += kThreads) {
      const int e = p.topk_idx[i];
      topk_s[i] = e;
      if (e >= 0 && e < p.E) atomicOr(&umask[e >> 5], 1u << (e & 31));
      else raise(kErrRouting);                         // its outputs are not written
    }
    __syncthreads();
    for (int i = tid; i < nr; i += kThreads) {         // each token lists distinct experts
      const int row0 = (i / p.topk) * p.topk;
      for (int j = row0; j < i; ++j)
        if (topk_s[j] == topk_s[i]) raise(kErrRouting);
    }
    if (warp == 0) {                                   // ascending list of the set bits
      int base = 0;
      for (int w0 = 0; w0 < nw; w0 += 32) {
        const int w = w0 + lane;
        const uint32_t bits = w < nw ? umask[w] : 0u;
        const int cnt = __popc(bits);
        int incl = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        int at = base + incl - cnt;
        for (uint32_t b = bits; b; b &= b - 1) used_s[at++] = static_cast<uint16_t>(32 * w + __ffs(b) - 1);
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) *n_used_s = base;
    }
    __syncthreads();
    n_used = *n_used_s;
  }

  if constexpr (GROUPED) sh = make_share(n_used);
  const int KT = geo.KT;
  const int n_units = sh.n_units, n_stages = sh.n_stages, t_first = sh.t_first, c_first = sh.c_first;
  // The next kernel on the stream may start its prologue (and, if it is this
  // one, its weight stream) as soon as SMs free up; whatever this grid reads
  // from or writes for earlier kernels waits on grid_dependency_wait below.
  grid_launch_dependents();

  uint32_t tbase = 0;
  if (warp == kProdWarp) {
    // -------------------------------------------------------- bulk producer --
    if (lane == 0) {
      int ta = t_first, ca = c_first;                 // first unit of stage j
      int slot = 0;
      uint32_t ph = 0;
      int issued = 0;
      const uint64_t pol = l2_evict_first_policy();
      int j0 = 0;
      if constexpr (!GROUPED) {
        if (n_stages > 0) {                            // stage 0 went out during setup
          geo.advance(ta, ca, kUnitsPerStage);
          slot = 1;                                    // NS >= 2
          issued = 1;
          j0 = 1;
        }
      }
      for (int j = j0; j < n_stages; ++j) {
        const int nu = min(kUnitsPerStage, n_units - j * kUnitsPerStage);
        const int ts = ta, cs = ca;                     // first unit of the stage
        geo.advance(ta, ca, kUnitsPerStage);
        if (j >= NS) {
          // the slot's previous stage must be decoded, and its copy landed
          // (always so after a normal release; checked so that no give-up
          // elsewhere can make a copy re-arm a barrier still in flight)
          if (!wait_bounded(&empty[slot], ph ^ 1u, abort_flag, wait_ns)) break;
          wait_drain(&full[slot], ph ^ 1u);
        }
        if constexpr (!GROUPED) {
          issue_dense_stage(ts, cs, nu, slot, pol);
        } else {
          // the stage's units in runs of one expert each (each run contiguous
          // in the stacked codes), back to back in the stage
          uint32_t total = 0;
          {
            int tr = ts, cr = cs;
            for (int k = 0; k < nu; ++k, geo.advance(tr, cr, 1)) total += geo.rows(tr) * RB;
          }
          mbar_arrive_expect_tx(&full[slot], total);
          int tr = ts, cr = cs, left = nu;
          uint32_t dst = 0;
          while (left > 0) {
            const int run_e = geo.by_tiles.div(tr);
            const long long src = geo.off(tr, cr);
            uint32_t run = 0;
            while (left > 0 && geo.by_tiles.div(tr) == run_e) {
              run += geo.rows(tr) * RB;
              geo.advance(tr, cr, 1);
              --left;
            }
            bulk_g2s(codes_s + slot * kStageBytes + dst, p.codes + src, run, &full[slot], pol);
            dst += run;
          }
        }
        ++issued;
        // stage 0 lands before the later stages' copies compete with it
        if (j == 1) wait_bounded(&full[0], 0, abort_flag, wait_ns);
        if (++slot == NS) {
          slot = 0;
          ph ^= 1u;
        }
      }
      // every copy this CTA issued has landed before it can leave
      for (int j = max(0, issued - NS); j < issued; ++j) wait_drain(&full[j % NS], (j / NS) & 1u);
    }
    __syncwarp();
  } else {
    if (warp == kAllocWarp) {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
    tc_fence_before();
    named_bar_sync(1, kThreads - 32);                  // everyone but the producer
    tc_fence_after();
    tbase = *tmem_slot;
    constexpr int S = TM::kSlots;

    if (warp >= kMmaWarp0 && warp < kMmaWarp0 + kGroups) {
      // ----------------------------------------------------------- MMA warps --
      // Group g's units g, g + 3, ... in order: 4 MMAs (K = 32 each) with A and
      // its scale factors from the unit's TMEM slot and B from shared memory,
      // into the group's accumulator for the unit's tile segment.  One warp
      // per group, each on its own sub-partition: an MMA thread whose
      // sub-partition also runs decode arithmetic issues at about half the
      // tensor core's rate, so three issue side by side.  The whole warp
      // follows the loop (its values stay warp-uniform); lane 0 issues,
      // always the same thread, so its commits track all of the group's
      // tensor-core work.
      const int g = warp - kMmaWarp0;
      named_bar_sync(3, 32 * kGroups + 32 * 4);        // the epilogue stored the B scale factors
      tc_fence_after();
      const uint64_t bd0 = umma_desc_kmajor_sw128(smem_u32(b_s));
      const uint32_t idesc = umma_idesc_mxf8(NTOK, 0, 0);
      const uint32_t sfb_col = tbase + kSfbCol;
      int t = t_first, c = c_first;
      geo.advance(t, c, g);
      int bsl = c - c_first;                           // B slot: (c - c_first) mod KT
      if (bsl < 0) bsl += KT;
      int cur_t = -1;
      uint32_t buf_par = 0;                            // bit b: parity of the uses of buffer b
      int su = 0;                                      // slot of the group's use: use % S
      uint32_t aph = 0;                                // its phase: (use / S) & 1
      for (int i = g; i < n_units; i += kGroups) {
        int t2 = t, c2 = c;
        geo.advance(t2, c2, kGroups);
        const int as = g * S + su;
        // this k-tile's activations landed (from unit 3 KT on, the group
        // waited for this slot at unit i - 3 KT)
        if (i < 3 * KT) wait_bounded(&b_full[bsl], 0, abort_flag, wait_ns);
        wait_bounded(&a_full[as], aph, abort_flag, wait_ns);    // the group's four warps stored it
        tc_fence_after();
        const bool seg_first = t != cur_t;              // the group's first unit of this tile
        const int b = (t - t_first) & 1;
        if (seg_first) {
          cur_t = t;
          wait_bounded(&acc_empty[2 * g + b], ((buf_par >> b) & 1u) ^ 1u, abort_flag, wait_ns);
          tc_fence_after();
        }
        const bool seg_last = t2 != t || i + kGroups >= n_units;   // the group's last unit of this tile
        if (lane == 0) {
          const uint32_t a_col = tbase + TM::kACol + 32 * as, sfa_col = tbase + TM::kSfaCol + 4 * as;
          const uint64_t bdu = bd0 + static_cast<uint64_t>(bsl * NTOK * 8);
          const uint32_t d_col = tbase + TM::acc(g, b);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            umma_mxf8_ts(d_col, a_col + 8 * j, bdu + static_cast<uint64_t>(2 * j), idesc | (uint32_t(j) << 29),
                         sfa_col, sfb_col, (seg_first && j == 0) ? 0u : 1u);
          umma_commit(&a_empty[as]);
          if (seg_last) umma_commit(&acc_full[2 * g + b]);
        }
        if (seg_last) buf_par ^= 1u << b;
        __syncwarp();
        t = t2;
        c = c2;
        bsl += kGroups;                                  // (bsl + 3) mod KT; KT may be 1 or 2
        while (bsl >= KT) bsl -= KT;
        if (++su == S) {
          su = 0;
          aph ^= 1u;
        }
      }
      // all of the group's tensor-core work is done before TMEM is freed
      if (lane == 0) {
        umma_commit(&drain[g]);
        wait_drain(&drain[g], 0);
      }
      __syncwarp();
    } else if (warp >= kDecWarp0 && warp < kEpiWarp0) {
      // ------------------------------------------------------------ decoders --
      // Warp 4 + 4 g + q: group g's units g, g + 3, ..., rows r = 32 q + lane
      // of each -- the warp's own TMEM lane quarter.  A unit's 128 decoded
      // bytes of row r go to 32 columns of one of the group's A slots, its
      // scale word to the slot's 4 scale-factor columns.
      const int g = (warp - kDecWarp0) >> 2, q = warp & 3;
      const int r = 32 * q + lane;                      // row inside the tile
      const uint32_t lane_base = tbase + (static_cast<uint32_t>(32 * q) << 16);
      const uint32_t codes_base = smem_u32(codes_s);
      const int gk = p.K / 32;
      // scale word and codebook of row r for the unit at (t, c)
      auto load_sc = [&](int t, int c, bool valid, uint32_t& sw, uint2& cb) {
        sw = 0x7F7F7F7Fu;
        cb = make_uint2(0, 0);
        if (valid && geo.local_tile(t) * kRows + r < p.N) {
          const long long n = geo.row_of(t, r);          // row of the (stacked) weight
          sw = __ldg(reinterpret_cast<const uint32_t*>(p.scales + static_cast<size_t>(n) * gk + 4 * c));
          if constexpr (BITS == 3)
            cb = __ldg(reinterpret_cast<const uint2*>(p.codebooks + static_cast<size_t>(n) * 8));
          else
            cb.x = __ldg(reinterpret_cast<const uint32_t*>(p.codebooks + static_cast<size_t>(n) * 4));
        }
      };
      // stage of unit i: i / 4, position i % 4; advanced by 3 units per step
      int slot = 0, pos = g;
      uint32_t ph = 0;
      int su = 0;                                       // the group's A slot: use % S
      uint32_t aph = 0;                                 // its phase: (use / S) & 1
      // With two slots per group a unit's TMEM stores complete while the warp
      // decodes its next unit; then the unit goes to the MMA warp (pend_as:
      // its slot, -1 if none).  With one slot the next store waits for the
      // MMAs of this unit, so it goes at once.
      int pend_as = -1;
      auto publish = [&]() {
        if (pend_as >= 0) {
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&a_full[pend_as]);
          pend_as = -1;
        }
      };
      auto process = [&](int t, int c, uint32_t sw, uint2 cb) {
        wait_bounded(&full[slot], ph, abort_flag, wait_ns);
        uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0, c2v = c0;
        const int rows_t = geo.rows(t);
        if (r < rows_t) {
          // rows of the pos units before this one in the stage: min(pos, c)
          // of them in tile t (rows_t rows each; t may be the ragged last
          // tile), the rest in full tiles before it -- or, grouped, in the
          // last tile of the previous expert, which may be ragged too
          int before;
          if constexpr (!GROUPED) {
            const int kin = min(pos, c);
            before = kin * rows_t + (pos - kin) * kRows;
          } else {
            before = 0;
            int tp = t, cp = c;
            for (int k = 0; k < pos; ++k) {
              if (cp == 0) {
                cp = KT - 1;
                --tp;
              } else {
                --cp;
              }
              before += geo.rows(tp);
            }
          }
          const uint32_t at = codes_base + slot * kStageBytes + (before + r) * RB;
          c0 = lds128(at);
          c1 = lds128(at + 16);
          if constexpr (BITS == 3) c2v = lds128(at + 32);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        uint32_t v[32];
        if constexpr (BITS == 3) {
          decode_group(c0.x, c0.y, c0.z, cb.x, cb.y, v);
          decode_group(c0.w, c1.x, c1.y, cb.x, cb.y, v + 8);
          decode_group(c1.z, c1.w, c2v.x, cb.x, cb.y, v + 16);
          decode_group(c2v.y, c2v.z, c2v.w, cb.x, cb.y, v + 24);
        } else {                                        // 8 bytes per group, 4-entry codebook in cb.x
          decode_group2(c0.x, c0.y, cb.x, v);
          decode_group2(c0.z, c0.w, cb.x, v + 8);
          decode_group2(c1.x, c1.y, cb.x, v + 16);
          decode_group2(c1.z, c1.w, cb.x, v + 24);
        }
        publish();                                      // the previous unit
        const int as = g * S + su;
        wait_bounded(&a_empty[as], aph ^ 1u, abort_flag, wait_ns);   // the MMAs of its last use are done
        tc_fence_after();
        tmem_st_x32(lane_base + TM::kACol + 32 * as, v);
        // row r's scale word in all 4 columns: the MMA finds it whichever
        // column of the 4 it reads for the row
        tmem_st_x4(lane_base + TM::kSfaCol + 4 * as, sw, sw, sw, sw);
        pend_as = as;
        if (S == 1) publish();
        if (++su == S) {
          su = 0;
          aph ^= 1u;
        }
        pos += kGroups;                                 // next unit of the group: 3 further
        if (pos >= kUnitsPerStage) {
          pos -= kUnitsPerStage;
          if (++slot == NS) {
            slot = 0;
            ph ^= 1u;
          }
        }
      };
      // Two register sets for the scale word and codebook, so the loads for
      // the group's next unit are in flight during the current one (the loop
      // is unrolled by two: no register copy waits for a load).
      int ta = t_first, ca = c_first;                   // unit i (set A)
      geo.advance(ta, ca, g);
      uint32_t swA, swB;
      uint2 cbA, cbB;
      load_sc(ta, ca, g < n_units, swA, cbA);
      for (int i = g; i < n_units; i += 2 * kGroups) {
        int tb = ta, cbb = ca;                          // unit i + 3 (set B)
        geo.advance(tb, cbb, kGroups);
        load_sc(tb, cbb, i + kGroups < n_units, swB, cbB);
        process(ta, ca, swA, cbA);
        if (i + kGroups >= n_units) break;
        ta = tb;                                        // unit i + 6 (set A)
        ca = cbb;
        geo.advance(ta, ca, kGroups);
        load_sc(ta, ca, i + 2 * kGroups < n_units, swA, cbA);
        process(tb, cbb, swB, cbB);
      }
      publish();                                        // the group's last unit
    } else if (warp >= kEpiWarp0) {
      // ------------------------------------------------------------ epilogue --
      const int q = warp & 3;
      const int r = 32 * q + lane;
      const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
      const bool leader = tid == kEpiWarp0 * 32;
      // Finished values of one 16-column chunk of tile t (row r, columns
      // c0..c0+15 = token rows): y = a_scale * v, or the gate-up product.
      // Every epilogue thread calls it (it may hold named barriers).
      auto emit = [&](int t, int c0, const float (&v)[16]) {
        if constexpr (GROUPED) {
          // y[m][j][n] for every slot j where token m chose this tile's expert:
          // lane k works out token c0 + k's slots, every lane learns them
          const int e = geo.expert(t);
          const int nl = geo.local_tile(t) * kRows + r;
          uint32_t mask = 0;
          if (lane < 16 && c0 + lane < p.M)
            for (int j = 0; j < p.topk; ++j)
              if (topk_s[(c0 + lane) * p.topk + j] == e) mask |= 1u << j;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            uint32_t mk = __shfl_sync(0xffffffffu, mask, k);
            if (nl < p.N && mk) {
              const float yv = v[k] * __ldg(p.a_scale + c0 + k);
              for (; mk; mk &= mk - 1)
                p.y[(static_cast<size_t>(c0 + k) * p.topk + (__ffs(mk) - 1)) * p.N + nl] = yv;
            }
          }
        } else if constexpr (!GATE_UP) {
          const int n = t * kRows + r;
          if (n < p.N) {
#pragma unroll
            for (int k = 0; k < 16; ++k)
              if (c0 + k < p.M) p.y[static_cast<size_t>(c0 + k) * p.N + n] = v[k] * __ldg(p.a_scale + c0 + k);
          }
        } else {
          const int R = geo.rows(t), half = R >> 1;
          if (r >= half && r < R) {
#pragma unroll
            for (int k = 0; k < 16; ++k)
              xchg[(r - half) * kXchgStride + k] = c0 + k < p.M ? v[k] * __ldg(p.a_scale + c0 + k) : 0.f;
          }
          named_bar_sync(2, 128);
          if (32 * q < half) {                          // warps holding gate rows
            const int f = 64 * t + r;
            float hv[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              hv[k] = 0.f;
              if (r < half && c0 + k < p.M) {
                const float gv = v[k] * __ldg(p.a_scale + c0 + k);
                hv[k] = gv / (1.f + expf(-gv)) * xchg[r * kXchgStride + k];
                p.h[static_cast<size_t>(c0 + k) * p.F + f] = hv[k];
              }
              hv[k] = fabsf(hv[k]);
            }
            // per token the warp's max|h| by a transposing butterfly (16
            // shuffles for the 16 tokens): at each step a lane keeps half of
            // its tokens and takes the partner's values of them; lane l ends
            // with token 8 b4 + 4 b3 + 2 b2 + b1 (b: the bits of l)
#pragma unroll
            for (int st = 0; st < 4; ++st) {
              const int mask = 16 >> st, hn = 8 >> st;
              const bool hi = (lane & mask) != 0;
#pragma unroll
              for (int i = 0; i < hn; ++i) {
                const float keep = hi ? hv[hn + i] : hv[i];
                const float send = hi ? hv[i] : hv[hn + i];
                hv[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, mask));
              }
            }
            hv[0] = fmaxf(hv[0], __shfl_xor_sync(0xffffffffu, hv[0], 1));
            const int tk = 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
            if ((lane & 1) == 0 && c0 + tk < p.M) atomicMax(p.h_amax + c0 + tk, __float_as_uint(hv[0]));
          }
          named_bar_sync(2, 128);                        // xchg is reused by the next chunk
        }
      };
      // scale factors of B: 2^0 in every byte of 8 columns, all 128 lanes
      for (int cc = 0; cc < 8; cc += 4)
        tmem_st_x4(tbase + lane_addr + kSfbCol + cc, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_st_wait();
      tc_fence_before();
      named_bar_sync(3, 32 * 4 + 32 * kGroups);        // B scale factors are in TMEM (with the MMA warps)
      grid_dependency_wait();                           // y, the workspace and the activations may still be in use
      if (warp == kEpiWarp0 && n_units > 0) {
        // Resident activations, written by an earlier kernel: k-tile c of this
        // CTA's share lands in slot (c - c_first) mod KT as NTOK rows of 128
        // bytes in the 128-byte swizzled K-major layout (one TMA box, one
        // barrier per slot, the warp's lanes issuing slots 0, 1, ... in the
        // order the MMAs take them); token rows >= M are outside the tensor
        // and arrive as zeros.
        const int nb = min(KT, n_units);
        for (int sl = lane; sl < nb; sl += 32) {
          int cc = c_first + sl;
          if (cc >= KT) cc -= KT;
          mbar_arrive_expect_tx(&b_full[sl], static_cast<uint32_t>(NTOK * 128));
          tma_load_2d(b_s + sl * NTOK * 128, &p.a_map, &b_full[sl], cc * 128, 0);
        }
      }
      uint32_t acc_par = 0;                             // bit 2 g + b: parity of (group, buffer) uses
      int t = t_first, c = c_first, s0 = 0;             // s0: first unit of the segment
      for (int i = 0; i < n_units; ++i, geo.advance(t, c, 1)) {
        if (c != KT - 1 && i != n_units - 1) continue;
        const int seg_c = (s0 == 0) ? c_first : 0;
        const bool complete = seg_c == 0 && c == KT - 1;
        const int span = i - s0;                          // units in the segment - 1
        const int b = (t - t_first) & 1;
        // groups with a unit in [s0, i] (unit u belongs to group u % 3): all
        // of them if the segment has 3 or more
        uint32_t part = 0;
#pragma unroll
        for (int g = 0; g < kGroups; ++g)
          if (span >= kGroups - 1 || (g - s0 % kGroups + kGroups) % kGroups <= span) part |= 1u << g;
        // A partial tile's parts: CTAs b_first .. b_first + nparts - 1, this
        // one part pme.  This CTA's last segment usually arrives after the
        // other parts (first segments of later CTAs, finished early): it reads
        // the tile's counter before its own accumulators are ready, so that
        // round trip overlaps the last MMAs.
        const long long tu = static_cast<long long>(t) * KT;
        const long long b_first = geo.owner(tu);
        const int nparts = complete ? 1 : static_cast<int>(geo.owner(tu + KT - 1) - b_first + 1);
        const int pme = static_cast<int>(blockIdx.x - b_first);
        bool last = false;
        if (!complete && i == n_units - 1) {
          if (leader) *last_flag = ld_acquire_gpu(p.counters + t) == static_cast<unsigned>(nparts - 1);
          named_bar_sync(2, 128);
          last = *last_flag;
          named_bar_sync(2, 128);
        }
#pragma unroll
        for (int g = 0; g < kGroups; ++g)
          if (part & (1u << g)) {
            wait_bounded(&acc_full[2 * g + b], (acc_par >> (2 * g + b)) & 1u, abort_flag, wait_ns);
            acc_par ^= 1u << (2 * g + b);
          }
        tc_fence_after();
        // the segment's accumulator, chunk c0: sum of the groups' parts in group order
        auto load_acc = [&](int c0, float (&v)[16]) {
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] = 0.f;
#pragma unroll
          for (int g = 0; g < kGroups; ++g)
            if (part & (1u << g)) {
              uint32_t tv[16];
              tmem_ld_x16(tbase + lane_addr + TM::acc(g, b) + c0, tv);
              tmem_ld_wait();
#pragma unroll
              for (int k = 0; k < 16; ++k) v[k] += __uint_as_float(tv[k]);
            }
        };
        if (complete) {
#pragma unroll 1
          for (int c0 = 0; c0 < NTOK; c0 += 16) {
            float v[16];
            load_acc(c0, v);
            emit(t, c0, v);
          }
        } else {
          // Partial tile.  Each part's fp32 tile goes to its workspace slot
          // and bumps the tile's counter; the part that finds every other part
          // published (by the read above, or by the value its own add
          // returns) sums all parts in part order and writes y.  One thread
          // releases the block's stores after a barrier, and acquires the
          // others' before one.
          const bool seg_is_first = s0 == 0;
          bool own_published = false;
          if (!last) {
            float* part_dst =
                p.partial + (static_cast<size_t>(2 * blockIdx.x + (seg_is_first ? 0 : 1)) * kRows + r) * NTOK;
#pragma unroll 1
            for (int c0 = 0; c0 < NTOK; c0 += 16) {
              float v[16];
              load_acc(c0, v);
              float4* dst = reinterpret_cast<float4*>(part_dst + c0);
#pragma unroll
              for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            }
            own_published = true;
            named_bar_sync(2, 128);                      // every thread's stores precede the release
            if (leader) *last_flag = atom_add_acq_rel_gpu(p.counters + t, 1u) == static_cast<unsigned>(nparts - 1);
            named_bar_sync(2, 128);
            last = *last_flag;
          }
          if (last) {
            // part pi's workspace slot: part 0's CTA reaches this tile as its
            // last segment if its share started in an earlier tile, every
            // later part as its first
            auto part_src = [&](int pi, int c0) {
              const long long bb = b_first + pi;
              const int pslot = 2 * static_cast<int>(bb) + ((pi == 0 && geo.first_unit(bb) < tu) ? 1 : 0);
              return reinterpret_cast<const float4*>(p.partial + (static_cast<size_t>(pslot) * kRows + r) * NTOK + c0);
            };
#pragma unroll 1
            for (int c0 = 0; c0 < NTOK; c0 += 16) {
              float mine[16];
              if (!own_published) load_acc(c0, mine);
              float acc[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) acc[k] = 0.f;
              // two parts' loads in flight at a time, summed in part order
#pragma unroll 1
              for (int pi = 0; pi < nparts; pi += 2) {
                const bool ld0 = pi != pme || own_published;
                const bool has1 = pi + 1 < nparts;
                const bool ld1 = has1 && (pi + 1 != pme || own_published);
                float4 f0[4], f1[4];
                if (ld0) {
                  const float4* src = part_src(pi, c0);
#pragma unroll
                  for (int k = 0; k < 4; ++k) f0[k] = __ldcg(src + k);
                }
                if (ld1) {
                  const float4* src = part_src(pi + 1, c0);
#pragma unroll
                  for (int k = 0; k < 4; ++k) f1[k] = __ldcg(src + k);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  if (ld0) {
                    acc[4 * k] += f0[k].x;
                    acc[4 * k + 1] += f0[k].y;
                    acc[4 * k + 2] += f0[k].z;
                    acc[4 * k + 3] += f0[k].w;
                  } else {
                    acc[4 * k] += mine[4 * k];
                    acc[4 * k + 1] += mine[4 * k + 1];
                    acc[4 * k + 2] += mine[4 * k + 2];
                    acc[4 * k + 3] += mine[4 * k + 3];
                  }
                }
                if (has1) {
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    if (ld1) {
                      acc[4 * k] += f1[k].x;
                      acc[4 * k + 1] += f1[k].y;
                      acc[4 * k + 2] += f1[k].z;
                      acc[4 * k + 3] += f1[k].w;
                    } else {
                      acc[4 * k] += mine[4 * k];
                      acc[4 * k + 1] += mine[4 * k + 1];
                      acc[4 * k + 2] += mine[4 * k + 2];
                      acc[4 * k + 3] += mine[4 * k + 3];
                    }
                  }
                }
              }
              emit(t, c0, acc);
            }
            if (leader) p.counters[t] = 0u;              // ready for the next call
          }
          named_bar_sync(2, 128);                        // last_flag is reused by the next segment
        }
        tc_fence_before();
        __syncwarp();
#pragma unroll
        for (int g = 0; g < kGroups; ++g)
          if ((part & (1u << g)) && lane == 0) mbar_arrive(&acc_empty[2 * g + b]);
        s0 = i + 1;
      }
      if (warp == kEpiWarp0)                             // the activations landed before the CTA can end
        for (int sl = lane; sl < min(KT, n_units); sl += 32) wait_drain(&b_full[sl], 0);
      if constexpr (GATE_UP) {
        // every product and maximum of this CTA is written: one release-
        // acquire add after a barrier counts the CTA; the last one learns
        // that all CTAs' are visible
        named_bar_sync(2, 128);
        if (leader) *last_flag = atom_add_acq_rel_gpu(p.h_done, 1u) == gridDim.x - 1u;
      }
    }
  }

  // ---- teardown: each group's MMA warp saw its tensor-core work complete,
  // the producer saw its copies land, the B loads landed, the epilogue
  // waited for its TMEM loads.
  tc_fence_before();
  __syncthreads();
  if constexpr (GATE_UP) {
    if (*last_flag) {
      // The last CTA: per token the scale s = max|h| / 448 (1 for an
      // all-zero token); with few products, every product h / s to E4M3
      // (nearest even, saturating), all threads over each token's row (else
      // gate_up_quant_kernel does that from the scales); then the maxima and
      // the count go back to zero for the next call.
      float* s_tok = xchg;                           // [M] scales
      if (tid < p.M) {
        const float a = __uint_as_float(__ldcg(p.h_amax + tid));
        const float sc = a > 0.f ? a / 448.f : 1.f;
        s_tok[tid] = sc;
        p.q_scale[tid] = sc;
      }
      __syncthreads();
      if (p.fuse_quant) {
      // the M x F products as one flat array (rows are contiguous in h and
      // q): four float4 loads in flight per thread, token of element i = i / F
      FastDiv by_f;
      by_f.init(static_cast<uint32_t>(p.F));
      const int total = p.M * p.F, n4 = total >> 2;
      const float4* h4 = reinterpret_cast<const float4*>(p.h);
      for (int i0 = tid; i0 < n4; i0 += 4 * kThreads) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (i0 + u * kThreads < n4) v[u] = __ldcg(h4 + i0 + u * kThreads);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = i0 + u * kThreads;
          if (j < n4) {
            const float e[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int i = 4 * j + c;
              p.q[i] = static_cast<uint8_t>(
                  __nv_cvt_float_to_fp8(e[c] / s_tok[by_f.div(i)], __NV_SATFINITE, __NV_E4M3));
            }
          }
        }
      }
      for (int i = 4 * n4 + tid; i < total; i += kThreads)   // the last total % 4 products
        p.q[i] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(__ldcg(p.h + i) / s_tok[by_f.div(i)], __NV_SATFINITE,
                                                             __NV_E4M3));
      }
      __syncthreads();
      if (tid < p.M) p.h_amax[tid] = 0u;
      if (tid == 0) *p.h_done = 0u;
    }
  }
  if (warp == kAllocWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, kTmemCols);
  }
}

int ntok_for(int M) { return M <= 16 ? 16 : (M <= 32 ? 32 : 64); }

constexpr int kQuantThreads = 256;
constexpr int kQuantChunk = 8 * kQuantThreads;        // products of one CTA: eight a thread

// The products of one token in chunks of 2048, eight consecutive products a
// thread: h / s to E4M3 (nearest even, saturating) with the token's scale s,
// which the matmul's last CTA wrote.
__global__ void __launch_bounds__(kQuantThreads) gate_up_quant_kernel(const float* __restrict__ h,
                                                                      const float* __restrict__ scale, int F,
                                                                      uint8_t* __restrict__ q) {
  grid_dependency_wait();                         // h and the scales of the matmul kernel
  const int m = blockIdx.y;
  const float s = scale[m];
  const float* hr = h + static_cast<size_t>(m) * F;
  uint8_t* qr = q + static_cast<size_t>(m) * F;
  const int f0 = blockIdx.x * kQuantChunk + 8 * threadIdx.x;
  const bool vec = (F & 7) == 0 && (reinterpret_cast<uintptr_t>(q) & 7) == 0;   // 32-byte rows of h, 8 of q
  if (vec && f0 + 8 <= F) {
    const float4 a = __ldcg(reinterpret_cast<const float4*>(hr + f0));
    const float4 b = __ldcg(reinterpret_cast<const float4*>(hr + f0 + 4));
    const float e[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t w[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i >> 2] |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(e[i] / s, __NV_SATFINITE, __NV_E4M3)) << (8 * (i & 3));
    *reinterpret_cast<uint2*>(qr + f0) = make_uint2(w[0], w[1]);
  } else {
    for (int f = f0; f < min(F, f0 + 8); ++f)
      qr[f] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(__ldcg(hr + f) / s, __NV_SATFINITE, __NV_E4M3));
  }
}

// Products up to which the last CTA of the matmul quantises them itself.
constexpr int kFusedQuant = 1 << 13;

struct Plan {
  int ntok = 0, grid = 0, stages = 0, b_ktiles = 0, smem = 0, tiles = 0;
};

// Tile arrival counters and the gate-up per-token maxima live in a fixed area
// at the start of the workspace, the same for every shape, so that partial
// tiles or products a call writes can never land where a later call with
// another shape expects zeros.
constexpr int kMaxTiles = 1 << 16;                    // N <= 8388608 rows
constexpr size_t kCountersBytes = static_cast<size_t>(kMaxTiles) * 4;
constexpr size_t kFixedBytes = kCountersBytes + 512;  // + gate-up maxima [64], finished-CTA count

enum Mode { kDense, kGateUp, kGrouped };

// Grouped calls: E experts stacked, each N x K; at most min(E, M topk) of
// them are used (the kernel finds which), and the plan is made for that many.
bool plan_for(int M, int N, int K, Mode mode, Plan& pl, int E = 1, int topk = 1) {
  if (M < 1 || M > 64 || N < 1 || K < 128 || K % 128 != 0) return false;
  if (mode == kGrouped && (E < 1 || E > 4096 || topk < 1 || topk > 8 || M * topk > kMaxRouted)) return false;
  const int KT = K / 128;
  const long long experts = mode == kGrouped ? std::min<long long>(E, static_cast<long long>(M) * topk) : 1;
  const long long tiles = experts * ((N + kRows - 1) / kRows);
  if (tiles > kMaxTiles) return false;
  const long long U = tiles * KT;
  if (U >= (1LL << 31)) return false;                 // unit numbers are 32-bit on the device
  // Stream-K shares (an equal number of units per CTA, tiles split between
  // CTAs) -- except where the tiles alone fill most of the GPU: then one
  // whole tile per CTA, which needs no partial-tile fix-up (decode 4096 x
  // 12288: 96 tiles on 152 SMs, 11.4-11.8 us against 12.1-12.3 us per call).
  // A grouped call's unit count is known on the device only: shares.
  const long long sms = device_sm_count();
  const long long G = (mode != kGrouped && tiles <= sms && 5 * tiles >= 3 * sms) ? tiles : std::min<long long>(U, sms);
  const long long per = (U + G - 1) / G;               // most units of any CTA
  pl.ntok = ntok_for(M);
  pl.b_ktiles = static_cast<int>(std::min<long long>(KT, per));
  if (pl.b_ktiles > kMaxBSlots) return false;
  const int fixed = pl.b_ktiles * pl.ntok * 128 + (mode == kGateUp ? kXchgBytes : 0) + kBarBytes +
                    (mode == kGrouped ? kRouteBytes : 0);
  pl.stages = std::min(kMaxStages, (kMaxSmem - fixed) / kStageBytes);
  if (pl.stages < 2) return false;
  pl.smem = std::max(pl.stages * kStageBytes + fixed, kMinSmem);
  pl.grid = static_cast<int>(G);
  pl.tiles = static_cast<int>(tiles);
  return true;
}

// Workspace layout: [tile counters, 256 KB][gate-up maxima, 64 x 4 B]
// [two partial tiles of 128 x ntok fp32 per CTA][gate-up products, M x F fp32].
size_t partial_bytes(const Plan& pl) { return static_cast<size_t>(2) * pl.grid * kRows * pl.ntok * sizeof(float); }
size_t workspace_bytes(const Plan& pl, int M, int F) {
  return kFixedBytes + partial_bytes(pl) + (F > 0 ? (static_cast<size_t>(M) * F * 4 + 255) / 256 * 256 : 0);
}

// cudaFuncSetAttribute once per (device, kernel).
template <int NTOK, bool GATE_UP, bool GROUPED, int BITS>
int configure() {
  static std::atomic<int> done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return CBQ_EDEVICE;
  if (done[dev].load(std::memory_order_acquire)) return CBQ_OK;
  if (cudaFuncSetAttribute(sk_kernel<NTOK, GATE_UP, GROUPED, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kMaxSmem) !=
      cudaSuccess)
    return CBQ_ECUDA;
  done[dev].store(1, std::memory_order_release);
  return CBQ_OK;
}

// Launch with programmatic stream serialisation: the kernel may start while
// the previous kernel on the stream finishes (it waits on the grid dependency
// before it touches what that kernel may write).
template <typename... Args>
cudaError_t launch_pdl(void (*kern)(Args...), dim3 grid, dim3 block, int smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
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

template <int NTOK, bool GATE_UP, bool GROUPED, int BITS = 3>
int launch_t(const SkParams& p, const Plan& pl, cudaStream_t stream) {
  if (const int st = configure<NTOK, GATE_UP, GROUPED, BITS>(); st != CBQ_OK) return st;
  return launch_pdl(sk_kernel<NTOK, GATE_UP, GROUPED, BITS>, dim3(pl.grid), dim3(kThreads), pl.smem, stream, p) ==
                 cudaSuccess
             ? CBQ_OK
             : CBQ_ECUDA;
}

// Activations a[M][K] as a TMA tensor whose box is one k-tile of `ntok`
// token rows: a 2-D view with a (128 B, ntok) box and the 128-byte swizzle;
// rows past M read as zeros.
int encode_a_map(SkParams& p, int ntok) { return encode_activation_map(&p.a_map, p.a, p.M, p.K, ntok); }

int launch_planned(const SkParams& p_in, const Plan& pl, float* partial, unsigned* counters, Mode mode,
                   cudaStream_t stream, int bits = 3) {
  SkParams p = p_in;
  p.partial = partial;
  p.counters = counters;
  p.stages = pl.stages;
  p.b_ktiles = pl.b_ktiles;
  const int em = encode_a_map(p, pl.ntok);
  if (em != CBQ_OK) return em;
  if (mode == kGateUp) {
    if (pl.ntok == 16) return launch_t<16, true, false>(p, pl, stream);
    if (pl.ntok == 32) return launch_t<32, true, false>(p, pl, stream);
    return launch_t<64, true, false>(p, pl, stream);
  }
  if (mode == kGrouped) {
    if (pl.ntok == 16) return launch_t<16, false, true>(p, pl, stream);
    if (pl.ntok == 32) return launch_t<32, false, true>(p, pl, stream);
    return launch_t<64, false, true>(p, pl, stream);
  }
  if (bits == 2) {
    if (pl.ntok == 16) return launch_t<16, false, false, 2>(p, pl, stream);
    if (pl.ntok == 32) return launch_t<32, false, false, 2>(p, pl, stream);
    return launch_t<64, false, false, 2>(p, pl, stream);
  }
  if (pl.ntok == 16) return launch_t<16, false, false>(p, pl, stream);
  if (pl.ntok == 32) return launch_t<32, false, false>(p, pl, stream);
  return launch_t<64, false, false>(p, pl, stream);
}

// Static scratch of the allocation-free entry point: partial tiles for up to
// kStaticCtas CTAs at 64 token columns, and counters for kStaticTiles tiles.
// Zero at module load; each call clears the counters it will use.
constexpr int kStaticCtas = 160;
constexpr int kStaticTiles = kMaxTiles;
__device__ __align__(256) float g_static_partial[2 * kStaticCtas * kRows * 64];
__device__ __align__(256) unsigned g_static_counters[kStaticTiles];

}  // namespace

bool sk_applicable(int M, int N, int K) {
  Plan pl;
  return plan_for(M, N, K, kDense, pl);
}

size_t sk_workspace_bytes(int M, int N, int K) {
  Plan pl;
  return plan_for(M, N, K, kDense, pl) ? workspace_bytes(pl, M, 0) : 0;
}

size_t sk_gate_up_workspace_bytes(int M, int F, int K) {
  Plan pl;
  return plan_for(M, 2 * F, K, kGateUp, pl) ? workspace_bytes(pl, M, F) : 0;
}

int launch_sk(const SkParams& p_in, void* workspace, size_t ws_bytes, cudaStream_t stream, int bits) {
  Plan pl;
  if (!plan_for(p_in.M, p_in.N, p_in.K, kDense, pl)) return CBQ_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || ws_bytes < workspace_bytes(pl, p_in.M, 0))
    return CBQ_EINVAL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return launch_planned(p_in, pl, reinterpret_cast<float*>(ws + kFixedBytes), reinterpret_cast<unsigned*>(ws),
                        kDense, stream, bits);
}

size_t sk_grouped_workspace_bytes(int E, int topk, int M, int N, int K) {
  Plan pl;
  return plan_for(M, N, K, kGrouped, pl, E, topk) ? workspace_bytes(pl, M, 0) : 0;
}

int launch_sk_grouped(const SkParams& p_in, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  Plan pl;
  if (!plan_for(p_in.M, p_in.N, p_in.K, kGrouped, pl, p_in.E, p_in.topk)) return CBQ_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || ws_bytes < workspace_bytes(pl, p_in.M, 0))
    return CBQ_EINVAL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  return launch_planned(p_in, pl, reinterpret_cast<float*>(ws + kFixedBytes), reinterpret_cast<unsigned*>(ws),
                        kGrouped, stream);
}

int launch_sk_gate_up(const SkParams& p_in, void* workspace, size_t ws_bytes, uint8_t* q, float* q_scale,
                      cudaStream_t stream) {
  Plan pl;
  const int F = p_in.N / 2;
  if (p_in.N % 2 != 0 || !plan_for(p_in.M, p_in.N, p_in.K, kGateUp, pl)) return CBQ_EINVAL;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      ws_bytes < workspace_bytes(pl, p_in.M, F))
    return CBQ_EINVAL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SkParams p = p_in;
  p.F = F;
  p.h_amax = reinterpret_cast<unsigned*>(ws + kCountersBytes);
  p.h_done = reinterpret_cast<unsigned*>(ws + kCountersBytes + 256);
  p.h = reinterpret_cast<float*>(ws + kFixedBytes + partial_bytes(pl));
  p.q = q;
  p.q_scale = q_scale;
  p.fuse_quant = static_cast<long long>(p.M) * F <= kFusedQuant ? 1 : 0;
  const int st = launch_planned(p, pl, reinterpret_cast<float*>(ws + kFixedBytes), reinterpret_cast<unsigned*>(ws),
                                kGateUp, stream);
  if (st != CBQ_OK || p.fuse_quant) return st;
  return launch_pdl(gate_up_quant_kernel, dim3((F + kQuantChunk - 1) / kQuantChunk, p.M), dim3(kQuantThreads), 0,
                    stream, static_cast<const float*>(p.h), static_cast<const float*>(q_scale), F, q) == cudaSuccess
             ? CBQ_OK
             : CBQ_ECUDA;
}

int launch_sk_static(const SkParams& p_in, cudaStream_t stream) {
  Plan pl;
  if (!plan_for(p_in.M, p_in.N, p_in.K, kDense, pl)) return CBQ_EINVAL;
  if (pl.grid > kStaticCtas || pl.tiles > kStaticTiles) return CBQ_EINVAL;
  // the static buffers' addresses on the current device (looked up on the
  // first call on each device)
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
  return launch_planned(p_in, pl, static_cast<float*>(partial), static_cast<unsigned*>(counters), kDense, stream);
}

unsigned take_status_sk(cudaStream_t stream) {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbolAsync(&v, g_status_sk, sizeof(v), 0, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return kErrTimeout;
  cudaMemcpyToSymbolAsync(g_status_sk, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  cudaStreamSynchronize(stream);
  return v;
}

}  // namespace cbq
