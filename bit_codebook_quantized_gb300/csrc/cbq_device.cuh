// cbq_device.cuh -- device-side building blocks shared by the libcbq kernels:
// the 3-bit code decode, mbarrier / TMA wrappers with bounded waits, and the
// library's sticky device status word.
//
// Format ("Hibana: Fast Agentic Inference on Unified-Memory Devices",
// section "Model surgery / Three-bit weights"): a group of 32 weights is 12
// bytes, a 96-bit little-endian number holding code j at bits 3j..3j+2; each
// code indexes the row's 8-entry E4M3 codebook; one E8M0 scale per group.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace cbq {

// Status bits a kernel can raise (each translation unit keeps its own sticky
// word; cbq_device_status() collects and clears them).
enum : unsigned { kErrTimeout = 1u, kErrRouting = 2u };

// Bounded waits give up after this many nanoseconds of the global timer
// (~2 s; the SM clock may not advance for a suspended warp, the global timer
// does).
constexpr long long kWaitLimitNs = 2000000000LL;

__device__ __forceinline__ long long global_ns() {
  long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Decode: 8 codes (a 24-bit field) -> 8 E4M3 bytes through the codebook.
// ---------------------------------------------------------------------------

// Spread 8 packed 3-bit codes (bits 3j..3j+2 of f, j = 0..7; bits 24..31 of f
// are ignored) so that code j lands in nibble j.  The result, and the result
// shifted right by 16, are byte-permute selectors for codes 0-3 and 4-7.
__device__ __forceinline__ uint32_t spread_codes8(uint32_t f) {
  uint32_t h = f & 0x00FFFFFFu;                   // the 8 codes, bits 0..23
  h += (h & 0x00FFF000u) * 15u;                   // codes 4-7 up by 4 bits
  h += (h & 0x0FC00FC0u) * 3u;                    // codes 2,3 and 6,7 up by 2
  return h + (h & 0x38383838u);                   // odd codes up by 1
}

// Four E4M3 codebook bytes for the four codes held in nibbles 0..3 of `sel`
// (each 0..7; nibble bit 3 clear).  cb_lo holds entries 0-3, cb_hi 4-7.
__device__ __forceinline__ uint32_t lookup4(uint32_t cb_lo, uint32_t cb_hi, uint32_t sel) {
  return __byte_perm(cb_lo, cb_hi, sel);
}

// x >> 16 as the high word of x * 2^16: a multiply-high runs on the
// integer multiply-add pipe, which the decode leaves mostly idle, instead of
// the shift/logic pipe that its masks and byte permutes keep busy.
__device__ __forceinline__ uint32_t upper_half(uint32_t x) {
  uint32_t r;
  asm("mul.hi.u32 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0x10000u));
  return r;
}

// Decode one group (three 32-bit words) of a row into 32 E4M3 bytes
// (8 TMEM columns):
// v[0..7] = E4M3 bytes of codes 0..31, four per column.
__device__ __forceinline__ void decode_group(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t cb_lo,
                                             uint32_t cb_hi, uint32_t* v) {
  const uint32_t s0 = spread_codes8(w0);
  const uint32_t s1 = spread_codes8(__funnelshift_r(w0, w1, 24));
  const uint32_t s2 = spread_codes8(__funnelshift_r(w1, w2, 16));
  const uint32_t s3 = spread_codes8(w2 >> 8);
  v[0] = lookup4(cb_lo, cb_hi, s0);
  v[1] = lookup4(cb_lo, cb_hi, upper_half(s0));
  v[2] = lookup4(cb_lo, cb_hi, s1);
  v[3] = lookup4(cb_lo, cb_hi, upper_half(s1));
  v[4] = lookup4(cb_lo, cb_hi, s2);
  v[5] = lookup4(cb_lo, cb_hi, upper_half(s2));
  v[6] = lookup4(cb_lo, cb_hi, s3);
  v[7] = lookup4(cb_lo, cb_hi, upper_half(s3));
}

// Two-bit codes (the draft head's format: code j of a 32-weight group at bits
// 2j..2j+1 of its 64-bit little-endian group).  Spread the 8 codes in bits
// 0..15 of f (bits 16..31 ignored) so that code j lands in nibble j (bits
// 4j, 4j+1; bits 4j+2, 4j+3 clear): three steps that each move the upper
// half of every field up by half the field's width, with a mask and a
// multiply-add (no two moved pieces overlap, so the adds carry nothing).
__device__ __forceinline__ uint32_t spread_codes2x8(uint32_t f) {
  uint32_t h = f & 0x0000FFFFu;
  h += (h & 0x0000FF00u) * 255u;                  // codes 4-7 up by 8 bits
  h += (h & 0x00F000F0u) * 15u;                   // codes 2, 3 and 6, 7 up by 4
  h += (h & 0x0C0C0C0Cu) * 3u;                    // odd codes up by 2
  return h;
}

// Decode one two-bit group (two 32-bit words, 32 codes) into 32 E4M3 bytes
// through the row's 4-entry codebook (one register): v[0..7] = the bytes of
// codes 0..31, four per column.
__device__ __forceinline__ void decode_group2(uint32_t w0, uint32_t w1, uint32_t cb, uint32_t* v) {
  const uint32_t s0 = spread_codes2x8(w0), s1 = spread_codes2x8(w0 >> 16);
  const uint32_t s2 = spread_codes2x8(w1), s3 = spread_codes2x8(w1 >> 16);
  v[0] = __byte_perm(cb, cb, s0);
  v[1] = __byte_perm(cb, cb, upper_half(s0));
  v[2] = __byte_perm(cb, cb, s1);
  v[3] = __byte_perm(cb, cb, upper_half(s1));
  v[4] = __byte_perm(cb, cb, s2);
  v[5] = __byte_perm(cb, cb, upper_half(s2));
  v[6] = __byte_perm(cb, cb, s3);
  v[7] = __byte_perm(cb, cb, upper_half(s3));
}

// E8M0 byte -> fp32 2^(s-127) (s = 0 gives the subnormal 2^-127).
__device__ __forceinline__ float e8m0_to_f32(uint32_t s) {
  return s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}

// Byte q (0..3, a compile-time constant after unrolling) of a word of four
// E8M0 scales -> fp32 2^(s-127): the byte is moved into the exponent field;
// s = 0 leaves the field empty and the unsigned max turns it into the
// subnormal 2^-127 (every other s gives a larger bit pattern).
__device__ __forceinline__ float e8m0_word_byte_to_f32(uint32_t word, int q) {
  const uint32_t e = (q < 3 ? (word << (23 - 8 * q)) : (word >> 1)) & 0x7F800000u;
  return __uint_as_float(max(e, 0x00400000u));
}

// Twenty-four bits of a group starting at bit 24*t: codes 8t..8t+7.  The
// group's three 32-bit words are w0, w1, w2.
__device__ __forceinline__ uint32_t group_field(uint32_t w0, uint32_t w1, uint32_t w2, int t) {
  switch (t) {
    case 0: return w0;
    case 1: return __funnelshift_r(w0, w1, 24);
    case 2: return __funnelshift_r(w1, w2, 16);
    default: return w2 >> 8;
  }
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers, TMA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the async (TMA / tensor-core) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of an mbarrier phase (try_wait may block the thread for a
// system-dependent time; test_wait returns at once).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Same, but the thread may be suspended (up to `hint_ns`) until the phase
// completes instead of returning at once: a waiting warp then takes no issue
// slots from the warps that do the work.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}


// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 32-bit load with acquire semantics at GPU scope.
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Add with release and acquire semantics at GPU scope: the caller's earlier
// writes -- and, after a CTA barrier, those of the threads that took part in
// it -- are visible to whoever acquires the new value; writes released by
// the earlier adders are visible to the caller (and, after a barrier, to the
// CTA).  Returns the old value.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their writes are visible / let dependent grids start.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0),
// completing `bytes` transaction bytes on `bar`.
// The packed weights are read once per call: their bulk copies carry an L2
// evict-first policy, so the stream does not push the kernel's instructions,
// the activations and the scratch out of L2 (cold instruction fetches at the
// start of a call queue behind the weight stream otherwise).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Code stream layout: rows in tiles of 128 (the last tile holds the
// remaining rows); tile t starts at byte 128 t (3K/8); inside a tile the
// 48-byte k-tile pieces (4 groups, 128 weights) of all its rows form one
// block per k-tile: block c at c * rows_t * 48, row i at i * 48.  K % 128 == 0.
__host__ __device__ __forceinline__ long long tile_base(int t, int K) {
  return static_cast<long long>(t) * 128 * (3LL * K / 8);
}
__host__ __device__ __forceinline__ int tile_rows(int t, int N) {
  return N - 128 * t < 128 ? N - 128 * t : 128;
}

// Named barrier over `nthreads` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

// ---------------------------------------------------------------------------
// Warp-level FP8 MMA: D(16x8 f32) = A(16x32 e4m3, row) * B(32x8 e4m3, col) + C.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_e4m3_16832(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f), "f"(0.f), "f"(0.f),
        "f"(0.f));
}


// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core, accumulators in tensor memory).
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor for tcgen05.mma, K-major, no swizzle:
// core matrices of 8 rows x 16 bytes (128 contiguous bytes); `lbo` = byte
// distance between core matrices adjacent along K, `sbo` = byte distance
// between core matrices adjacent along M/N.  Bits: start>>4 [0,14),
// lbo>>4 [16,30), sbo>>4 [32,46), version 1 at [46,48), swizzle 0 at [61,64).
__device__ __forceinline__ uint64_t umma_desc_kmajor(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Same for a K-major operand stored with the 128-byte swizzle (what a TMA
// load with CU_TENSOR_MAP_SWIZZLE_128B writes): rows of 128 bytes, the 16-byte
// chunk j of row r at chunk j ^ (r % 8), 8-row atoms of 1024 bytes (1024-byte
// aligned); sbo = 1024, layout type 2 at [61,64).  An MMA reading K bytes
// [32 i, 32 i + 32) of the atom starts at atom + 32 i.
__device__ __forceinline__ uint64_t umma_desc_kmajor_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor of a block-scaled kind::mxf8f6f4 MMA with E4M3 A
// and B (both K-major), E8M0 scale factors, M = 128 and N = n (multiple of
// 16, <= 256); a_sf_id / b_sf_id pick the scale byte inside a 32-bit TMEM
// column.  Bits: b_sf_id [4,6), a/b format [7,10)/[10,13) (E4M3 = 0),
// N>>3 [17,23), scale type [23] (1 = E8M0), M>>4 [24,29), a_sf_id [29,31).
__host__ __device__ constexpr uint32_t umma_idesc_mxf8(int n, int a_sf_id, int b_sf_id) {
  return (uint32_t(b_sf_id & 3) << 4) | (uint32_t(n >> 3) << 17) | (1u << 23) |
         (uint32_t(128 >> 4) << 24) | (uint32_t(a_sf_id & 3) << 29);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D(tmem) (+)= A(smem) x B(smem)^T with per-32-K block scales from tmem.
__device__ __forceinline__ void umma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Same with A read from tensor memory: row m of A in lane m, K along the
// columns, 4 E4M3 values per 32-bit column (K = 32 -> 8 columns).
__device__ __forceinline__ void umma_mxf8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], [%1], %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Copy a 128-row x 16-byte matrix from shared memory (described like an MMA
// operand: 8-row x 16-byte core matrices, `sdesc`) into 4 TMEM columns of all
// 128 lanes (row r -> lane r).  Asynchronous, in order with this thread's MMAs.
__device__ __forceinline__ void tmem_cp_128x128b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x128b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Arrive (once) on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_st_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_st_x4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
               "r"(v2), "r"(v3)
               : "memory");
}
// 32 consecutive columns of the warp's lane quadrant, one lane per thread.
__device__ __forceinline__ void tmem_st_x32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
      "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
      "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
        "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---- clusters / distributed shared memory --------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t raddr, float a, float b, float c, float d) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(raddr), "f"(a), "f"(b), "f"(c), "f"(d)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t raddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(raddr) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same with a suspend-time hint (ns): the waiting thread may sleep in the
// barrier instead of polling.
__device__ __forceinline__ bool mbar_try_wait_cluster_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

}  // namespace cbq
