/*
 * cbq.h -- C ABI of the 3.25-bit codebook-quantised matmul library (libcbq).
 *
 * Method: "Hibana: Fast Agentic Inference on Unified-Memory Devices",
 * section "Model surgery / Three-bit weights": every group of 32 weights is a
 * 3-bit index into an 8-entry FP8 codebook plus one 8-bit scale per group,
 * 3 + 8/32 = 3.25 bits per weight; the matmul turns each code into its FP8
 * codebook value on the fly and multiplies on the FP8 tensor cores.  Section "Adaptive speculation / Expert sharing": a
 * speculative-verify round of a mixture-of-experts layer reads only the
 * experts its tokens route to.
 *
 * Packed format (fixed by this library; the pages leave it open):
 *   codes     uint8 [3KN/8]  one group (row n, g = k/32) is 12 bytes, a
 *             96-bit little-endian number with code j = k%32 at bits
 *             3j..3j+2.  Groups are ordered in tiles of 128 rows (the last
 *             tile holds the remaining R rows): tile t starts at byte
 *             128*t*(3K/8); inside it, k-tile c (four groups, k in
 *             [128c, 128c+128)) is a block of R rows x 48 bytes at c*R*48,
 *             row n%128 at (n%128)*48, group g%4 at (g%4)*12.  A tile's
 *             consecutive k-tiles are therefore contiguous bytes.
 *   scales    uint8 [rows][K/32]  E8M0: value 2^(s-127); 255 (NaN) not allowed.
 *   codebooks uint8 [rows][8]     OCP FP8 E4M3 ("fn"), one codebook per row.
 *   w[n,k] = E4M3(codebooks[n][code(n,k)]) * 2^(scales[n][k/32] - 127)
 *
 * Matmul: activations a uint8 E4M3 [M][K] row-major, a_scale fp32 [M],
 *   y[m,n] = a_scale[m] * sum_k E4M3(a[m,k]) * w[n,k]   (fp32 out [M][N]),
 *   accumulated in fp32 on tensor cores; the summation order is free, so
 *   results agree with an exact evaluation within 1e-3*a_scale*sum|a*w| + 1e-6.
 *
 * Conventions for every entry point:
 *   - the caller owns every buffer; no entry point allocates device memory
 *     (the fastest dense path takes scratch from a caller-owned workspace,
 *     see cbq_gemm_ws; cbq_gemm_noalloc uses a fixed static buffer of the
 *     library instead);
 *   - device pointers must be 16-byte aligned (cudaMalloc gives 256);
 *   - calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream) and never synchronise the host;
 *   - the return value is CBQ_OK or a negative CBQ_E* code; on an argument
 *     error nothing is launched; nothing throws across the ABI;
 *   - requires an sm_103 (GB300) or sm_100 class GPU; K % 128 == 0;
 *   - the stream-K kernel (every call that takes a workspace and runs it)
 *     is launched as a programmatic dependent of the previous kernel on
 *     `stream`: it may start streaming the packed weights before that kernel
 *     has finished, and reads activations, routing and scratch or writes
 *     outputs only after it has; so the packed weights must not be written
 *     by the kernel launched just before the call on the same stream (copies
 *     and host writes are fine).
 */
#ifndef CBQ_H
#define CBQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CBQ_OK 0
#define CBQ_EINVAL (-1)      /* bad argument: null/misaligned pointer, bad size */
#define CBQ_ECUDA (-2)       /* a CUDA runtime/driver call failed */
#define CBQ_EDEVICE (-3)     /* no supported GPU on the current device */
#define CBQ_ETIMEOUT (-4)    /* a kernel gave up waiting (see cbq_device_status) */
#define CBQ_EROUTING (-5)    /* grouped call: an expert id outside [0,E) or a
                                token listing one expert twice was seen */

/* Which kernel cbq_gemm_path / cbq_grouped_gemm_ws runs. */
#define CBQ_PATH_AUTO 0      /* dense: see cbq_gemm_auto_path; grouped:
                                M <= 4 GEMV, else the tile kernel */
#define CBQ_PATH_GEMV 1      /* register-decode + warp MMA kernel, any M <= 64 */
#define CBQ_PATH_MMA 2       /* tcgen05 block-scaled FP8 tile kernel (K split
                                over a cluster), any M <= 64 */
#define CBQ_PATH_STREAMK 3   /* tcgen05 kernel with an equal contiguous share
                                of the weights per SM; needs ntok(M) *
                                min(K/128, share) * 128 bytes of activations
                                to fit next to a 2-stage ring (ntok =
                                16/32/64), and a caller workspace of
                                cbq_gemm_workspace_size (dense) or
                                cbq_grouped_workspace_size (grouped) bytes,
                                else CBQ_EINVAL */

/* One packed matrix in device memory (all three arrays 16-byte aligned). */
typedef struct cbq_weight {
    const uint8_t *codes;      /* [3K*rows/8], tile order */
    const uint8_t *scales;     /* [rows][K/32]  */
    const uint8_t *codebooks;  /* [rows][8]     */
} cbq_weight_t;

/* Byte sizes of the three packed arrays for an N x K matrix:
 * 3KN/8, KN/32 and 8N (3.25 bits per weight plus an 8-byte codebook per row,
 * section "Model surgery / Three-bit weights").  Any pointer may be NULL.
 * Errors: CBQ_EINVAL if N < 0, K < 0 or K % 128 != 0. */
int cbq_packed_sizes(int32_t N, int32_t K, size_t *codes_bytes,
                     size_t *scales_bytes, size_t *codebook_bytes);

/* Quantise fp32 weights W (HOST, [N][K] row-major) into the packed format
 * (HOST outputs, sized by cbq_packed_sizes).  Runs on the calling thread, is
 * deterministic, and implements the rule this library fixes for choosing the
 * codebooks and codes (the pages do not give one):
 *   1. per group of 32: s = clamp(127 + ceil(log2 max|w|), 0, 254), 127 if all
 *      zero, so |w| / 2^(s-127) <= 1;
 *   2. u = w / 2^(s-127);
 *   3. per row, 1-D Lloyd with 8 centroids over u: start at the sorted values
 *      at index floor((i+0.5)K/8); 16 rounds of nearest assignment (ties to the
 *      lower index) and mean update in k order (empty clusters keep theirs);
 *   4. round centroids to E4M3 (nearest, ties to even, saturate at 448), sort;
 *   5. code = nearest rounded centroid (ties to the lower index).
 * Not on the matmul path (weights are packed once, offline).
 * Errors: CBQ_EINVAL on NULL pointers, N < 0, K <= 0 or K % 128 != 0, or a
 * non-finite weight. */
int cbq_pack(const float *W, int32_t N, int32_t K, uint8_t *codes,
             uint8_t *scales, uint8_t *codebooks);

/* Decode a packed matrix to fp32 W_out (DEVICE, [N][K]); every value is exact
 * (an E4M3 value times a power of two).  One kernel launch on `stream`.
 * Errors: CBQ_EINVAL (null/misaligned pointer, N < 0, K % 128 != 0),
 * CBQ_EDEVICE, CBQ_ECUDA. */
int cbq_unpack(const cbq_weight_t *w, int32_t N, int32_t K, float *W_out,
               void *stream);

/* y[M][N] = a_scale * (a[M][K] x W^T): the decode-step / verify-round matmul
 * against packed weights.  a, a_scale, y and w's arrays are DEVICE pointers.
 * 1 <= M <= 64 (M == 0 or N == 0 is a no-op); N >= 0; K % 128 == 0 (K == 0
 * writes y = 0).  Picks among the kernels that need no scratch memory
 * (cbq_gemm_auto_path(M, N, K, 0)); one launch, no allocation.  For the
 * fastest kernel on most shapes pass a workspace to cbq_gemm_ws.
 * Errors: CBQ_EINVAL, CBQ_EDEVICE, CBQ_ECUDA. */
int cbq_gemm(const uint8_t *a, const float *a_scale, const cbq_weight_t *w,
             int32_t M, int32_t N, int32_t K, float *y, void *stream);

/* Bytes of the workspace cbq_gemm_ws needs for an M x N x K call (0 when
 * no kernel that uses one takes the shape; cbq_gemm_ws then needs none).
 * Host only.  Errors: CBQ_EINVAL (NULL `bytes`, sizes cbq_gemm rejects). */
int cbq_gemm_workspace_size(int32_t M, int32_t N, int32_t K, size_t *bytes);

/* cbq_gemm with a caller-owned DEVICE workspace (256-byte aligned, at least
 * cbq_gemm_workspace_size bytes; NULL/0 = none, which is cbq_gemm).  With it
 * the stream-K kernel runs where it fits: every SM streams an equal contiguous
 * share of the packed weights and a 128-row tile split between SMs is summed
 * through the workspace, in a fixed order (the result is deterministic).
 * The workspace starts with a fixed area (the first 262 656 bytes = 256.5 KB,
 * the same for every shape: tile counters, and the gate-up step's per-token
 * maxima and finished-CTA count); that area must be zero-filled before the
 * workspace's first use (cudaMemset) and every call leaves it zero again, so
 * one workspace serves calls of any shape in turn.  Calls that share one workspace must not run at
 * the same time (one workspace per stream).  The stream-K kernel is launched
 * as a programmatic dependent of the previous kernel on `stream`: it may
 * start streaming the packed weights before that kernel has finished (a,
 * a_scale, y and the workspace are touched only after it has), so the weights
 * must not be written by the kernel launched just before it on the same
 * stream (copies and host writes are fine).
 * Errors: CBQ_EINVAL (also a workspace that is misaligned or too small for
 * the kernel chosen), CBQ_EDEVICE, CBQ_ECUDA. */
int cbq_gemm_ws(const uint8_t *a, const float *a_scale, const cbq_weight_t *w,
                int32_t M, int32_t N, int32_t K, float *y, void *workspace,
                size_t workspace_bytes, void *stream);

/* Fused gate-up projection of a feed-forward layer, for the verify round
 * ("Adaptive speculation": the drafted tokens run through the model's FFN):
 * the packed weight has N = 2F rows in blocks of 64 features -- block b is
 * rows [128 b, 128 b + 2 R) with R = min(64, F - 64 b): its R gate rows, then
 * its R up rows -- so a 128-row tile pairs each gate row with its up row.
 * With g, u the matmul outputs of a feature's gate and up rows (a_scale
 * applied, fp32 accumulation), the call writes
 *   h_scale[m] = max_f |SiLU(g[m,f]) * u[m,f]| / 448   (1 if that max is 0),
 *   h[m][f]    = E4M3(SiLU(g) * u / h_scale[m])  (nearest, ties to even,
 *                saturating at +-448; SiLU(x) = x / (1 + e^-x)),
 * the activations and per-token scale the down projection takes.
 *   a, a_scale, w  as for cbq_gemm (w: 2F rows); 1 <= M <= 64, F >= 1
 *   h        DEVICE uint8 [M][F] out, E4M3
 *   h_scale  DEVICE fp32 [M] out
 *   workspace, workspace_bytes: as for cbq_gemm_ws, at least
 *            cbq_gate_up_workspace_size bytes (it also holds h in fp32)
 * One launch on `stream` up to M * F = 8192 products (the stream-K matmul
 * with the SiLU-product epilogue; the CTA that finishes last quantises every
 * product), else two (the matmul's last CTA writes the per-token scales,
 * and a quantisation kernel over chunks of 2048 products per token follows);
 * each a programmatic dependent of the kernel before it.
 * Errors: CBQ_EINVAL (also when the stream-K kernel cannot take the shape:
 * the size query then gives 0), CBQ_EDEVICE, CBQ_ECUDA. */
int cbq_gemm_gate_up(const uint8_t *a, const float *a_scale, const cbq_weight_t *w,
                     int32_t M, int32_t F, int32_t K, uint8_t *h, float *h_scale,
                     void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of the workspace cbq_gemm_gate_up needs (0 if it cannot take the
 * shape).  Host only.  Errors: CBQ_EINVAL. */
int cbq_gate_up_workspace_size(int32_t M, int32_t F, int32_t K, size_t *bytes);

/* The kernel (CBQ_PATH_GEMV / _MMA / _STREAMK) that cbq_gemm_ws picks for an
 * M x N x K call with (with_workspace != 0) or without a workspace, chosen by
 * measured speed on GB300; CBQ_EINVAL for sizes cbq_gemm rejects.  (If the
 * tile kernel's activations do not fit in shared memory, the call then runs
 * the GEMV kernel instead of CBQ_PATH_MMA.)  Host only: no device access. */
int cbq_gemm_auto_path(int32_t M, int32_t N, int32_t K, int32_t with_workspace);

/* Same as cbq_gemm_ws with an explicit kernel choice (CBQ_PATH_*); used by
 * the tests and the benchmark to exercise each kernel at every M.
 * CBQ_PATH_STREAMK needs the workspace. */
int cbq_gemm_path(const uint8_t *a, const float *a_scale, const cbq_weight_t *w,
                  int32_t M, int32_t N, int32_t K, float *y, void *workspace,
                  size_t workspace_bytes, void *stream, int32_t path);

/* The stream-K matmul (CBQ_PATH_STREAMK) with no allocation at all and no
 * workspace argument, for callers that can neither allocate device memory
 * nor hold a workspace of their own: its scratch (fp32 partial tiles and
 * per-tile arrival counters) is a fixed static device buffer of the library
 * (10.5 MB of partials for up to 160 SMs at 64 token columns, 65536 tile
 * counters, i.e. N <= 8388608), which every GPU that loads the library holds
 * until the process exits.  The pages have no counterpart: this is a
 * deployment variant of the same kernel.
 * The first call on a device looks up the buffer's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  Each call first clears the counters of the
 * tiles it uses (one cudaMemsetAsync on `stream`, no allocation), then
 * launches the kernel.  The buffer is shared by every call on the device and
 * keeps the last call's contents: two calls that may run at the same time
 * (different streams, overlapping graph replays) race on it and give wrong
 * results; serialise them.
 * Errors: CBQ_EINVAL (bad argument, K == 0, or a problem the stream-K kernel
 * or the static buffer cannot take), CBQ_EDEVICE, CBQ_ECUDA. */
int cbq_gemm_noalloc(const uint8_t *a, const float *a_scale, const cbq_weight_t *w,
                     int32_t M, int32_t N, int32_t K, float *y, void *stream);

/* Mixture-of-experts verify round ("Adaptive speculation / Expert sharing"):
 * the E experts' packed matrices are stacked in ONE cbq_weight_t (expert e:
 * codes from byte e*3KN/8, scales and codebooks from row e*N) rather than
 * passed as an array of E separate matrices, so the one kernel launch finds
 * every expert from a single set of base pointers; topk_idx is DEVICE int32
 * [M][topk] and
 *   y[t][j][:] = a_scale[t] * a[t] x W_{topk_idx[t][j]}^T   (fp32 [M][topk][N]),
 * with no gate weight and no combine.  Only experts that appear in topk_idx
 * are read from memory.  Picks the kernel by M (GEMV up to 4 token rows, the
 * tile kernel beyond, the GEMV kernel again where every token's activations
 * do not fit the tile kernel's shared memory).  The routing is read on the device inside the one
 * kernel launch.  1 <= M <= 64, 1 <= topk <= 8, 1 <= E <= 4096, each row of
 * topk_idx must list distinct experts in [0, E); a violation seen on the
 * device is reported by cbq_device_status as CBQ_EROUTING.
 * Errors: CBQ_EINVAL, CBQ_EDEVICE, CBQ_ECUDA. */
int cbq_grouped_gemm(const uint8_t *a, const float *a_scale,
                     const cbq_weight_t *experts, int32_t E,
                     const int32_t *topk_idx, int32_t topk, int32_t M,
                     int32_t N, int32_t K, float *y, void *stream);

/* Same as cbq_grouped_gemm with an explicit kernel choice (CBQ_PATH_GEMV or
 * CBQ_PATH_MMA; CBQ_PATH_STREAMK needs a workspace: cbq_grouped_gemm_ws). */
int cbq_grouped_gemm_path(const uint8_t *a, const float *a_scale,
                          const cbq_weight_t *experts, int32_t E,
                          const int32_t *topk_idx, int32_t topk, int32_t M,
                          int32_t N, int32_t K, float *y, void *stream,
                          int32_t path);

/* Workspace of a grouped stream-K call: bytes for (E, topk, M, N, K), 0 if
 * the stream-K kernel cannot take the shape.  Arguments as in
 * cbq_grouped_gemm.  Errors: CBQ_EINVAL. */
int cbq_grouped_workspace_size(int32_t E, int32_t topk, int32_t M, int32_t N,
                               int32_t K, size_t *bytes);

/* cbq_grouped_gemm with a caller-owned DEVICE workspace (the same layout and
 * rules as cbq_gemm_ws's: 256-byte aligned, at least
 * cbq_grouped_workspace_size bytes, its first 256.5 KB zero-filled once before
 * first use, one call at a time) and a kernel choice.  CBQ_PATH_STREAMK runs
 * the stream-K kernel (CBQ_PATH_AUTO picks as cbq_grouped_gemm does):
 * every SM takes an equal contiguous share of the (used expert, tile,
 * k-tile) units of the experts the routing names -- each used expert
 * multiplied by all M token rows, only the routed (token, slot) outputs
 * written.  workspace may be NULL for the other paths.  No allocation.
 * Errors: CBQ_EINVAL, CBQ_EDEVICE, CBQ_ECUDA; routing errors as in
 * cbq_grouped_gemm (reported by cbq_device_status). */
int cbq_grouped_gemm_ws(const uint8_t *a, const float *a_scale,
                        const cbq_weight_t *experts, int32_t E,
                        const int32_t *topk_idx, int32_t topk, int32_t M,
                        int32_t N, int32_t K, float *y, void *workspace,
                        size_t workspace_bytes, void *stream, int32_t path);

/* ---- Two-bit draft head ("Hibana: Fast Agentic Inference on Unified-Memory
 * Devices", section "Model surgery / Two-bit draft head"): the drafter's
 * vocabulary head scores every token from a 2-bit copy of its weights, keeps
 * a shortlist of 16 and rescores only those with the FP8 head.
 *
 * The 2-bit head (this library's reading; the pages fix no format): per row
 * a 4-entry E4M3 codebook, 2-bit codes (code j of a 32-weight group at bits
 * 2j..2j+1 of its 64-bit little-endian group), one E8M0 scale per group;
 * groups in the same tile order as the 3-bit codes with 32 bytes per row and
 * 128-wide k-tile (8 bytes per group): 2 + 8/32 = 2.25 bits per weight.  A
 * cbq_weight_t describes it: codes KN/4 bytes, scales [N][K/32],
 * codebooks [N][4].  The FP8 head: head8 DEVICE uint8 E4M3 [N][K] row-major
 * (16-byte aligned) with row_scale DEVICE fp32 [N]. */

/* Byte sizes of a 2-bit head's codes, scales and codebooks.  Host only.
 * Errors: CBQ_EINVAL (K not a multiple of 128, NULL outputs). */
int cbq_head2_sizes(int32_t N, int32_t K, size_t *codes_bytes,
                    size_t *scales_bytes, size_t *codebook_bytes);

/* 2-bit scores s[m][n] = a_scale[m] * sum_k a[m,k] w2[n,k] (fp32 out,
 * DEVICE [M][N]) on the stream-K kernel; the workspace is as for
 * cbq_gemm_ws, at least cbq_gemm_workspace_size(M, N, K) bytes (required).
 * Errors: CBQ_EINVAL (also when the stream-K kernel cannot take the shape),
 * CBQ_EDEVICE, CBQ_ECUDA. */
int cbq_gemm2_ws(const uint8_t *a, const float *a_scale, const cbq_weight_t *head2,
                 int32_t M, int32_t N, int32_t K, float *y, void *workspace,
                 size_t workspace_bytes, void *stream);

/* Workspace of cbq_draft_head (0: the shape cannot be taken).  1 <= M <= 64,
 * 16 <= N <= 262144 (at most 256 chunks of 1024 vocabulary rows), K a
 * positive multiple of 128.  Host only.  Errors: CBQ_EINVAL. */
int cbq_draft_head_workspace_size(int32_t M, int32_t N, int32_t K, size_t *bytes);

/* The draft head's step for M token rows a (E4M3 [M][K], a_scale fp32 [M]):
 *   shortlist DEVICE int32 [M][16]: the 16 rows with the highest 2-bit
 *             scores, descending, equal scores -> lower row first;
 *   logits    DEVICE fp32 [M][16]: their FP8 logits
 *             a_scale[m] * row_scale[n] * sum_k a[m,k] E4M3(head8[n,k]);
 *   pick      DEVICE int32 [M]: the shortlisted row with the highest logit,
 *             equal logits -> the earlier one in the shortlist.
 * The workspace (DEVICE, 256-byte aligned, at least
 * cbq_draft_head_workspace_size bytes; its first 256.5 KB zero-filled once
 * before first use and left zero by every call; one call at a time) holds
 * the stream-K scratch, the scores and the shortlist candidates.  Three
 * launches on `stream` (2-bit scores, the 16 best of every 1024-row chunk,
 * shortlist + rescoring + pick), each a programmatic dependent of the one
 * before.  Shapes as for cbq_draft_head_workspace_size.
 * Errors: CBQ_EINVAL, CBQ_EDEVICE, CBQ_ECUDA. */
int cbq_draft_head(const uint8_t *a, const float *a_scale, const cbq_weight_t *head2,
                   const uint8_t *head8, const float *row_scale, int32_t M,
                   int32_t N, int32_t K, int32_t *shortlist, float *logits,
                   int32_t *pick, void *workspace, size_t workspace_bytes,
                   void *stream);

/* Diagnostic: every kernel launched after this call gives up a bounded wait
 * (for a copy, a tensor-core result or another role of its block) after `ns`
 * nanoseconds instead of the default 2 s, returns early and reports
 * CBQ_ETIMEOUT through cbq_device_status; ns <= 0 restores the default.  A
 * wait that gives up never leaves the block's own copies or tensor-core work
 * behind: those are waited for before the block ends. */
int cbq_set_wait_limit(int64_t ns);

/* Synchronise `stream`, then return and clear the sticky device status of
 * this library on the current device: CBQ_OK, CBQ_ETIMEOUT (a kernel's
 * bounded wait for a copy or a tensor-core op ran out; the kernel returned
 * early and its output is incomplete) or CBQ_EROUTING. */
int cbq_device_status(void *stream);

/* Kernel launches made by this library since load (all entry points). */
uint64_t cbq_launch_count(void);

/* Human-readable text for a status code (static storage). */
const char *cbq_status_str(int status);

/* Shared expert budget of one MoE verify round ("Hibana: Fast Agentic
 * Inference on Unified-Memory Devices", section "Adaptive speculation /
 * Expert sharing"): the round reads only B experts, and a token's choice
 * outside them gives way to the token's best expert inside.  Rule (the page
 * illustrates the idea on a small example only):
 * each token ranks experts by its logit (higher first, ties -> lower id) and
 * takes its own top-k; expert e scores sum_t (k - rank of e in t's top-k);
 * the budget is the B best-scoring experts (ties -> lower id); each token
 * then takes its top-k among the budget.  Logits compare as numbers (-0 and
 * +0 are equal); a NaN logit ranks below every other value, so any input
 * gives k distinct in-budget ids per token.
 *   logits   device fp32 [T][E] router logits
 *   T        tokens of the round, >= 1
 *   E        experts, 1 <= E <= 4096
 *   k        choices per token, 1 <= k <= min(B, 8) (cbq_grouped_gemm takes
 *            at most 8 choices per token)
 *   B        budget, k <= B <= E
 *   budget   device int32 [B] out: the budget's expert ids, ascending
 *   topk_idx device int32 [T][k] out: each token's choices in rank order
 *            (the routing cbq_grouped_gemm takes)
 * One kernel launch on `stream`; CBQ_EINVAL on bad arguments (no launch). */
int cbq_select_budget(const float *logits, int32_t T, int32_t E, int32_t k,
                      int32_t B, int32_t *budget, int32_t *topk_idx,
                      void *stream);

/* Draft length of the next speculative round ("Hibana: Fast Agentic
 * Inference on Unified-Memory Devices", section "Adaptive speculation /
 * Adaptive draft length"): d* = argmax over 1 <= d <= dmax of
 * E[N_d] / T(d), with E[N_d] = sum_{j=0..d} q^j the expected tokens a round
 * yields (the drafted tokens accepted before the first rejection, plus the
 * token the target model produces itself) and T(d) = 1 + c (d - 1)
 * its time relative to d = 1.  The verify round that follows multiplies
 * d* + 1 token rows per request.
 *   q      acceptance probability of a drafted token, in [0, 1]
 *   c      added relative cost of one more draft token, finite and >= 0
 *   dmax   longest draft allowed, 1 <= dmax <= 63 (the verify round of one
 *          request then has at most 64 token rows, the most cbq_gemm takes)
 *   d_star out: the chosen length (ties go to the shorter draft)
 *   expected_tokens, tokens_per_time: out, may be NULL: E[N_d*] and
 *          E[N_d*] / T(d*)
 * Host only (no device work); CBQ_EINVAL on arguments out of range. */
int cbq_draft_length(double q, double c, int32_t dmax, int32_t *d_star,
                     double *expected_tokens, double *tokens_per_time);

#ifdef __cplusplus
}
#endif

#endif /* CBQ_H */
