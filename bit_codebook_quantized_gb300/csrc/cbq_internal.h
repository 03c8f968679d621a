// cbq_internal.h -- host-side glue between the C entry points (cbq_api.cu)
// and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/cbq.h"

namespace cbq {

// Kernel parameters of the small-M kernel (dense and grouped).
struct GemvParams {
  const uint8_t* codes;       // code stream (tile order), expert stack for grouped calls
  const uint8_t* a;           // [M][K] E4M3
  const float* a_scale;       // [M]
  const uint8_t* scales;      // [rows][K/32]
  const uint8_t* codebooks;   // [rows][8]
  float* y;                   // dense [M][N]; grouped [M][topk][N]
  const int32_t* topk_idx;    // grouped only: [M][topk]
  int M, N, K;
  int E, topk;                // grouped only
  long long wait_ns;          // bounded waits give up after this many ns
};

// Kernel parameters of the tcgen05 kernel (dense and grouped).
struct UmmaParams {
  CUtensorMap a_map;          // activations a[M][K]: box of ntok rows x 128 B (one k-tile), 128-byte swizzle
  const uint8_t* codes;       // code stream (tile order), expert stack for grouped calls
  const uint8_t* a;
  const float* a_scale;
  const uint8_t* scales;
  const uint8_t* codebooks;
  float* y;
  const int32_t* topk_idx;
  int M, N, K;
  int E, topk;
  int ksplit;                 // K-range split factor (cluster size along K)
  int b_bytes;                // shared bytes of the resident activation tile
  int red_bytes;              // shared bytes of the split-K partial tiles (leader CTA)
  int code_stages;            // depth of the code-stage ring (<= kMaxCodeStages)
  long long wait_ns;          // bounded waits give up after this many ns
};

// Kernel parameters of the stream-K kernel (dense calls, cbq_sk.cu).
struct SkParams {
  CUtensorMap a_map;          // activations a[M][K]: box of ntok rows x 128 B, 128-byte swizzle
  const uint8_t* codes;       // code stream (tile order)
  const uint8_t* a;           // [M][K] E4M3
  const float* a_scale;       // [M]
  const uint8_t* scales;      // [N][K/32]
  const uint8_t* codebooks;   // [N][8]
  float* y;                   // [M][N]
  float* partial;             // workspace: 2 x grid partial tiles of 128 x NTOK fp32
  unsigned* counters;         // workspace: one arrival counter per 128-row tile, zero between calls
  long long wait_ns;          // bounded waits give up after this many ns
  float* h;                   // gate-up only: workspace products h [M][F] fp32
  unsigned* h_amax;           // gate-up only: workspace running max |h| per token (fp32 bits)
  unsigned* h_done;           // gate-up only: workspace count of CTAs whose products are written
  uint8_t* q;                 // gate-up only: E4M3 products [M][F] out
  float* q_scale;             // gate-up only: per-token scales [M] out
  int fuse_quant;             // gate-up only: the last CTA quantises (else a second kernel does)
  int M, N, K;
  int F;                      // gate-up only: features, N / 2
  int stages;                 // depth of the code-stage ring
  int b_ktiles;               // k-tiles of resident activations
  const int32_t* topk_idx;    // grouped only: [M][topk] expert ids; codes/scales/codebooks stack E experts
  int E, topk;                // grouped only
};

// cuTensorMapEncodeTiled from the driver (nullptr if unavailable).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();
// Activations a[M][K] (E4M3 bytes, row-major) as a TMA tensor whose box is one
// 128-byte k-tile of `ntok` token rows, landed with the 128-byte swizzle (rows
// past M read as zeros).  The map depends on (a, M, K, ntok) only, so the
// calling thread keeps the last maps it encoded.  CBQ_OK or CBQ_ECUDA.
int encode_activation_map(CUtensorMap* out, const uint8_t* a, int M, int K, int ntok);

int device_sm_count();
void note_launch();
long long wait_limit_ns();   // current bound of the kernels' mbarrier waits (cbq_set_wait_limit)

int launch_gemv(const GemvParams& p, bool grouped, cudaStream_t stream);
int launch_unpack(const uint8_t* codes, const uint8_t* scales, const uint8_t* codebooks, int N,
                  int K, float* W, cudaStream_t stream);
unsigned take_status_gemv(cudaStream_t stream);

int launch_umma(const UmmaParams& p, bool grouped, cudaStream_t stream);
unsigned take_status_umma(cudaStream_t stream);

bool sk_applicable(int M, int N, int K);
size_t sk_workspace_bytes(int M, int N, int K);   // 0 if the stream-K kernel cannot take the shape
// bits: 3 (the 3.25-bit weights) or 2 (the two-bit draft head: 4-entry
// codebooks [N][4], 8 code bytes per group)
int launch_sk(const SkParams& p, void* workspace, size_t workspace_bytes, cudaStream_t stream, int bits = 3);
int launch_sk_static(const SkParams& p, cudaStream_t stream);
size_t sk_gate_up_workspace_bytes(int M, int F, int K);   // 0 if the kernel cannot take the shape
int launch_sk_gate_up(const SkParams& p, void* workspace, size_t workspace_bytes, uint8_t* q, float* q_scale,
                      cudaStream_t stream);
size_t sk_grouped_workspace_bytes(int E, int topk, int M, int N, int K);   // 0 if the kernel cannot take it
int launch_sk_grouped(const SkParams& p, void* workspace, size_t workspace_bytes, cudaStream_t stream);
unsigned take_status_sk(cudaStream_t stream);

// Two-bit draft head (cbq_head.cu): the 16-row shortlist of every token from
// its 2-bit scores [M][N], the FP8 rescoring and the pick.  cand: scratch of
// M x (row chunks) x 16 words.
constexpr int kHeadShortlist = 16;
constexpr int kHeadChunkRows = 1024;
constexpr int kHeadMaxChunks = 256;
constexpr int kHeadMaxRows = kHeadChunkRows * kHeadMaxChunks;   // 262144 vocabulary rows
int head_chunks(int N);                 // number of 1024-row chunks
int launch_head_select(const float* scores, int M, int N, int K, const uint8_t* a, const float* a_scale,
                       const uint8_t* head8, const float* row_scale, uint64_t* cand, int32_t* rows, float* logits,
                       int32_t* pick, cudaStream_t stream);

// Host quantiser (cbq_pack.cpp).
int pack_host(const float* W, int N, int K, uint8_t* codes, uint8_t* scales,
              uint8_t* codebooks);

}  // namespace cbq
