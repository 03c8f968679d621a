// cbq_api.cu -- the C entry points declared in include/cbq.h: argument
// checks and kernel selection.  All device work is done by the kernels in
// cbq_sk.cu, cbq_gemv.cu, cbq_umma.cu and cbq_budget.cu; this file launches them on the
// caller's stream and never synchronises (except cbq_device_status).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "cbq_budget.h"
#include "cbq_internal.h"

namespace cbq {

namespace {

std::atomic<uint64_t> g_launches{0};
constexpr long long kDefaultWaitNs = 2000000000LL;   // 2 s
std::atomic<long long> g_wait_ns{kDefaultWaitNs};

struct DeviceInfo {
  int sm_count = 0;
  int supported = -1;  // -1 unknown, 0 no, 1 yes
};

constexpr int kMaxDevices = 64;
DeviceInfo g_devices[kMaxDevices];
std::mutex g_dev_mutex;

int current_device_checked(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CBQ_EDEVICE;
  std::lock_guard<std::mutex> lk(g_dev_mutex);
  DeviceInfo& d = g_devices[dev];
  if (d.supported < 0) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return CBQ_EDEVICE;
    // The kernels are compiled for sm_103a only.
    d.supported = (prop.major == 10 && prop.minor == 3) ? 1 : 0;
    d.sm_count = prop.multiProcessorCount;
  }
  if (!d.supported) return CBQ_EDEVICE;
  if (out) *out = &d;
  return CBQ_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool weight_ok(const cbq_weight_t* w) {
  return w && w->codes && w->scales && w->codebooks && aligned(w->codes, 16) &&
         aligned(w->scales, 16) && aligned(w->codebooks, 16);
}

}  // namespace

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

int encode_activation_map(CUtensorMap* out, const uint8_t* a, int M, int K, int ntok) {
  // the last maps this thread encoded (encoding is host work on every call
  // otherwise); a small direct-mapped table keyed on (a, M, K, ntok)
  struct Entry {
    const uint8_t* a = nullptr;
    int M = 0, K = 0, ntok = 0;
    CUtensorMap map;
  };
  constexpr int kEntries = 16;
  thread_local Entry table[kEntries];
  const uintptr_t h = (reinterpret_cast<uintptr_t>(a) >> 8) ^ static_cast<uintptr_t>(M) * 31u ^
                      static_cast<uintptr_t>(K) * 131u ^ static_cast<uintptr_t>(ntok) * 7u;
  Entry& e = table[h % kEntries];
  if (e.a == a && e.M == M && e.K == K && e.ntok == ntok) {
    *out = e.map;
    return CBQ_OK;
  }
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return CBQ_ECUDA;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(ntok)};
  const cuuint32_t estr[2] = {1, 1};
  if (enc(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return CBQ_ECUDA;
  e.a = a;
  e.M = M;
  e.K = K;
  e.ntok = ntok;
  e.map = *out;
  return CBQ_OK;
}

int device_sm_count() {
  DeviceInfo* d = nullptr;
  if (current_device_checked(&d) != CBQ_OK) return 1;
  return d->sm_count;
}

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

long long wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

}  // namespace cbq

using namespace cbq;

extern "C" {

int cbq_packed_sizes(int32_t N, int32_t K, size_t* codes_bytes, size_t* scales_bytes,
                     size_t* codebook_bytes) {
  if (N < 0 || K < 0 || K % 128 != 0) return CBQ_EINVAL;
  const size_t n = static_cast<size_t>(N), k = static_cast<size_t>(K);
  if (codes_bytes) *codes_bytes = 3 * k * n / 8;
  if (scales_bytes) *scales_bytes = k * n / 32;
  if (codebook_bytes) *codebook_bytes = 8 * n;
  return CBQ_OK;
}

int cbq_pack(const float* W, int32_t N, int32_t K, uint8_t* codes, uint8_t* scales,
             uint8_t* codebooks) {
  if (N < 0 || K <= 0 || K % 128 != 0) return CBQ_EINVAL;
  if (N == 0) return CBQ_OK;
  if (!W || !codes || !scales || !codebooks) return CBQ_EINVAL;
  return pack_host(W, N, K, codes, scales, codebooks);
}

int cbq_unpack(const cbq_weight_t* w, int32_t N, int32_t K, float* W_out, void* stream) {
  if (N < 0 || K < 0 || K % 128 != 0) return CBQ_EINVAL;
  if (N == 0 || K == 0) return CBQ_OK;
  if (!weight_ok(w) || !W_out || !aligned(W_out, 16)) return CBQ_EINVAL;
  int st = current_device_checked(nullptr);
  if (st != CBQ_OK) return st;
  return launch_unpack(w->codes, w->scales, w->codebooks, N, K, W_out,
                       static_cast<cudaStream_t>(stream));
}

int cbq_gemm_auto_path(int32_t M, int32_t N, int32_t K, int32_t with_workspace) {
  if (M < 1 || M > 64 || N < 1 || K < 128 || K % 128 != 0) return CBQ_EINVAL;
  // Measured on GB300 (CUDA graphs of back-to-back calls, weights beyond L2).
  // Up to 8 token rows the GEMV kernel has the least fixed cost per call and
  // wins up to ~32 M weights (2048 x 2048: 3.9 us against 8.9 us for the
  // stream-K kernel; the two meet near 2^25 weights).  Otherwise, with a
  // workspace, the stream-K kernel (equal contiguous weight share per SM)
  // takes every shape it fits.  Without one: up to 8 token rows the GEMV
  // kernel on matrices up to ~64 M weights and the tile kernel beyond; from 9
  // rows the tile kernel.  The tile kernel needs its activations resident;
  // where they do not fit, the GEMV kernel runs (see cbq_gemm_path).
  const long long weights = static_cast<long long>(N) * K;
  if (M <= 8 && weights <= (1LL << 25)) return CBQ_PATH_GEMV;
  if (with_workspace && sk_applicable(M, N, K)) return CBQ_PATH_STREAMK;
  if (M <= 8) return weights <= (1LL << 26) ? CBQ_PATH_GEMV : CBQ_PATH_MMA;
  return CBQ_PATH_MMA;
}

int cbq_gemm_workspace_size(int32_t M, int32_t N, int32_t K, size_t* bytes) {
  if (!bytes || M < 0 || M > 64 || N < 0 || K < 0 || K % 128 != 0) return CBQ_EINVAL;
  *bytes = (M == 0 || N == 0 || K == 0) ? 0 : sk_workspace_bytes(M, N, K);
  return CBQ_OK;
}

int cbq_set_wait_limit(int64_t ns) {
  g_wait_ns.store(ns > 0 ? static_cast<long long>(ns) : kDefaultWaitNs, std::memory_order_relaxed);
  return CBQ_OK;
}

int cbq_gemm_path(const uint8_t* a, const float* a_scale, const cbq_weight_t* w, int32_t M,
                  int32_t N, int32_t K, float* y, void* workspace, size_t workspace_bytes, void* stream,
                  int32_t path) {
  if (M < 0 || M > 64 || N < 0 || K < 0 || K % 128 != 0) return CBQ_EINVAL;
  if (path < CBQ_PATH_AUTO || path > CBQ_PATH_STREAMK) return CBQ_EINVAL;
  if (M == 0 || N == 0) return CBQ_OK;
  if (!y || !aligned(y, 4)) return CBQ_EINVAL;
  int st = current_device_checked(nullptr);
  if (st != CBQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    return cudaMemsetAsync(y, 0, sizeof(float) * size_t(M) * size_t(N), s) == cudaSuccess
               ? CBQ_OK
               : CBQ_ECUDA;
  }
  if (!a || !aligned(a, 16) || !a_scale || !aligned(a_scale, 4) || !weight_ok(w))
    return CBQ_EINVAL;
  const bool automatic = path == CBQ_PATH_AUTO;
  if (automatic) path = cbq_gemm_auto_path(M, N, K, workspace != nullptr);
  if (path == CBQ_PATH_STREAMK) {
    if (!sk_applicable(M, N, K)) return CBQ_EINVAL;
    SkParams p;
    std::memset(&p, 0, sizeof(p));
    p.codes = w->codes;
    p.a = a;
    p.a_scale = a_scale;
    p.scales = w->scales;
    p.codebooks = w->codebooks;
    p.y = y;
    p.M = M;
    p.N = N;
    p.K = K;
    p.wait_ns = wait_limit_ns();
    return launch_sk(p, workspace, workspace_bytes, s);
  }
  if (path == CBQ_PATH_GEMV) {
    GemvParams p;
    std::memset(&p, 0, sizeof(p));
    p.codes = w->codes;
    p.a = a;
    p.a_scale = a_scale;
    p.scales = w->scales;
    p.codebooks = w->codebooks;
    p.y = y;
    p.M = M;
    p.N = N;
    p.K = K;
    p.wait_ns = wait_limit_ns();
    return launch_gemv(p, false, s);
  }
  UmmaParams p;
  std::memset(&p, 0, sizeof(p));
  p.codes = w->codes;
  p.a = a;
  p.a_scale = a_scale;
  p.scales = w->scales;
  p.codebooks = w->codebooks;
  p.y = y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.wait_ns = wait_limit_ns();
  const int r = launch_umma(p, false, s);
  if (r != CBQ_EINVAL || !automatic) return r;
  // the tile kernel's resident activations do not fit either: GEMV kernel
  GemvParams g;
  std::memset(&g, 0, sizeof(g));
  g.codes = w->codes;
  g.a = a;
  g.a_scale = a_scale;
  g.scales = w->scales;
  g.codebooks = w->codebooks;
  g.y = y;
  g.M = M;
  g.N = N;
  g.K = K;
  g.wait_ns = wait_limit_ns();
  return launch_gemv(g, false, s);
}

int cbq_gemm_noalloc(const uint8_t* a, const float* a_scale, const cbq_weight_t* w, int32_t M,
                     int32_t N, int32_t K, float* y, void* stream) {
  if (M < 0 || M > 64 || N < 0 || K < 0 || K % 128 != 0) return CBQ_EINVAL;
  if (M == 0 || N == 0) return CBQ_OK;
  if (K == 0 || !sk_applicable(M, N, K)) return CBQ_EINVAL;
  if (!y || !aligned(y, 4) || !a || !aligned(a, 16) || !a_scale || !aligned(a_scale, 4) || !weight_ok(w))
    return CBQ_EINVAL;
  int st = current_device_checked(nullptr);
  if (st != CBQ_OK) return st;
  SkParams p;
  std::memset(&p, 0, sizeof(p));
  p.codes = w->codes;
  p.a = a;
  p.a_scale = a_scale;
  p.scales = w->scales;
  p.codebooks = w->codebooks;
  p.y = y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.wait_ns = wait_limit_ns();
  return launch_sk_static(p, static_cast<cudaStream_t>(stream));
}

int cbq_gate_up_workspace_size(int32_t M, int32_t F, int32_t K, size_t* bytes) {
  if (!bytes || M < 1 || M > 64 || F < 1 || K < 128 || K % 128 != 0 || static_cast<int64_t>(F) * 2 > INT32_MAX)
    return CBQ_EINVAL;
  *bytes = sk_gate_up_workspace_bytes(M, F, K);
  return CBQ_OK;
}

int cbq_gemm_gate_up(const uint8_t* a, const float* a_scale, const cbq_weight_t* w, int32_t M, int32_t F,
                     int32_t K, uint8_t* h, float* h_scale, void* workspace, size_t workspace_bytes,
                     void* stream) {
  if (M < 1 || M > 64 || F < 1 || K < 128 || K % 128 != 0 || static_cast<int64_t>(F) * 2 > INT32_MAX)
    return CBQ_EINVAL;
  if (!a || !aligned(a, 16) || !a_scale || !aligned(a_scale, 4) || !weight_ok(w) || !h || !h_scale ||
      !aligned(h_scale, 4))
    return CBQ_EINVAL;
  int st = current_device_checked(nullptr);
  if (st != CBQ_OK) return st;
  SkParams p;
  std::memset(&p, 0, sizeof(p));
  p.codes = w->codes;
  p.a = a;
  p.a_scale = a_scale;
  p.scales = w->scales;
  p.codebooks = w->codebooks;
  p.M = M;
  p.N = 2 * F;
  p.K = K;
  p.wait_ns = wait_limit_ns();
  return launch_sk_gate_up(p, workspace, workspace_bytes, h, h_scale, static_cast<cudaStream_t>(stream));
}

int cbq_gemm_ws(const uint8_t* a, const float* a_scale, const cbq_weight_t* w, int32_t M, int32_t N,
                int32_t K, float* y, void* workspace, size_t workspace_bytes, void* stream) {
  return cbq_gemm_path(a, a_scale, w, M, N, K, y, workspace, workspace_bytes, stream, CBQ_PATH_AUTO);
}

int cbq_gemm(const uint8_t* a, const float* a_scale, const cbq_weight_t* w, int32_t M, int32_t N,
             int32_t K, float* y, void* stream) {
  return cbq_gemm_path(a, a_scale, w, M, N, K, y, nullptr, 0, stream, CBQ_PATH_AUTO);
}

int cbq_grouped_workspace_size(int32_t E, int32_t topk, int32_t M, int32_t N, int32_t K, size_t* bytes) {
  if (!bytes || M < 0 || M > 64 || N < 0 || K < 0 || K % 128 != 0 || E < 1 || E > 4096 || topk < 1 || topk > 8 ||
      topk > E)
    return CBQ_EINVAL;
  *bytes = (M == 0 || N == 0 || K == 0) ? 0 : sk_grouped_workspace_bytes(E, topk, M, N, K);
  return CBQ_OK;
}

int cbq_grouped_gemm_ws(const uint8_t* a, const float* a_scale, const cbq_weight_t* experts, int32_t E,
                        const int32_t* topk_idx, int32_t topk, int32_t M, int32_t N, int32_t K, float* y,
                        void* workspace, size_t workspace_bytes, void* stream, int32_t path) {
  if (M < 0 || M > 64 || N < 0 || K < 0 || K % 128 != 0 || E < 1 || E > 4096 || topk < 1 ||
      topk > 8 || topk > E)
    return CBQ_EINVAL;
  if (path < CBQ_PATH_AUTO || path > CBQ_PATH_STREAMK) return CBQ_EINVAL;
  if (M == 0 || N == 0) return CBQ_OK;
  if (!y || !aligned(y, 4) || !topk_idx || !aligned(topk_idx, 4)) return CBQ_EINVAL;
  if (static_cast<int64_t>(E) * N > INT32_MAX) return CBQ_EINVAL;
  int st = current_device_checked(nullptr);
  if (st != CBQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0) {
    return cudaMemsetAsync(y, 0, sizeof(float) * size_t(M) * topk * size_t(N), s) == cudaSuccess
               ? CBQ_OK
               : CBQ_ECUDA;
  }
  if (!a || !aligned(a, 16) || !a_scale || !aligned(a_scale, 4) || !weight_ok(experts))
    return CBQ_EINVAL;
  const bool automatic = path == CBQ_PATH_AUTO;
  // By M: the GEMV kernel up to 4 token rows, the tile kernel beyond.  (The
  // stream-K kernel, taken only when asked for, measured 31.6 us against the
  // tile kernel's 21.9 us on the 128-expert, 64-token round.)
  if (automatic) path = (M <= 4) ? CBQ_PATH_GEMV : CBQ_PATH_MMA;
  if (path == CBQ_PATH_STREAMK) {
    SkParams p;
    std::memset(&p, 0, sizeof(p));
    p.codes = experts->codes;
    p.a = a;
    p.a_scale = a_scale;
    p.scales = experts->scales;
    p.codebooks = experts->codebooks;
    p.y = y;
    p.topk_idx = topk_idx;
    p.M = M;
    p.N = N;
    p.K = K;
    p.E = E;
    p.topk = topk;
    p.wait_ns = wait_limit_ns();
    return launch_sk_grouped(p, workspace, workspace_bytes, s);
  }
  if (path == CBQ_PATH_GEMV) {
    GemvParams p;
    std::memset(&p, 0, sizeof(p));
    p.codes = experts->codes;
    p.a = a;
    p.a_scale = a_scale;
    p.scales = experts->scales;
    p.codebooks = experts->codebooks;
    p.y = y;
    p.topk_idx = topk_idx;
    p.M = M;
    p.N = N;
    p.K = K;
    p.wait_ns = wait_limit_ns();
    p.E = E;
    p.topk = topk;
    return launch_gemv(p, true, s);
  }
  UmmaParams p;
  std::memset(&p, 0, sizeof(p));
  p.codes = experts->codes;
  p.a = a;
  p.a_scale = a_scale;
  p.scales = experts->scales;
  p.codebooks = experts->codebooks;
  p.y = y;
  p.topk_idx = topk_idx;
  p.M = M;
  p.N = N;
  p.K = K;
  p.wait_ns = wait_limit_ns();
  p.E = E;
  p.topk = topk;
  const int r = launch_umma(p, true, s);
  if (r != CBQ_EINVAL || !automatic) return r;
  // every token's activations do not fit the tile kernel's shared memory
  // (long K): the GEMV kernel's grouped variant takes any K
  GemvParams g;
  std::memset(&g, 0, sizeof(g));
  g.codes = experts->codes;
  g.a = a;
  g.a_scale = a_scale;
  g.scales = experts->scales;
  g.codebooks = experts->codebooks;
  g.y = y;
  g.topk_idx = topk_idx;
  g.M = M;
  g.N = N;
  g.K = K;
  g.wait_ns = wait_limit_ns();
  g.E = E;
  g.topk = topk;
  return launch_gemv(g, true, s);
}

int cbq_grouped_gemm_path(const uint8_t* a, const float* a_scale, const cbq_weight_t* experts,
                          int32_t E, const int32_t* topk_idx, int32_t topk, int32_t M, int32_t N,
                          int32_t K, float* y, void* stream, int32_t path) {
  if (path == CBQ_PATH_STREAMK) return CBQ_EINVAL;    // needs a workspace: cbq_grouped_gemm_ws
  return cbq_grouped_gemm_ws(a, a_scale, experts, E, topk_idx, topk, M, N, K, y, nullptr, 0, stream, path);
}

int cbq_grouped_gemm(const uint8_t* a, const float* a_scale, const cbq_weight_t* experts,
                     int32_t E, const int32_t* topk_idx, int32_t topk, int32_t M, int32_t N,
                     int32_t K, float* y, void* stream) {
  return cbq_grouped_gemm_path(a, a_scale, experts, E, topk_idx, topk, M, N, K, y, stream,
                               CBQ_PATH_AUTO);
}

// ---- two-bit draft head ---------------------------------------------------

int cbq_head2_sizes(int32_t N, int32_t K, size_t* codes_bytes, size_t* scales_bytes, size_t* codebook_bytes) {
  if (N < 0 || K < 0 || K % 128 != 0 || !codes_bytes || !scales_bytes || !codebook_bytes) return CBQ_EINVAL;
  *codes_bytes = static_cast<size_t>(K) * N / 4;
  *scales_bytes = static_cast<size_t>(K) * N / 32;
  *codebook_bytes = static_cast<size_t>(4) * N;
  return CBQ_OK;
}

int cbq_gemm2_ws(const uint8_t* a, const float* a_scale, const cbq_weight_t* head2, int32_t M, int32_t N, int32_t K,
                 float* y, void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 0 || M > 64 || N < 0 || K < 0 || K % 128 != 0) return CBQ_EINVAL;
  if (M == 0 || N == 0) return CBQ_OK;
  if (!y || !aligned(y, 4)) return CBQ_EINVAL;
  int st = current_device_checked(nullptr);
  if (st != CBQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0)
    return cudaMemsetAsync(y, 0, sizeof(float) * size_t(M) * size_t(N), s) == cudaSuccess ? CBQ_OK : CBQ_ECUDA;
  if (!a || !aligned(a, 16) || !a_scale || !aligned(a_scale, 4) || !weight_ok(head2) || !sk_applicable(M, N, K))
    return CBQ_EINVAL;
  SkParams p;
  std::memset(&p, 0, sizeof(p));
  p.codes = head2->codes;
  p.a = a;
  p.a_scale = a_scale;
  p.scales = head2->scales;
  p.codebooks = head2->codebooks;
  p.y = y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.wait_ns = wait_limit_ns();
  return launch_sk(p, workspace, workspace_bytes, s, 2);
}

namespace {
// Draft-head workspace: [the stream-K workspace][scores M x N fp32]
// [chunk candidates M x chunks x 16 x 8 bytes], each part 256-byte aligned.
size_t round256(size_t b) { return (b + 255) / 256 * 256; }
size_t head_parts(int M, int N, int K, size_t* sk, size_t* scores) {
  *sk = round256(sk_workspace_bytes(M, N, K));
  *scores = round256(static_cast<size_t>(M) * N * sizeof(float));
  const int nchunks = head_chunks(N);
  return *sk == 0 ? 0 : *sk + *scores + round256(static_cast<size_t>(M) * nchunks * kHeadShortlist * 8);
}
}  // namespace

int cbq_draft_head_workspace_size(int32_t M, int32_t N, int32_t K, size_t* bytes) {
  if (!bytes || M < 1 || M > 64 || N < kHeadShortlist || N > kHeadMaxRows || K < 128 || K % 128 != 0)
    return CBQ_EINVAL;
  size_t sk = 0, sc = 0;
  *bytes = head_parts(M, N, K, &sk, &sc);
  return CBQ_OK;
}

int cbq_draft_head(const uint8_t* a, const float* a_scale, const cbq_weight_t* head2, const uint8_t* head8,
                   const float* row_scale, int32_t M, int32_t N, int32_t K, int32_t* shortlist, float* logits,
                   int32_t* pick, void* workspace, size_t workspace_bytes, void* stream) {
  if (M < 1 || M > 64 || N < kHeadShortlist || N > kHeadMaxRows || K < 128 || K % 128 != 0) return CBQ_EINVAL;
  if (!a || !aligned(a, 16) || !a_scale || !aligned(a_scale, 4) || !weight_ok(head2) || !head8 ||
      !aligned(head8, 16) || !row_scale || !aligned(row_scale, 4) || !shortlist || !aligned(shortlist, 4) ||
      !logits || !aligned(logits, 4) || !pick || !aligned(pick, 4) || !workspace || !aligned(workspace, 256))
    return CBQ_EINVAL;
  size_t sk = 0, sc = 0;
  const size_t need = head_parts(M, N, K, &sk, &sc);
  if (need == 0 || workspace_bytes < need) return CBQ_EINVAL;
  int st = current_device_checked(nullptr);
  if (st != CBQ_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* scores = reinterpret_cast<float*>(ws + sk);
  st = cbq_gemm2_ws(a, a_scale, head2, M, N, K, scores, ws, sk, stream);
  if (st != CBQ_OK) return st;
  return launch_head_select(scores, M, N, K, a, a_scale, head8, row_scale, reinterpret_cast<uint64_t*>(ws + sk + sc),
                            shortlist, logits, pick, s);
}

int cbq_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return CBQ_ECUDA;
  unsigned v = take_status_gemv(s) | take_status_umma(s) | take_status_sk(s);
  if (v & 1u) return CBQ_ETIMEOUT;
  if (v & 2u) return CBQ_EROUTING;
  return CBQ_OK;
}

int cbq_select_budget(const float* logits, int32_t T, int32_t E, int32_t k, int32_t B, int32_t* budget,
                      int32_t* topk_idx, void* stream) {
  if (T < 1 || E < 1 || E > kMaxBudgetExperts || k < 1 || k > kMaxBudgetK || B < k || B > E) return CBQ_EINVAL;
  if (!logits || !aligned(logits, 4) || !budget || !aligned(budget, 4) || !topk_idx || !aligned(topk_idx, 4))
    return CBQ_EINVAL;
  const int st = current_device_checked(nullptr);
  if (st != CBQ_OK) return st;
  return launch_budget(logits, T, E, k, B, budget, topk_idx, static_cast<cudaStream_t>(stream));
}

uint64_t cbq_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* cbq_status_str(int status) {
  switch (status) {
    case CBQ_OK: return "ok";
    case CBQ_EINVAL: return "invalid argument";
    case CBQ_ECUDA: return "CUDA call failed";
    case CBQ_EDEVICE: return "no supported GPU (needs sm_103)";
    case CBQ_ETIMEOUT: return "a kernel gave up waiting; its output is incomplete";
    case CBQ_EROUTING: return "routing indices out of range or repeated within a token";
    default: return "unknown status";
  }
}

}  // extern "C"
