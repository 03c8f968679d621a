"""ctypes binding of libcbq (include/cbq.h).  Argument marshalling only: every
step of the matmul runs in the library's CUDA kernels; torch supplies device
memory and streams.  Each function has the name of its C entry point without
the ``cbq_`` prefix.

The library must have been built (``python -m bit_codebook_quantized_gb300.build``
or ``__graft_entry__.build()``); loading raises ``CbqError`` otherwise.  There
is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcbq.so")

PATH_AUTO, PATH_GEMV, PATH_MMA, PATH_STREAMK = 0, 1, 2, 3
OK, EINVAL, ECUDA, EDEVICE, ETIMEOUT, EROUTING = 0, -1, -2, -3, -4, -5

# Every symbol include/cbq.h declares.
EXPORTS = ("cbq_packed_sizes", "cbq_pack", "cbq_unpack", "cbq_gemm", "cbq_gemm_ws", "cbq_gemm_workspace_size",
           "cbq_gemm_path", "cbq_gemm_auto_path", "cbq_gemm_noalloc", "cbq_set_wait_limit",
           "cbq_gemm_gate_up", "cbq_gate_up_workspace_size",
           "cbq_grouped_gemm", "cbq_grouped_gemm_path", "cbq_grouped_gemm_ws", "cbq_grouped_workspace_size",
           "cbq_device_status", "cbq_launch_count", "cbq_status_str", "cbq_draft_length", "cbq_select_budget",
           "cbq_head2_sizes", "cbq_gemm2_ws", "cbq_draft_head_workspace_size", "cbq_draft_head")


class CbqError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_str(status)} ({status})")


class _Weight(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("codebooks", ctypes.c_void_p)]


_lib = None
_lock = threading.RLock()


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise CbqError(ECUDA, f"libcbq.so not built at {LIB_PATH}; run the build first")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        L.cbq_packed_sizes.argtypes = [i32, i32, ctypes.POINTER(sz), ctypes.POINTER(sz),
                                       ctypes.POINTER(sz)]
        L.cbq_pack.argtypes = [vp, i32, i32, vp, vp, vp]
        L.cbq_unpack.argtypes = [ctypes.POINTER(_Weight), i32, i32, vp, vp]
        L.cbq_gemm.argtypes = [vp, vp, ctypes.POINTER(_Weight), i32, i32, i32, vp, vp]
        L.cbq_gemm_ws.argtypes = [vp, vp, ctypes.POINTER(_Weight), i32, i32, i32, vp, vp, sz, vp]
        L.cbq_gemm_workspace_size.argtypes = [i32, i32, i32, ctypes.POINTER(sz)]
        L.cbq_gemm_path.argtypes = [vp, vp, ctypes.POINTER(_Weight), i32, i32, i32, vp, vp, sz, vp, i32]
        L.cbq_gemm_auto_path.argtypes = [i32, i32, i32, i32]
        L.cbq_set_wait_limit.argtypes = [ctypes.c_int64]
        L.cbq_gemm_gate_up.argtypes = [vp, vp, ctypes.POINTER(_Weight), i32, i32, i32, vp, vp, vp, sz, vp]
        L.cbq_gate_up_workspace_size.argtypes = [i32, i32, i32, ctypes.POINTER(sz)]
        L.cbq_gemm_noalloc.argtypes = [vp, vp, ctypes.POINTER(_Weight), i32, i32, i32, vp, vp]
        L.cbq_grouped_gemm.argtypes = [vp, vp, ctypes.POINTER(_Weight), i32, vp, i32, i32, i32,
                                       i32, vp, vp]
        L.cbq_grouped_gemm_path.argtypes = [vp, vp, ctypes.POINTER(_Weight), i32, vp, i32, i32,
                                            i32, i32, vp, vp, i32]
        L.cbq_grouped_gemm_ws.argtypes = [vp, vp, ctypes.POINTER(_Weight), i32, vp, i32, i32, i32, i32, vp, vp,
                                          sz, vp, i32]
        L.cbq_grouped_workspace_size.argtypes = [i32, i32, i32, i32, i32, ctypes.POINTER(sz)]
        L.cbq_head2_sizes.argtypes = [i32, i32, ctypes.POINTER(sz), ctypes.POINTER(sz), ctypes.POINTER(sz)]
        L.cbq_gemm2_ws.argtypes = [vp, vp, ctypes.POINTER(_Weight), i32, i32, i32, vp, vp, sz, vp]
        L.cbq_draft_head_workspace_size.argtypes = [i32, i32, i32, ctypes.POINTER(sz)]
        L.cbq_draft_head.argtypes = [vp, vp, ctypes.POINTER(_Weight), vp, vp, i32, i32, i32, vp, vp, vp, vp, sz, vp]
        L.cbq_device_status.argtypes = [vp]
        L.cbq_launch_count.argtypes = []
        L.cbq_launch_count.restype = ctypes.c_uint64
        L.cbq_status_str.argtypes = [ctypes.c_int]
        L.cbq_status_str.restype = ctypes.c_char_p
        dp = ctypes.POINTER(ctypes.c_double)
        L.cbq_draft_length.argtypes = [ctypes.c_double, ctypes.c_double, i32, ctypes.POINTER(i32), dp, dp]
        L.cbq_select_budget.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp]
        for name in ("cbq_packed_sizes", "cbq_pack", "cbq_unpack", "cbq_gemm", "cbq_gemm_ws",
                     "cbq_gemm_workspace_size", "cbq_gemm_path", "cbq_gemm_auto_path", "cbq_gemm_noalloc",
                     "cbq_set_wait_limit", "cbq_gemm_gate_up", "cbq_gate_up_workspace_size",
                     "cbq_grouped_gemm", "cbq_grouped_gemm_path", "cbq_grouped_gemm_ws",
                     "cbq_grouped_workspace_size", "cbq_device_status", "cbq_draft_length", "cbq_select_budget",
                     "cbq_head2_sizes", "cbq_gemm2_ws", "cbq_draft_head_workspace_size", "cbq_draft_head"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
        return L


def auto_path(M: int, N: int, K: int, with_workspace: bool = True) -> int:
    """The kernel cbq_gemm_ws picks for an M x N x K call with or without a
    workspace (PATH_GEMV/_MMA/_STREAMK)."""
    p = lib().cbq_gemm_auto_path(M, N, K, int(bool(with_workspace)))
    _check(p if p < 0 else OK, "cbq_gemm_auto_path")
    return p


def workspace_size(M: int, N: int, K: int) -> int:
    """Bytes of the workspace cbq_gemm_ws needs for an M x N x K call."""
    b = ctypes.c_size_t()
    _check(lib().cbq_gemm_workspace_size(M, N, K, ctypes.byref(b)), "cbq_gemm_workspace_size")
    return b.value


def set_wait_limit(ns: int) -> None:
    """cbq_set_wait_limit: bound of the kernels' waits (<= 0: the default 2 s)."""
    _check(lib().cbq_set_wait_limit(int(ns)), "cbq_set_wait_limit")


# One zero-filled workspace per (device, stream), allocated by torch (the
# caller side of the C ABI) on first use and large enough for any call (the
# library leaves it zero after every call), so that it never has to grow while
# a CUDA graph is being captured.
_WS_MIN = 16 << 20
_workspaces: dict = {}


def workspace_for(device: torch.device, stream, need: int) -> torch.Tensor:
    key = (device.index, stream.cuda_stream)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(max(need, _WS_MIN), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def select_budget(logits: torch.Tensor, k: int, B: int, stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """(budget [B] ascending expert ids, topk_idx [T, k]) of cbq_select_budget
    for router logits [T, E] (fp32, on the GPU)."""
    if logits.dtype != torch.float32 or logits.dim() != 2 or not logits.is_cuda:
        raise CbqError(EINVAL, "select_budget: logits must be a CUDA float32 [T, E] tensor")
    logits = logits.contiguous()
    T, E = logits.shape
    budget = torch.empty(max(B, 0), dtype=torch.int32, device=logits.device)
    topk = torch.empty((T, max(k, 0)), dtype=torch.int32, device=logits.device)
    _check(lib().cbq_select_budget(logits.data_ptr(), T, E, int(k), int(B), budget.data_ptr(),
                                   topk.data_ptr(), _stream(stream)), "cbq_select_budget")
    return budget, topk


def draft_length(q: float, c: float, dmax: int) -> tuple[int, float, float]:
    """(d*, E[N_d*], E[N_d*] / T(d*)) of cbq_draft_length: the draft length
    that maximises expected tokens per unit of round time."""
    d = ctypes.c_int32(0)
    e, r = ctypes.c_double(0.0), ctypes.c_double(0.0)
    _check(lib().cbq_draft_length(float(q), float(c), int(dmax), ctypes.byref(d), ctypes.byref(e),
                                  ctypes.byref(r)), "cbq_draft_length")
    return d.value, e.value, r.value


def status_str(status: int) -> str:
    if _lib is None:                      # never load (or wait on the loader) from an error path
        return "library not loaded"
    return _lib.cbq_status_str(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != OK:
        raise CbqError(status, what)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


@dataclass
class PackedWeights:
    """Packed matrix resident on the GPU (rows = N, or E*N for stacked experts)."""
    codes: torch.Tensor      # uint8 [rows, 3K/8]
    scales: torch.Tensor     # uint8 [rows, K/32]
    codebooks: torch.Tensor  # uint8 [rows, 8]
    N: int
    K: int

    @classmethod
    def from_host(cls, codes: np.ndarray, scales: np.ndarray, codebooks: np.ndarray, N: int,
                  K: int, device="cuda") -> "PackedWeights":
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(device)  # noqa: E731
        return cls(t(codes), t(scales), t(codebooks), N, K)

    def struct(self) -> _Weight:
        return _Weight(self.codes.data_ptr(), self.scales.data_ptr(), self.codebooks.data_ptr())

    @property
    def nbytes(self) -> int:
        return self.codes.numel() + self.scales.numel() + self.codebooks.numel()


def packed_sizes(N: int, K: int) -> tuple[int, int, int]:
    c, s, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().cbq_packed_sizes(N, K, ctypes.byref(c), ctypes.byref(s), ctypes.byref(b)),
           "cbq_packed_sizes")
    return c.value, s.value, b.value


def pack(W: np.ndarray):
    """Host quantiser: fp32 [N, K] -> (codes, scales, codebooks) numpy uint8."""
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    cs, ss, bs = packed_sizes(N, K)
    codes = np.zeros(cs, np.uint8)
    scales = np.zeros(ss, np.uint8)
    cbs = np.zeros(bs, np.uint8)
    _check(lib().cbq_pack(W.ctypes.data, N, K, codes.ctypes.data, scales.ctypes.data,
                          cbs.ctypes.data), "cbq_pack")
    return codes.reshape(N, -1), scales.reshape(N, -1), cbs.reshape(N, 8)


def unpack(w: PackedWeights, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    if out is None:
        out = torch.empty((w.N, w.K), dtype=torch.float32, device=w.codes.device)
    ws = w.struct()
    _check(lib().cbq_unpack(ctypes.byref(ws), w.N, w.K, out.data_ptr(), _stream(stream)),
           "cbq_unpack")
    return out


def gemm(a: torch.Tensor, a_scale: torch.Tensor, w: PackedWeights,
         out: torch.Tensor | None = None, path: int = PATH_AUTO, stream=None,
         workspace="auto") -> torch.Tensor:
    """y[M, N] = a_scale * (a[M, K] @ W^T); a is uint8 E4M3 bytes on the GPU.

    workspace: "auto" (a cached zero-filled buffer per device and stream, the
    cbq_gemm_ws path), None (cbq_gemm: no workspace) or a CUDA uint8 tensor."""
    M = a.shape[0]
    if out is None:
        out = torch.empty((M, w.N), dtype=torch.float32, device=a.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    if isinstance(workspace, str):
        need = workspace_size(M, w.N, w.K) if M > 0 and w.N > 0 else 0
        workspace = workspace_for(a.device, st, need) if need > 0 else None
    ws_ptr, ws_bytes = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    wt = w.struct()
    _check(lib().cbq_gemm_path(a.data_ptr(), a_scale.data_ptr(), ctypes.byref(wt), M, w.N, w.K,
                               out.data_ptr(), ws_ptr, ws_bytes, _stream(st), path), "cbq_gemm")
    return out


def gate_up(a: torch.Tensor, a_scale: torch.Tensor, w: PackedWeights, out: torch.Tensor | None = None,
            out_scale: torch.Tensor | None = None, stream=None, workspace="auto"):
    """cbq_gemm_gate_up: (h uint8 E4M3 [M, F], h_scale fp32 [M]) for the fused
    gate-up weight w (2F rows in blocks of 64 gate then 64 up rows)."""
    M, F = a.shape[0], w.N // 2
    if out is None:
        out = torch.empty((M, F), dtype=torch.uint8, device=a.device)
    if out_scale is None:
        out_scale = torch.empty(M, dtype=torch.float32, device=a.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    if isinstance(workspace, str):
        b = ctypes.c_size_t()
        _check(lib().cbq_gate_up_workspace_size(M, F, w.K, ctypes.byref(b)), "cbq_gate_up_workspace_size")
        if b.value == 0:
            raise CbqError(EINVAL, "cbq_gemm_gate_up: the stream-K kernel cannot take this shape")
        workspace = workspace_for(a.device, st, b.value)
    wt = w.struct()
    _check(lib().cbq_gemm_gate_up(a.data_ptr(), a_scale.data_ptr(), ctypes.byref(wt), M, F, w.K, out.data_ptr(),
                                  out_scale.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(st)),
           "cbq_gemm_gate_up")
    return out, out_scale


def gemm_noalloc(a: torch.Tensor, a_scale: torch.Tensor, w: PackedWeights,
                 out: torch.Tensor, stream=None) -> torch.Tensor:
    """cbq_gemm_noalloc: the stream-K matmul on the library's static scratch
    (no allocation; concurrent calls on one device race)."""
    ws = w.struct()
    _check(lib().cbq_gemm_noalloc(a.data_ptr(), a_scale.data_ptr(), ctypes.byref(ws), a.shape[0], w.N,
                                  w.K, out.data_ptr(), _stream(stream)), "cbq_gemm_noalloc")
    return out


def grouped_workspace_size(E: int, topk: int, M: int, N: int, K: int) -> int:
    """Bytes of workspace a grouped stream-K call needs (0: it cannot take the shape)."""
    b = ctypes.c_size_t()
    _check(lib().cbq_grouped_workspace_size(E, topk, M, N, K, ctypes.byref(b)), "cbq_grouped_workspace_size")
    return b.value


def grouped_gemm(a: torch.Tensor, a_scale: torch.Tensor, experts: PackedWeights, E: int,
                 topk_idx: torch.Tensor, out: torch.Tensor | None = None,
                 path: int = PATH_AUTO, stream=None, workspace="auto") -> torch.Tensor:
    """y[M, topk, N] for stacked experts (experts.N = rows per expert).
    workspace: "auto" (a cached one per device and stream, for the paths
    that use it), None (no workspace: cbq_grouped_gemm_path) or a device
    tensor."""
    M, topk = topk_idx.shape
    if out is None:
        out = torch.empty((M, topk, experts.N), dtype=torch.float32, device=a.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    if isinstance(workspace, str):
        need = grouped_workspace_size(E, topk, M, experts.N, experts.K) if path == PATH_STREAMK else 0
        workspace = workspace_for(a.device, st, need) if need > 0 else None
    ws = experts.struct()
    wp, wb = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    _check(lib().cbq_grouped_gemm_ws(a.data_ptr(), a_scale.data_ptr(), ctypes.byref(ws), E, topk_idx.data_ptr(),
                                     topk, M, experts.N, experts.K, out.data_ptr(), wp, wb, _stream(st), path),
           "cbq_grouped_gemm")
    return out


def gemm2(a: torch.Tensor, a_scale: torch.Tensor, head2: PackedWeights, out: torch.Tensor | None = None,
          stream=None, workspace="auto") -> torch.Tensor:
    """cbq_gemm2_ws: the two-bit head's scores [M, N] (head2: codes KN/4 bytes,
    scales [N][K/32], codebooks [N][4])."""
    M = a.shape[0]
    if out is None:
        out = torch.empty((M, head2.N), dtype=torch.float32, device=a.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    if isinstance(workspace, str):
        need = workspace_size(M, head2.N, head2.K) if M > 0 and head2.N > 0 else 0
        workspace = workspace_for(a.device, st, need) if need > 0 else None
    wp, wb = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    wt = head2.struct()
    _check(lib().cbq_gemm2_ws(a.data_ptr(), a_scale.data_ptr(), ctypes.byref(wt), M, head2.N, head2.K,
                              out.data_ptr(), wp, wb, _stream(st)), "cbq_gemm2_ws")
    return out


def draft_head(a: torch.Tensor, a_scale: torch.Tensor, head2: PackedWeights, head8: torch.Tensor,
               row_scale: torch.Tensor, stream=None, workspace="auto"):
    """cbq_draft_head: (shortlist int32 [M, 16], FP8 logits fp32 [M, 16],
    pick int32 [M]) of the two-bit draft head and the FP8 head."""
    M, N, K = a.shape[0], head2.N, head2.K
    rows = torch.empty((M, 16), dtype=torch.int32, device=a.device)
    logits = torch.empty((M, 16), dtype=torch.float32, device=a.device)
    pick = torch.empty(M, dtype=torch.int32, device=a.device)
    st = stream if stream is not None else torch.cuda.current_stream()
    if isinstance(workspace, str):
        b = ctypes.c_size_t()
        _check(lib().cbq_draft_head_workspace_size(M, N, K, ctypes.byref(b)), "cbq_draft_head_workspace_size")
        if b.value == 0:
            raise CbqError(EINVAL, "cbq_draft_head: the stream-K kernel cannot take this shape")
        workspace = workspace_for(a.device, st, b.value)
    wt = head2.struct()
    _check(lib().cbq_draft_head(a.data_ptr(), a_scale.data_ptr(), ctypes.byref(wt), head8.data_ptr(),
                                row_scale.data_ptr(), M, N, K, rows.data_ptr(), logits.data_ptr(), pick.data_ptr(),
                                workspace.data_ptr(), workspace.numel(), _stream(st)), "cbq_draft_head")
    return rows, logits, pick


def device_status(stream=None) -> int:
    return int(lib().cbq_device_status(_stream(stream)))


def launch_count() -> int:
    return int(lib().cbq_launch_count())
