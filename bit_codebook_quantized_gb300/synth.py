"""Seeded synthetic inputs for the codebook-quantised matmul.

This module only draws random inputs of the right shapes and distributions;
it holds none of the method's arithmetic (no decoding, no packing, no
products).  Tests and the benchmark feed the same arrays to the CUDA library
and to the CPU oracle.

Packed weights are drawn directly in packed form: the code stream is uniform
random bytes, which makes every 3-bit field uniform over 0..7 and independent,
whatever the bit layout.  Scale bytes are uniform integers in a range,
codebooks are 8 sorted N(0,1) values per row rounded to E4M3, activations are
N(0,1) (or |N(0,1)|) rounded to E4M3.  The E4M3 rounding is torch's
``float8_e4m3fn`` cast, after clipping to +-448.

Workload shapes follow the decode / speculative-verify matmuls of "Hibana:
Fast Agentic Inference on Unified-Memory Devices" (sections "Model surgery /
Three-bit weights" and "Adaptive speculation / Expert sharing").
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def rng_for(seed: int) -> np.random.Generator:
    """Counter-based generator (Philox) so every stream is reproducible."""
    return np.random.Generator(np.random.Philox(seed))


def to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    """Round float values to OCP E4M3 bytes with torch's cast (RNE), clipped
    to the finite range first."""
    t = torch.from_numpy(np.clip(np.asarray(x, dtype=np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


@dataclass
class PackedWeights:
    """Host copy of one packed matrix (or a stack of experts: rows = E*N)."""
    codes: np.ndarray      # uint8 [rows, 3K/8]
    scales: np.ndarray     # uint8 [rows, K/32]
    codebooks: np.ndarray  # uint8 [rows, 8]
    N: int                 # rows
    K: int

    @property
    def nbytes(self) -> int:
        return self.codes.nbytes + self.scales.nbytes + self.codebooks.nbytes


def gen_weights(N: int, K: int, seed: int, scale_lo: int = 120, scale_hi: int = 127,
                codebook: str = "draws") -> PackedWeights:
    """Packed weights with uniform codes, uniform scale bytes in
    [scale_lo, scale_hi] and one sorted N(0,1) codebook per row.

    codebook="draws": 8 sorted N(0,1) draws per row (a different lookup table
    on every row); codebook="quantiles": the 8 N(0,1) quantiles at
    (i + 0.5)/8, the same on every row."""
    assert K % 32 == 0
    rng = rng_for(seed)
    codes = rng.integers(0, 256, size=(N, K // 32 * 12), dtype=np.uint8)
    scales = rng.integers(scale_lo, scale_hi + 1, size=(N, K // 32), dtype=np.uint8)
    if codebook == "draws":
        vals = np.sort(rng.standard_normal((N, 8)), axis=1)
    elif codebook == "quantiles":
        from scipy.special import ndtri
        q = ndtri((np.arange(8) + 0.5) / 8.0)
        vals = np.broadcast_to(q, (N, 8))
    else:
        raise ValueError(codebook)
    cbs = to_e4m3_bytes(vals).reshape(N, 8)
    return PackedWeights(codes, scales, np.ascontiguousarray(cbs), N, K)


def gen_head2(N: int, K: int, seed: int, scale_lo: int = 120, scale_hi: int = 127) -> PackedWeights:
    """A two-bit draft head: uniform 2-bit codes (random bytes: every 2-bit
    field uniform over 0..3), uniform scale bytes in [scale_lo, scale_hi] and
    one sorted 4-entry N(0,1) codebook per row, rounded to E4M3."""
    assert K % 32 == 0
    rng = rng_for(seed)
    codes = rng.integers(0, 256, size=(N, K // 32 * 8), dtype=np.uint8)
    scales = rng.integers(scale_lo, scale_hi + 1, size=(N, K // 32), dtype=np.uint8)
    cbs = to_e4m3_bytes(np.sort(rng.standard_normal((N, 4)), axis=1)).reshape(N, 4)
    return PackedWeights(codes, scales, np.ascontiguousarray(cbs), N, K)


def gen_head8(N: int, K: int, seed: int) -> tuple[np.ndarray, np.ndarray]:
    """An FP8 head: (E4M3 bytes [N, K] of N(0,1) draws, fp32 per-row scales
    uniform in [0.01, 0.05])."""
    rng = rng_for(seed)
    w = to_e4m3_bytes(rng.standard_normal((N, K))).reshape(N, K)
    rs = rng.uniform(0.01, 0.05, size=N).astype(np.float32)
    return np.ascontiguousarray(w), rs


def gen_activations(M: int, K: int, seed: int, half_normal: bool = False) -> np.ndarray:
    rng = rng_for(seed)
    x = rng.standard_normal((M, K))
    if half_normal:
        x = np.abs(x)
    return to_e4m3_bytes(x).reshape(M, K)


def gen_a_scale(M: int, seed: int, mode: str = "one") -> np.ndarray:
    if mode == "one":
        return np.ones(M, dtype=np.float32)
    if mode == "uniform":
        return rng_for(seed).uniform(0.5, 2.0, size=M).astype(np.float32)
    raise ValueError(mode)


def gen_router_logits(T: int, E: int, seed: int) -> np.ndarray:
    """Router logits of a verify round: fp32 N(0,1) draws [T, E]."""
    return rng_for(seed).standard_normal((T, E)).astype(np.float32)


def budget_workloads() -> dict[str, tuple[int, int, int, int]]:
    """(tokens T, experts E, per-token top-k, budget B) of a verify round's
    expert budget: the MoE round of the grouped workload (64 tokens, 128
    experts, top-8 inside 24) and a wide router (4096 experts, budget 64)."""
    return {"budget_t64_e128": (64, 128, 8, 24), "budget_t64_e4096": (64, 4096, 8, 64)}


def gen_moe_routing(M: int, E: int, budget: int, topk: int, seed: int) -> np.ndarray:
    """Per-round shared expert budget: `budget` distinct experts drawn
    uniformly; every token takes the top-`topk` of its N(0,1) router logits
    restricted to the budget, by descending logit (ties: lower expert id).
    Returns int32 [M, topk]."""
    assert topk <= budget <= E
    rng = rng_for(seed)
    chosen = np.sort(rng.choice(E, size=budget, replace=False))
    logits = rng.standard_normal((M, E))
    out = np.empty((M, topk), dtype=np.int32)
    for t in range(M):
        lg = logits[t, chosen]
        order = np.lexsort((chosen, -lg))   # primary: -logit, secondary: id
        out[t] = chosen[order[:topk]]
    return out


def gen_dense_weights_fp32(N: int, K: int, seed: int) -> np.ndarray:
    """Unquantised fp32 weights for the packer: N(0,1) per row times a random
    per-group magnitude, so group scales vary."""
    rng = rng_for(seed)
    w = rng.standard_normal((N, K))
    mag = np.exp2(rng.integers(-8, 4, size=(N, K // 32)))
    return (w * np.repeat(mag, 32, axis=1)).astype(np.float32)


# ---- the workloads ----------------------------------------------------------

@dataclass
class Workload:
    name: str
    M: int
    N: int
    K: int
    a_scale: str = "one"          # "one" | "uniform"
    half_normal: bool = False
    experts: int = 0              # >0: grouped MoE verify round
    budget: int = 0
    topk: int = 0
    tags: dict = field(default_factory=dict)


def workloads() -> dict[str, Workload]:
    w = {}
    w["gemv_2048"] = Workload("gemv_2048", 1, 2048, 2048)
    for m in (1, 2, 4, 8):
        w[f"decode_4096x12288_m{m}"] = Workload(f"decode_4096x12288_m{m}", m, 12288, 4096,
                                                a_scale="uniform")
    w["verify_up_5120x25600_m16"] = Workload("verify_up_5120x25600_m16", 16, 25600, 5120)
    w["verify_down_25600x5120_m16"] = Workload("verify_down_25600x5120_m16", 16, 5120, 25600,
                                               half_normal=True)
    w["moe_verify_e128_2048x1536_m64"] = Workload("moe_verify_e128_2048x1536_m64", 64, 1536, 2048,
                                                  experts=128, budget=24, topk=8)
    for m in (1, 8, 64):
        w[f"vocab_head_2048x151936_m{m}"] = Workload(f"vocab_head_2048x151936_m{m}", m, 151936,
                                                     2048)
    return w


def draft_head_workloads() -> dict[str, Workload]:
    """The two-bit draft head on the vocabulary-head shape (the drafter
    proposes one token per step; M = 8 covers a batch of requests)."""
    return {f"draft_head_2048x151936_m{m}": Workload(f"draft_head_2048x151936_m{m}", m, 151936, 2048)
            for m in (1, 8)}
