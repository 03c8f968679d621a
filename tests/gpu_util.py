"""Helpers shared by the GPU parity tests: seeded cases, device copies, the
oracle on a subset of rows, and the fp32 tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_codebook_quantized_gb300 import ops, synth

# |y_gpu - y_ref| <= REL * |a_scale| * sum_k |a*w| + ABS
REL, ABS = 1e-3, 1e-6


def ensure_built():
    from bit_codebook_quantized_gb300 import build
    build.build()
    ops.lib()


class Case:
    def __init__(self, M, N, K, seed, a_scale="uniform", half_normal=False, scale_lo=120,
                 scale_hi=127, codebook="draws"):
        self.M, self.N, self.K = M, N, K
        self.pw = synth.gen_weights(N, K, seed, scale_lo, scale_hi, codebook)
        self.a = synth.gen_activations(M, K, seed + 1, half_normal)
        self.s = synth.gen_a_scale(M, seed + 2, a_scale)
        self._dev = None

    def device(self):
        if self._dev is None:
            w = ops.PackedWeights.from_host(self.pw.codes, self.pw.scales, self.pw.codebooks,
                                            self.N, self.K)
            self._dev = (torch.from_numpy(self.a).cuda(), torch.from_numpy(self.s).cuda(), w)
        return self._dev

    def run(self, path=ops.PATH_AUTO):
        a, s, w = self.device()
        y = ops.gemm(a, s, w, path=path)
        torch.cuda.synchronize()
        return y.cpu().numpy()

    def oracle_rows(self, rows):
        return oracle.gemm_rows(self.a, self.s, self.pw.codes, self.pw.scales, self.pw.codebooks,
                                self.M, self.N, self.K, np.asarray(rows))

    def oracle(self):
        return oracle.gemm(self.a, self.s, self.pw.codes, self.pw.scales, self.pw.codebooks,
                           self.M, self.N, self.K)


def assert_close(y, yref, bound, what=""):
    y = np.asarray(y, np.float64)
    err = np.abs(y - yref)
    lim = REL * bound + ABS
    bad = err > lim
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at "
                             f"{tuple(i)}: got {y[tuple(i)]!r} want {yref[tuple(i)]!r} "
                             f"limit {lim[tuple(i)]!r}")
    assert np.all(np.isfinite(y))


def sample_rows(N, count, seed):
    rng = synth.rng_for(seed)
    pick = rng.choice(N, size=min(count, N), replace=False)
    # always include both ends and a slab boundary
    extra = [0, N - 1, min(N - 1, 15), min(N - 1, 16), min(N - 1, 127), min(N - 1, 128)]
    return np.unique(np.concatenate([pick, extra]))
