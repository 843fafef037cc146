"""Shared helpers of the GPU tests: build a device layer from the seeded fp32 weights (packed on the GPU from fp32
with the library's own encoder) and the matching oracle references (encoded on the CPU with the oracle's encoder).
The two sides share only the seeded input generators."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
from moe_inputs import expert_matrix_f32, router_f16_bits, x_bf16_bits

FMTS = [1, 2, 3, 4]
FMT_NAME = {1: "mxfp4", 2: "int4g32", 3: "q2k", 4: "q8_0"}


def tol_check(y_gpu: np.ndarray, y_ref: np.ndarray, absterm: np.ndarray, what: str = ""):
    """|y_gpu - y_ref| <= 1e-3 * sum|terms| + 1e-6 per element; NaN must match NaN. Returns max err/bound."""
    y = np.asarray(y_gpu, dtype=np.float64)
    nan_ref = np.isnan(y_ref)
    assert np.array_equal(np.isnan(y), nan_ref), "%s: NaN pattern differs" % what
    ok = ~nan_ref
    err = np.abs(y[ok] - y_ref[ok])
    bound = 1e-3 * absterm[ok] + 1e-6
    ratio = float(np.max(err / bound)) if err.size else 0.0
    assert np.all(err <= bound), "%s: max err/bound %.3g" % (what, ratio)
    return ratio


class Weights:
    """Seeded fp32 source weights of one layer, generated lazily per expert."""

    def __init__(self, seed: int, H: int, I: int, layer: int = 0):
        self.seed, self.H, self.I, self.layer = seed, H, I, layer

    @functools.lru_cache(maxsize=None)
    def f32(self, e: int, which: int) -> np.ndarray:
        return expert_matrix_f32(self.seed, self.layer, e, which, self.H, self.I)

    @functools.lru_cache(maxsize=None)
    def blocks(self, fmt: int, e: int, which: int) -> np.ndarray:
        return oracle.encode(fmt, self.f32(e, which))


def make_layer(m, fmt: int, W: Weights, E: int, experts, dev, layout: int = 0) -> "m.Layer":
    """Device layer with E expert slots; the listed experts are packed from fp32 on the GPU."""
    layer = m.Layer(fmt, W.H, W.I, E, layout=layout, device=dev)
    for e in sorted(set(int(v) for v in experts)):
        g = torch.from_numpy(W.f32(e, 0)).to(dev)[None]
        u = torch.from_numpy(W.f32(e, 1)).to(dev)[None]
        d = torch.from_numpy(W.f32(e, 2)).to(dev)[None]
        layer.pack(m.MOE_SRC_F32, g, u, d, e0=e)
    return layer


def oracle_moe(fmt: int, W: Weights, idx: np.ndarray, w: np.ndarray, x: np.ndarray):
    return oracle.moe_tokens(fmt, W.H, W.I, lambda e: W.blocks(fmt, e, 0), lambda e: W.blocks(fmt, e, 1),
                             lambda e: W.blocks(fmt, e, 2), idx, w, x)


def dev_bits(a: np.ndarray, dev):
    """uint16 bit patterns (bf16 / fp16) -> int16 device tensor with the same bits."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)


def near_tie_ok(gpu_idx, ref_idx, logits, absl, H):
    """True if the GPU top-k list differs from the oracle's only by swaps of candidates whose exact logits are
    within the fp32 summation error bound of each other (H * 2^-24 * sum|terms| each)."""
    if np.array_equal(gpu_idx, ref_idx):
        return True
    tol = H * 2.0 ** -24 * absl
    k = len(ref_idx)
    chosen = list(gpu_idx)
    if len(set(chosen)) != k:
        return False
    others = [e for e in range(len(logits)) if e not in chosen]
    for r in range(k):
        a = chosen[r]
        for b in chosen[r + 1:] + others:
            if logits[a] < logits[b] - (tol[a] + tol[b]):
                return False
    return True
