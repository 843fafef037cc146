"""Seeded synthetic inputs for the routed-MoE decode path.

This module is shared by the CUDA path's callers (tests, bench) and the CPU oracle. It only draws random
numbers and rounds them to the storage types the workloads name (fp32 weights, fp16 router, bf16
activations). It holds none of the method's arithmetic: no quantisation, routing or FFN.

Recipes (numpy PCG64 seeded through SeedSequence, so every array depends only on its key):
  * expert weights, key (seed, layer, expert, which):  fp32( fp32(N(0,1)) * 0.02f ),
    which = 0 gate [I,H], 1 up [I,H], 2 down [H,I];
  * router weights, key (seed, layer, 7777):  fp16 RNE of float64 N(0,1) * 0.02, shape [E,H];
  * activations, key (seed, 9999, token):  bf16 RNE of fp32 N(0,1), shape [H] per token;
  * token ids: uniform over the vocabulary;  tid2eid: k distinct experts per id (random keys, arg-sorted);
  * prefill routing: k distinct experts per token without replacement, p(expert at Zipf rank r) ~ r^-s
    over a seeded permutation of the experts (Gumbel top-k), and weights = u / sum(u), u ~ U(0.5, 1.5).
"""
from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

GATE, UP, DOWN = 0, 1, 2


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def expert_matrix_f32(seed: int, layer: int, expert: int, which: int, H: int, I: int) -> np.ndarray:
    """fp32 source weights of one expert matrix: gate/up are [I, H], down is [H, I] (row-major, K last)."""
    rows, cols = (I, H) if which in (GATE, UP) else (H, I)
    z = _rng(seed, layer, expert, which).standard_normal(rows * cols, dtype=np.float32)
    return (z * np.float32(0.02)).reshape(rows, cols)


def expert_stack_f32(seed: int, layer: int, experts, which: int, H: int, I: int, threads: int | None = None) -> np.ndarray:
    """[len(experts), rows, cols] fp32 for a list of experts, generated on a thread pool."""
    experts = list(experts)
    rows, cols = (I, H) if which in (GATE, UP) else (H, I)
    out = np.empty((len(experts), rows, cols), dtype=np.float32)

    def one(j):
        out[j] = expert_matrix_f32(seed, layer, experts[j], which, H, I)

    nthr = threads or min(32, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(nthr) as ex:
        list(ex.map(one, range(len(experts))))
    return out


def router_f16_bits(seed: int, layer: int, E: int, H: int) -> np.ndarray:
    """Router weights [E, H] as binary16 bit patterns (uint16)."""
    z = _rng(seed, layer, 7777).standard_normal(E * H)
    return (z * 0.02).astype(np.float16).view(np.uint16).reshape(E, H)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bfloat16 (nearest, ties to even) and return the bit patterns as uint16."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    r = np.where(nan, (u >> 16) | 0x40, r)
    return r.astype(np.uint16)


def x_bf16_bits(seed: int, tokens, H: int) -> np.ndarray:
    """Activations [len(tokens), H] as bf16 bit patterns; token t uses key (seed, 9999, t)."""
    tokens = list(tokens)
    out = np.empty((len(tokens), H), dtype=np.uint16)
    for j, t in enumerate(tokens):
        out[j] = f32_to_bf16_bits(_rng(seed, 9999, t).standard_normal(H, dtype=np.float32))
    return out


def token_ids(seed: int, T: int, vocab: int) -> np.ndarray:
    return _rng(seed, 4242).integers(0, vocab, size=T, dtype=np.int64).astype(np.int32)


def tid2eid(seed: int, layer: int, vocab: int, E: int, k: int) -> np.ndarray:
    """[vocab, k] int32: k distinct experts per token id."""
    keys = _rng(seed, layer, 5151).random((vocab, E), dtype=np.float32)
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def zipf_routing(seed: int, T: int, E: int, k: int, s: float = 1.1):
    """Prefill routing: (idx [T,k] int32, w [T,k] fp32). Experts are drawn without replacement with
    p(expert of Zipf rank r) proportional to r^-s, ranks assigned by a seeded permutation."""
    rng = _rng(seed, 3131)
    perm = rng.permutation(E)
    logp = np.empty(E)
    logp[perm] = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    g = rng.gumbel(size=(T, E))
    keys = logp[None, :] + g
    idx = np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)
    u = rng.uniform(0.5, 1.5, size=(T, k))
    w = (u / u.sum(axis=1, keepdims=True)).astype(np.float32)
    return idx, w


def spec_inputs(seed: int, K: int, V: int, spread: float = 2.0, noise: float = 0.5):
    """Synthetic speculative-decoding inputs: target distributions p [K+1, V] and draft distributions q [K, V]
    (fp32, each row the fp32 rounding of a float64 softmax of N(0, spread) logits; a draft row's logits are the
    target row's plus N(0, noise)), K drafted tokens drawn from the q rows, and K + 1 uniforms u in [0, 1) with
    24 random bits each."""
    rng = _rng(seed, 8181, K, V)
    lp = rng.normal(0.0, spread, size=(K + 1, V))
    lq = lp[:K] + rng.normal(0.0, noise, size=(K, V))

    def softmax(l):
        e = np.exp(l - l.max(axis=1, keepdims=True))
        return e / e.sum(axis=1, keepdims=True)

    p64, q64 = softmax(lp), softmax(lq) if K else np.zeros((0, V))
    draft = np.array([rng.choice(V, p=q64[k]) for k in range(K)], dtype=np.int32)
    u = (rng.integers(0, 1 << 24, size=K + 1) * 2.0 ** -24).astype(np.float32)
    return p64.astype(np.float32), q64.astype(np.float32), draft, u
