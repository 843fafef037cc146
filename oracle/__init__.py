"""CPU oracle for the routed-MoE low-bit decode path -- TEST INFRASTRUCTURE.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg may import this package.
The CUDA library never calls it and shares no code with it. The arithmetic lives in oracle.c (plain C,
fp64 accumulation, built with -O2 -ffp-contract=off); this file only builds it and marshals numpy arrays.

Formats: fmt 1 = MXFP4 (17-byte blocks of 32), 2 = INT4 group-32 (18-byte blocks), 3 = Q2_K (84-byte blocks
of 256), 4 = Q8_0 (34-byte blocks of 32, the shared expert's format as the library defines it). A matrix
[rows, K] is rows*K/bs consecutive canonical blocks (blocks run along K).

Parity pins: every function here is pinned by tests/test_oracle_*.py against values the pages print
(E2M1 table, E8M0 rule, block sizes), closed forms, brute force on tiny inputs or library routines.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MXFP4, INT4G32, Q2K, Q8_0 = 1, 2, 3, 4
BLOCK = {MXFP4: (32, 17), INT4G32: (32, 18), Q2K: (256, 84), Q8_0: (32, 34)}


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def bind(path: str) -> C.CDLL:
    """Load a build of oracle.c and set the argument and result types of its functions."""
    L = C.CDLL(path)
    P = C.c_void_p
    i64, i32, dbl = C.c_int64, C.c_int, C.c_double
    sig = {
        "orc_f16_to_f64": (dbl, [C.c_uint16]),
        "orc_bf16_to_f64": (dbl, [C.c_uint16]),
        "orc_round_f32": (dbl, [dbl]),
        "orc_round_f16": (dbl, [dbl]),
        "orc_round_bf16": (dbl, [dbl]),
        "orc_f32_to_f16_rne": (C.c_uint16, [C.c_float]),
        "orc_e2m1_value": (dbl, [i32]),
        "orc_e8m0_scale": (dbl, [i32]),
        "orc_e4m3_value": (dbl, [i32]),
        "orc_decode_mxfp4": (None, [P, i64, P]),
        "orc_decode_int4": (None, [P, i64, P]),
        "orc_decode_q2k": (None, [P, i64, P]),
        "orc_decode_q8_0": (None, [P, i64, P]),
        "orc_encode_mxfp4": (None, [P, i64, P]),
        "orc_encode_int4": (None, [P, i64, P]),
        "orc_encode_q2k": (None, [P, i64, P]),
        "orc_encode_q8_0": (None, [P, i64, P]),
        "orc_quant_mxfp8": (None, [P, i64, P, P]),
        "orc_mxfp4_half_lut": (None, [P]),
        "orc_router_logits": (None, [P, P, i32, i32, i32, P, P]),
        "orc_topk_from_logits": (None, [P, i32, i32, i32, P, P]),
        "orc_route_topk": (None, [P, P, i32, i32, i32, i32, P, P, P, P]),
        "orc_route_hash": (None, [P, P, i32, i32, P, P]),
        "orc_rms_norm": (None, [P, i32, i32, C.c_double, P]),
        "orc_weight_at": (dbl, [i32, P, i32, i64, i32]),
        "orc_expert_ffn": (None, [i32, i32, i32, P, P, P, P, P, P, P, P, P]),
        "orc_moe_token": (None, [i32, i32, i32, i32, P, P, P, P, P, P, P]),
        "orc_moe_batch": (None, [i32, i32, i32, i32, i32, P, P, P, i32, P, P, P, P, P, i32]),
        "orc_prefill_token": (None, [i32, i32, i32, P, P, P, P, P, P, P, P, P, P, P, P]),
        "orc_max_threads": (i32, []),
        "orc_spec_accept": (None, [P, P, i32, i32, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = bind(_LIB)
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def max_threads() -> int:
    return lib().orc_max_threads()


# ---------------------------------------------------------------- scalar helpers
def f16_to_f64(bits: int) -> float:
    return lib().orc_f16_to_f64(bits)


def bf16_to_f64(bits: int) -> float:
    return lib().orc_bf16_to_f64(bits)


def e2m1_value(code: int) -> float:
    return lib().orc_e2m1_value(code)


def e8m0_scale(e: int) -> float:
    return lib().orc_e8m0_scale(e)


def e4m3_value(code: int) -> float:
    return lib().orc_e4m3_value(code)


def round_f32(x: float) -> float:
    return lib().orc_round_f32(x)


def round_f16(x: float) -> float:
    return lib().orc_round_f16(x)


def round_bf16(x: float) -> float:
    return lib().orc_round_bf16(x)


def f32_to_f16_rne(x: float) -> int:
    return lib().orc_f32_to_f16_rne(x)


# ---------------------------------------------------------------- formats
def decode(fmt: int, blocks: np.ndarray) -> np.ndarray:
    """Canonical blocks (uint8, any shape with total size a multiple of the block bytes) -> fp32 weights."""
    bs, nb = BLOCK[fmt]
    b = _c(blocks, np.uint8).reshape(-1)
    n = b.size // nb
    out = np.empty(n * bs, dtype=np.float32)
    fn = {MXFP4: lib().orc_decode_mxfp4, INT4G32: lib().orc_decode_int4, Q2K: lib().orc_decode_q2k,
          Q8_0: lib().orc_decode_q8_0}[fmt]
    fn(_p(b), n, _p(out))
    return out


def encode(fmt: int, w: np.ndarray) -> np.ndarray:
    """fp32 weights [..., K] -> canonical blocks [..., K/bs * block_bytes] (uint8)."""
    bs, nb = BLOCK[fmt]
    a = _c(w, np.float32)
    shape = a.shape
    assert shape[-1] % bs == 0
    n = a.size // bs
    out = np.empty(n * nb, dtype=np.uint8)
    fn = {MXFP4: lib().orc_encode_mxfp4, INT4G32: lib().orc_encode_int4, Q2K: lib().orc_encode_q2k,
          Q8_0: lib().orc_encode_q8_0}[fmt]
    fn(_p(a), n, _p(out))
    return out.reshape(*shape[:-1], shape[-1] // bs * nb)


def quant_mxfp8(v: np.ndarray):
    """values (float64, already in the precision the decision is taken in) [..., 32n] -> (codes u8, scales u8)."""
    a = _c(v, np.float64)
    n = a.size // 32
    codes = np.empty(a.size, dtype=np.uint8)
    scales = np.empty(n, dtype=np.uint8)
    lib().orc_quant_mxfp8(_p(a), n, _p(codes), _p(scales))
    return codes.reshape(a.shape), scales.reshape(*a.shape[:-1], a.shape[-1] // 32)


def mxfp4_half_lut() -> np.ndarray:
    lut = np.empty(256 * 16, dtype=np.uint16)
    lib().orc_mxfp4_half_lut(_p(lut))
    return lut.reshape(256, 16)


def weight_at(fmt: int, mat: np.ndarray, K: int, row: int, col: int) -> float:
    m = _c(mat, np.uint8)
    return lib().orc_weight_at(fmt, _p(m), K, row, col)


# ---------------------------------------------------------------- router
def router_logits(wr_f16: np.ndarray, x_bf16: np.ndarray):
    wr = _c(wr_f16, np.uint16)
    x = _c(x_bf16, np.uint16).reshape(-1, wr.shape[1])
    T, H = x.shape
    E = wr.shape[0]
    logits = np.empty((T, E))
    absl = np.empty((T, E))
    lib().orc_router_logits(_p(wr), _p(x), T, H, E, _p(logits), _p(absl))
    return logits, absl


def topk_from_logits(logits: np.ndarray, k: int):
    l = _c(logits, np.float64)
    T, E = l.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    lib().orc_topk_from_logits(_p(l), T, E, k, _p(idx), _p(w))
    return idx, w


def route_topk(wr_f16: np.ndarray, x_bf16: np.ndarray, k: int):
    """-> idx [T,k] int32, w [T,k] fp32, logits [T,E] fp64, abs_terms [T,E] fp64"""
    logits, absl = router_logits(wr_f16, x_bf16)
    idx, w = topk_from_logits(logits, k)
    return idx, w, logits, absl


def route_hash(token_ids: np.ndarray, tid2eid: np.ndarray, k: int):
    tok = _c(token_ids, np.int32)
    tab = _c(tid2eid, np.int32)
    T = tok.size
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    lib().orc_route_hash(_p(tok), _p(tab), T, k, _p(idx), _p(w))
    return idx, w


def rms_norm(y: np.ndarray, eps: float) -> np.ndarray:
    """y [T, H] fp32 -> y / sqrt(mean(y^2) + eps) per row, exact in fp64 (the library rounds it to bf16)."""
    yy = _c(y, np.float32)
    T, H = yy.shape
    out = np.empty((T, H))
    lib().orc_rms_norm(_p(yy), T, H, float(eps), _p(out))
    return out


# ---------------------------------------------------------------- FFN
def expert_ffn(fmt: int, H: int, I: int, gate: np.ndarray, up: np.ndarray, down: np.ndarray, x: np.ndarray):
    """One expert on one activation vector x (float64 [H]). -> dict g,u,h [I], d,dabs [H]."""
    g, u, h = (np.empty(I) for _ in range(3))
    d, da = np.empty(H), np.empty(H)
    G, U, D = (_c(a, np.uint8) for a in (gate, up, down))
    xx = _c(x, np.float64)
    lib().orc_expert_ffn(fmt, H, I, _p(G), _p(U), _p(D), _p(xx), _p(g), _p(u), _p(h), _p(d), _p(da))
    return dict(g=g, u=u, h=h, d=d, dabs=da)


def moe_tokens(fmt: int, H: int, I: int, gate_of, up_of, down_of, idx: np.ndarray, w: np.ndarray,
               x_bf16: np.ndarray):
    """Per-token MoE output where gate_of(e)/up_of(e)/down_of(e) return an expert's canonical blocks.
    -> y [T,H] fp64, absterm [T,H] fp64."""
    idx = np.asarray(idx, dtype=np.int32).reshape(len(x_bf16), -1)
    w = _c(w, np.float32).reshape(idx.shape)
    x = _c(x_bf16, np.uint16).reshape(-1, H)
    T, k = idx.shape
    y = np.empty((T, H))
    ab = np.empty((T, H))
    for t in range(T):
        mats = [(_c(gate_of(e), np.uint8), _c(up_of(e), np.uint8), _c(down_of(e), np.uint8)) for e in idx[t]]
        ptr = lambda j: (C.c_void_p * k)(*[m[j].ctypes.data for m in mats])
        lib().orc_moe_token(fmt, H, I, k, ptr(0), ptr(1), ptr(2), _p(w[t]), _p(x[t]),
                            _p(y[t]), _p(ab[t]))
    return y, ab


def moe_batch(fmt: int, H: int, I: int, gate_all: np.ndarray, up_all: np.ndarray, down_all: np.ndarray,
              idx: np.ndarray, w: np.ndarray, x_bf16: np.ndarray, threads: int = 1):
    """All experts resident: gate_all/up_all [E, I, H/bs*nb] and down_all [E, H, I/bs*nb] canonical blocks."""
    G, U, D = (_c(a, np.uint8) for a in (gate_all, up_all, down_all))
    x = _c(x_bf16, np.uint16).reshape(-1, H)
    T = x.shape[0]
    idx = _c(idx, np.int32).reshape(T, -1)
    k = idx.shape[1]
    w = _c(w, np.float32).reshape(T, k)
    E = G.shape[0]
    y = np.empty((T, H))
    ab = np.empty((T, H))
    lib().orc_moe_batch(fmt, H, I, E, k, _p(G), _p(U), _p(D), T, _p(idx), _p(w), _p(x), _p(y), _p(ab), threads)
    return y, ab


def prefill_token(H: int, I: int, gate_of, up_of, down_of, idx_t, w_t, x_t_bf16):
    """One prefill token (MXFP4 weights, MXFP8 activations). -> dict y, absterm, xq codes/scales,
    hq codes/scales per rank, h (fp64) per rank."""
    k = len(idx_t)
    mats = [(_c(gate_of(e), np.uint8), _c(up_of(e), np.uint8), _c(down_of(e), np.uint8)) for e in idx_t]
    ptr = lambda j: (C.c_void_p * k)(*[m[j].ctypes.data for m in mats])
    w = _c(w_t, np.float32)
    x = _c(x_t_bf16, np.uint16)
    y, ab = np.empty(H), np.empty(H)
    xc, xs = np.empty(H, np.uint8), np.empty(H // 32, np.uint8)
    hc, hs = np.empty(k * I, np.uint8), np.empty(k * I // 32, np.uint8)
    h = np.empty(k * I)
    lib().orc_prefill_token(H, I, k, ptr(0), ptr(1), ptr(2), _p(w), _p(x), _p(y), _p(ab), _p(xc), _p(xs),
                            _p(hc), _p(hs), _p(h))
    return dict(y=y, absterm=ab, xq_codes=xc, xq_scales=xs, hq_codes=hc.reshape(k, I),
                hq_scales=hs.reshape(k, I // 32), h=h.reshape(k, I))


# ---------------------------------------------------------------- speculative acceptance
def spec_accept(p: np.ndarray, q: np.ndarray, draft, u) -> tuple[int, int]:
    """The chain of K drafted tokens under the acceptance rule of "Mixed-precision compression of DeepSeek-V4-Flash"
    (lumirain.cn), "What compression does not solve"
    (accept draft k with probability min(1, p_k(d)/q_k(d)); at the first rejection draw from max(p_k - q_k, 0)
    normalised; after K acceptances draw from p_K). p [K+1, V] fp32, q [K, V] fp32, draft [K] int32,
    u [K+1] fp32 (u[K] drives the draw). -> (accepted drafts n, drawn token); (-1, -1) for a draft id outside
    [0, V). The arithmetic of the decision and of the draw is fixed in oracle.c (fp32 quotient, exact integer
    inverse CDF)."""
    pp = _c(p, np.float32)
    K1, V = pp.shape
    K = K1 - 1
    qq = _c(q, np.float32).reshape(K, V) if K > 0 else np.zeros((1, V), np.float32)
    d = _c(np.asarray(draft, dtype=np.int32).reshape(-1), np.int32) if K > 0 else np.zeros(1, np.int32)
    uu = _c(np.asarray(u, dtype=np.float32).reshape(-1), np.float32)
    assert uu.size == K + 1 and (K == 0 or d.size == K)
    out = np.empty(2, dtype=np.int32)
    lib().orc_spec_accept(_p(pp), _p(qq), K, V, _p(d), _p(uu), _p(out))
    return int(out[0]), int(out[1])
