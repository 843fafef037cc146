"""Full-shape parity (hidden 4096, expert intermediate 2048, 256 experts, top-6) of every decode path against the
CPU oracle, on 16 seeded tokens per format and on activations built to stress the tensor-core path's E2M1-part
representation of x and h (one E8M0 exponent per 32 values): outlier channels, an outlier on a column whose
weights are zero in some rows, heavy-tailed (Student-t, 3 degrees of freedom) tokens, and exact zeros and bf16
subnormals.

The bar is the per-element tolerance of the decode path ("Mixed-precision compression of DeepSeek-V4-Flash",
"What compression does not solve": the expert FFN output of every routed token):
    |y_gpu - y_ref| <= 1e-3 * sum_r |w_r| sum_i |Down_r[j,i] h_r[i]| + 1e-6.
Each case prints its largest err/bound.
"""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import oracle
from moe_inputs import GATE, UP, DOWN, expert_stack_f32, f32_to_bf16_bits, router_f16_bits, x_bf16_bits
from tests._harness import FMTS, FMT_NAME, Weights, dev_bits, near_tie_ok, tol_check

pytestmark = pytest.mark.gpu
DEV = "cuda"
E, H, I, K = 256, 4096, 2048, 6
SEED = 31
NTOK = 16


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


def _rng(*key):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def _pack_all(m, layer, W):
    for e0 in range(0, E, 16):
        ex = range(e0, min(E, e0 + 16))
        g, u, d = (torch.from_numpy(expert_stack_f32(W.seed, 0, ex, which, H, I)).to(DEV) for which in (GATE, UP, DOWN))
        layer.pack(m.MOE_SRC_F32, g, u, d, e0=e0)


def _pack_some(m, layer, W, experts):
    for e in sorted(set(int(v) for v in experts)):
        g, u, d = (torch.from_numpy(W.f32(e, which)).to(DEV)[None] for which in (GATE, UP, DOWN))
        layer.pack(m.MOE_SRC_F32, g, u, d, e0=e)


@pytest.fixture(scope="module")
def full(m):
    W = Weights(SEED, H, I)
    wr = router_f16_bits(SEED, 0, E, H)
    x = x_bf16_bits(SEED, range(NTOK), H)
    idx, w, _, _ = oracle.route_topk(wr, x, K)
    tc = m.Layer(1, H, I, E, layout=m.MOE_LAYOUT_TC, device=DEV)
    _pack_all(m, tc, W)
    dec = {}
    for fmt in FMTS:
        dec[fmt] = m.Layer(fmt, H, I, E, device=DEV)
        _pack_some(m, dec[fmt], W, idx.ravel())
    torch.cuda.synchronize()
    return dict(W=W, wr=wr, x=x, idx=idx, w=w, tc=tc, dec=dec)


def _oracle(fmt, W, idx, w, x):
    """The oracle on every token in parallel (one token per host thread)."""
    def one(t):
        return oracle.moe_tokens(fmt, H, I, lambda e: W.blocks(fmt, e, 0), lambda e: W.blocks(fmt, e, 1),
                                 lambda e: W.blocks(fmt, e, 2), idx[t:t + 1], w[t:t + 1], x[t:t + 1])
    for e in sorted(set(int(v) for v in np.asarray(idx).ravel())):   # encode once, outside the threads
        for which in range(3):
            W.blocks(fmt, e, which)
    with cf.ThreadPoolExecutor(16) as ex:
        res = list(ex.map(one, range(len(x))))
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def _decode_all(m, layer, x, idx, w):
    ws = layer.workspace(1, K)
    ys = []
    for t in range(len(x)):
        y = torch.full((1, H), float("nan"), device=DEV)
        m.moe_expert_ffn_decode(layer, dev_bits(x[t:t + 1], DEV), torch.from_numpy(np.ascontiguousarray(idx[t], np.int32)).to(DEV),
                                torch.from_numpy(np.ascontiguousarray(w[t], np.float32)).to(DEV), K, y, None, False, ws)
        ys.append(y)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws) == 0
    return torch.cat(ys).cpu().numpy()


def _check_all(y, yr, ab, what):
    worst = max(tol_check(y[t], yr[t], ab[t], "%s token %d" % (what, t)) for t in range(len(y)))
    print("%s: %d tokens, max err/bound %.4g" % (what, len(y), worst))
    return worst


# ---------------------------------------------------------------- 16 seeded tokens per format and layout
def test_tc_layout_16_tokens(m, full):
    y = _decode_all(m, full["tc"], full["x"], full["idx"], full["w"])
    yr, ab = _oracle(1, full["W"], full["idx"], full["w"], full["x"])
    _check_all(y, yr, ab, "tc mxfp4")


@pytest.mark.parametrize("fmt", FMTS, ids=[FMT_NAME[f] for f in FMTS])
def test_decode_layout_16_tokens(m, full, fmt):
    y = _decode_all(m, full["dec"][fmt], full["x"], full["idx"], full["w"])
    yr, ab = _oracle(fmt, full["W"], full["idx"], full["w"], full["x"])
    _check_all(y, yr, ab, "decode layout %s" % FMT_NAME[fmt])


def test_fused_router_ffn_16_tokens(m, full):
    """router + FFN in one launch at full shape: routing equals the oracle's (up to proven near-ties), y within
    tolerance of the oracle with that routing"""
    tc, x, wr = full["tc"], full["x"], full["wr"]
    ws = tc.workspace(1, K)
    logits, absl = oracle.router_logits(wr, x)
    fi, fw, fy = [], [], []
    for t in range(NTOK):
        it = torch.full((1, K), -1, dtype=torch.int32, device=DEV)
        wt = torch.zeros((1, K), device=DEV)
        y = torch.full((1, H), float("nan"), device=DEV)
        m.moe_route_expert_ffn(tc, dev_bits(wr, DEV), dev_bits(x[t:t + 1], DEV), 1, K, it, wt, y, None, False, ws)
        fi.append(it)
        fw.append(wt)
        fy.append(y)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws) == 0
    fi = torch.cat(fi).cpu().numpy()
    fw = torch.cat(fw).cpu().numpy()
    fy = torch.cat(fy).cpu().numpy()
    for t in range(NTOK):
        assert near_tie_ok(fi[t], full["idx"][t], logits[t], absl[t], H), "token %d routing" % t
    yr, ab = _oracle(1, full["W"], fi, fw, x)
    _check_all(fy, yr, ab, "fused router+ffn")


# ---------------------------------------------------------------- activations that stress a shared block exponent
def _outliers(x, p, seed):
    """one element per 32-block multiplied by 2^p (exact in bf16 while it stays finite)"""
    xo = x.copy()
    r = _rng(seed, p)
    f = np.frombuffer(((xo.astype(np.uint32)) << 16).tobytes(), dtype=np.float32).reshape(xo.shape).copy()
    for t in range(len(xo)):
        cols = np.arange(0, H, 32) + r.integers(0, 32, size=H // 32)
        f[t, cols] *= np.float32(2.0 ** p)
    return f32_to_bf16_bits(f)


def _student_t(n, seed):
    f = _rng(seed, 3).standard_t(3, size=(n, H)).astype(np.float32)
    return f32_to_bf16_bits(f)


def _zeros_subnormals(x, seed):
    r = _rng(seed, 77)
    xz = x.copy()
    for t in range(len(xz)):
        sel = r.random(H)
        xz[t, sel < 0.15] = 0x0000                                    # +0
        xz[t, (sel >= 0.15) & (sel < 0.25)] = 0x8000                  # -0
        sub = (sel >= 0.25) & (sel < 0.40)
        xz[t, sub] = (r.integers(1, 0x80, size=int(sub.sum())) | (r.integers(0, 2, size=int(sub.sum())) << 15)).astype(np.uint16)
        xz[t, 64:96] = 0                                              # one block of zeros
        xz[t, 128:160] = r.integers(1, 0x80, size=32).astype(np.uint16)   # one block of subnormals only
    return xz


def _cases(full):
    x4 = full["x"][:4]
    out = [("outliers x2^%d" % p, _outliers(x4, p, 5)) for p in (8, 10, 12)]
    out.append(("student-t(3)", _student_t(4, 6)))
    out.append(("zeros and subnormals", _zeros_subnormals(x4, 7)))
    return out


@pytest.mark.parametrize("case", range(5), ids=["x2^8", "x2^10", "x2^12", "student_t3", "zeros_subnormals"])
def test_tc_layout_stress_activations(m, full, case):
    name, xs = _cases(full)[case]
    idx, w = full["idx"][:4], full["w"][:4]   # routing is an input: the seeded tokens' experts
    y = _decode_all(m, full["tc"], xs, idx, w)
    yr, ab = _oracle(1, full["W"], idx, w, xs)
    _check_all(y, yr, ab, "tc %s" % name)


@pytest.mark.parametrize("case", range(5), ids=["x2^8", "x2^10", "x2^12", "student_t3", "zeros_subnormals"])
def test_fused_router_ffn_stress_activations(m, full, case):
    """the same activations through router + FFN in one launch, each token routed by its own logits"""
    name, xs = _cases(full)[case]
    tc, wr = full["tc"], full["wr"]
    ws = tc.workspace(4, K)
    it = torch.full((4, K), -1, dtype=torch.int32, device=DEV)
    wt = torch.zeros((4, K), device=DEV)
    y = torch.full((4, H), float("nan"), device=DEV)
    m.moe_route_expert_ffn(tc, dev_bits(wr, DEV), dev_bits(xs, DEV), 4, K, it, wt, y, None, False, ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws) == 0
    fi, fw, fy = it.cpu().numpy(), wt.cpu().numpy(), y.cpu().numpy()
    ri, _, logits, absl = oracle.route_topk(wr, xs, K)
    for t in range(4):
        assert near_tie_ok(fi[t], ri[t], logits[t], absl[t], H), "%s token %d routing" % (name, t)
    yr, ab = _oracle(1, full["W"], fi, fw, xs)
    _check_all(fy, yr, ab, "fused %s" % name)


@pytest.mark.parametrize("fmt", FMTS, ids=[FMT_NAME[f] for f in FMTS])
def test_decode_layout_stress_activations(m, full, fmt):
    idx, w = full["idx"][:4], full["w"][:4]
    for name, xs in _cases(full):
        y = _decode_all(m, full["dec"][fmt], xs, idx, w)
        yr, ab = _oracle(fmt, full["W"], idx, w, xs)
        _check_all(y, yr, ab, "decode layout %s %s" % (FMT_NAME[fmt], name))


def test_tc_outlier_on_a_column_with_zero_weights(m, full):
    """an outlier (x 2^12) on column c of every block, where Gate and Up of the routed experts hold zeros in every
    other row at column c: the rows without the outlier's contribution must still be exact to the tolerance"""
    W0 = full["W"]
    idx, w = full["idx"][:2], full["w"][:2]
    experts = sorted(set(int(v) for v in idx.ravel()))

    class Zeroed(Weights):
        def f32(self, e, which):
            a = W0.f32(e, which).copy()
            if which in (GATE, UP):
                a[0::2, 5::32] = 0.0
            return a

    Wz = Zeroed(SEED, H, I)
    layer = m.Layer(1, H, I, E, layout=m.MOE_LAYOUT_TC, device=DEV)
    _pack_some(m, layer, Wz, experts)
    xo = full["x"][:2].copy()
    f = np.frombuffer((xo.astype(np.uint32) << 16).tobytes(), dtype=np.float32).reshape(xo.shape).copy()
    f[:, 5::32] *= np.float32(4096.0)
    xo = f32_to_bf16_bits(f)
    y = _decode_all(m, layer, xo, idx, w)
    yr, ab = _oracle(1, Wz, idx, w, xo)
    _check_all(y, yr, ab, "tc outlier on zeroed column")
