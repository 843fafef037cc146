"""Fused decode / verify FFN on the GPU against the oracle, and the width-1 invariant (verify row t == decode of
token t, bit for bit) from "Mixed-precision compression of DeepSeek-V4-Flash", "Width drift".

Tolerance (per output element): |y_gpu - y_ref| <= 1e-3 * sum_r |w_r| sum_i |Down_r[j,i] h_r[i]| + 1e-6.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import router_f16_bits, x_bf16_bits
from tests._harness import FMTS, FMT_NAME, Weights, dev_bits, make_layer, oracle_moe, tol_check

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


def _decode(m, layer, ws, x_row, idx_row, w_row, k, accumulate=False, y0=None, want_bf16=False):
    H = layer.H
    y = (y0.clone() if y0 is not None else torch.full((1, H), float("nan"), device=DEV))
    yb = torch.zeros((1, H), dtype=torch.int16, device=DEV) if want_bf16 else None
    m.moe_expert_ffn_decode(layer, dev_bits(x_row, DEV), torch.from_numpy(np.ascontiguousarray(idx_row, np.int32)).to(DEV),
                            torch.from_numpy(np.ascontiguousarray(w_row, np.float32)).to(DEV), k, y, yb, accumulate, ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws) == 0
    return y.cpu().numpy()[0], (yb.cpu().numpy()[0] if want_bf16 else None)


def _verify(m, layer, ws, x, idx, w, k):
    T, H = x.shape
    y = torch.full((T, H), float("nan"), device=DEV)
    m.moe_expert_ffn_verify(layer, dev_bits(x, DEV), T, torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(DEV),
                            torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(DEV), k, y, None, False, ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws) == 0
    return y.cpu().numpy()


def _routing(E, H, k, T, seed):
    wr = router_f16_bits(seed, 0, E, H)
    x = x_bf16_bits(seed, range(T), H)
    idx, w, _, _ = oracle.route_topk(wr, x, k)
    return x, idx, w


# ---------------------------------------------------------------- small layer (8 experts, hidden 512, top-2)
@pytest.mark.parametrize("fmt", FMTS, ids=[FMT_NAME[f] for f in FMTS])
def test_decode_small_layer(m, fmt):
    E, H, I, k, T = 8, 512, 256, 2, 8
    W = Weights(0, H, I)
    layer = make_layer(m, fmt, W, E, range(E), DEV)
    ws = layer.workspace(1, k)
    x, idx, w = _routing(E, H, k, T, seed=0)
    yr, ab = oracle_moe(fmt, W, idx, w, x)
    worst = 0.0
    for t in range(T):
        y, _ = _decode(m, layer, ws, x[t:t + 1], idx[t], w[t], k)
        worst = max(worst, tol_check(y, yr[t], ab[t], "token %d" % t))
    print("%s small decode: max err/bound %.3g" % (FMT_NAME[fmt], worst))


@pytest.mark.parametrize("fmt", FMTS, ids=[FMT_NAME[f] for f in FMTS])
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 8])
def test_verify_small_layer_width_exact(m, fmt, T):
    E, H, I, k = 8, 512, 256, 2
    W = Weights(0, H, I)
    layer = make_layer(m, fmt, W, E, range(E), DEV)
    ws = layer.workspace(8, k)
    x, idx, w = _routing(E, H, k, T, seed=10 + T)
    yv = _verify(m, layer, ws, x, idx, w, k)
    yr, ab = oracle_moe(fmt, W, idx, w, x)
    for t in range(T):
        yd, _ = _decode(m, layer, ws, x[t:t + 1], idx[t], w[t], k)
        assert np.array_equal(yv[t].view(np.uint32), yd.view(np.uint32)), "row %d differs from width-1 decode" % t
        tol_check(yv[t], yr[t], ab[t], "verify row %d" % t)


# ---------------------------------------------------------------- DS4-Flash-shaped layer (256 experts, 4096/2048, top-6)
@pytest.fixture(scope="module")
def big():
    E, H, I, k = 256, 4096, 2048, 6
    x, idx, w = _routing(E, H, k, 8, seed=1000)
    return dict(E=E, H=H, I=I, k=k, x=x, idx=idx, w=w, W=Weights(1, H, I))


@pytest.mark.parametrize("fmt", FMTS, ids=[FMT_NAME[f] for f in FMTS])
def test_full_shape_decode_and_verify(m, big, fmt):
    E, H, I, k, x, idx, w, W = (big[n] for n in ("E", "H", "I", "k", "x", "idx", "w", "W"))
    layer = make_layer(m, fmt, W, E, np.unique(idx), DEV)
    ws = layer.workspace(8, k)
    yv = _verify(m, layer, ws, x, idx, w, k)
    ys = []
    for t in range(8):
        yd, _ = _decode(m, layer, ws, x[t:t + 1], idx[t], w[t], k)
        assert np.array_equal(yv[t].view(np.uint32), yd.view(np.uint32)), "row %d differs from width-1 decode" % t
        ys.append(yd)
    sample = [0, 5]
    yr, ab = oracle_moe(fmt, W, idx[sample], w[sample], x[sample])
    for j, t in enumerate(sample):
        r = tol_check(ys[t], yr[j], ab[j], "token %d" % t)
        print("%s full-shape token %d: max err/bound %.3g" % (FMT_NAME[fmt], t, r))


def test_full_shape_shared_routing_verify(m, big):
    """all T tokens routed to the same 6 experts (the shared-routing reading of verify)"""
    E, H, I, k, x, idx, w, W = (big[n] for n in ("E", "H", "I", "k", "x", "idx", "w", "W"))
    fmt = 1
    sidx = np.tile(idx[0], (8, 1))
    layer = make_layer(m, fmt, W, E, np.unique(sidx), DEV)
    ws = layer.workspace(8, k)
    yv = _verify(m, layer, ws, x, sidx, w, k)
    for t in range(8):
        yd, _ = _decode(m, layer, ws, x[t:t + 1], sidx[t], w[t], k)
        assert np.array_equal(yv[t].view(np.uint32), yd.view(np.uint32))
    yr, ab = oracle_moe(fmt, W, sidx[[3]], w[[3]], x[[3]])
    tol_check(yv[3], yr[0], ab[0], "shared row 3")


# ---------------------------------------------------------------- edge cases
def test_accumulate_and_bf16_output(m):
    E, H, I, k = 8, 512, 256, 2
    W = Weights(0, H, I)
    layer = make_layer(m, 1, W, E, range(E), DEV)
    ws = layer.workspace(1, k)
    x, idx, w = _routing(E, H, k, 1, seed=3)
    y0 = torch.linspace(-1, 1, H, device=DEV)[None].contiguous()
    y, yb = _decode(m, layer, ws, x, idx[0], w[0], k, accumulate=True, y0=y0, want_bf16=True)
    yplain, _ = _decode(m, layer, ws, x, idx[0], w[0], k)
    assert np.array_equal(y, (y0.cpu().numpy()[0] + yplain).astype(np.float32))
    ref_b = torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(yb, ref_b)


def test_k1_and_duplicate_experts(m):
    E, H, I = 8, 512, 256
    W = Weights(0, H, I)
    layer = make_layer(m, 1, W, E, range(E), DEV)
    x = x_bf16_bits(4, [0], H)
    ws = layer.workspace(1, 3)
    y1, _ = _decode(m, layer, ws, x, np.array([5]), np.array([1.0]), 1)
    yr, ab = oracle_moe(1, W, np.array([[5]]), np.array([[1.0]], np.float32), x)
    tol_check(y1, yr[0], ab[0], "k=1")
    idx = np.array([2, 2, 6])
    w = np.array([0.25, 0.5, 0.25], np.float32)
    y3, _ = _decode(m, layer, ws, x, idx, w, 3)
    yr3, ab3 = oracle_moe(1, W, idx[None], w[None], x)
    tol_check(y3, yr3[0], ab3[0], "duplicate experts")


def test_special_exponents_propagate(m):
    """an E8M0 exponent of 0 zeroes its block; 255 makes every output NaN (NaN h reaches all of Down)"""
    E, H, I, k = 2, 512, 256, 1
    rng = np.random.default_rng(9)
    g = oracle.encode(1, (rng.standard_normal((E, I, H)) * 0.02).astype(np.float32))
    u = oracle.encode(1, (rng.standard_normal((E, I, H)) * 0.02).astype(np.float32))
    d = oracle.encode(1, (rng.standard_normal((E, H, I)) * 0.02).astype(np.float32))
    g = g.reshape(E, I, H // 32, 17)
    g[0, :, 3, 0] = 0          # expert 0: one block column zeroed
    g[1, 7, 5, 0] = 255        # expert 1: one NaN block
    g = g.reshape(E, I, -1)
    layer = m.Layer(1, H, I, E)
    layer.pack(m.MOE_SRC_BLOCKS, torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda(), torch.from_numpy(d).cuda())
    ws = layer.workspace(1, k)
    x = x_bf16_bits(9, [0], H)
    for e in range(E):
        y, _ = _decode(m, layer, ws, x, np.array([e]), np.array([1.0]), 1)
        yr, ab = oracle.moe_tokens(1, H, I, lambda q: g[q], lambda q: u[q], lambda q: d[q], np.array([[e]]),
                                   np.array([[1.0]], np.float32), x)
        tol_check(y, yr[0], ab[0], "expert %d" % e)
    assert np.all(np.isnan(y))


def test_invalid_expert_id_reports_status(m):
    E, H, I, k = 8, 512, 256, 2
    layer = m.Layer(1, H, I, E)
    layer.gate_up.zero_()
    layer.down.zero_()
    ws = layer.workspace(1, k)
    y = torch.zeros((1, H), device=DEV)
    x = torch.zeros((1, H), dtype=torch.int16, device=DEV)
    m.moe_expert_ffn_decode(layer, x, torch.tensor([[1, 9]], dtype=torch.int32, device=DEV),
                            torch.tensor([[0.5, 0.5]], device=DEV), k, y, None, False, ws)
    assert m.moe_get_device_status(ws) == 1
    m.moe_workspace_init(ws)
    # the workspace is usable again
    m.moe_expert_ffn_decode(layer, x, torch.tensor([[1, 3]], dtype=torch.int32, device=DEV),
                            torch.tensor([[0.5, 0.5]], device=DEV), k, y, None, False, ws)
    assert m.moe_get_device_status(ws) == 0
    assert torch.all(y == 0)


def test_host_side_errors(m):
    E, H, I, k = 8, 512, 256, 2
    layer = m.Layer(1, H, I, E)
    ws = layer.workspace(1, k)
    y = torch.zeros((9, H), device=DEV)
    x = torch.zeros((9, H), dtype=torch.int16, device=DEV)
    idx = torch.zeros((9, k), dtype=torch.int32, device=DEV)
    w = torch.zeros((9, k), device=DEV)
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_ffn_verify(layer, x, 9, idx, w, k, y, None, False, ws)
    assert ei.value.status == 2
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_ffn_verify(layer, x, 2, idx, w, k, y, None, False, ws)   # workspace sized for T=1
    assert ei.value.status == 5


def test_bounded_wait_timeout_probe(m):
    layer = m.Layer(1, 512, 256, 2)
    ws = layer.workspace(1, 1)
    m.moe_debug_timeout_probe(ws, 2000)
    assert m.moe_get_device_status(ws) == 7
    assert m.moe_get_device_status(ws) == 0   # read clears it
    # the context is still healthy
    a = torch.ones(1000, device=DEV)
    assert float(a.sum()) == 1000.0
