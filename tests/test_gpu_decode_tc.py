"""Decode and verify of MXFP4 experts held in the tensor-core layout (block-scaled tcgen05 MMA path) against the
oracle, and the width-1 invariant of "Mixed-precision compression of DeepSeek-V4-Flash", "Width drift": row t of a
verify of width T is bit-identical to the decode of token t alone.

Tolerance (per output element): |y_gpu - y_ref| <= 1e-3 * sum_r |w_r| sum_i |Down_r[j,i] h_r[i]| + 1e-6.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import router_f16_bits, x_bf16_bits
from tests._harness import Weights, dev_bits, make_layer, oracle_moe, tol_check
from tests.test_gpu_ffn import _decode, _routing, _verify

pytestmark = pytest.mark.gpu
DEV = "cuda"
MXFP4, TC = 1, 1


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


@pytest.fixture(scope="module")
def small(m):
    E, H, I = 8, 512, 256
    W = Weights(0, H, I)
    return W, make_layer(m, MXFP4, W, E, range(E), DEV, layout=TC)


def test_tc_decode_small_layer(m, small):
    W, layer = small
    E, H, k, T = 8, 512, 2, 8
    ws = layer.workspace(1, k)
    x, idx, w = _routing(E, H, k, T, seed=0)
    yr, ab = oracle_moe(MXFP4, W, idx, w, x)
    worst = 0.0
    for t in range(T):
        y, _ = _decode(m, layer, ws, x[t:t + 1], idx[t], w[t], k)
        worst = max(worst, tol_check(y, yr[t], ab[t], "token %d" % t))
    print("tc small decode: max err/bound %.3g" % worst)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_tc_verify_small_layer_width_exact(m, small, T):
    W, layer = small
    E, H, k = 8, 512, 2
    ws = layer.workspace(8, k)
    x, idx, w = _routing(E, H, k, T, seed=10 + T)
    yv = _verify(m, layer, ws, x, idx, w, k)
    yr, ab = oracle_moe(MXFP4, W, idx, w, x)
    for t in range(T):
        yd, _ = _decode(m, layer, ws, x[t:t + 1], idx[t], w[t], k)
        assert np.array_equal(yv[t].view(np.uint32), yd.view(np.uint32)), "row %d differs from width-1 decode" % t
        tol_check(yv[t], yr[t], ab[t], "verify row %d" % t)


@pytest.fixture(scope="module")
def big(m):
    E, H, I, k = 256, 4096, 2048, 6
    x, idx, w = _routing(E, H, k, 8, seed=1000)
    W = Weights(1, H, I)
    shared = np.tile(idx[0], (8, 1))
    layer = make_layer(m, MXFP4, W, E, np.unique(np.concatenate([idx.ravel(), shared.ravel()])), DEV, layout=TC)
    return dict(E=E, H=H, I=I, k=k, x=x, idx=idx, w=w, W=W, layer=layer, shared=shared)


def test_tc_full_shape_decode_and_verify(m, big):
    H, k, x, idx, w, W, layer = (big[n] for n in ("H", "k", "x", "idx", "w", "W", "layer"))
    ws = layer.workspace(8, k)
    yv = _verify(m, layer, ws, x, idx, w, k)
    ys = []
    for t in range(8):
        yd, _ = _decode(m, layer, ws, x[t:t + 1], idx[t], w[t], k)
        assert np.array_equal(yv[t].view(np.uint32), yd.view(np.uint32)), "row %d differs from width-1 decode" % t
        ys.append(yd)
    sample = [0, 5]
    yr, ab = oracle_moe(MXFP4, W, idx[sample], w[sample], x[sample])
    for j, t in enumerate(sample):
        r = tol_check(ys[t], yr[j], ab[j], "token %d" % t)
        print("tc full-shape token %d: max err/bound %.3g" % (t, r))


def test_tc_full_shape_shared_routing_verify(m, big):
    k, x, w, W, layer, sidx = (big[n] for n in ("k", "x", "w", "W", "layer", "shared"))
    ws = layer.workspace(8, k)
    yv = _verify(m, layer, ws, x, sidx, w, k)
    for t in range(8):
        yd, _ = _decode(m, layer, ws, x[t:t + 1], sidx[t], w[t], k)
        assert np.array_equal(yv[t].view(np.uint32), yd.view(np.uint32))
    yr, ab = oracle_moe(MXFP4, W, sidx[[3]], w[[3]], x[[3]])
    tol_check(yv[3], yr[0], ab[0], "shared row 3")


def test_tc_decode_workspace_for_one_token_repeats_bitwise(m, big):
    """consecutive calls reuse the workspace counters (reset by the last CTA): same inputs, same bits"""
    k, x, idx, w, layer = (big[n] for n in ("k", "x", "idx", "w", "layer"))
    ws = layer.workspace(1, k)
    y1, _ = _decode(m, layer, ws, x[2:3], idx[2], w[2], k)
    y2, _ = _decode(m, layer, ws, x[2:3], idx[2], w[2], k)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


def test_tc_accumulate_bf16_k1_duplicates(m, small):
    W, layer = small
    E, H, k = 8, 512, 2
    ws = layer.workspace(1, 3)
    x, idx, w = _routing(E, H, k, 1, seed=3)
    y0 = torch.linspace(-1, 1, H, device=DEV)[None].contiguous()
    y, yb = _decode(m, layer, ws, x, idx[0], w[0], k, accumulate=True, y0=y0, want_bf16=True)
    yplain, _ = _decode(m, layer, ws, x, idx[0], w[0], k)
    assert np.array_equal(y, (y0.cpu().numpy()[0] + yplain).astype(np.float32))
    assert np.array_equal(yb, torch.from_numpy(y).to(torch.bfloat16).view(torch.int16).numpy())
    x1 = x_bf16_bits(4, [0], H)
    y1, _ = _decode(m, layer, ws, x1, np.array([5]), np.array([1.0]), 1)
    yr, ab = oracle_moe(MXFP4, W, np.array([[5]]), np.array([[1.0]], np.float32), x1)
    tol_check(y1, yr[0], ab[0], "k=1")
    idx3, w3 = np.array([2, 2, 6]), np.array([0.25, 0.5, 0.25], np.float32)
    y3, _ = _decode(m, layer, ws, x1, idx3, w3, 3)
    yr3, ab3 = oracle_moe(MXFP4, W, idx3[None], w3[None], x1)
    tol_check(y3, yr3[0], ab3[0], "duplicate experts")


def test_tc_invalid_expert_id_reports_status(m, small):
    _, layer = small
    H, k = 512, 2
    ws = layer.workspace(1, k)
    y = torch.zeros((1, H), device=DEV)
    x = torch.zeros((1, H), dtype=torch.int16, device=DEV)
    m.moe_expert_ffn_decode(layer, x, torch.tensor([[1, 9]], dtype=torch.int32, device=DEV),
                            torch.tensor([[0.5, 0.5]], device=DEV), k, y, None, False, ws)
    assert m.moe_get_device_status(ws) == 1
    m.moe_workspace_init(ws)
    m.moe_expert_ffn_decode(layer, x, torch.tensor([[1, 3]], dtype=torch.int32, device=DEV),
                            torch.tensor([[0.5, 0.5]], device=DEV), k, y, None, False, ws)
    assert m.moe_get_device_status(ws) == 0
    assert torch.all(y == 0)


def test_tc_special_exponents(m):
    """E8M0 e = 0 blocks contribute (next to) nothing; e = 255 makes the outputs NaN"""
    E, H, I, k = 2, 512, 256, 1
    rng = np.random.default_rng(9)
    g = oracle.encode(1, (rng.standard_normal((E, I, H)) * 0.02).astype(np.float32))
    u = oracle.encode(1, (rng.standard_normal((E, I, H)) * 0.02).astype(np.float32))
    d = oracle.encode(1, (rng.standard_normal((E, H, I)) * 0.02).astype(np.float32))
    g = g.reshape(E, I, H // 32, 17)
    g[0, :, 3, 0] = 0
    g[1, 7, 5, 0] = 255
    g = g.reshape(E, I, -1)
    layer = m.Layer(1, H, I, E, layout=TC)
    layer.pack(m.MOE_SRC_BLOCKS, torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda(), torch.from_numpy(d).cuda())
    ws = layer.workspace(1, k)
    x = x_bf16_bits(9, [0], H)
    for e in range(E):
        y, _ = _decode(m, layer, ws, x, np.array([e]), np.array([1.0]), 1)
        yr, ab = oracle.moe_tokens(1, H, I, lambda q: g[q], lambda q: u[q], lambda q: d[q], np.array([[e]]),
                                   np.array([[1.0]], np.float32), x)
        tol_check(y, yr[0], ab[0], "expert %d" % e)
    assert np.all(np.isnan(y))


# ---------------------------------------------------------------- router and FFN in one launch
def _route_ffn(m, layer, ws, wr, x, k):
    T, H = x.shape
    idx = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
    w = torch.zeros((T, k), dtype=torch.float32, device=DEV)
    y = torch.full((T, H), float("nan"), device=DEV)
    m.moe_route_expert_ffn(layer, dev_bits(wr, DEV), dev_bits(x, DEV), T, k, idx, w, y, None, False, ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws) == 0
    return idx.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()


def _route_sep(m, wr, x, k):
    T, H = x.shape
    idx = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
    w = torch.zeros((T, k), dtype=torch.float32, device=DEV)
    m.moe_route_topk(dev_bits(wr, DEV), dev_bits(x, DEV), T, H, wr.shape[0], k, None, None, 0, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T", [1, 3, 8])
def test_tc_route_ffn_equals_route_then_verify_full_shape(m, big, T):
    """the fused call routes exactly as moe_route_topk and computes exactly what verify computes with that routing"""
    E, H, k, x, layer = (big[n] for n in ("E", "H", "k", "x", "layer"))
    wr = router_f16_bits(1000, 0, E, H)  # the router the fixture's routing came from
    ws = layer.workspace(8, k)
    fi, fw, fy = _route_ffn(m, layer, ws, wr, x[:T], k)
    si, sw = _route_sep(m, wr, x[:T], k)
    assert np.array_equal(fi, si) and np.array_equal(fw.view(np.uint32), sw.view(np.uint32))
    assert np.array_equal(fi, big["idx"][:T])
    yv = _verify(m, layer, ws, x[:T], si, sw, k)
    assert np.array_equal(fy.view(np.uint32), yv.view(np.uint32))


def test_tc_route_ffn_small_layer(m, small):
    W, layer = small
    E, H, k, T = 8, 512, 2, 5
    wr = router_f16_bits(7, 0, E, H)
    x = x_bf16_bits(7, range(T), H)
    ws = layer.workspace(8, k)
    fi, fw, fy = _route_ffn(m, layer, ws, wr, x, k)
    si, sw = _route_sep(m, wr, x, k)
    assert np.array_equal(fi, si) and np.array_equal(fw.view(np.uint32), sw.view(np.uint32))
    yr, ab = oracle_moe(MXFP4, W, si, sw, x)
    for t in range(T):
        tol_check(fy[t], yr[t], ab[t], "fused row %d" % t)
    # repeated calls reuse the workspace (its router counter is reset by the last CTA)
    fi2, fw2, fy2 = _route_ffn(m, layer, ws, wr, x, k)
    assert np.array_equal(fy2.view(np.uint32), fy.view(np.uint32))
