"""The always-on shared expert in Q8_0 added to the routed output: the routed layer writes y (fp32), then the shared
expert runs as a one-expert layer (idx = 0, w = 1) with accumulate = 1 and writes the bf16 copy
("Mixed-precision compression of DeepSeek-V4-Flash", "The recipe": the shared expert stays in 8 bits while the
routed experts are quantised harder). Each token against the oracle's routed output plus its shared-expert output
(|y - y_ref| <= 1e-3 * (sum|routed terms| + sum|shared terms|) + 1e-6), verify rows bit-identical to decoding each
token alone, and the bf16 copy equal to the round-to-nearest-even of the fp32 result."""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import router_f16_bits, x_bf16_bits
from tests._harness import Weights, dev_bits, make_layer, oracle_moe, tol_check

pytestmark = pytest.mark.gpu
DEV = "cuda"
MXFP4, Q8_0, TC = 1, 4, 1


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


def _t(a, dt):
    return torch.from_numpy(np.ascontiguousarray(a, dt)).to(DEV)


def _routed_plus_shared(m, routed, shared, ws_r, ws_s, x, idx, w, k, verify):
    """routed FFN (y only), then the shared expert accumulated into y with the bf16 copy written"""
    T, H = x.shape
    y = torch.full((T, H), float("nan"), device=DEV)
    yb = torch.zeros((T, H), dtype=torch.int16, device=DEV)
    xd = dev_bits(x, DEV)
    one_i, one_w = _t(np.zeros((T, 1)), np.int32), _t(np.ones((T, 1)), np.float32)
    if verify:
        m.moe_expert_ffn_verify(routed, xd, T, _t(idx, np.int32), _t(w, np.float32), k, y, None, False, ws_r)
        m.moe_expert_ffn_verify(shared, xd, T, one_i, one_w, 1, y, yb, True, ws_s)
    else:
        assert T == 1
        m.moe_expert_ffn_decode(routed, xd, _t(idx, np.int32), _t(w, np.float32), k, y, None, False, ws_r)
        m.moe_expert_ffn_decode(shared, xd, one_i, one_w, 1, y, yb, True, ws_s)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws_r) == 0 and m.moe_get_device_status(ws_s) == 0
    return y.cpu().numpy(), yb.cpu().numpy().view(np.uint16)


def _bf16_rne(y):
    b = np.ascontiguousarray(y, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _reference(W, Ws, idx, w, x):
    T = x.shape[0]
    yr, ab = oracle_moe(MXFP4, W, idx, w, x)
    ys, abs_ = oracle_moe(Q8_0, Ws, np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32), x)
    return yr + ys, ab + abs_


@pytest.mark.parametrize("layout", [0, TC], ids=["decode_layout", "tc_layout"])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_routed_plus_shared_small(m, layout, T):
    E, H, I, k = 16, 1024, 512, 4
    W, Ws = Weights(3, H, I), Weights(31, H, I)
    routed = make_layer(m, MXFP4, W, E, range(E), DEV, layout=layout)
    shared = make_layer(m, Q8_0, Ws, 1, [0], DEV)
    ws_r, ws_s = routed.workspace(8, k), shared.workspace(8, 1)
    x = x_bf16_bits(40 + T, range(T), H)
    idx, w, _, _ = oracle.route_topk(router_f16_bits(40 + T, 0, E, H), x, k)
    yv, ybv = _routed_plus_shared(m, routed, shared, ws_r, ws_s, x, idx, w, k, verify=True)
    yref, ab = _reference(W, Ws, idx, w, x)
    worst = 0.0
    for t in range(T):
        worst = max(worst, tol_check(yv[t], yref[t], ab[t], "token %d" % t))
        yd, ybd = _routed_plus_shared(m, routed, shared, ws_r, ws_s, x[t:t + 1], idx[t:t + 1], w[t:t + 1], k,
                                      verify=False)
        assert np.array_equal(yv[t].view(np.uint32), yd[0].view(np.uint32)), "verify row %d differs" % t
        assert np.array_equal(ybd[0], ybv[t])
    assert np.array_equal(ybv, _bf16_rne(yv))
    print("routed + shared, layout %d, T=%d: max err/bound %.3g" % (layout, T, worst))


def test_routed_plus_shared_full_shape(m):
    """hidden 4096, intermediate 2048, 256 routed experts (top-6, tensor-core layout) plus one Q8_0 shared expert of
    the same intermediate size, two tokens"""
    E, H, I, k, T = 256, 4096, 2048, 6, 2
    W, Ws = Weights(5, H, I), Weights(55, H, I)
    x = x_bf16_bits(77, range(T), H)
    idx, w, _, _ = oracle.route_topk(router_f16_bits(77, 0, E, H), x, k)
    routed = make_layer(m, MXFP4, W, E, np.unique(idx), DEV, layout=TC)
    shared = make_layer(m, Q8_0, Ws, 1, [0], DEV)
    ws_r, ws_s = routed.workspace(8, k), shared.workspace(8, 1)
    yv, ybv = _routed_plus_shared(m, routed, shared, ws_r, ws_s, x, idx, w, k, verify=True)
    yref, ab = _reference(W, Ws, idx, w, x)
    for t in range(T):
        r = tol_check(yv[t], yref[t], ab[t], "token %d" % t)
        yd, _ = _routed_plus_shared(m, routed, shared, ws_r, ws_s, x[t:t + 1], idx[t:t + 1], w[t:t + 1], k,
                                    verify=False)
        assert np.array_equal(yv[t].view(np.uint32), yd[0].view(np.uint32))
        print("full shape token %d: max err/bound %.3g" % (t, r))
    assert np.array_equal(ybv, _bf16_rne(yv))


def test_shared_expert_alone_matches_oracle_expert_ffn(m):
    """the shared layer by itself (accumulate = 0) equals the oracle's single-expert FFN d, full shape"""
    H, I = 4096, 2048
    Ws = Weights(56, H, I)
    shared = make_layer(m, Q8_0, Ws, 1, [0], DEV)
    ws = shared.workspace(1, 1)
    x = x_bf16_bits(78, range(1), H)
    y = torch.full((1, H), float("nan"), device=DEV)
    m.moe_expert_ffn_decode(shared, dev_bits(x, DEV), _t([[0]], np.int32), _t([[1.0]], np.float32), 1, y, None, False,
                            ws)
    torch.cuda.synchronize()
    assert m.moe_get_device_status(ws) == 0
    out = oracle.expert_ffn(Q8_0, H, I, Ws.blocks(Q8_0, 0, 0), Ws.blocks(Q8_0, 0, 1), Ws.blocks(Q8_0, 0, 2),
                            (x.astype(np.uint32) << 16).view(np.float32)[0].astype(np.float64))
    tol_check(y.cpu().numpy()[0], out["d"], out["dabs"], "shared expert alone")


def test_q8_0_has_no_tc_layout(m):
    assert m.moe_packed_bytes(Q8_0, TC, 0, 1, 4096, 2048) == 0
    with pytest.raises(m.MoeError):
        m.Layer(Q8_0, 4096, 2048, 1, layout=TC, device=DEV)
