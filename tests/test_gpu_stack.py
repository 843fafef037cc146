"""The routed-expert stack end to end at a small shape: 3 hash-routed layers ("quant surgery", section 4: tid2eid)
then 2 softmax-routed layers ("Mixed-precision compression of DeepSeek-V4-Flash", "The recipe"), layer L + 1's x
= bf16(y_L / rms(y_L)) (the model normalises before each MoE layer). Every layer is checked against the oracle on
the GPU's own input to that layer: routing exactly (hash) or up to proven near-ties (softmax), y within
1e-3 * sum|terms| + 1e-6 per element, and the next layer's x within bf16 rounding of the oracle's normalised y. A verify pass of T tokens gives, at every layer, rows bit-identical to
decoding each token alone ("Width drift")."""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import router_f16_bits, tid2eid, token_ids, x_bf16_bits
from tests._harness import Weights, dev_bits, near_tie_ok, oracle_moe, tol_check

pytestmark = pytest.mark.gpu
DEV = "cuda"
MXFP4 = 1
H, I, E, K, V, NL, NH = 512, 256, 16, 6, 1000, 5, 3
SEED = 3


@pytest.fixture(scope="module")
def stack():
    import bit_moe_decode_gb300 as m
    from bit_moe_decode_gb300.stack import RoutedStack
    st = RoutedStack(H, I, E, K, NL, NH, V, T_max=8, device=DEV)
    Ws = [Weights(SEED, H, I, layer=L) for L in range(NL)]
    for L in range(NL):
        g = torch.from_numpy(np.stack([Ws[L].f32(e, 0) for e in range(E)])).to(DEV)
        u = torch.from_numpy(np.stack([Ws[L].f32(e, 1) for e in range(E)])).to(DEV)
        d = torch.from_numpy(np.stack([Ws[L].f32(e, 2) for e in range(E)])).to(DEV)
        st.layers[L].pack(m.MOE_SRC_F32, g, u, d, e0=0)
        if L < NH:
            st.tid2eid[L] = torch.from_numpy(tid2eid(SEED, L, V, E, K)).to(DEV)
        else:
            st.router[L] = dev_bits(router_f16_bits(SEED, L, E, H), DEV)
    torch.cuda.synchronize()
    return st, Ws


def _next_x_ok(x_bits: np.ndarray, y: np.ndarray) -> bool:
    """the next layer's bf16 x against the oracle's exact y / sqrt(mean(y^2) + eps), within bf16 rounding"""
    x = (x_bits.astype(np.uint32) << 16).view(np.float32)
    ref = oracle.rms_norm(y, 1e-6)
    return bool(np.all(np.abs(x - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30))


def _run(st, T, tok, x0):
    st.run(T, token_ids=torch.from_numpy(tok).to(DEV), x0=dev_bits(x0, DEV))
    torch.cuda.synchronize()
    xs = [x0] + [st.x[L + 1][:T].cpu().numpy().view(np.uint16) for L in range(NL)]
    return (xs, [st.idx[L][:T].cpu().numpy() for L in range(NL)], [st.w[L][:T].cpu().numpy() for L in range(NL)],
            [st.y[L][:T].cpu().numpy() for L in range(NL)])


def test_stack_layers_against_oracle(stack):
    st, Ws = stack
    T = 4
    tok = token_ids(SEED, T, V)
    x0 = x_bf16_bits(SEED, range(T), H)
    xs, idx, w, ys = _run(st, T, tok, x0)
    worst = 0.0
    for L in range(NL):
        if L < NH:
            ri, rw = oracle.route_hash(tok, tid2eid(SEED, L, V, E, K), K)
            assert np.array_equal(idx[L], ri), "layer %d: hash routing differs" % L
            assert np.array_equal(w[L].view(np.uint32), rw.view(np.uint32)), "layer %d: hash weights differ" % L
        else:
            ri, rw, lg, ab = oracle.route_topk(router_f16_bits(SEED, L, E, H), xs[L], K)
            for t in range(T):
                assert near_tie_ok(idx[L][t], ri[t], lg[t], ab[t], H), "layer %d token %d: routing differs" % (L, t)
        yr, yab = oracle_moe(MXFP4, Ws[L], idx[L], w[L], xs[L])
        for t in range(T):
            worst = max(worst, tol_check(ys[L][t], yr[t], yab[t], "layer %d token %d" % (L, t)))
        assert _next_x_ok(xs[L + 1], ys[L]), "layer %d: next x is not the normalised y" % L
    print("stack of %d layers (%d hash), T=%d: max err/bound %.3g" % (NL, NH, T, worst))


def test_stack_verify_rows_equal_decode(stack):
    st, _ = stack
    T = 5
    tok = token_ids(SEED + 1, T, V)
    x0 = x_bf16_bits(SEED + 1, range(T), H)
    xv, iv, _, yv = _run(st, T, tok, x0)
    for t in range(T):
        xd, idd, _, yd = _run(st, 1, tok[t:t + 1], x0[t:t + 1])
        for L in range(NL):
            assert np.array_equal(idd[L][0], iv[L][t]), "layer %d token %d: routing differs in the verify" % (L, t)
            assert np.array_equal(yd[L][0].view(np.uint32), yv[L][t].view(np.uint32)), \
                "layer %d: verify row %d differs from its decode" % (L, t)


# ---------------------------------------------------------------- the same stack with a Q8_0 shared expert per layer
Q8_0, IS = 4, 512   # the shared expert's format and intermediate size


@pytest.fixture(scope="module")
def stack_shared():
    import bit_moe_decode_gb300 as m
    from bit_moe_decode_gb300.stack import RoutedStack
    st = RoutedStack(H, I, E, K, NL, NH, V, T_max=8, device=DEV, shared_I=IS)
    Ws = [Weights(SEED, H, I, layer=L) for L in range(NL)]
    Wsh = [Weights(SEED + 50, H, IS, layer=L) for L in range(NL)]
    for L in range(NL):
        g, u, d = (torch.from_numpy(np.stack([Ws[L].f32(e, which) for e in range(E)])).to(DEV) for which in range(3))
        st.layers[L].pack(m.MOE_SRC_F32, g, u, d, e0=0)
        gs, us, ds = (torch.from_numpy(Wsh[L].f32(0, which)[None]).to(DEV) for which in range(3))
        st.shared[L].pack(m.MOE_SRC_F32, gs, us, ds, e0=0)
        if L < NH:
            st.tid2eid[L] = torch.from_numpy(tid2eid(SEED, L, V, E, K)).to(DEV)
        else:
            st.router[L] = dev_bits(router_f16_bits(SEED, L, E, H), DEV)
    torch.cuda.synchronize()
    return st, Ws, Wsh


def test_stack_with_shared_experts_against_oracle(stack_shared):
    st, Ws, Wsh = stack_shared
    T = 3
    tok = token_ids(SEED + 2, T, V)
    x0 = x_bf16_bits(SEED + 2, range(T), H)
    xs, idx, w, ys = _run(st, T, tok, x0)
    worst = 0.0
    for L in range(NL):
        if L < NH:
            ri, _ = oracle.route_hash(tok, tid2eid(SEED, L, V, E, K), K)
            assert np.array_equal(idx[L], ri), "layer %d: hash routing differs" % L
        else:
            ri, _, lg, ab = oracle.route_topk(router_f16_bits(SEED, L, E, H), xs[L], K)
            for t in range(T):
                assert near_tie_ok(idx[L][t], ri[t], lg[t], ab[t], H), "layer %d token %d: routing differs" % (L, t)
        yr, yab = oracle_moe(MXFP4, Ws[L], idx[L], w[L], xs[L])
        ysh, ysab = oracle_moe(Q8_0, Wsh[L], np.zeros((T, 1), np.int32), np.ones((T, 1), np.float32), xs[L])
        for t in range(T):
            worst = max(worst, tol_check(ys[L][t], yr[t] + ysh[t], yab[t] + ysab[t], "layer %d token %d" % (L, t)))
        assert _next_x_ok(xs[L + 1], ys[L]), "layer %d: next x is not the normalised y" % L
    print("stack with shared experts, T=%d: max err/bound %.3g" % (T, worst))


def test_stack_with_shared_experts_verify_rows_equal_decode(stack_shared):
    st, _, _ = stack_shared
    T = 4
    tok = token_ids(SEED + 3, T, V)
    x0 = x_bf16_bits(SEED + 3, range(T), H)
    _, iv, _, yv = _run(st, T, tok, x0)
    for t in range(T):
        _, idd, _, yd = _run(st, 1, tok[t:t + 1], x0[t:t + 1])
        for L in range(NL):
            assert np.array_equal(idd[L][0], iv[L][t])
            assert np.array_equal(yd[L][0].view(np.uint32), yv[L][t].view(np.uint32)), \
                "layer %d: verify row %d differs from its decode" % (L, t)
