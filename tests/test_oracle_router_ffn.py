"""Pins of the oracle's router, expert FFN, MoE combine and prefill path.

Expected values come from brute force (sorting), closed forms on hand-built integer cases, and an
independent numpy/scipy/torch computation of the same definition (decode -> float64 matmul -> SiLU ->
matmul -> weighted sum), which would catch a transposed operand, a dropped term, a wrong sign or index.
"""
import numpy as np
import pytest
import scipy.special
import torch

import oracle
from moe_inputs import f32_to_bf16_bits, router_f16_bits, x_bf16_bits, expert_matrix_f32, tid2eid, token_ids

# ---------------------------------------------------------------- helpers (independent numpy path)


def _bf16_values(bits):
    return torch.from_numpy(np.asarray(bits, np.uint16).view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def _f16_values(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _np_expert(fmt, H, I, gate, up, down, x):
    G = oracle.decode(fmt, gate).astype(np.float64).reshape(I, H)
    U = oracle.decode(fmt, up).astype(np.float64).reshape(I, H)
    D = oracle.decode(fmt, down).astype(np.float64).reshape(H, I)
    g, u = G @ x, U @ x
    h = g * scipy.special.expit(g) * u
    return g, u, h, D @ h, np.abs(D) @ np.abs(h)


def _layer(fmt, E, H, I, seed=0):
    enc = lambda which: np.stack([oracle.encode(fmt, expert_matrix_f32(seed, 0, e, which, H, I)) for e in range(E)])
    return enc(0), enc(1), enc(2)


# ---------------------------------------------------------------- router
def test_router_matches_sort_and_scipy_softmax():
    E, H, T, k = 16, 96, 12, 4
    wr = router_f16_bits(3, 0, E, H)
    x = x_bf16_bits(3, range(T), H)
    idx, w, logits, absl = oracle.route_topk(wr, x, k)
    ref_l = _bf16_values(x) @ _f16_values(wr).T
    assert np.allclose(logits, ref_l, rtol=0, atol=1e-12 * np.abs(absl).max())
    assert np.allclose(absl, np.abs(_bf16_values(x)) @ np.abs(_f16_values(wr)).T, rtol=1e-12)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t]))[:k]   # by -logit, then index
        assert np.array_equal(idx[t], order)
        sm = scipy.special.softmax(logits[t])
        ref_w = sm[order] / sm[order].sum()
        assert np.allclose(w[t], ref_w.astype(np.float32), rtol=1e-6, atol=0)
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) < 1e-6


def test_router_ties_go_to_lower_index():
    E, H, k = 8, 64, 3
    rng = np.random.default_rng(0)
    row = (rng.standard_normal(H) * 0.02).astype(np.float16).view(np.uint16)
    wr = np.tile(row, (E, 1))                      # all logits equal
    x = f32_to_bf16_bits(rng.standard_normal((2, H)).astype(np.float32))
    idx, w, _, _ = oracle.route_topk(wr, x, k)
    assert np.array_equal(idx, [[0, 1, 2], [0, 1, 2]])
    assert np.allclose(w, 1.0 / 3, rtol=1e-7)
    # expert 5 strictly larger, 2 and 6 tied second: order 5, 2, 6
    wr2 = np.zeros((E, H), np.uint16)
    one = np.float16(1.0).view(np.uint16)
    xx = np.zeros((1, H), np.uint16)
    xx[0, 0] = f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    wr2[5, 0] = np.float16(3.0).view(np.uint16)
    wr2[2, 0] = one
    wr2[6, 0] = one
    idx2, w2, l2, _ = oracle.route_topk(wr2, xx, 3)
    assert list(idx2[0]) == [5, 2, 6]
    e = np.exp(np.array([3.0, 1.0, 1.0]) - 3.0)
    assert np.allclose(w2[0], (e / e.sum()).astype(np.float32), rtol=1e-7)


def test_hash_routing_gathers_table_with_equal_weights():
    V, E, k, T = 1000, 64, 6, 50
    tab = tid2eid(1, 0, V, E, k)
    assert all(len(set(r)) == k for r in tab)
    tok = token_ids(1, T, V)
    idx, w = oracle.route_hash(tok, tab, k)
    assert np.array_equal(idx, tab[tok])
    assert np.all(w == np.float32(1.0 / 6))


# ---------------------------------------------------------------- expert FFN
def test_ffn_integer_case_is_exact():
    """MXFP4 with e = 127 and codes of +-1, +-2, x small integers: g and u are exact integers."""
    H, I = 64, 32
    rng = np.random.default_rng(1)
    tab_codes = np.array([2, 4, 10, 12])          # 1, 2, -1, -2

    def mat(rows, K):
        c = rng.choice(tab_codes, size=(rows, K))
        raw = np.zeros((rows, K // 32, 17), np.uint8)
        raw[..., 0] = 127
        cc = c.reshape(rows, K // 32, 16, 2)
        raw[..., 1:] = (cc[..., 0] << 4) | cc[..., 1]
        vals = np.select([c == 2, c == 4, c == 10, c == 12], [1.0, 2.0, -1.0, -2.0])
        return raw.reshape(rows, -1), vals

    gb, gv = mat(I, H)
    ub, uv = mat(I, H)
    db, dv = mat(H, I)
    xi = rng.integers(-3, 4, size=H).astype(np.float64)
    out = oracle.expert_ffn(oracle.MXFP4, H, I, gb, ub, db, xi)
    assert np.array_equal(out["g"], gv @ xi) and np.array_equal(out["u"], uv @ xi)
    h = (gv @ xi) / (1 + np.exp(-(gv @ xi))) * (uv @ xi)
    assert np.allclose(out["h"], h, rtol=1e-15, atol=0)
    assert np.allclose(out["d"], dv @ h, rtol=1e-13, atol=1e-12)


@pytest.mark.parametrize("fmt", [oracle.MXFP4, oracle.INT4G32, oracle.Q2K, oracle.Q8_0])
def test_ffn_random_matches_numpy_path(fmt):
    H, I = 512, 256
    g, u, d = (oracle.encode(fmt, expert_matrix_f32(7, 0, 3, which, H, I)) for which in range(3))
    x = _bf16_values(x_bf16_bits(7, [0], H)[0])
    out = oracle.expert_ffn(fmt, H, I, g, u, d, x)
    rg, ru, rh, rd, rabs = _np_expert(fmt, H, I, g, u, d, x)
    scale = np.abs(oracle.decode(fmt, g).reshape(I, H)) @ np.abs(x)
    assert np.all(np.abs(out["g"] - rg) <= 1e-13 * scale)
    assert np.allclose(out["h"], rh, rtol=1e-10, atol=1e-14)
    assert np.all(np.abs(out["d"] - rd) <= 1e-12 * rabs + 1e-15)
    assert np.allclose(out["dabs"], rabs, rtol=1e-12)


@pytest.mark.parametrize("fmt", [oracle.MXFP4, oracle.Q2K, oracle.Q8_0])
def test_moe_combine_batch_and_token_agree_with_numpy(fmt):
    E, H, I, k, T = 8, 512, 256, 2, 5
    G, U, D = _layer(fmt, E, H, I, seed=2)
    wr = router_f16_bits(2, 0, E, H)
    x = x_bf16_bits(2, range(T), H)
    idx, w, _, _ = oracle.route_topk(wr, x, k)
    y, ab = oracle.moe_batch(fmt, H, I, G, U, D, idx, w, x, threads=2)
    y2, ab2 = oracle.moe_tokens(fmt, H, I, lambda e: G[e], lambda e: U[e], lambda e: D[e], idx, w, x)
    assert np.array_equal(y, y2) and np.array_equal(ab, ab2)
    for t in range(T):
        xv = _bf16_values(x[t])
        ref = np.zeros(H)
        rab = np.zeros(H)
        for r in range(k):
            e = idx[t, r]
            *_, rd, rabs = _np_expert(fmt, H, I, G[e], U[e], D[e], xv)
            ref += np.float64(w[t, r]) * rd
            rab += abs(np.float64(w[t, r])) * rabs
        assert np.all(np.abs(y[t] - ref) <= 1e-12 * rab + 1e-15)
        assert np.allclose(ab[t], rab, rtol=1e-12)


def test_single_expert_weight_one_is_the_expert_output():
    E, H, I = 4, 256, 128
    G, U, D = _layer(oracle.MXFP4, E, H, I, seed=4)
    x = x_bf16_bits(4, [0], H)
    y, _ = oracle.moe_batch(oracle.MXFP4, H, I, G, U, D, np.array([[2]]), np.array([[1.0]], np.float32), x)
    d = oracle.expert_ffn(oracle.MXFP4, H, I, G[2], U[2], D[2], _bf16_values(x[0]))["d"]
    assert np.array_equal(y[0], d)


# ---------------------------------------------------------------- prefill (MXFP8 activations)
def _q8_torch(v64):
    """MXFP8 of a float64 vector via torch's float8_e4m3fn conversion (library routine)."""
    v = v64.reshape(-1, 32)
    out = np.empty_like(v)
    for b in range(v.shape[0]):
        amax = np.max(np.abs(v[b]))
        k = int(np.ceil(np.log2(amax / 448.0))) if amax > 0 else -200
        while amax > 448 * 2.0 ** k:
            k += 1
        while amax > 0 and amax <= 448 * 2.0 ** (k - 1):
            k -= 1
        e = min(max(k + 127, 1), 254)
        q = torch.from_numpy(v[b] * 2.0 ** (127 - e)).to(torch.float8_e4m3fn).double().numpy()
        out[b] = q * 2.0 ** (e - 127)
    return out.reshape(-1)


def test_prefill_token_matches_torch_float8_path():
    E, H, I, k = 6, 512, 256, 2
    G, U, D = _layer(oracle.MXFP4, E, H, I, seed=5)
    x = x_bf16_bits(5, [0], H)[0]
    idx = [4, 1]
    w = np.array([0.3, 0.7], np.float32)
    out = oracle.prefill_token(H, I, lambda e: G[e], lambda e: U[e], lambda e: D[e], idx, w, x)
    xq = _q8_torch(_bf16_values(x))
    ref = np.zeros(H)
    flips = 0
    for r, e in enumerate(idx):
        Gm = oracle.decode(oracle.MXFP4, G[e]).astype(np.float64).reshape(I, H)
        Um = oracle.decode(oracle.MXFP4, U[e]).astype(np.float64).reshape(I, H)
        Dm = oracle.decode(oracle.MXFP4, D[e]).astype(np.float64).reshape(H, I)
        g, u = Gm @ xq, Um @ xq
        h = (g * scipy.special.expit(g) * u).astype(np.float32).astype(np.float64)
        hq = _q8_torch(h)
        ohq = np.array([oracle.e4m3_value(c) for c in out["hq_codes"][r]]) * \
            np.repeat([oracle.e8m0_scale(s) for s in out["hq_scales"][r]], 32)
        flips += int(np.sum(ohq != hq))
        ref += np.float64(w[r]) * (Dm @ ohq)
    assert flips <= 2                      # fp64 sum-order differences may flip a rounding of h, rarely
    assert np.all(np.abs(out["y"] - ref) <= 1e-12 * out["absterm"] + 1e-15)
    oxq = np.array([oracle.e4m3_value(c) for c in out["xq_codes"]]) * \
        np.repeat([oracle.e8m0_scale(s) for s in out["xq_scales"]], 32)
    assert np.array_equal(oxq, xq)


# ---------------------------------------------------------------- RMS normalisation between stacked layers
def test_rms_norm_closed_forms():
    """[3, 4]: mean square 12.5; a constant row c: every output c / sqrt(c^2 + eps); zeros stay zeros; the result
    has unit mean square when eps = 0; scaling a row does not change it (eps = 0)."""
    y = np.array([[3.0, 4.0], [2.5, 2.5], [0.0, 0.0]], np.float32)
    out = oracle.rms_norm(y, 1e-6)
    assert np.allclose(out[0], np.array([3.0, 4.0]) / np.sqrt(12.5 + 1e-6), rtol=1e-15, atol=0)
    assert np.allclose(out[1], 2.5 / np.sqrt(6.25 + 1e-6), rtol=1e-15, atol=0)
    assert np.array_equal(out[2], [0.0, 0.0])
    rng = np.random.default_rng(5)
    z = (rng.standard_normal((4, 1000)) * 7.0).astype(np.float32)
    n0 = oracle.rms_norm(z, 0.0)
    assert np.allclose(np.mean(n0 ** 2, axis=1), 1.0, rtol=1e-13)
    assert np.allclose(oracle.rms_norm(z * np.float32(0.25), 0.0), n0, rtol=1e-13)   # exact power-of-two scale
