"""Prefill grouped GEMM (block-scaled MXFP4 x MXFP8 on the tensor cores) against the oracle, stage by stage.

The oracle quantises x and h to MXFP8 per 32 exactly as the library does ("quantization" glossary, "V4.1 Flash":
E4M3 codes with one E8M0 exponent per 32), but computes g, u and h in fp64. Checks:
  (a) the MXFP8 codes and exponents of x: bit-exact;
  (b) g and u (fp32 accumulators of the gate/up GEMM): |gpu - ref| <= 1e-3 * sum_k |W_ik xq_k| + 1e-6;
  (c) the MXFP8 codes and exponents of h: equal except where an ulp-level difference of g or u moves h across a
      rounding boundary of E4M3 ("flips"), which are counted, must be rare and at most one code step;
  (d) the down GEMM on the GPU's own quantised h: |gpu - ref| <= 1e-3 * sum_i |Down_ji hq_i| + 1e-6;
  (e) y end to end within 1e-3 * sum|terms| + 1e-6 (flips included), and y_bf16 == RNE(y) bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import x_bf16_bits, zipf_routing
from tests._harness import Weights, dev_bits, make_layer, tol_check

pytestmark = pytest.mark.gpu
DEV = "cuda"
MXFP4, PREFILL = 1, 1


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


def _bf16_values(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _e4m3(codes):
    tab = np.array([oracle.e4m3_value(c) for c in range(256)])
    return tab[np.asarray(codes, np.int64)]


def _e8m0(scales):
    return np.ldexp(1.0, np.asarray(scales, np.int64) - 127)


def _unpermute_sf(blocks, rows_in_tile):
    """[tiles, KG, 512] permuted exponents -> [tiles*128, KG*4] (row, 32-block)."""
    tiles, KG, _ = blocks.shape
    b = blocks.reshape(tiles, KG, 32, 4, 4)           # [tile][kg][l][c][kb], row = l + 32c
    return b.transpose(0, 3, 2, 1, 4).reshape(tiles * 128, KG * 4)


def _act_tiles(r, name, tiles, K):
    """Tile-major MXFP8 buffer -> (codes [tiles*128, K], exponents [tiles*128, K/32])."""
    KG = K // 128
    a = _ws_view(r, name, np.uint8, tiles * KG * 16896, (tiles, KG, 16896))
    codes = a[:, :, :16384].reshape(tiles, KG, 128, 128).transpose(0, 2, 1, 3).reshape(tiles * 128, K)
    return codes, _unpermute_sf(np.ascontiguousarray(a[:, :, 16384:]), 128)


def _rne_bf16_bits(y32):
    b = np.asarray(y32, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _run(m, layer, x, idx, w, k, gu=True):
    T, H = x.shape
    I = layer.I
    ws = layer.prefill_workspace(T, k)
    assert ws.numel() == m.moe_prefill_workspace_bytes(layer, T, k)
    y = torch.full((T, H), float("nan"), device=DEV)
    yb = torch.zeros((T, H), dtype=torch.int16, device=DEV)
    gud = None
    if gu:
        # rows of the sorted buffers: 128 per tile, at most ceil(T k / 128) + min(E, T k) tiles
        npairs = T * k
        rows_max = ((npairs + 127) // 128 + min(layer.E, npairs)) * 128
        gud = torch.full((rows_max, 2 * I), float("nan"), device=DEV)
    off = m.moe_debug_prefill(layer, dev_bits(x, DEV), T, torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(DEV),
                              torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(DEV), k, y, yb, ws, gud)
    torch.cuda.synchronize()
    status = m.moe_get_device_status(ws)
    wsn = ws.cpu().numpy()
    return dict(y=y.cpu().numpy(), yb=yb.cpu().numpy().view(np.uint16), ws=wsn, off=off, status=status,
                gu=None if gud is None else gud.cpu().numpy())


def _ws_view(r, name, dtype, count, shape=None):
    a = np.frombuffer(r["ws"][r["off"][name]:].tobytes()[:count * np.dtype(dtype).itemsize], dtype=dtype)
    return a.reshape(shape) if shape is not None else a


def _stages(m, W, E, H, I, T, k, idx, w, x, r, sample):
    off = r["off"]
    rows_max, tiles_max = off["rows_max"], off["tiles_max"]
    n_tiles = int(_ws_view(r, "n_tiles", np.uint32, 1)[0])
    pair_row = _ws_view(r, "pair_row", np.int32, T * k).reshape(T, k)
    tile_first = _ws_view(r, "tile_first", np.int32, tiles_max)
    xq, xsf = _act_tiles(r, "xq", tiles_max, H)
    hq, hsf = _act_tiles(r, "hq", tiles_max, I)
    dout = _ws_view(r, "dout", np.float32, T * k * H, (T * k, H))
    # bucketing: rows are distinct, inside the used tiles, grouped by expert in (token, rank) order
    rows = pair_row.reshape(-1)
    assert np.all(rows >= 0) and len(set(rows.tolist())) == rows.size and rows.max() < n_tiles * 128
    for e in np.unique(idx):
        pr = rows[idx.reshape(-1) == e]
        assert np.all(np.diff(pr) == 1), "expert %d rows not contiguous in pair order" % e
        assert pr[0] % 128 == 0
    flips = 0
    nh = 0
    dec = {}

    def mats(e):
        if e not in dec:
            dec[e] = [oracle.decode(MXFP4, W.blocks(MXFP4, e, j)).astype(np.float64).reshape(
                (I, H) if j < 2 else (H, I)) for j in range(3)]
        return dec[e]

    for t in sample:
        out = oracle.prefill_token(H, I, lambda e: W.blocks(MXFP4, e, 0), lambda e: W.blocks(MXFP4, e, 1),
                                   lambda e: W.blocks(MXFP4, e, 2), idx[t], w[t], x[t])
        xqv = _e4m3(out["xq_codes"]) * np.repeat(_e8m0(out["xq_scales"]), 32)
        for rk in range(k):
            row = pair_row[t, rk]
            # (a) x codes and exponents
            assert np.array_equal(xq[row], out["xq_codes"]), "x codes token %d" % t
            assert np.array_equal(xsf[row], out["xq_scales"]), "x exponents token %d" % t
            G, U, D = mats(int(idx[t, rk]))
            # (b) g and u
            if r["gu"] is not None:
                g_ref, u_ref = G @ xqv, U @ xqv
                tol_check(r["gu"][row, :I], g_ref, np.abs(G) @ np.abs(xqv), "g token %d rank %d" % (t, rk))
                tol_check(r["gu"][row, I:], u_ref, np.abs(U) @ np.abs(xqv), "u token %d rank %d" % (t, rk))
            # (c) h codes: count flips, each at most one code step within the same exponent
            hc, hs = out["hq_codes"][rk], out["hq_scales"][rk]
            nh += I
            if not np.array_equal(hsf[row], hs):
                flips += int(np.sum(np.repeat(hsf[row] != hs, 32)))
            same = np.repeat(hsf[row] == hs, 32)
            dc = np.abs(hq[row].astype(np.int64) - hc.astype(np.int64))
            assert np.all(dc[same] <= 1), "h code off by more than one step"
            flips += int(np.sum(dc[same] != 0))
            # (d) down GEMM on the GPU's own h
            hqv = _e4m3(hq[row]) * np.repeat(_e8m0(hsf[row]), 32)
            crow = tile_first[row // 128] + row % 128
            tol_check(dout[crow], D @ hqv, np.abs(D) @ np.abs(hqv) + 0.0, "down token %d rank %d" % (t, rk))
        # (e) end to end
        tol_check(r["y"][t], out["y"], out["absterm"], "y token %d" % t)
    assert flips <= max(2, nh // 1000), "%d h flips out of %d" % (flips, nh)
    assert np.array_equal(r["yb"], _rne_bf16_bits(r["y"]))
    return flips, nh


@pytest.mark.parametrize("T,k,seed", [(300, 2, 0), (1, 1, 1), (64, 8, 2)])
def test_prefill_small_stagewise(m, T, k, seed):
    E, H, I = 8, 512, 256
    W = Weights(40 + seed, H, I)
    layer = make_layer(m, MXFP4, W, E, range(E), DEV, layout=PREFILL)
    x = x_bf16_bits(40 + seed, range(T), H)
    idx, w = zipf_routing(40 + seed, T, E, k)
    r = _run(m, layer, x, idx, w, k)
    assert r["status"] == 0
    flips, nh = _stages(m, W, E, H, I, T, k, idx, w, x, r, range(T))
    print("prefill small T=%d k=%d: %d h flips / %d" % (T, k, flips, nh))


def test_prefill_tile_boundaries(m):
    """Experts with exactly 128, 129 and 127 pairs, one with 1, and one with none."""
    E, H, I, k = 8, 512, 256, 1
    W = Weights(47, H, I)
    layer = make_layer(m, MXFP4, W, E, range(E), DEV, layout=PREFILL)
    counts = {0: 128, 3: 129, 5: 127, 6: 1}
    idx = np.concatenate([np.full(c, e, np.int32) for e, c in counts.items()])
    rng = np.random.default_rng(47)
    idx = idx[rng.permutation(idx.size)].reshape(-1, 1)
    T = idx.shape[0]
    w = np.ones((T, 1), np.float32)
    x = x_bf16_bits(47, range(T), H)
    r = _run(m, layer, x, idx, w, k)
    assert r["status"] == 0
    _stages(m, W, E, H, I, T, k, idx, w, x, r, [int(i) for i in rng.choice(T, 24, replace=False)])


def test_prefill_full_shape_sampled(m):
    """Hidden 4096, intermediate 2048, 256 expert slots, top-6, 1024 tokens routed (Zipf) over 16 of the experts
    so that every expert spans several 128-row tiles with a ragged last tile; 6 tokens checked stage by stage."""
    E, H, I, k, T = 256, 4096, 2048, 6, 1024
    W = Weights(48, H, I)
    used = np.random.default_rng(48).choice(E, 16, replace=False)
    sub, w = zipf_routing(48, T, 16, k)
    idx = used[sub].astype(np.int32)
    layer = make_layer(m, MXFP4, W, E, used, DEV, layout=PREFILL)
    x = x_bf16_bits(48, range(T), H)
    r = _run(m, layer, x, idx, w, k)
    assert r["status"] == 0
    assert np.all(np.isfinite(r["y"]))
    flips, nh = _stages(m, W, E, H, I, T, k, idx, w, x, r, [0, 1, 511, 777, 1022, 1023])
    print("prefill full shape: %d h flips / %d" % (flips, nh))


def test_prefill_duplicate_and_invalid_ids(m):
    E, H, I, k, T = 8, 512, 256, 2, 4
    W = Weights(49, H, I)
    layer = make_layer(m, MXFP4, W, E, range(E), DEV, layout=PREFILL)
    x = x_bf16_bits(49, range(T), H)
    idx = np.array([[3, 3], [1, 2], [2, 9], [0, 7]], np.int32)
    w = np.array([[0.25, 0.75], [0.5, 0.5], [0.6, 0.4], [0.9, 0.1]], np.float32)
    r = _run(m, layer, x, idx, w, k, gu=False)
    assert r["status"] == 2 - 1  # MOE_ERR_INVALID_ARG: expert 9 is not < E
    for t in (0, 1, 3):
        out = oracle.prefill_token(H, I, lambda e: W.blocks(MXFP4, e, 0), lambda e: W.blocks(MXFP4, e, 1),
                                   lambda e: W.blocks(MXFP4, e, 2), idx[t], w[t], x[t])
        tol_check(r["y"][t], out["y"], out["absterm"], "token %d" % t)
    # token 2: only its valid pair (expert 2, weight 0.6) contributes
    out = oracle.prefill_token(H, I, lambda e: W.blocks(MXFP4, e, 0), lambda e: W.blocks(MXFP4, e, 1),
                               lambda e: W.blocks(MXFP4, e, 2), idx[2, :1], w[2, :1], x[2])
    tol_check(r["y"][2], out["y"], out["absterm"], "token 2")


def test_prefill_layout_unpacks_to_oracle_values(m):
    E, H, I = 2, 512, 256
    W = Weights(50, H, I)
    for src in (m.MOE_SRC_F32, m.MOE_SRC_BLOCKS):
        layer = m.Layer(MXFP4, H, I, E, layout=PREFILL, device=DEV)
        for e in range(E):
            if src == m.MOE_SRC_F32:
                mats = [torch.from_numpy(W.f32(e, j)).to(DEV)[None] for j in range(3)]
            else:
                mats = [torch.from_numpy(np.ascontiguousarray(W.blocks(MXFP4, e, j))).to(DEV)[None] for j in range(3)]
            layer.pack(src, *mats, e0=e)
        for e in range(E):
            gu = torch.empty((2, I, H), device=DEV)
            dn = torch.empty((H, I), device=DEV)
            m.moe_debug_unpack(MXFP4, PREFILL, m.MOE_MAT_GATE_UP, layer.gate_up, H, I, e, gu)
            m.moe_debug_unpack(MXFP4, PREFILL, m.MOE_MAT_DOWN, layer.down, H, I, e, dn)
            torch.cuda.synchronize()
            for j, got in ((0, gu[0]), (1, gu[1]), (2, dn)):
                ref = oracle.decode(MXFP4, W.blocks(MXFP4, e, j))
                assert np.array_equal(got.cpu().numpy().reshape(-1).view(np.uint32), ref.view(np.uint32))


def test_prefill_host_errors(m):
    E, H, I, k, T = 8, 512, 256, 2, 4
    dec = m.Layer(MXFP4, H, I, E, device=DEV)
    pre = m.Layer(MXFP4, H, I, E, layout=PREFILL, device=DEV)
    ws = pre.prefill_workspace(T, k)
    x = torch.zeros((T, H), dtype=torch.int16, device=DEV)
    idx = torch.zeros((T, k), dtype=torch.int32, device=DEV)
    w = torch.zeros((T, k), device=DEV)
    y = torch.zeros((T, H), device=DEV)
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_grouped_gemm_prefill(dec, x, T, idx, w, k, y, None, ws)
    assert ei.value.status == 3
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_grouped_gemm_prefill(pre, x, T, idx, w, k, y, None, ws[:ws.numel() // 2])
    assert ei.value.status == 5
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_grouped_gemm_prefill(pre, x, T, idx, w, 9, y, None, ws)
    assert ei.value.status == 2
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_grouped_gemm_prefill(pre, x, T, idx, w, k, None, None, ws)
    assert ei.value.status == 1
    assert m.moe_packed_bytes(2, PREFILL, 0, 1, H, I) == 0  # INT4 has no prefill layout
