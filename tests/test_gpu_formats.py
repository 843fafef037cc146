"""GPU encoders and the packed layout against the oracle, bit for bit (integer/byte work: exact)."""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import expert_matrix_f32
from tests._harness import FMTS, FMT_NAME

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


def _edge_rows(rng, K):
    rows = [rng.standard_normal(K) * 0.02, rng.standard_normal(K) * 1e-30, rng.standard_normal(K) * 1e30,
            np.zeros(K), -np.zeros(K), rng.standard_normal(K) * 10.0 ** rng.integers(-8, 8, K)]
    ties = np.tile(np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -2.5, -5.0, 3.0, -6.0, 0.5, 1.0]), K // 16)
    rows.append(ties * 2.0 ** -7)
    r = rng.standard_normal(K)
    r[::7] = 0.0
    r[3::11] = -0.0
    rows.append(r * 0.02)
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("fmt", FMTS, ids=[FMT_NAME[f] for f in FMTS])
def test_gpu_encoder_bit_exact(m, fmt):
    rng = np.random.default_rng(100 + fmt)
    K = 512
    w = np.concatenate([_edge_rows(rng, K), (rng.standard_normal((56, K)) * 0.02).astype(np.float32)])
    ref = oracle.encode(fmt, w)
    src = torch.from_numpy(w).cuda()
    dst = torch.zeros(ref.size, dtype=torch.uint8, device="cuda")
    m.moe_encode_blocks(fmt, src, w.shape[0], K, dst)
    got = dst.cpu().numpy().reshape(ref.shape)
    bad = np.argwhere(got != ref)
    if bad.size:
        bs, nb = oracle.BLOCK[fmt]
        r, c = bad[0]
        b0 = (c // nb) * nb
        msg = "first mismatch row %d block %d: gpu %s oracle %s (of %d bytes)" % (
            r, c // nb, got[r, b0:b0 + nb].tobytes().hex(), ref[r, b0:b0 + nb].tobytes().hex(), bad.shape[0])
        raise AssertionError(msg)


@pytest.mark.parametrize("fmt", FMTS, ids=[FMT_NAME[f] for f in FMTS])
def test_gpu_encoder_full_matrix(m, fmt):
    """one full [2048, 4096] expert matrix of the DS4-Flash shape"""
    w = expert_matrix_f32(1, 0, 17, 0, 4096, 2048)
    ref = oracle.encode(fmt, w)
    dst = torch.zeros(ref.size, dtype=torch.uint8, device="cuda")
    m.moe_encode_blocks(fmt, torch.from_numpy(w).cuda(), 2048, 4096, dst)
    assert np.array_equal(dst.cpu().numpy().reshape(ref.shape), ref)


def _random_blocks(rng, fmt, rows, K):
    bs, nb = oracle.BLOCK[fmt]
    b = rng.integers(0, 256, size=(rows, K // bs, nb), dtype=np.uint8)
    if fmt == 1:
        b[..., 0] = rng.choice(np.array([0, 1, 100, 119, 120, 121, 127, 140, 200, 252, 255], np.uint8), size=b.shape[:-1])
    if fmt == 3:
        b[..., 80:84] = np.frombuffer((np.abs(rng.standard_normal(rows * (K // bs) * 2)) * 0.01).astype(np.float16)
                                      .tobytes(), np.uint8).reshape(rows, K // bs, 4)
    return b.reshape(rows, -1)


def _same(a, b):
    a = np.asarray(a)
    b = np.asarray(b)
    return np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(
        np.where(np.isnan(a), 0, a).view(np.uint32), np.where(np.isnan(b), 0, b).view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS, ids=[FMT_NAME[f] for f in FMTS])
@pytest.mark.parametrize("H,I", [(512, 256), (256, 512)])
def test_pack_blocks_roundtrip(m, fmt, H, I):
    """random canonical blocks (all exponents, incl. 0 and 255) -> packed layout -> debug unpack == oracle decode"""
    rng = np.random.default_rng(7 * fmt + H)
    E = 3
    g = _random_blocks(rng, fmt, E * I, H).reshape(E, I, -1)
    u = _random_blocks(rng, fmt, E * I, H).reshape(E, I, -1)
    d = _random_blocks(rng, fmt, E * H, I).reshape(E, H, -1)
    layer = m.Layer(fmt, H, I, E)
    layer.pack(m.MOE_SRC_BLOCKS, torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda(), torch.from_numpy(d).cuda())
    for e in range(E):
        out = torch.empty((2, I, H), dtype=torch.float32, device="cuda")
        m.moe_debug_unpack(fmt, m.MOE_LAYOUT_DECODE, m.MOE_MAT_GATE_UP, layer.gate_up, H, I, e, out)
        got = out.cpu().numpy()
        assert _same(got[0], oracle.decode(fmt, g[e]).reshape(I, H))
        assert _same(got[1], oracle.decode(fmt, u[e]).reshape(I, H))
        outd = torch.empty((H, I), dtype=torch.float32, device="cuda")
        m.moe_debug_unpack(fmt, m.MOE_LAYOUT_DECODE, m.MOE_MAT_DOWN, layer.down, H, I, e, outd)
        assert _same(outd.cpu().numpy(), oracle.decode(fmt, d[e]).reshape(H, I))


@pytest.mark.parametrize("fmt", FMTS, ids=[FMT_NAME[f] for f in FMTS])
def test_pack_f32_equals_oracle_encode_decode(m, fmt):
    H, I, E = 512, 256, 2
    rng = np.random.default_rng(fmt)
    g = (rng.standard_normal((E, I, H)) * 0.02).astype(np.float32)
    u = (rng.standard_normal((E, I, H)) * 0.02).astype(np.float32)
    d = (rng.standard_normal((E, H, I)) * 0.02).astype(np.float32)
    layer = m.Layer(fmt, H, I, E)
    layer.pack(m.MOE_SRC_F32, torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda(), torch.from_numpy(d).cuda())
    for e in range(E):
        out = torch.empty((2, I, H), dtype=torch.float32, device="cuda")
        m.moe_debug_unpack(fmt, m.MOE_LAYOUT_DECODE, m.MOE_MAT_GATE_UP, layer.gate_up, H, I, e, out)
        assert _same(out.cpu().numpy()[0], oracle.decode(fmt, oracle.encode(fmt, g[e])).reshape(I, H))
        assert _same(out.cpu().numpy()[1], oracle.decode(fmt, oracle.encode(fmt, u[e])).reshape(I, H))


def test_packed_bytes_equal_canonical_bytes(m):
    for fmt in FMTS:
        for (H, I) in [(4096, 2048), (512, 256)]:
            gu = m.moe_packed_bytes(fmt, 0, 0, 256, H, I)
            dn = m.moe_packed_bytes(fmt, 0, 1, 256, H, I)
            assert gu == 256 * 2 * m.moe_canonical_bytes(fmt, I, H)
            assert dn == 256 * m.moe_canonical_bytes(fmt, H, I)
    # active bytes per token-layer, DS4-Flash shape, top-6
    per_tok = {f: 6 * (m.moe_packed_bytes(f, 0, 0, 1, 4096, 2048) + m.moe_packed_bytes(f, 0, 1, 1, 4096, 2048))
               for f in FMTS}
    assert per_tok == {1: 80216064, 2: 84934656, 3: 49545216, 4: 160432128}
