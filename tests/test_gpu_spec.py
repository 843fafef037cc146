"""Speculative acceptance on the GPU against the oracle: the kept-draft count and the drawn token must match
exactly (integer results; the decision and the draw are defined in fp32 and exact integers on both sides)."""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import spec_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


def _gpu(m, p, q, draft, u):
    K, V = p.shape[0] - 1, p.shape[1]
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).cuda()
    res = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    m.moe_spec_accept(dev(p, np.float32), dev(q, np.float32) if K else None, K, V,
                      dev(np.asarray(draft).reshape(-1), np.int32) if K else None,
                      dev(np.asarray(u).reshape(-1), np.float32), res)
    torch.cuda.synchronize()
    r = res.cpu().numpy()
    return int(r[0]), int(r[1])


@pytest.mark.parametrize("K,V", [(0, 1), (0, 7), (1, 4), (2, 1027), (3, 1000), (5, 4099), (7, 32768), (8, 32768),
                                 (7, 129280)])
def test_spec_matches_oracle(m, K, V):
    for seed in (range(40) if V <= 32768 else range(8)):
        p, q, d, u = spec_inputs(seed, K, V)
        got = _gpu(m, p, q, d, u)
        assert got == oracle.spec_accept(p, q, d, u), seed


def test_spec_sharp_and_flat_distributions(m):
    for spread, noise in ((8.0, 0.1), (8.0, 4.0), (0.1, 0.1), (0.0, 0.0)):
        for seed in range(10):
            p, q, d, u = spec_inputs(100 + seed, 7, 5000, spread=spread, noise=noise)
            assert _gpu(m, p, q, d, u) == oracle.spec_accept(p, q, d, u), (spread, noise, seed)


def test_spec_edge_cases(m):
    V = 64
    rng = np.random.default_rng(9)
    p = rng.random((4, V)).astype(np.float32)
    p /= p.sum(axis=1, keepdims=True)
    # p = q: everything kept, the draw comes from the last row
    for us in (0.0, 0.5, 0.9999999, 1.0):
        d = np.array([1, 2, 3], np.int32)
        u = np.array([0.9999999, 0.9, 0.0, us], np.float32)
        want = oracle.spec_accept(p, p[:3], d, u)
        assert want[0] == 3 and _gpu(m, p, p[:3], d, u) == want
    # q = 0 < p keeps; p = q = 0 rejects and, with no residual mass, draws from p
    q = p[:3].copy()
    q[0, 5] = 0.0
    p2 = p.copy()
    p2[1, 7] = 0.0
    q[1] = p2[1]
    for u0 in (0.0, 0.9999999):
        u = np.array([u0, 0.3, 0.3, 0.61], np.float32)
        d = np.array([5, 7, 0], np.int32)
        assert _gpu(m, p2, q, d, u) == oracle.spec_accept(p2, q, d, u)
    # greedy: one-hot rows
    a = np.array([3, 9, 9, 40])
    pg = np.zeros((4, V), np.float32)
    pg[np.arange(4), a] = 1
    for d in ([3, 9, 9], [3, 8, 9], [0, 9, 9]):
        qg = np.zeros((3, V), np.float32)
        qg[np.arange(3), d] = 1
        u = np.array([0.2, 0.7, 0.99, 0.4], np.float32)
        assert _gpu(m, pg, qg, np.array(d, np.int32), u) == oracle.spec_accept(pg, qg, d, u)
    # odd uniforms: negative, NaN, >= 1
    for us in (-0.5, float("nan"), 1.5, 1e-30):
        u = np.array([0.1, 0.2, 0.3, us], np.float32)
        d = np.array([1, 2, 3], np.int32)
        assert _gpu(m, p, p[:3] * 0.5, d, u) == oracle.spec_accept(p, p[:3] * 0.5, d, u)
    # draft ids outside [0, V)
    for bad in (-1, V, 1 << 30):
        d = np.array([1, bad, 3], np.int32)
        assert _gpu(m, p, p[:3], d, np.zeros(4, np.float32)) == (-1, -1)


def test_spec_largest_vocabulary(m):
    V = 1 << 22
    p, q, d, u = spec_inputs(3, 1, V, spread=1.0)
    assert _gpu(m, p, q, d, u) == oracle.spec_accept(p, q, d, u)
