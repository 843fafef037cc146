"""Router top-k and hash routing on the GPU against the oracle (indices exact up to proven near-ties)."""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import router_f16_bits, tid2eid, token_ids, x_bf16_bits
from tests._harness import dev_bits, near_tie_ok

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


def _route(m, wr, x, k):
    T, H = x.shape
    E = wr.shape[0]
    idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    m.moe_route_topk(dev_bits(wr, "cuda"), dev_bits(x, "cuda"), T, H, E, k, None, None, 0, idx, w)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("E,H,k,T", [(8, 512, 2, 1), (8, 512, 2, 13), (256, 4096, 6, 1), (256, 4096, 6, 8),
                                     (256, 4096, 6, 37), (64, 256, 8, 5), (1024, 512, 4, 3)])
def test_route_matches_oracle(m, E, H, k, T):
    wr = router_f16_bits(11, 3, E, H)
    x = x_bf16_bits(11, range(T), H)
    gi, gw = _route(m, wr, x, k)
    ri, rw, logits, absl = oracle.route_topk(wr, x, k)
    ties = 0
    for t in range(T):
        if not np.array_equal(gi[t], ri[t]):
            assert near_tie_ok(gi[t], ri[t], logits[t], absl[t], H), (t, gi[t], ri[t])
            ties += 1
            continue
        assert np.all(np.abs(gw[t] - rw[t]) <= 1e-6 + 1e-5 * rw[t]), (t, gw[t], rw[t])
    assert ties <= max(1, T // 10)


def test_route_ties_lower_index(m):
    E, H, k = 32, 256, 4
    rng = np.random.default_rng(2)
    row = (rng.standard_normal(H) * 0.02).astype(np.float16).view(np.uint16)
    wr = np.tile(row, (E, 1))
    wr[9] = (rng.standard_normal(H) * 0.5).astype(np.float16).view(np.uint16)
    x = x_bf16_bits(2, range(3), H)
    gi, gw = _route(m, wr, x, k)
    ri, rw, logits, _ = oracle.route_topk(wr, x, k)
    assert np.array_equal(gi, ri)
    for t in range(3):
        rest = [e for e in gi[t] if e != 9]
        assert rest == sorted(rest)


def test_route_batch_equals_single(m):
    """routing T tokens in one call gives bit-identical results to routing each token alone"""
    E, H, k, T = 256, 4096, 6, 11
    wr = router_f16_bits(5, 0, E, H)
    x = x_bf16_bits(5, range(T), H)
    bi, bw = _route(m, wr, x, k)
    for t in range(T):
        si, sw = _route(m, wr, x[t:t + 1], k)
        assert np.array_equal(si[0], bi[t]) and np.array_equal(sw[0].view(np.uint32), bw[t].view(np.uint32))


def test_hash_routing(m):
    V, E, k, T = 32768, 256, 6, 100
    tab = tid2eid(3, 0, V, E, k)
    tok = token_ids(3, T, V)
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    m.moe_route_topk(None, None, T, 4096, E, k, torch.from_numpy(tok).cuda(), torch.from_numpy(tab).cuda(), V, idx, w)
    ri, rw = oracle.route_hash(tok, tab, k)
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert np.array_equal(w.cpu().numpy(), rw)


def test_route_argument_errors(m):
    idx = torch.empty((1, 6), dtype=torch.int32, device="cuda")
    w = torch.empty((1, 6), dtype=torch.float32, device="cuda")
    x = torch.zeros((1, 4096), dtype=torch.int16, device="cuda")
    wr = torch.zeros((256, 4096), dtype=torch.int16, device="cuda")
    with pytest.raises(m.MoeError) as ei:
        m.moe_route_topk(wr, x, 1, 4096, 256, 9, None, None, 0, idx, w)
    assert ei.value.status == 2
    with pytest.raises(m.MoeError) as ei:
        m.moe_route_topk(wr, x, 1, 4000, 256, 6, None, None, 0, idx, w)
    assert ei.value.status == 2
