"""Host-side helpers of bench.py that run without a GPU."""
import bench


def test_peak_of_reads_numbers_and_value_objects_and_falls_back():
    assert bench.peak_of({"hbm_gbs": 6780}, "hbm_gbs") == 6780.0
    assert bench.peak_of({"hbm_gbs": "6780.5"}, "hbm_gbs") == 6780.5
    assert bench.peak_of({"hbm_gbs": {"value": 6700, "unit": "GB/s"}}, "hbm_gbs") == 6700.0
    for bad in (None, [], {}, {"hbm_gbs": None}, {"hbm_gbs": "n/a"}, {"hbm_gbs": 0}, {"hbm_gbs": {"unit": "GB/s"}},
                {"bf16_tflops": 1900}):
        assert bench.peak_of(bad, "hbm_gbs") is None


def test_rank_seeds_and_single_process_max():
    assert bench.rank_token_seed(1, 0) == 1 and bench.rank_token_seed(1, 1) != bench.rank_token_seed(1, 0)
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25


def _bf16_rne(y):
    import numpy as np
    b = np.ascontiguousarray(y, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_parity_leg_accepts_the_oracle_and_rejects_a_wrong_row():
    """the bench's parity check (routed, and routed + shared expert) passes the oracle's own rows and fails a
    perturbed element, a wrong routing and a bf16 copy that is not the rounding of y"""
    import numpy as np
    co = bench.CpuOracle(1, 2, n_experts=16)
    n = 2
    idx, w = co.idx[:n], co.w[:n]
    co._encode(1, idx)
    y = np.concatenate([co._moe(1, idx[t:t + 1], w[t:t + 1], co.x[t:t + 1])[0] for t in range(n)]).astype(np.float32)
    assert co.parity(1, y, idx, w)["ok"]
    bad = y.copy()
    bad[1, 7] += 1.0
    assert not co.parity(1, bad, idx, w)["ok"]
    swapped = idx.copy()
    swapped[0, 0] = next(e for e in range(16) if e not in idx[0])   # not a near tie
    assert not co.parity(1, y, swapped, w)["ok"]
    sidx = np.array([0, 1])
    ys = y + np.concatenate([co._shared(int(sidx[t]), t)[0] for t in range(n)]).astype(np.float32)
    assert co.parity_shared(ys, idx, w, sidx, _bf16_rne(ys))["ok"]
    assert not co.parity_shared(y, idx, w, sidx, _bf16_rne(y))["ok"]        # the shared expert left out
    yb = _bf16_rne(ys)
    yb[0, 3] ^= 1
    assert not co.parity_shared(ys, idx, w, sidx, yb)["ok"]
