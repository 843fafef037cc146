"""RMS normalisation between stacked layers against the oracle's exact values: the bf16 output within the bf16
rounding of the exact value plus the fp32 arithmetic (|x - exact| <= 2^-8 |exact|), a token's row independent of
the other tokens (bit for bit), zeros kept, NaN and infinity propagated."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda"
EPS = 1e-6


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


def _gpu(m, y):
    T, H = y.shape
    x = torch.zeros((T, H), dtype=torch.int16, device=DEV)
    m.moe_rms_norm_bf16(torch.from_numpy(np.ascontiguousarray(y, np.float32)).to(DEV), T, H, EPS, x)
    torch.cuda.synchronize()
    b = x.cpu().numpy().view(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


@pytest.mark.parametrize("H", [1, 7, 512, 4096, 7168])
def test_rms_norm_matches_oracle(m, H):
    rng = np.random.default_rng(H)
    y = np.concatenate([rng.standard_normal((3, H)) * s for s in (1e-20, 1.0, 1e20)]).astype(np.float32)
    y = np.concatenate([y, np.zeros((1, H), np.float32), (rng.standard_t(3, (2, H)) * 5).astype(np.float32)])
    got = _gpu(m, y)
    ref = oracle.rms_norm(y, EPS)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-30), H
    assert np.array_equal(got[9], np.zeros(H, np.float32))
    for t in (0, 4, 10):   # a row alone gives the same bits as in the batch
        assert np.array_equal(_gpu(m, y[t:t + 1])[0].view(np.uint32), got[t].view(np.uint32))


def test_rms_norm_propagates_nan_and_inf(m):
    y = np.ones((2, 64), np.float32)
    y[0, 3] = np.nan
    y[1, 5] = np.inf
    got = _gpu(m, y)
    assert np.all(np.isnan(got[0]))
    assert np.isnan(got[1, 5]) and np.all(got[1, :5] == 0) and np.all(got[1, 6:] == 0)


def test_rms_norm_rejects_bad_arguments(m):
    y = torch.zeros((2, 8), device=DEV)
    x = torch.zeros((2, 8), dtype=torch.int16, device=DEV)
    with pytest.raises(m.MoeError):
        m.moe_rms_norm_bf16(y, 0, 8, EPS, x)
    with pytest.raises(m.MoeError):
        m.moe_rms_norm_bf16(y, 2, 8, -1.0, x)
