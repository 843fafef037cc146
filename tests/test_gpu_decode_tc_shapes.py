"""The tensor-core decode path on shapes that exercise the other branches of its work split: every slice split
across CTAs (no whole slice), an odd number of down row pairs (one down chunk per unit), three and eight gate/up
segments, and a call whose slices divide evenly among the CTAs (no split slice at all). Each token against the
oracle (|y - y_ref| <= 1e-3 * sum|terms| + 1e-6), and verify rows bit-identical to decoding each token alone
("Mixed-precision compression of DeepSeek-V4-Flash", "Width drift")."""
import numpy as np
import pytest

from tests._harness import Weights, make_layer, oracle_moe, tol_check
from tests.test_gpu_ffn import _decode, _routing, _verify

pytestmark = pytest.mark.gpu
DEV = "cuda"
MXFP4, TC = 1, 1


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


def _check(m, layer, W, x, idx, w, k, what):
    T = x.shape[0]
    ws = layer.workspace(8, k)
    yv = _verify(m, layer, ws, x, idx, w, k)
    yr, ab = oracle_moe(MXFP4, W, idx, w, x)
    worst = 0.0
    for t in range(T):
        yd, _ = _decode(m, layer, ws, x[t:t + 1], idx[t], w[t], k)
        worst = max(worst, tol_check(yd, yr[t], ab[t], "%s token %d" % (what, t)))
        assert np.array_equal(yv[t].view(np.uint32), yd.view(np.uint32)), "%s: verify row %d differs" % (what, t)
    print("%s: max err/bound %.3g" % (what, worst))


# H = 768: 6 k-tiles in 3 segments, 3 down row pairs (one chunk per down unit); H = 2048, I = 1280: 8 segments of
# 2 k-tiles, 20 slices per expert
@pytest.mark.parametrize("H,I,E,k", [(768, 768, 16, 4), (2048, 1280, 32, 6)], ids=["h768_i768", "h2048_i1280"])
@pytest.mark.parametrize("T", [1, 3, 8])
def test_tc_odd_shapes(m, H, I, E, k, T):
    W = Weights(5, H, I)
    layer = make_layer(m, MXFP4, W, E, range(E), DEV, layout=TC)
    x, idx, w = _routing(E, H, k, T, seed=100 + T)
    _check(m, layer, W, x, idx, w, k, "H=%d I=%d T=%d" % (H, I, T))


def test_tc_full_shape_slices_divide_evenly(m):
    # 19 distinct experts x 32 slices = 608 = 4 x 152 whole slices per CTA on a 152-SM GB300: no split slice
    H, I, E, k, T = 4096, 2048, 256, 6, 4
    rng = np.random.default_rng(7)
    experts = rng.choice(E, 19, replace=False)
    idx = np.stack([experts[[0, 1, 2, 3, 4, 5]], experts[[6, 7, 8, 9, 10, 11]], experts[[12, 13, 14, 15, 16, 17]],
                    experts[[18, 0, 6, 12, 1, 7]]]).astype(np.int32)
    w = rng.uniform(0.5, 1.5, size=(T, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    from moe_inputs import x_bf16_bits
    x = x_bf16_bits(9, range(T), H)
    W = Weights(1, H, I)
    layer = make_layer(m, MXFP4, W, E, np.unique(idx), DEV, layout=TC)
    _check(m, layer, W, x, idx, w, k, "full shape, 19 experts")
