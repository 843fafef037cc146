"""The scratch-free decode entry point (for callers that cannot allocate device memory, such as a plugin that is
handed only its input and output buffers) against the regular decode with a caller-provided workspace.

Two calls in a row through the C ABI for each weight format: each result must be bit-identical to
moe_expert_ffn_decode's on the same inputs (both run the same kernel) and within the suite's tolerance of the CPU
oracle (|y - y_ref| <= 1e-3 * sum|terms| + 1e-6 per element); the static call's device status word must read OK.
This file is collected last so a stop at the first failure has already run every other test; it also passes
alone.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import router_f16_bits, x_bf16_bits
from tests._harness import FMTS, FMT_NAME, Weights, dev_bits, make_layer, oracle_moe, tol_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


@pytest.mark.parametrize("fmt", FMTS, ids=[FMT_NAME[f] for f in FMTS])
@pytest.mark.parametrize("E,H,I,k", [(8, 512, 256, 2), (256, 4096, 2048, 6)])
def test_static_scratch_decode_matches_workspace_decode(m, fmt, E, H, I, k):
    W = Weights(21, H, I)
    x = x_bf16_bits(21, range(2), H)
    idx, w, _, _ = oracle.route_topk(router_f16_bits(21, 0, E, H), x, k)
    layer = make_layer(m, fmt, W, E, np.unique(idx), "cuda")
    ws = layer.workspace(1, k)
    y_or, absterm = oracle_moe(fmt, W, idx, w, x)
    for t in range(2):  # two calls in a row share the library's scratch array
        xt = dev_bits(x[t:t + 1], "cuda")
        it = torch.from_numpy(idx[t:t + 1]).cuda()
        wt = torch.from_numpy(w[t:t + 1]).cuda()
        y_ref = torch.full((1, H), float("nan"), device="cuda")
        y_static = torch.full((1, H), float("nan"), device="cuda")
        m.moe_expert_ffn_decode(layer, xt, it, wt, k, y_ref, None, False, ws)
        m.moe_expert_ffn_decode_static(layer, xt, it, wt, k, y_static)
        torch.cuda.synchronize()
        assert m.moe_get_device_status(ws) == 0
        assert m.moe_static_device_status() == 0
        ys, yr = y_static.cpu().numpy()[0], y_ref.cpu().numpy()[0]
        assert np.array_equal(ys.view(np.uint32), yr.view(np.uint32)), "token %d: static != workspace decode" % t
        tol_check(ys, y_or[t], absterm[t], "token %d vs oracle" % t)


def test_static_scratch_reports_invalid_expert_in_its_status(m):
    E, H, I, k = 8, 512, 256, 2
    layer = make_layer(m, 1, Weights(22, H, I), E, range(E), "cuda")
    x = torch.zeros((1, H), dtype=torch.int16, device="cuda")
    y = torch.zeros((1, H), device="cuda")
    w = torch.tensor([[0.5, 0.5]], device="cuda")
    m.moe_expert_ffn_decode_static(layer, x, torch.tensor([[1, 9]], dtype=torch.int32, device="cuda"), w, k, y)
    assert m.moe_static_device_status() == 1   # MOE_ERR_INVALID_ARG: expert id 9 >= E
    m.moe_expert_ffn_decode_static(layer, x, torch.tensor([[1, 3]], dtype=torch.int32, device="cuda"), w, k, y)
    assert m.moe_static_device_status() == 0   # the next call starts from a cleared status word


def test_static_scratch_rejects_sizes_beyond_its_maximum(m):
    layer = m.Layer(1, 512, 256, 16)
    x = torch.zeros((1, 512), dtype=torch.int16, device="cuda")
    idx = torch.zeros((1, 9), dtype=torch.int32, device="cuda")
    w = torch.zeros((1, 9), device="cuda")
    y = torch.zeros((1, 512), device="cuda")
    with pytest.raises(m.MoeError) as ei:
        m.moe_expert_ffn_decode_static(layer, x, idx, w, 9, y)   # k = 9 > 8
    assert ei.value.status == 2
