"""The call order of RoutedStack.run (host logic only; the library calls are replaced by recorders): per layer the
hash router and a verify call, or the fused router + FFN call; then the layer's shared expert when there is one,
accumulating into y; then the normalisation into the next layer's x. The FFN calls never write the bf16 copy
themselves, and every call goes to the given stream."""
import pytest
import torch

import bit_moe_decode_gb300.stack as stack_mod
from bit_moe_decode_gb300.stack import RoutedStack


class FakeLayer:
    """stands in for Layer: no device memory, a workspace that is a host tensor"""

    def __init__(self, fmt, H, I, E, layout=0, device="cpu"):
        self.fmt, self.H, self.I, self.E, self.layout = fmt, H, I, E, layout
        self.gate_up = torch.zeros(1, dtype=torch.uint8)
        self.down = torch.zeros(1, dtype=torch.uint8)

    def workspace(self, T_max, k):
        return torch.zeros(256, dtype=torch.uint8)


@pytest.fixture
def calls(monkeypatch):
    monkeypatch.setattr(stack_mod, "Layer", FakeLayer)
    log = []

    def rec(name):
        def f(*args, **kw):
            log.append((name, args, kw))
        return f
    for name in ("moe_route_topk", "moe_expert_ffn_verify", "moe_route_expert_ffn", "moe_rms_norm_bf16"):
        monkeypatch.setattr(stack_mod, name, rec(name))
    return log


def _stack(shared_I=0):
    st = RoutedStack(512, 256, 16, 6, n_layers=4, n_hash=2, vocab=100, T_max=8, device="cpu", shared_I=shared_I)
    for L in range(4):
        st.router[L] = torch.zeros((16, 512), dtype=torch.int16)
        st.tid2eid[L] = torch.zeros((100, 6), dtype=torch.int32)
    return st


@pytest.mark.parametrize("shared_I", [0, 256])
@pytest.mark.parametrize("use_shared", [None, False])
def test_call_order_per_layer(calls, shared_I, use_shared):
    st = _stack(shared_I)
    stream = object()
    x0 = torch.zeros((3, 512), dtype=torch.int16)
    st.run(3, token_ids=torch.zeros(3, dtype=torch.int32), x0=x0, stream=stream, shared=use_shared)
    with_shared = shared_I > 0 and use_shared is None
    names = [c[0] for c in calls]
    per_layer = []
    for L in range(4):
        seq = ["moe_route_topk", "moe_expert_ffn_verify"] if L < 2 else ["moe_route_expert_ffn"]
        if with_shared:
            seq.append("moe_expert_ffn_verify")
        seq.append("moe_rms_norm_bf16")
        per_layer += seq
    assert names == per_layer
    assert all(kw.get("stream") is stream for _, _, kw in calls)
    i = 0
    for L in range(4):
        xin = x0 if L == 0 else st.x[L][:3]
        if L < 2:
            _, a, _ = calls[i + 1]          # verify: (layer, x, T, idx, w, k, y, y_bf16, accumulate, ws)
            assert a[0] is st.layers[L] and a[1].data_ptr() == xin.data_ptr() and a[7] is None and a[8] is False
            i += 2
        else:
            _, a, _ = calls[i]              # fused: (layer, router, x, T, k, idx, w, y, y_bf16, accumulate, ws)
            assert a[0] is st.layers[L] and a[2].data_ptr() == xin.data_ptr() and a[8] is None and a[9] is False
            i += 1
        if with_shared:
            _, a, _ = calls[i]
            assert a[0] is st.shared[L] and a[5] == 1 and a[7] is None and a[8] is True   # k = 1, accumulate
            assert a[6].data_ptr() == st.y[L].data_ptr()
            i += 1
        _, a, _ = calls[i]                  # norm: (y, T, H, eps, x_next)
        assert a[0].data_ptr() == st.y[L].data_ptr() and a[4].data_ptr() == st.x[L + 1].data_ptr()
        i += 1
    assert st.launches_per_run(shared=with_shared) == 2 * 2 + 2 + 4 + (4 if with_shared else 0)
