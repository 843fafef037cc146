"""Guard canaries around every buffer a call writes: each output and workspace is the middle of a larger device
allocation whose 4 KB guard bands on both sides hold a byte pattern; after the call the bands must be unchanged.
An out-of-bounds write by any kernel of the path (decode, verify, the fused router + FFN, the shared expert,
prefill, routing, speculative acceptance) shows up here even where the outputs inside the buffer are right."""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import router_f16_bits, spec_inputs, x_bf16_bits, zipf_routing
from tests._harness import Weights, dev_bits, make_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"
GUARD, PAT = 4096, 0xA5


@pytest.fixture(scope="module")
def m():
    import bit_moe_decode_gb300 as mod
    return mod


class Guarded:
    """nbytes of device memory (aligned to `align`) between two guard bands of PAT bytes."""

    def __init__(self, nbytes: int, align: int = 256, fill: int = 0):
        self.raw = torch.full((nbytes + 2 * GUARD + align,), PAT, dtype=torch.uint8, device=DEV)
        off = (-(self.raw.data_ptr() + GUARD)) % align
        self.lo, self.hi = GUARD + off, GUARD + off + nbytes
        self.body = self.raw[self.lo:self.hi]
        self.body.fill_(fill)

    def view(self, dtype, shape):
        return self.body.view(dtype).reshape(shape)

    def intact(self) -> bool:
        return bool((self.raw[:self.lo] == PAT).all()) and bool((self.raw[self.hi:] == PAT).all())


def _outs(T, H, k=None):
    g = {"y": Guarded(T * H * 4), "yb": Guarded(T * H * 2)}
    if k:
        g["idx"] = Guarded(T * k * 4)
        g["w"] = Guarded(T * k * 4)
    return g


def _check(guards, what):
    torch.cuda.synchronize()
    for name, g in guards.items():
        assert g.intact(), "%s: a guard band of %s was overwritten" % (what, name)


@pytest.mark.parametrize("layout,T", [(0, 1), (0, 8), (1, 1), (1, 5)], ids=["decode_T1", "decode_T8", "tc_T1", "tc_T5"])
def test_decode_verify_write_inside_their_buffers(m, layout, T):
    E, H, I, k = 16, 1024, 512, 4
    W = Weights(61, H, I)
    layer = make_layer(m, 1, W, E, range(E), DEV, layout=layout)
    x = x_bf16_bits(62, range(T), H)
    idx, w, _, _ = oracle.route_topk(router_f16_bits(62, 0, E, H), x, k)
    g = _outs(T, H)
    g["ws"] = Guarded(m.moe_workspace_bytes(layer, 8, k))
    y, yb, ws = g["y"].view(torch.float32, (T, H)), g["yb"].view(torch.int16, (T, H)), g["ws"].body
    it = torch.from_numpy(idx).to(DEV)
    wt = torch.from_numpy(w).to(DEV)
    if T == 1:
        m.moe_expert_ffn_decode(layer, dev_bits(x, DEV), it, wt, k, y, yb, False, ws)
    else:
        m.moe_expert_ffn_verify(layer, dev_bits(x, DEV), T, it, wt, k, y, yb, False, ws)
    _check(g, "layout %d T=%d" % (layout, T))
    assert m.moe_get_device_status(ws) == 0
    assert torch.isfinite(y).all()


@pytest.mark.parametrize("T", [1, 3])
def test_fused_router_ffn_writes_inside_its_buffers(m, T):
    E, H, I, k = 32, 1024, 512, 6
    W = Weights(63, H, I)
    layer = make_layer(m, 1, W, E, range(E), DEV, layout=1)
    x = x_bf16_bits(64, range(T), H)
    g = _outs(T, H, k)
    g["ws"] = Guarded(m.moe_workspace_bytes(layer, 8, k))
    m.moe_route_expert_ffn(layer, dev_bits(router_f16_bits(64, 0, E, H), DEV), dev_bits(x, DEV), T, k,
                           g["idx"].view(torch.int32, (T, k)), g["w"].view(torch.float32, (T, k)),
                           g["y"].view(torch.float32, (T, H)), g["yb"].view(torch.int16, (T, H)), False, g["ws"].body)
    _check(g, "fused T=%d" % T)
    assert m.moe_get_device_status(g["ws"].body) == 0


@pytest.mark.parametrize("fmt", [2, 3, 4], ids=["int4g32", "q2k", "q8_0"])
def test_other_formats_write_inside_their_buffers(m, fmt):
    E, H, I, k, T = 8, 768, 512, 2, 8
    W = Weights(65, H, I)
    layer = make_layer(m, fmt, W, E, range(E), DEV)
    x = x_bf16_bits(66, range(T), H)
    idx, w, _, _ = oracle.route_topk(router_f16_bits(66, 0, E, H), x, k)
    g = _outs(T, H)
    g["ws"] = Guarded(m.moe_workspace_bytes(layer, 8, k))
    m.moe_expert_ffn_verify(layer, dev_bits(x, DEV), T, torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV), k,
                            g["y"].view(torch.float32, (T, H)), g["yb"].view(torch.int16, (T, H)), True, g["ws"].body)
    _check(g, "format %d" % fmt)
    assert m.moe_get_device_status(g["ws"].body) == 0


def test_router_writes_inside_its_buffers(m):
    E, H, k, T = 256, 4096, 6, 8
    g = {"idx": Guarded(T * k * 4), "w": Guarded(T * k * 4)}
    m.moe_route_topk(dev_bits(router_f16_bits(67, 0, E, H), DEV), dev_bits(x_bf16_bits(67, range(T), H), DEV), T, H,
                     E, k, None, None, 0, g["idx"].view(torch.int32, (T, k)), g["w"].view(torch.float32, (T, k)))
    _check(g, "router")


def test_prefill_writes_inside_its_buffers(m):
    E, H, I, k, T = 8, 512, 256, 2, 300
    W = Weights(68, H, I)
    layer = make_layer(m, 1, W, E, range(E), DEV, layout=1)
    x = x_bf16_bits(68, range(T), H)
    idx, w = zipf_routing(68, T, E, k)
    g = _outs(T, H)
    g["ws"] = Guarded(m.moe_prefill_workspace_bytes(layer, T, k))
    m.moe_expert_grouped_gemm_prefill(layer, dev_bits(x, DEV), T, torch.from_numpy(np.ascontiguousarray(idx, np.int32))
                                      .to(DEV), torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(DEV), k,
                                      g["y"].view(torch.float32, (T, H)), g["yb"].view(torch.int16, (T, H)),
                                      g["ws"].body)
    _check(g, "prefill")


def test_spec_accept_writes_inside_its_buffer(m):
    p, q, d, u = spec_inputs(69, 7, 32768)
    g = {"res": Guarded(8)}
    dev = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).to(DEV)
    m.moe_spec_accept(dev(p, np.float32), dev(q, np.float32), 7, 32768, dev(np.asarray(d).reshape(-1), np.int32),
                      dev(np.asarray(u).reshape(-1), np.float32), g["res"].view(torch.int32, (2,)))
    _check(g, "spec accept")
    assert tuple(int(v) for v in g["res"].view(torch.int32, (2,)).cpu()) == oracle.spec_accept(p, q, d, u)


@pytest.mark.parametrize("T", [1, 8])
def test_tc_full_shape_writes_inside_its_buffers(m, T):
    """hidden 4096, intermediate 2048, 256 experts, top-6 (split slices, exports, imports, the h images): the
    tensor-core decode / verify with the routing given, workspace sized for 8 tokens"""
    E, H, I, k = 256, 4096, 2048, 6
    W = Weights(70, H, I)
    x = x_bf16_bits(70, range(T), H)
    idx, w, _, _ = oracle.route_topk(router_f16_bits(70, 0, E, H), x, k)
    layer = make_layer(m, 1, W, E, np.unique(idx), DEV, layout=1)
    g = _outs(T, H)
    g["ws"] = Guarded(m.moe_workspace_bytes(layer, 8, k))
    m.moe_expert_ffn_verify(layer, dev_bits(x, DEV), T, torch.from_numpy(idx).to(DEV), torch.from_numpy(w).to(DEV), k,
                            g["y"].view(torch.float32, (T, H)), g["yb"].view(torch.int16, (T, H)), False, g["ws"].body)
    _check(g, "tc full shape T=%d" % T)
    assert m.moe_get_device_status(g["ws"].body) == 0
