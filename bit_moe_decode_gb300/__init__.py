"""bit_moe_decode_gb300 -- thin Python binding of libmoe.so (the C ABI in include/moe.h).

Every function here only marshals arguments (torch tensors -> device pointers, the current torch stream) and
calls the C entry point of the same name; all computation runs in the library's CUDA kernels. There is no
fallback: if libmoe.so is missing or the device is not sm_103 the calls raise.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_FMT_MXFP4, MOE_FMT_INT4G32, MOE_FMT_Q2K, MOE_FMT_Q8_0 = 1, 2, 3, 4
MOE_SRC_BLOCKS, MOE_SRC_F32 = 0, 1
MOE_LAYOUT_DECODE, MOE_LAYOUT_TC = 0, 1
MOE_LAYOUT_PREFILL = MOE_LAYOUT_TC
MOE_MAT_GATE_UP, MOE_MAT_DOWN = 0, 1

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_SHAPE", 3: "MOE_ERR_UNSUPPORTED_FORMAT",
          4: "MOE_ERR_UNSUPPORTED_ARCH", 5: "MOE_ERR_WORKSPACE_TOO_SMALL", 6: "MOE_ERR_CUDA",
          7: "MOE_ERR_DEVICE_TIMEOUT", 8: "MOE_ERR_FAULT_INJECTED"}
# canonical block geometry: (weights per block, bytes per block)
BLOCK = {MOE_FMT_MXFP4: (32, 17), MOE_FMT_INT4G32: (32, 18), MOE_FMT_Q2K: (256, 84), MOE_FMT_Q8_0: (32, 34)}

# every symbol include/moe.h declares
EXPORTS = ["moe_status_string", "moe_version", "moe_check_device", "moe_canonical_bytes", "moe_packed_bytes",
           "moe_encode_blocks", "moe_pack_weights", "moe_route_topk", "moe_workspace_bytes", "moe_workspace_init",
           "moe_get_device_status", "moe_expert_ffn_decode", "moe_expert_ffn_verify", "moe_route_expert_ffn",
           "moe_debug_unpack", "moe_debug_timeout_probe", "moe_expert_ffn_decode_static", "moe_static_device_status",
           "moe_prefill_workspace_bytes",
           "moe_expert_grouped_gemm_prefill", "moe_debug_prefill", "moe_spec_accept", "moe_rms_norm_bf16"]


class MoeError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__("%s failed: %s (%d)" % (call, STATUS.get(status, "?"), status))


class moe_layer_t(C.Structure):
    _fields_ = [("fmt", C.c_int), ("layout", C.c_int), ("H", C.c_int32), ("I", C.c_int32), ("E", C.c_int32),
                ("gate_up", C.c_void_p), ("down", C.c_void_p)]


_lib = None


def lib() -> C.CDLL:
    """Load libmoe.so (built by bit_moe_decode_gb300.build.build() / __graft_entry__.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoe.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = C.CDLL(LIB_PATH)
        P, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
        LP = C.POINTER(moe_layer_t)
        sig = {
            "moe_status_string": (C.c_char_p, [C.c_int]),
            "moe_version": (i32, []),
            "moe_check_device": (C.c_int, []),
            "moe_canonical_bytes": (sz, [C.c_int, i64, i64]),
            "moe_packed_bytes": (sz, [C.c_int, C.c_int, C.c_int, i64, i64, i64]),
            "moe_encode_blocks": (C.c_int, [C.c_int, P, i64, i64, P, P]),
            "moe_pack_weights": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_int, i64, i64, i64, P, P, P, sz, P]),
            "moe_route_topk": (C.c_int, [P, P, i32, i32, i32, i32, P, P, i32, P, P, P]),
            "moe_spec_accept": (C.c_int, [P, P, i32, i32, P, P, P, P]),
            "moe_rms_norm_bf16": (C.c_int, [P, i32, i32, C.c_float, P, P]),
            "moe_workspace_bytes": (sz, [LP, i32, i32]),
            "moe_workspace_init": (C.c_int, [P, sz, P]),
            "moe_get_device_status": (C.c_int, [P, P]),
            "moe_expert_ffn_decode": (C.c_int, [LP, P, P, P, i32, P, P, i32, P, sz, P]),
            "moe_expert_ffn_verify": (C.c_int, [LP, P, i32, P, P, i32, P, P, i32, P, sz, P]),
            "moe_route_expert_ffn": (C.c_int, [LP, P, P, i32, i32, P, P, P, P, i32, P, sz, P]),
            "moe_debug_unpack": (C.c_int, [C.c_int, C.c_int, C.c_int, P, i64, i64, i64, P, P]),
            "moe_debug_timeout_probe": (C.c_int, [P, sz, i32, P]),
            "moe_expert_ffn_decode_static": (C.c_int, [LP, P, P, P, i32, P, P, i32, P]),
            "moe_static_device_status": (C.c_int, [P]),
            "moe_prefill_workspace_bytes": (sz, [LP, i32, i32]),
            "moe_expert_grouped_gemm_prefill": (C.c_int, [LP, P, i32, P, P, i32, P, P, P, sz, P]),
            "moe_debug_prefill": (C.c_int, [LP, P, i32, P, P, i32, P, P, P, sz, P, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _ptr(t):
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "expected a contiguous CUDA tensor"
    return C.c_void_p(t.data_ptr())


def _check(st: int, call: str):
    if st != 0:
        raise MoeError(st, call)


# ------------------------------------------------------------------------------------------------ plain calls
def moe_status_string(st: int) -> str:
    return lib().moe_status_string(st).decode()


def moe_version() -> int:
    return lib().moe_version()


def moe_check_device() -> int:
    return lib().moe_check_device()


def moe_canonical_bytes(fmt: int, rows: int, k: int) -> int:
    return lib().moe_canonical_bytes(fmt, rows, k)


def moe_packed_bytes(fmt: int, layout: int, kind: int, n_experts: int, H: int, I: int) -> int:
    return lib().moe_packed_bytes(fmt, layout, kind, n_experts, H, I)


def moe_encode_blocks(fmt: int, src: torch.Tensor, rows: int, k: int, dst: torch.Tensor, stream=None):
    assert src.dtype == torch.float32 and dst.dtype == torch.uint8
    assert dst.numel() >= moe_canonical_bytes(fmt, rows, k)
    _check(lib().moe_encode_blocks(fmt, _ptr(src), rows, k, _ptr(dst), _stream(stream)), "moe_encode_blocks")


def moe_pack_weights(fmt: int, src_kind: int, layout: int, kind: int, n_experts: int, H: int, I: int,
                     src_a: torch.Tensor, src_b, dst: torch.Tensor, stream=None):
    _check(lib().moe_pack_weights(fmt, src_kind, layout, kind, n_experts, H, I, _ptr(src_a), _ptr(src_b), _ptr(dst),
                                  dst.numel() * dst.element_size(), _stream(stream)), "moe_pack_weights")


def moe_route_topk(router_w_f16, x_bf16, T: int, H: int, E: int, k: int, token_ids, tid2eid, V: int,
                   idx: torch.Tensor, weights: torch.Tensor, stream=None):
    _check(lib().moe_route_topk(_ptr(router_w_f16), _ptr(x_bf16), T, H, E, k, _ptr(token_ids), _ptr(tid2eid), V,
                                _ptr(idx), _ptr(weights), _stream(stream)), "moe_route_topk")


def moe_spec_accept(p, q, K: int, V: int, draft, u, result, stream=None):
    """Acceptance of K drafted tokens (see include/moe.h): result[0] = drafts kept, result[1] = the drawn token."""
    _check(lib().moe_spec_accept(_ptr(p), _ptr(q), K, V, _ptr(draft), _ptr(u), _ptr(result), _stream(stream)),
           "moe_spec_accept")


def moe_rms_norm_bf16(y, T: int, H: int, eps: float, x_bf16, stream=None):
    """x_bf16[t] = bf16(y[t] / sqrt(mean(y[t]^2) + eps)) (see include/moe.h)."""
    _check(lib().moe_rms_norm_bf16(_ptr(y), T, H, eps, _ptr(x_bf16), _stream(stream)), "moe_rms_norm_bf16")


def moe_workspace_bytes(layer: "Layer", T_max: int, k: int) -> int:
    return lib().moe_workspace_bytes(C.byref(layer.c), T_max, k)


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_workspace_init")


def moe_get_device_status(ws: torch.Tensor, stream=None) -> int:
    return lib().moe_get_device_status(_ptr(ws), _stream(stream))


def moe_expert_ffn_decode(layer: "Layer", x_bf16, idx, w, k: int, y, y_bf16=None, accumulate: bool = False,
                          ws=None, stream=None):
    _check(lib().moe_expert_ffn_decode(C.byref(layer.c), _ptr(x_bf16), _ptr(idx), _ptr(w), k, _ptr(y), _ptr(y_bf16),
                                       int(accumulate), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_expert_ffn_decode")


def moe_expert_ffn_verify(layer: "Layer", x_bf16, T: int, idx, w, k: int, y, y_bf16=None, accumulate: bool = False,
                          ws=None, stream=None):
    _check(lib().moe_expert_ffn_verify(C.byref(layer.c), _ptr(x_bf16), T, _ptr(idx), _ptr(w), k, _ptr(y),
                                       _ptr(y_bf16), int(accumulate), _ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream)), "moe_expert_ffn_verify")


def moe_route_expert_ffn(layer: "Layer", router_w_f16, x_bf16, T: int, k: int, idx, w, y, y_bf16=None,
                         accumulate: bool = False, ws=None, stream=None):
    """Router top-k and expert FFN in one launch (tensor-core layout, MXFP4, E <= 256): writes idx [T, k] and
    w [T, k] (equal to moe_route_topk's) and y (equal to moe_expert_ffn_verify's with that routing)."""
    _check(lib().moe_route_expert_ffn(C.byref(layer.c), _ptr(router_w_f16), _ptr(x_bf16), T, k, _ptr(idx), _ptr(w),
                                      _ptr(y), _ptr(y_bf16), int(accumulate), _ptr(ws), ws.numel() * ws.element_size(),
                                      _stream(stream)), "moe_route_expert_ffn")


def moe_expert_ffn_decode_static(layer: "Layer", x_bf16, idx, w, k: int, y, y_bf16=None, accumulate: bool = False,
                                 stream=None):
    """Decode one token without a workspace: the library uses its own fixed scratch array (for callers that
    cannot allocate device memory). See include/moe.h for the limits and the first-call set-up."""
    _check(lib().moe_expert_ffn_decode_static(C.byref(layer.c), _ptr(x_bf16), _ptr(idx), _ptr(w), k, _ptr(y),
                                              _ptr(y_bf16), int(accumulate), _stream(stream)),
           "moe_expert_ffn_decode_static")


def moe_static_device_status(stream=None) -> int:
    """Device status word of the last moe_expert_ffn_decode_static call on the current device (syncs `stream`)."""
    return lib().moe_static_device_status(_stream(stream))


def moe_prefill_workspace_bytes(layer: "Layer", T_max: int, k: int) -> int:
    return lib().moe_prefill_workspace_bytes(C.byref(layer.c), T_max, k)


def moe_expert_grouped_gemm_prefill(layer: "Layer", x_bf16, T: int, idx, w, k: int, y, y_bf16=None, ws=None,
                                    stream=None):
    _check(lib().moe_expert_grouped_gemm_prefill(C.byref(layer.c), _ptr(x_bf16), T, _ptr(idx), _ptr(w), k, _ptr(y),
                                                 _ptr(y_bf16), _ptr(ws), ws.numel() * ws.element_size(),
                                                 _stream(stream)), "moe_expert_grouped_gemm_prefill")


PREFILL_OFFSETS = ("rows_max", "tiles_max", "n_tiles", "tile_first", "pair_row", "xq", "hq", "dout")


def moe_debug_prefill(layer: "Layer", x_bf16, T: int, idx, w, k: int, y, y_bf16=None, ws=None, gu_dump=None,
                      stream=None) -> dict:
    """The prefill call with test hooks; returns the workspace layout (see include/moe.h)."""
    off = (C.c_int64 * 8)()
    _check(lib().moe_debug_prefill(C.byref(layer.c), _ptr(x_bf16), T, _ptr(idx), _ptr(w), k, _ptr(y), _ptr(y_bf16),
                                   _ptr(ws), ws.numel() * ws.element_size(), _ptr(gu_dump), off, _stream(stream)),
           "moe_debug_prefill")
    return dict(zip(PREFILL_OFFSETS, list(off)))


def moe_debug_unpack(fmt: int, layout: int, kind: int, packed: torch.Tensor, H: int, I: int, expert: int,
                     out: torch.Tensor, stream=None):
    _check(lib().moe_debug_unpack(fmt, layout, kind, _ptr(packed), H, I, expert, _ptr(out), _stream(stream)),
           "moe_debug_unpack")


def moe_debug_timeout_probe(ws: torch.Tensor, limit_us: int, stream=None):
    _check(lib().moe_debug_timeout_probe(_ptr(ws), ws.numel() * ws.element_size(), limit_us, _stream(stream)),
           "moe_debug_timeout_probe")


# ------------------------------------------------------------------------------------------------ a packed layer
class Layer:
    """Device-resident packed experts of one layer plus the moe_layer_t that describes them."""

    def __init__(self, fmt: int, H: int, I: int, E: int, layout: int = MOE_LAYOUT_DECODE, device="cuda"):
        self.fmt, self.H, self.I, self.E, self.layout = fmt, H, I, E, layout
        gu = moe_packed_bytes(fmt, layout, MOE_MAT_GATE_UP, E, H, I)
        dn = moe_packed_bytes(fmt, layout, MOE_MAT_DOWN, E, H, I)
        if gu == 0 or dn == 0:
            raise MoeError(2, "moe_packed_bytes")
        self.gate_up = torch.empty(gu, dtype=torch.uint8, device=device)
        self.down = torch.empty(dn, dtype=torch.uint8, device=device)
        self.gu_stride = moe_packed_bytes(fmt, layout, MOE_MAT_GATE_UP, 1, H, I)
        self.dn_stride = moe_packed_bytes(fmt, layout, MOE_MAT_DOWN, 1, H, I)
        self.c = moe_layer_t(fmt, layout, H, I, E, self.gate_up.data_ptr(), self.down.data_ptr())

    def pack(self, src_kind: int, gate, up, down, e0: int = 0, stream=None):
        """Pack experts [e0, e0 + n) from canonical blocks (uint8) or fp32 weights ([n, I, H] / [n, H, I])."""
        n = gate.shape[0]
        gsl = self.gate_up[e0 * self.gu_stride:(e0 + n) * self.gu_stride]
        dsl = self.down[e0 * self.dn_stride:(e0 + n) * self.dn_stride]
        moe_pack_weights(self.fmt, src_kind, self.layout, MOE_MAT_GATE_UP, n, self.H, self.I, gate, up, gsl, stream)
        moe_pack_weights(self.fmt, src_kind, self.layout, MOE_MAT_DOWN, n, self.H, self.I, down, None, dsl, stream)

    def workspace(self, T_max: int, k: int, stream=None) -> torch.Tensor:
        """Zeroed, 256-byte aligned workspace for decode / verify of up to T_max tokens."""
        return self._ws(moe_workspace_bytes(self, T_max, k), stream)

    def prefill_workspace(self, T_max: int, k: int, stream=None) -> torch.Tensor:
        """Zeroed, 256-byte aligned workspace for the prefill grouped GEMM of up to T_max tokens (TC layout)."""
        return self._ws(moe_prefill_workspace_bytes(self, T_max, k), stream)

    def _ws(self, nbytes: int, stream) -> torch.Tensor:
        if nbytes == 0:
            raise MoeError(2, "workspace size")
        ws = torch.empty(nbytes + 256, dtype=torch.uint8, device=self.gate_up.device)
        off = (-ws.data_ptr()) % 256
        ws = ws[off:off + nbytes]
        moe_workspace_init(ws, stream)
        return ws
