"""The C-ABI library builds, loads and exports every symbol include/moe.h declares; host-side logic (sizes, status
strings, argument checks, fault injection) works without a GPU."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    from bit_moe_decode_gb300 import build
    build.build()
    import bit_moe_decode_gb300 as mod
    mod.lib()
    return mod


def _declared():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(m):
    names = _declared()
    assert len(names) >= 15
    L = C.CDLL(m.LIB_PATH)
    for n in names:
        assert hasattr(L, n), n
    assert sorted(m.EXPORTS) == names


def test_status_strings_and_version(m):
    assert m.moe_status_string(0) == "ok"
    assert "timed" in m.moe_status_string(7) or "time" in m.moe_status_string(7)
    assert m.moe_version() >= 100


def test_sizes_host_only(m):
    # canonical bytes: 17 B / 32, 18 B / 32, 84 B / 256
    assert m.moe_canonical_bytes(1, 2048, 4096) == 2048 * 128 * 17
    assert m.moe_canonical_bytes(2, 2048, 4096) == 2048 * 128 * 18
    assert m.moe_canonical_bytes(3, 2048, 4096) == 2048 * 16 * 84
    assert m.moe_canonical_bytes(3, 2048, 4000) == 0
    # packed layout holds exactly the canonical bytes
    for f in (1, 2, 3):
        assert m.moe_packed_bytes(f, 0, 0, 256, 4096, 2048) == 256 * 2 * m.moe_canonical_bytes(f, 2048, 4096)
        assert m.moe_packed_bytes(f, 0, 1, 256, 4096, 2048) == 256 * m.moe_canonical_bytes(f, 4096, 2048)
    # active bytes per token-layer at top-6
    per_tok = {f: 6 * (m.moe_packed_bytes(f, 0, 0, 1, 4096, 2048) + m.moe_packed_bytes(f, 0, 1, 1, 4096, 2048))
               for f in (1, 2, 3)}
    assert per_tok == {1: 80216064, 2: 84934656, 3: 49545216}
    # unsupported shapes
    assert m.moe_packed_bytes(1, 0, 0, 1, 4096 + 128, 2048) == 0
    assert m.moe_packed_bytes(1, 0, 0, 1, 8192, 2048) == 0


def test_workspace_bytes(m):
    class FakeLayer:
        pass
    lay = FakeLayer()
    lay.c = m.moe_layer_t(1, 0, 4096, 2048, 256, None, None)
    one = m.moe_workspace_bytes(lay, 1, 6)
    eight = m.moe_workspace_bytes(lay, 8, 6)
    assert one == 4096 + 6 * 8 * 2048 * 4 + 6 * 4096 * 8 * 4
    assert eight == 4096 + 48 * 8 * 2048 * 4 + 48 * 4096 * 8 * 4
    assert m.moe_workspace_bytes(lay, 9, 6) == 0


def test_fault_injection_and_argument_checks(m, monkeypatch):
    L = m.lib()
    monkeypatch.setenv("MOE_FAULT", "decode,pack")
    assert L.moe_pack_weights(1, 0, 0, 0, 1, 512, 256, None, None, None, 0, None) == 8
    lay = m.moe_layer_t(1, 0, 512, 256, 8, None, None)
    assert L.moe_expert_ffn_decode(C.byref(lay), None, None, None, 2, None, None, 0, None, 0, None) == 8
    # a call not named still runs its own checks: null pointers are rejected before any launch
    assert L.moe_expert_ffn_verify(C.byref(lay), None, 1, None, None, 2, None, None, 0, None, 0, None) == 1
    monkeypatch.setenv("MOE_FAULT", "")
    assert L.moe_pack_weights(1, 0, 0, 0, 1, 512, 256, None, None, None, 0, None) == 1
    assert L.moe_pack_weights(9, 0, 0, 0, 1, 512, 256, None, None, None, 0, None) == 3
    assert L.moe_route_topk(None, None, 1, 4096, 256, 6, None, None, 0, None, None, None) == 1
    # speculative acceptance: pointers, then K and V, are checked on the host before any launch
    buf = (C.c_float * 16)()
    ib = (C.c_int32 * 16)()
    assert L.moe_spec_accept(None, buf, 1, 4, ib, buf, ib, None) == 1
    assert L.moe_spec_accept(buf, None, 1, 4, ib, buf, ib, None) == 1       # q is needed when K > 0
    assert L.moe_spec_accept(buf, buf, 9, 4, ib, buf, ib, None) == 2
    assert L.moe_spec_accept(buf, buf, 1, 0, ib, buf, ib, None) == 2
    assert L.moe_spec_accept(buf, buf, 1, (1 << 22) + 1, ib, buf, ib, None) == 2
    monkeypatch.setenv("MOE_FAULT", "spec")
    assert L.moe_spec_accept(buf, buf, 1, 4, ib, buf, ib, None) == 8


def _aligned(nbytes: int, align: int):
    """A host buffer and an address inside it aligned to `align` (only for checks that precede any launch)."""
    buf = (C.c_uint8 * (nbytes + align))()
    addr = C.addressof(buf)
    return buf, addr + (-addr) % align


def test_ffn_and_fused_call_argument_checks(m):
    """Every argument error of the decode / verify / fused calls is found on the host, before the device check, so
    these run without a GPU."""
    L = m.lib()
    keep = []
    def ptr(n=1 << 12, align=256):
        b, a = _aligned(n, align)
        keep.append(b)
        return C.c_void_p(a)
    gu, dn, x, ws, y, idx, w, wr = (ptr() for _ in range(8))
    def layer(fmt=1, layout=1, H=4096, I=2048, E=256, g=gu, d=dn):
        return m.moe_layer_t(fmt, layout, H, I, E, g, d)
    lay = layer()
    ver = L.moe_expert_ffn_verify
    # verify: null pointers, bad format / layout, sizes
    assert ver(C.byref(lay), None, 1, idx, w, 6, y, None, 0, ws, 1 << 20, None) == 1
    assert ver(C.byref(layer(fmt=4)), x, 1, idx, w, 6, y, None, 0, ws, 1 << 20, None) == 3
    assert ver(C.byref(layer(layout=5)), x, 1, idx, w, 6, y, None, 0, ws, 1 << 20, None) == 3
    assert ver(C.byref(lay), x, 9, idx, w, 6, y, None, 0, ws, 1 << 20, None) == 2
    assert ver(C.byref(lay), x, 0, idx, w, 6, y, None, 0, ws, 1 << 20, None) == 2
    assert ver(C.byref(lay), x, 1, idx, w, 9, y, None, 0, ws, 1 << 20, None) == 2
    assert ver(C.byref(layer(H=4096 + 64)), x, 1, idx, w, 6, y, None, 0, ws, 1 << 20, None) == 2
    assert ver(C.byref(layer(fmt=2)), x, 1, idx, w, 6, y, None, 0, ws, 1 << 20, None) == 3   # INT4 has no TC layout
    assert ver(C.byref(lay), x, 1, idx, w, 6, y, None, 0, C.c_void_p(ws.value + 8), 1 << 20, None) == 1  # ws alignment
    # fused router + FFN: MXFP4 in the tensor-core layout, E <= 256, 16-byte aligned router and x
    fused = L.moe_route_expert_ffn
    assert fused(C.byref(lay), None, x, 1, 6, idx, w, y, None, 0, ws, 1 << 20, None) == 1
    assert fused(C.byref(layer(layout=0)), wr, x, 1, 6, idx, w, y, None, 0, ws, 1 << 20, None) == 3
    assert fused(C.byref(layer(E=300)), wr, x, 1, 6, idx, w, y, None, 0, ws, 1 << 20, None) == 2
    assert fused(C.byref(layer(E=4)), wr, x, 1, 6, idx, w, y, None, 0, ws, 1 << 20, None) == 2          # E < k
    assert fused(C.byref(lay), wr, C.c_void_p(x.value + 4), 1, 6, idx, w, y, None, 0, ws, 1 << 20, None) == 1
    assert fused(C.byref(lay), wr, x, 9, 6, idx, w, y, None, 0, ws, 1 << 20, None) == 2


def test_prefill_argument_checks(m):
    """The prefill call's argument and size errors, found on the host before the device check."""
    L = m.lib()
    keep = []
    def ptr(n=1 << 12, align=256):
        b, a = _aligned(n, align)
        keep.append(b)
        return C.c_void_p(a)
    gu, dn, x, ws, y, idx, w = (ptr() for _ in range(7))
    def layer(fmt=1, layout=1, H=4096, I=2048, E=256):
        return m.moe_layer_t(fmt, layout, H, I, E, gu, dn)
    pre = L.moe_expert_grouped_gemm_prefill
    lay = layer()
    assert pre(C.byref(lay), None, 16, idx, w, 6, y, None, ws, 1 << 20, None) == 1
    assert pre(C.byref(lay), x, 16, idx, w, 6, None, None, ws, 1 << 20, None) == 1      # neither y nor y_bf16
    assert pre(C.byref(layer(fmt=3)), x, 16, idx, w, 6, y, None, ws, 1 << 20, None) == 3
    assert pre(C.byref(layer(layout=0)), x, 16, idx, w, 6, y, None, ws, 1 << 20, None) == 3
    assert pre(C.byref(layer(H=4096 + 64)), x, 16, idx, w, 6, y, None, ws, 1 << 20, None) == 2
    assert pre(C.byref(lay), x, 0, idx, w, 6, y, None, ws, 1 << 20, None) == 2
    assert pre(C.byref(lay), x, 16, idx, w, 9, y, None, ws, 1 << 20, None) == 2
    assert pre(C.byref(layer(E=4)), x, 16, idx, w, 6, y, None, ws, 1 << 20, None) == 2     # k > E
    assert pre(C.byref(lay), C.c_void_p(x.value + 4), 16, idx, w, 6, y, None, ws, 1 << 20, None) == 1
    assert pre(C.byref(lay), x, 16, idx, w, 6, y, None, ws, 16, None) == 5                # workspace too small


def test_header_is_plain_c_and_links(m, tmp_path):
    """include/moe.h compiles as C11 with warnings as errors, and a C program that calls through it links against
    libmoe.so: the boundary needs no C++ and no torch"""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    prog = tmp_path / "use_moe.c"
    prog.write_text('#include "moe.h"\n#include <stdio.h>\n'
                    'int main(void) { printf("%d %s\\n", (int)moe_version(), moe_status_string(MOE_OK));\n'
                    '  return moe_canonical_bytes(MOE_FMT_Q8_0, 4, 64) == 4 * 2 * 34 ? 0 : 1; }\n')
    exe = tmp_path / "use_moe"
    lib_dir = os.path.dirname(m.LIB_PATH)
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    str(prog), "-o", str(exe), "-L", lib_dir, "-lmoe", "-Wl,-rpath," + lib_dir], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.split() == [str(m.lib().moe_version()), m.lib().moe_status_string(0).decode()]
