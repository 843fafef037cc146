"""The speculative-acceptance pins catch plausible mistakes: each test plants one mistake in a copy of the oracle's
C source (on the CPU, in a temporary directory), builds it, and checks that a pin of tests/test_oracle_spec.py
fails on it while the unmodified oracle passes."""
import ctypes as C
import os
import subprocess

import numpy as np
import pytest

import oracle
from moe_inputs import spec_inputs
from tests.test_oracle_spec import _draw_law, _first_token_law

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    # keep a draft when u > p/q instead of u < p/q
    "accept_inverted": ("if (!(u[n] < ratio)) break;", "if (!(u[n] > ratio)) break;"),
    # residual q - p instead of p - q
    "residual_swapped": ("float r = q ? p[v] - q[v] : p[v];", "float r = q ? q[v] - p[v] : p[v];"),
    # residual not clamped at 0 (negative weights count)
    "residual_unclamped": ("if (!(r > 0.0f)) r = 0.0f;  /* negative or NaN: no mass */", "if (r != r) r = 0.0f;"),
    # the extra token after K acceptances drawn from the last draft position instead of the row after it
    "bonus_row_off_by_one": ("tok = spec_draw(p + (int64_t)K * V, NULL, V, u[K]);",
                             "tok = spec_draw(p + (int64_t)(K - 1) * V, NULL, V, u[K]);"),
}


def _build(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / (name + ".c")
    path.write_text(src.replace(old, new))
    lib = tmp_path / ("lib" + name + ".so")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                    str(path), "-o", str(lib), "-lm"], check=True)
    L = C.CDLL(str(lib))
    f = L.orc_spec_accept
    f.restype = None
    f.argtypes = [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p]

    def accept(p, q, draft, u):
        pp = np.ascontiguousarray(p, np.float32)
        K, V = pp.shape[0] - 1, pp.shape[1]
        qq = np.ascontiguousarray(q, np.float32).reshape(K, V) if K else np.zeros((1, V), np.float32)
        d = np.ascontiguousarray(np.asarray(draft, np.int32).reshape(-1)) if K else np.zeros(1, np.int32)
        uu = np.ascontiguousarray(np.asarray(u, np.float32).reshape(-1))
        out = np.empty(2, np.int32)
        f(pp.ctypes.data, qq.ctypes.data, K, V, d.ctypes.data, uu.ctypes.data, out.ctypes.data)
        return int(out[0]), int(out[1])
    return accept


def _lossless_holds(accept) -> bool:
    p, q, _, _ = spec_inputs(5, 1, 6, spread=1.0, noise=1.0)
    return np.allclose(_first_token_law(p, q, accept), p[0], atol=1e-6)


def _bonus_law_holds(accept) -> bool:
    p, _, d, _ = spec_inputs(7, 3, 6, spread=1.0)
    return np.allclose(_draw_law(p, p[:3].copy(), d, [0.9999999, 0.5, 0.0], accept), p[3], atol=1e-6)


def test_unmodified_oracle_passes_the_pins():
    assert _lossless_holds(oracle.spec_accept) and _bonus_law_holds(oracle.spec_accept)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_fails_a_pin(tmp_path, name):
    accept = _build(tmp_path, name, *MUTANTS[name])
    assert not (_lossless_holds(accept) and _bonus_law_holds(accept)), name
