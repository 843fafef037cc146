"""Pins of the oracle's number formats against what the pages print and what the mathematics fixes.

Each test names the page passage it checks. None of them re-types the oracle's own formula: the
expected values come from printed tables, hand-built blocks worked out by hand, closed forms, brute
force on small inputs or independent library routines (numpy / torch conversions).
"""
import math
import os
import warnings

import numpy as np
import pytest
import torch

import oracle
from moe_inputs import f32_to_bf16_bits

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _table():
    vals = {}
    for line in open(os.path.join(GOLD, "e2m1_table.txt")):
        if line.startswith("#") or not line.strip():
            continue
        c, v = line.split()
        vals[int(c)] = float(v)
    return vals


def _handbuilt(name):
    rows = [l.split(None, 1) for l in open(os.path.join(GOLD, name)) if l.strip() and not l.startswith("#")]
    out = {}
    for key, payload in rows:
        out.setdefault(key, []).append(payload.strip())
    return {k: (bytes.fromhex(v[0]), np.array([float(x) for x in v[1].split()])) for k, v in out.items()}


# ---------------------------------------------------------------- scalar conversions vs library routines
def test_f16_bits_to_value_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(b)) for b in bits[::7]])
    r = ref[::7]
    assert np.array_equal(np.isnan(got), np.isnan(r))
    m = ~np.isnan(r)
    assert np.array_equal(got[m], r[m]) and np.array_equal(np.signbit(got[m]), np.signbit(r[m]))


def test_bf16_bits_to_value_matches_torch():
    bits = np.arange(0, 65536, 5, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    m = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), ~m)
    assert np.array_equal(got[m], ref[m])


def test_rounding_helpers_match_numpy_and_torch():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-12, 12, 4000),
                        rng.standard_normal(500) * 1e-6, [65519.99, 65520.0, 65504.0, 6.1e-5, 5.96e-8, 2.98e-8]])
    f32 = np.array([oracle.round_f32(float(v)) for v in x])
    assert np.array_equal(f32, x.astype(np.float32).astype(np.float64))
    f16 = np.array([oracle.round_f16(float(v)) for v in x])
    ref16 = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(f16, ref16)
    xb = x.astype(np.float32)
    bf = np.array([oracle.round_bf16(float(v)) for v in xb])
    refb = torch.from_numpy(xb).to(torch.bfloat16).double().numpy()
    assert np.array_equal(bf, refb)
    # fp32 -> fp16 bits equals numpy's conversion
    for v in xb[:800]:
        assert oracle.f32_to_f16_rne(float(v)) == int(np.float16(v).view(np.uint16))


# ---------------------------------------------------------------- MXFP4
def test_e2m1_table_printed_on_pages():
    t = _table()
    for c in range(16):
        v = oracle.e2m1_value(c)
        assert v == t[c] and math.copysign(1, v) == math.copysign(1, t[c]), c


def test_e8m0_rule():
    """glossary "MXFP4": 2^(e-127), e=0 treated as zero; LUT section: the 0xff row is NaN."""
    assert oracle.e8m0_scale(0) == 0.0
    assert math.isnan(oracle.e8m0_scale(255))
    assert oracle.e8m0_scale(127) == 1.0 and oracle.e8m0_scale(128) == 2.0 and oracle.e8m0_scale(126) == 0.5
    for e in range(1, 255):
        assert oracle.e8m0_scale(e) == math.ldexp(1.0, e - 127)


def test_mxfp4_block_size_and_rate():
    w = np.random.default_rng(0).standard_normal((3, 64)).astype(np.float32)
    blk = oracle.encode(oracle.MXFP4, w)
    assert blk.shape == (3, 2 * 17)
    assert blk.size * 8 / w.size == 4.25


def test_mxfp4_handbuilt_blocks():
    for key, (raw, vals) in _handbuilt("mxfp4_handbuilt.txt").items():
        got = oracle.decode(oracle.MXFP4, np.frombuffer(raw, np.uint8))
        assert np.array_equal(got, vals.astype(np.float32)), key
        assert np.array_equal(np.signbit(got), np.signbit(vals)), key


def test_mxfp4_decode_exhaustive_vs_numpy_ldexp():
    """every (e, code) pair: value = table[code] * 2^(e-127) rounded to fp32 (numpy ldexp in float32)."""
    t = _table()
    raw = np.zeros((256 * 8, 17), np.uint8)
    for e in range(256):
        for j in range(8):
            raw[e * 8 + j, 0] = e
            raw[e * 8 + j, 1:] = ((2 * j) << 4) | (2 * j + 1)   # codes 2j, 2j+1 repeated
    got = oracle.decode(oracle.MXFP4, raw).reshape(256 * 8, 32)
    for e in range(256):
        for j in range(8):
            for c, col in ((2 * j, 0), (2 * j + 1, 1)):
                g = got[e * 8 + j, col]
                if e == 255:
                    assert np.isnan(g)
                elif e == 0:
                    assert g == 0.0
                else:
                    ref = np.ldexp(np.float32(t[c]), e - 127).astype(np.float32)
                    assert g == ref and np.signbit(g) == np.signbit(ref), (e, c)


def test_mxfp4_element_order_follows_printed_unpack():
    """model card step 1: vals = stack([TABLE[byte >> 4], TABLE[byte & 0xF]]).flatten()."""
    t = _table()
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, size=16, dtype=np.uint8)
    raw = np.concatenate([[127], codes]).astype(np.uint8)
    got = oracle.decode(oracle.MXFP4, raw)
    ref = np.stack([[t[b >> 4] for b in codes], [t[b & 15] for b in codes]], -1).reshape(-1)
    assert np.array_equal(got, ref.astype(np.float32))


def _e2m1_brute(v):
    """nearest of the 16 table values, ties to the even code, sign of v kept on zero"""
    t = _table()
    mags = [t[c] for c in range(8)]
    a = abs(v)
    d = [abs(a - m) for m in mags]
    best = min(range(8), key=lambda c: (d[c], c % 2))
    return best | (8 if math.copysign(1, v) < 0 else 0)


def test_mxfp4_encoder_brute_force_small():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((40, 32)) * 10.0 ** rng.integers(-3, 2, (40, 1))).astype(np.float32)
    w[0, :] = 0.0
    w[1, 5] = -0.0
    blk = oracle.encode(oracle.MXFP4, w).reshape(40, 17)
    for b in range(40):
        amax = float(np.max(np.abs(w[b].astype(np.float64))))
        if amax == 0:
            e = 1
        else:
            k = math.ceil(math.log2(amax / 6.0))
            # exact correction of the float log at powers of two
            while amax > 6 * 2.0 ** k:
                k += 1
            while amax <= 6 * 2.0 ** (k - 1):
                k -= 1
            e = min(max(k + 127, 1), 254)
        assert blk[b, 0] == e
        for j in range(32):
            v = float(w[b, j]) * 2.0 ** (127 - e)
            code = (blk[b, 1 + j // 2] >> 4) if j % 2 == 0 else (blk[b, 1 + j // 2] & 15)
            assert code == _e2m1_brute(v), (b, j, v)


def test_mxfp4_encoder_ties_and_roundtrip():
    """ties go to the even code (0.25->0, 0.75->1, 1.25->1, 1.75->2, 2.5->2, 3.5->4, 5->4); grid values
    round-trip exactly; the error bound is half a step."""
    ties = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    expect = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    w = np.zeros(32, np.float32)
    w[0] = 6.0                                 # amax 6 -> e = 127, scale 1
    w[1:8] = ties
    w[8:15] = [-t for t in ties]
    dec = oracle.decode(oracle.MXFP4, oracle.encode(oracle.MXFP4, w))
    assert np.array_equal(dec[1:8], np.array(expect, np.float32))
    assert np.array_equal(dec[8:15], -np.array(expect, np.float32))
    t = _table()
    rng = np.random.default_rng(9)
    grid = np.array([t[c] for c in rng.integers(0, 16, 32 * 50)], np.float32).reshape(50, 32)
    grid[:, 0] = 6.0
    scale = np.ldexp(np.float32(1), rng.integers(-20, 20, (50, 1))).astype(np.float32)
    g = grid * scale
    assert np.array_equal(oracle.decode(oracle.MXFP4, oracle.encode(oracle.MXFP4, g)).reshape(50, 32), g)
    # half-step bound on random data (spacing of E2M1 near |v|: 0.5 below 2, 1 below 4, 2 above)
    x = rng.standard_normal((200, 32)).astype(np.float32) * 0.02
    blk = oracle.encode(oracle.MXFP4, x).reshape(200, 17)
    dec = oracle.decode(oracle.MXFP4, blk).reshape(200, 32)
    s = np.ldexp(1.0, blk[:, :1].astype(np.int64) - 127)
    v = np.abs(x / s)
    step = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0))
    assert np.all(np.abs(dec - x) <= step / 2 * s + 1e-30)


# ---------------------------------------------------------------- INT4 g32
def test_int4_layout_and_decode_closed_form():
    rng = np.random.default_rng(11)
    q = rng.integers(-8, 8, size=32)
    scale = np.float32(0.0123)
    sb = int(f32_to_bf16_bits(np.array([scale]))[0])
    raw = np.zeros(18, np.uint8)
    for j in range(32):
        n = int(q[j]) & 15
        raw[j // 2] |= (n << 4) if j % 2 == 0 else n
    raw[16], raw[17] = sb & 255, sb >> 8
    got = oracle.decode(oracle.INT4G32, raw)
    sval = torch.tensor([scale]).to(torch.bfloat16).float().item()
    assert np.array_equal(got, (q * np.float64(sval)).astype(np.float32))


def test_int4_encoder_is_grid_argmin():
    """model card step 2: for each r in the grid, s = amax*r/7, q = clamp(round(w/s), -8, 7); keep the (q, s)
    of smallest MSE. Checked with torch fp32 ops (torch.round rounds half to even)."""
    grid = [6 / 7, 0.9, 0.95, 1.0, 1.05, 1.1]
    rng = np.random.default_rng(13)
    w = (rng.standard_normal((300, 32)) * 0.02).astype(np.float32)
    w[0] = 0.0
    blk = oracle.encode(oracle.INT4G32, w).reshape(300, 18)
    assert blk.shape[1] * 8 / 32 == 4.5
    W = torch.from_numpy(w)
    amax = W.abs().amax(-1, keepdim=True).clamp(min=1e-8)
    mses, qs, ss = [], [], []
    for r in grid:
        s = amax * torch.tensor(r, dtype=torch.float32) / 7
        qq = torch.clamp(torch.round(W / s), -8, 7)
        mses.append(((W - qq * s) ** 2).sum(-1))
        qs.append(qq)
        ss.append(s)
    M = torch.stack(mses, 1)
    dec = torch.from_numpy(oracle.decode(oracle.INT4G32, blk).reshape(300, 32))
    codes = np.zeros((300, 32), np.int64)
    for j in range(32):
        n = (blk[:, j // 2] >> 4) if j % 2 == 0 else (blk[:, j // 2] & 15)
        codes[:, j] = np.where(n >= 8, n.astype(np.int64) - 16, n)
    assert codes.min() >= -8 and codes.max() <= 7
    for b in range(300):
        best = int(torch.argmin(M[b]))
        # the chosen candidate is the argmin, or within summation-order rounding of it
        stored = int(blk[b, 16]) | (int(blk[b, 17]) << 8)
        bf = lambda i: int(torch.tensor([ss[i][b, 0].item()]).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF
        chosen = [i for i in range(6)
                  if torch.equal(qs[i][b].long(), torch.from_numpy(codes[b])) and bf(i) == stored]
        assert chosen, b
        assert min(float(M[b, i]) for i in chosen) <= float(M[b, best]) * (1 + 1e-5) + 1e-30
        sb = torch.tensor([ss[chosen[0]][b, 0].item()]).to(torch.bfloat16).float()
        assert torch.equal(dec[b], (torch.from_numpy(codes[b]).float() * sb).float())
    # the grid search never does worse than plain r = 1 on the stored codes' own fp32 scale
    assert float(M.min(1).values.sum()) <= float(M[:, 3].sum())


# ---------------------------------------------------------------- Q8_0 (the shared expert's format, defined by the library)
def test_q8_0_layout_and_decode_closed_form():
    """34 bytes per 32 weights (8.5 bits): fp16 d little-endian, then 32 two's-complement codes; w = d * q."""
    rng = np.random.default_rng(21)
    q = rng.integers(-127, 128, size=32)
    d = np.float16(0.0123)
    raw = np.zeros(34, np.uint8)
    raw[0:2] = np.frombuffer(d.tobytes(), np.uint8)
    raw[2:] = q.astype(np.int8).view(np.uint8)
    assert oracle.BLOCK[oracle.Q8_0] == (32, 34) and 34 * 8 / 32 == 8.5
    got = oracle.decode(oracle.Q8_0, raw)
    assert np.array_equal(got, (q * np.float64(d)).astype(np.float32))


def test_q8_0_encoder_against_torch():
    """d = fp16(amax / 127), q = clamp(round_half_even(w / d), -127, 127), in fp32 (torch.round is half-even)."""
    rng = np.random.default_rng(22)
    w = (rng.standard_normal((400, 32)) * 0.02).astype(np.float32)
    w[0] = 0.0                                # d = 0: all codes 0
    w[1, 5] = -w[1].__abs__().max() * 2       # the largest magnitude negative: code -127
    blk = oracle.encode(oracle.Q8_0, w).reshape(400, 34)
    W = torch.from_numpy(w)
    d = (W.abs().amax(-1, keepdim=True) / 127).to(torch.float16)
    df = d.float()
    qq = torch.where(df == 0, torch.zeros_like(W), torch.clamp(torch.round(W / torch.where(df == 0, 1, df)), -127, 127))
    assert np.array_equal(blk[:, 0:2].copy().view(np.float16)[:, 0], d[:, 0].numpy())
    assert np.array_equal(blk[:, 2:].view(np.int8).astype(np.int64), qq.long().numpy())
    assert np.all(blk[0] == 0) and blk[1, 2 + 5].view(np.int8) == -127
    dec = oracle.decode(oracle.Q8_0, blk).reshape(400, 32)
    # every weight within half a step of its code (d / 2), the step being the stored fp16 d
    assert np.all(np.abs(dec - w) <= df.numpy() / 2 * (1 + 1e-6) + 1e-30)


def test_q8_0_encoder_ties_go_to_even_and_clamp():
    """Exact half steps round to the even code (d a power of two, so w / d is exact); values past 127 d clamp."""
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = 127.0 * 0.25                    # amax: d = 0.25 exactly
    halves = [0.5, 1.5, 2.5, -0.5, -2.5, 126.5]
    for i, h in enumerate(halves):
        w[0, 1 + i] = h * 0.25
    blk = oracle.encode(oracle.Q8_0, w)[0]
    assert blk[0:2].view(np.float16)[0] == np.float16(0.25)
    codes = blk[2:].view(np.int8)
    assert codes[0] == 127
    assert list(codes[1:7]) == [0, 2, 2, 0, -2, 126]


# ---------------------------------------------------------------- Q2_K
def test_q2k_handbuilt_block():
    (raw, vals), = _handbuilt("q2k_handbuilt.txt").values()
    got = oracle.decode(oracle.Q2K, np.frombuffer(raw, np.uint8))
    assert np.array_equal(got, vals.astype(np.float32))


def test_q2k_size_and_encoder_bounds():
    rng = np.random.default_rng(17)
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    blk = oracle.encode(oracle.Q2K, w).reshape(64, 84)
    assert blk.size * 8 / w.size == 2.625
    dec = oracle.decode(oracle.Q2K, blk).reshape(64, 256)
    d = np.frombuffer(blk[:, 80:82].tobytes(), np.float16).astype(np.float64)
    dmin = np.frombuffer(blk[:, 82:84].tobytes(), np.float16).astype(np.float64)
    for b in range(64):
        for g in range(16):
            sc, m = blk[b, g] & 15, blk[b, g] >> 4
            step = d[b] * sc
            seg = w[b, g * 16:(g + 1) * 16].astype(np.float64)
            rec = dec[b, g * 16:(g + 1) * 16].astype(np.float64)
            lo = -dmin[b] * m
            hi = lo + 3 * step
            inside = (seg >= lo) & (seg <= hi)
            # inside the representable range: at most half a step (+ fp32 rounding) off
            assert np.all(np.abs(seg - rec)[inside] <= step / 2 + 1e-6 * max(step, 1e-30) + 1e-9)
            # outside it: reconstruction is the nearest end of the range
            assert np.all(rec[~inside] == np.clip(rec[~inside], lo - 1e-7, hi + 1e-7))
    # relative reconstruction error of a 2.6-bit code on Gaussian data: well below 1, well above 0
    rel = np.linalg.norm(dec - w) / np.linalg.norm(w)
    assert 0.1 < rel < 0.6


def test_q2k_decode_matches_closed_form_random_blocks():
    """w = d*sc*q - dmin*m evaluated independently with numpy from the raw bytes."""
    rng = np.random.default_rng(19)
    blk = rng.integers(0, 256, size=(30, 84), dtype=np.uint8)
    blk[:, 80:84] = np.frombuffer(np.abs(rng.standard_normal(60)).astype(np.float16).tobytes(), np.uint8).reshape(30, 4)
    got = oracle.decode(oracle.Q2K, blk).reshape(30, 256)
    d = np.frombuffer(blk[:, 80:82].tobytes(), np.float16).astype(np.float32)
    dmin = np.frombuffer(blk[:, 82:84].tobytes(), np.float16).astype(np.float32)
    for b in range(30):
        i = np.arange(256)
        sc = (blk[b, i // 16] & 15).astype(np.float32)
        m = (blk[b, i // 16] >> 4).astype(np.float32)
        q = ((blk[b, 16 + i // 4] >> (2 * (i % 4))) & 3).astype(np.float32)
        ref = (np.float32(d[b]) * sc) * q - np.float32(dmin[b]) * m
        assert np.array_equal(got[b], ref.astype(np.float32))


# ---------------------------------------------------------------- MXFP8 (prefill activations)
def test_e4m3_values_and_quantiser_vs_torch():
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0x08) == 2.0 ** -6 and oracle.e4m3_value(0x01) == 2.0 ** -9
    assert math.isnan(oracle.e4m3_value(0x7F))
    allc = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        v = oracle.e4m3_value(c)
        assert (math.isnan(v) and math.isnan(allc[c])) or v == allc[c]
    rng = np.random.default_rng(23)
    v = rng.standard_normal((100, 32)) * 10.0 ** rng.integers(-4, 4, (100, 1))
    v = v.astype(np.float32).astype(np.float64)
    codes, scales = oracle.quant_mxfp8(v)
    for b in range(100):
        amax = np.max(np.abs(v[b]))
        e = int(scales[b, 0])
        assert amax <= 448 * 2.0 ** (e - 127) and amax > 448 * 2.0 ** (e - 128)
        scaled = torch.from_numpy(v[b] * 2.0 ** (127 - e))
        ref = scaled.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(codes[b], ref), b


def test_mxfp8_quantiser_ties_go_to_even_codes_vs_torch():
    # values exactly halfway between neighbouring E4M3 values (normal and subnormal), in blocks whose largest
    # value is 448 so that the scale is 2^0 and the quantiser sees them unscaled; torch's float8_e4m3fn
    # conversion rounds them to the even code
    pos = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()   # 0 .. 448
    mids = (pos[:-1] + pos[1:]) / 2.0
    vals = np.concatenate([mids, -mids])
    nb = (len(vals) + 30) // 31
    blocks = np.zeros((nb, 32))
    blocks[:, 0] = 448.0
    flat = np.zeros(nb * 31)
    flat[:len(vals)] = vals
    blocks[:, 1:] = flat.reshape(nb, 31)
    codes, scales = oracle.quant_mxfp8(blocks)
    assert np.all(scales[:, 0] == 127)
    ref = torch.from_numpy(blocks).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


# ---------------------------------------------------------------- the half LUT of the Metal section
def test_mxfp4_half_lut_hash_has_not_drifted():
    # the generated 4096-entry table is pinned by its SHA-256, written by tests/golden/make_lut_hash.py from the
    # oracle when the table was checked entry by entry (test_mxfp4_half_lut_properties)
    import hashlib
    lut = oracle.mxfp4_half_lut()
    want = open(os.path.join(GOLD, "mxfp4_half_lut.sha256")).read().split()[0]
    assert hashlib.sha256(lut.astype("<u2").tobytes()).hexdigest() == want


def test_mxfp4_half_lut_properties():
    lut = oracle.mxfp4_half_lut()
    assert lut.shape == (256, 16) and lut.size == 4096
    t = _table()
    f = lut.view(np.float16).astype(np.float64)
    assert np.all(f[0] == 0)
    assert np.all(np.isnan(f[255]))
    for e in range(1, 255):
        exact = np.array([t[c] * 2.0 ** (e - 127) for c in range(16)])
        ref = exact.astype(np.float16)          # numpy: one RNE rounding to binary16
        assert np.array_equal(lut[e], ref.view(np.uint16)), e
        if 104 <= e <= 140:
            assert np.array_equal(f[e], exact), e   # exactly representable window
    # outside the window at least one product is rounded (not exact)
    assert not np.array_equal(f[103], np.array([t[c] * 2.0 ** (103 - 127) for c in range(16)]))
    assert not np.array_equal(f[141], np.array([t[c] * 2.0 ** (141 - 127) for c in range(16)]))
