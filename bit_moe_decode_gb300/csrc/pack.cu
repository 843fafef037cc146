// pack.cu -- GPU encoders (fp32 -> canonical blocks) and the packer (canonical blocks or fp32 -> device layout).
//
// Formats: "quantization" glossary (ds4-learning.pages.dev), sections "MXFP4" and "core principle" (Q2_K);
// INT4 group 32: "DeepSeek-V4-Flash-0731-W4A16" model card (alphaneural.io), "FP4 -> INT4 conversion" step 2.
// Q8_0 (the shared expert's "Q8" of "Mixed-precision compression of DeepSeek-V4-Flash", "The recipe"; the pages
// give no layout, so the library defines one scale per 32 weights like the other formats).
// All encoder arithmetic is fp32 with round-to-nearest-even and no contraction (explicit __f*_rn intrinsics).
#include "common.cuh"
#include "layout.cuh"
#include "api_internal.h"

namespace moe {

// ------------------------------------------------------------------ encoders (one canonical block per call)

// MXFP4: exponent e = clamp(k + 127, 1, 254), k the smallest integer with amax <= 6 * 2^k. With amax = m * 2^E
// (1 <= m < 2), 6 * 2^k = 1.5 * 2^(k+2), so k = E - 2 if m <= 1.5 and E - 1 otherwise.
__device__ void enc_mxfp4(const float* w, uint8_t* out /*17*/) {
  float amax = 0.f;
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(w[j]));
  uint32_t ab = __float_as_uint(amax);
  int ef = (int)(ab >> 23);
  int e;
  if (ef == 0) e = 1;  // zero or subnormal amax: k + 127 < 1
  else e = ef - 2 + ((ab & 0x7FFFFF) > 0x400000 ? 1 : 0);
  e = e < 1 ? 1 : (e > 254 ? 254 : e);
  out[0] = (uint8_t)e;
  for (int j = 0; j < 32; j += 2) {
    uint8_t byte = 0;
    for (int h = 0; h < 2; ++h) {
      float v = scalbnf(w[j + h], 127 - e);   // exact power-of-two scaling
      float a = fabsf(v);
      // nearest E2M1 magnitude, ties to even code: count the decision points passed (strict at ties that
      // round down to the even code, inclusive at ties that round up to it)
      int c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) + (a > 5.0f);
      c |= (__float_as_uint(v) >> 28) & 8;
      byte |= (uint8_t)(h == 0 ? (c << 4) : c);  // element 2i in the high nibble
    }
    out[1 + j / 2] = byte;
  }
}

// INT4 g32 with the six-candidate round-rate grid; first candidate with the strictly smallest fp32 error wins.
__device__ void enc_int4(const float* w, uint8_t* out /*18*/) {
  const float grid[6] = {6.0f / 7.0f, 0.9f, 0.95f, 1.0f, 1.05f, 1.1f};
  float amax = 0.f;
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(w[j]));
  amax = fmaxf(amax, 1e-8f);
  float best = __int_as_float(0x7f800000);
  float best_s = 0.f;
  for (int i = 0; i < 6; ++i) {
    float s = __fdiv_rn(__fmul_rn(amax, grid[i]), 7.0f);
    float mse = 0.f;
    for (int j = 0; j < 32; ++j) {
      float q = fminf(fmaxf(rintf(__fdiv_rn(w[j], s)), -8.f), 7.f);
      float d = __fsub_rn(w[j], __fmul_rn(q, s));
      mse = __fadd_rn(mse, __fmul_rn(d, d));
    }
    if (i == 0 || mse < best) { best = mse; best_s = s; }  // first candidate is the initial best
  }
  for (int j = 0; j < 32; j += 2) {
    int q0 = (int)fminf(fmaxf(rintf(__fdiv_rn(w[j], best_s)), -8.f), 7.f);
    int q1 = (int)fminf(fmaxf(rintf(__fdiv_rn(w[j + 1], best_s)), -8.f), 7.f);
    out[j / 2] = (uint8_t)(((q0 & 15) << 4) | (q1 & 15));
  }
  // bf16 round-to-nearest-even of the positive finite scale, on the bit pattern
  const uint32_t sbits = __float_as_uint(best_s);
  const uint32_t bits = (sbits + 0x7FFFu + ((sbits >> 16) & 1u)) >> 16;
  out[16] = (uint8_t)(bits & 255u);
  out[17] = (uint8_t)((bits >> 8) & 255u);
}

// Q2_K (the library's own encoder; the pages give none): per 16-weight group lo = min(0, min), s = (max-lo)/3,
// o = -lo; d, dmin = fp16 of the largest s, o over 15; integer sc, m by rounding; q by rounding (w + dmin m)/(d sc).
__device__ void enc_q2k(const float* w, uint8_t* out /*84*/) {
  float s[16], o[16];
  float smax = 0.f, omax = 0.f;
  for (int g = 0; g < 16; ++g) {
    float lo = 0.f, hi = -__int_as_float(0x7f800000);
    for (int j = 0; j < 16; ++j) { lo = fminf(lo, w[g * 16 + j]); hi = fmaxf(hi, w[g * 16 + j]); }
    s[g] = __fdiv_rn(__fsub_rn(hi, lo), 3.0f);
    o[g] = -lo;
    smax = fmaxf(smax, s[g]);
    omax = fmaxf(omax, o[g]);
  }
  __half dh = __float2half_rn(__fdiv_rn(smax, 15.0f));
  __half mh = __float2half_rn(__fdiv_rn(omax, 15.0f));
  float d = __half2float(dh), dmin = __half2float(mh);
  for (int i = 0; i < 84; ++i) out[i] = 0;
  for (int g = 0; g < 16; ++g) {
    float a = d > 0.f ? rintf(__fdiv_rn(s[g], d)) : 0.f;
    float c = dmin > 0.f ? rintf(__fdiv_rn(o[g], dmin)) : 0.f;
    int sc = (int)fminf(fmaxf(a, 0.f), 15.f), m = (int)fminf(fmaxf(c, 0.f), 15.f);
    out[g] = (uint8_t)(sc | (m << 4));
    float step = __fmul_rn(d, (float)sc), off = __fmul_rn(dmin, (float)m);
    for (int j = 0; j < 16; ++j) {
      int q = 0;
      if (step > 0.f) q = (int)fminf(fmaxf(rintf(__fdiv_rn(__fadd_rn(w[g * 16 + j], off), step)), 0.f), 3.f);
      int i = g * 16 + j;
      out[16 + i / 4] |= (uint8_t)(q << (2 * (i % 4)));
    }
  }
  uint16_t db = __half_as_ushort(dh), mb = __half_as_ushort(mh);
  out[80] = (uint8_t)(db & 255); out[81] = (uint8_t)(db >> 8);
  out[82] = (uint8_t)(mb & 255); out[83] = (uint8_t)(mb >> 8);
}

// Q8_0: d = fp16(amax / 127); q = clamp(rint(w / d), -127, 127), 0 where d = 0 or the quotient is NaN.
__device__ void enc_q8_0(const float* w, uint8_t* out /*34*/) {
  float amax = 0.f;
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(w[j]));   // NaN inputs do not raise amax
  const __half dh = __float2half_rn(__fdiv_rn(amax, 127.0f));
  const float d = __half2float(dh);
  const uint16_t db = __half_as_ushort(dh);
  out[0] = (uint8_t)(db & 255);
  out[1] = (uint8_t)(db >> 8);
  for (int j = 0; j < 32; ++j) {
    float q = 0.f;
    if (d != 0.f) {
      q = rintf(__fdiv_rn(w[j], d));
      if (q != q) q = 0.f;                 // before the clamp: fminf / fmaxf would turn NaN into a bound
      q = fminf(fmaxf(q, -127.f), 127.f);
    }
    out[2 + j] = (uint8_t)(int8_t)(int)q;
  }
}

template <int FMT>
__device__ __forceinline__ void get_block(const void* src, moe_src_t kind, int64_t blk, uint8_t* out) {
  constexpr int BS = Fmt<FMT>::BS, BB = Fmt<FMT>::BB;
  if (kind == MOE_SRC_BLOCKS) {
    const uint8_t* p = (const uint8_t*)src + blk * BB;
    for (int i = 0; i < BB; ++i) out[i] = p[i];
  } else {
    float w[BS];
    const float* p = (const float*)src + blk * BS;
    for (int i = 0; i < BS; ++i) w[i] = p[i];
    if (FMT == MOE_FMT_MXFP4) enc_mxfp4(w, out);
    else if (FMT == MOE_FMT_INT4G32) enc_int4(w, out);
    else if (FMT == MOE_FMT_Q8_0) enc_q8_0(w, out);
    else enc_q2k(w, out);
  }
}

template <int FMT>
__global__ void encode_kernel(const float* src, int64_t nblk, uint8_t* dst) {
  constexpr int BB = Fmt<FMT>::BB;
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblk; b += (int64_t)gridDim.x * blockDim.x) {
    uint32_t words[(BB + 3) / 4];
    uint8_t* blk = reinterpret_cast<uint8_t*>(words);
    get_block<FMT>(src, MOE_SRC_F32, b, blk);
    volatile uint8_t* out = dst + b * BB;
    for (int i = 0; i < BB; ++i) out[i] = blk[i];
  }
}

// OR `bits` (at bit position `bit` of the 32-bit word at byte offset `off`) into the packed buffer.
__device__ __forceinline__ void or_bits(uint8_t* base, int64_t off, uint32_t bits) {
  atomicOr((unsigned int*)(base + off), bits);
}

// One thread per canonical block. dst is zeroed beforehand; each block ORs its bits into place.
//   kind GATE_UP: matrix index mi = 0 (gate) / 1 (up) selects src_a / src_b; rows are [n_e, I, H]
//   kind DOWN:    rows are [n_e, H, I]
template <int FMT>
__global__ void pack_kernel(moe_src_t skind, moe_matrix_t kind, int64_t n_e, int64_t H, int64_t I, const void* src_a,
                            const void* src_b, uint8_t* dst) {
  constexpr int BS = Fmt<FMT>::BS, BB = Fmt<FMT>::BB, CK = Fmt<FMT>::CK, CB = Fmt<FMT>::CB, CODE = Fmt<FMT>::CODE;
  const int64_t K = kind == MOE_MAT_GATE_UP ? H : I;
  const int64_t rows = kind == MOE_MAT_GATE_UP ? I : H;
  const int64_t nmat = kind == MOE_MAT_GATE_UP ? 2 : 1;
  const int64_t bpr = K / BS;  // blocks per row
  const int64_t total = n_e * nmat * rows * bpr;
  const int64_t tbytes = (K / CK) * CB;
  const int64_t estride = kind == MOE_MAT_GATE_UP ? (I / 8) * tbytes : (H / 16) * tbytes;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    int64_t bk = t % bpr;
    int64_t row = (t / bpr) % rows;
    int64_t mi = (t / bpr / rows) % nmat;
    int64_t e = t / bpr / rows / nmat;
    const void* src = (mi == 0) ? src_a : src_b;
    int64_t sblk = (e * rows + row) * bpr + bk;
    uint8_t blk[BB];
    get_block<FMT>(src, skind, sblk, blk);
    // tile and tile row
    int64_t tile, tr;
    if (kind == MOE_MAT_GATE_UP) { tile = row / 8; tr = row % 8 + 8 * mi; }
    else { tile = row / 16; tr = row % 16; }
    uint8_t* tb = dst + e * estride + tile * tbytes;
    const int k0 = (int)(bk * BS);
    if (FMT == MOE_FMT_MXFP4 || FMT == MOE_FMT_INT4G32) {
      for (int j = 0; j < 32; ++j) {
        int k = k0 + j;
        int code = (j % 2 == 0) ? (blk[(FMT == MOE_FMT_MXFP4 ? 1 : 0) + j / 2] >> 4)
                                : (blk[(FMT == MOE_FMT_MXFP4 ? 1 : 0) + j / 2] & 15);
        CodePos p = code_pos(FMT, (int)tr, k);
        int64_t cbase = (int64_t)p.chunk * CB;
        if (FMT == MOE_FMT_MXFP4) {
          int64_t byte = cbase + p.lane * 16 + p.step * 4 + p.reg;
          int shift = 8 * (int)(byte & 3) + (p.hi ? 4 : 0);
          or_bits(tb, byte & ~3LL, (uint32_t)code << shift);
        } else {
          int64_t word = cbase + p.lane * 16 + p.step * 4;
          int shift = (p.hi ? 16 : 0) + 4 * p.reg;
          or_bits(tb, word, (uint32_t)code << shift);
        }
      }
      // scale of this (row, 32-block)
      int chunk = k0 / CK, blk_in_chunk = (k0 % CK) / 32;
      int r = (int)(tr % 8), hi_row = tr >= 8 ? 1 : 0;
      int64_t sbase = (int64_t)chunk * CB + CODE;
      if (FMT == MOE_FMT_MXFP4) {
        int64_t byte = sbase + r * 4 + blk_in_chunk * 2 + hi_row;
        or_bits(tb, byte & ~3LL, (uint32_t)blk[0] << (8 * (int)(byte & 3)));
      } else {
        int64_t half = sbase + r * 8 + (blk_in_chunk * 2 + hi_row) * 2;
        uint32_t v = (uint32_t)blk[16] | ((uint32_t)blk[17] << 8);
        or_bits(tb, half & ~3LL, v << (8 * (int)(half & 3)));
      }
    } else if (FMT == MOE_FMT_Q8_0) {
      for (int j = 0; j < 32; ++j) {
        CodePos p = code_pos(FMT, (int)tr, k0 + j);
        int64_t byte = (int64_t)p.chunk * CB + p.lane * 32 + p.step * 8 + 2 * p.reg + p.hi;
        or_bits(tb, byte & ~3LL, (uint32_t)blk[2 + j] << (8 * (int)(byte & 3)));
      }
      int chunk = k0 / CK, blk_in_chunk = (k0 % CK) / 32;
      int r = (int)(tr % 8), hi_row = tr >= 8 ? 1 : 0;
      int64_t half = (int64_t)chunk * CB + CODE + r * 8 + (blk_in_chunk * 2 + hi_row) * 2;
      uint32_t v = (uint32_t)blk[0] | ((uint32_t)blk[1] << 8);
      or_bits(tb, half & ~3LL, v << (8 * (int)(half & 3)));
    } else {  // Q2_K: one super-block = one chunk row
      int chunk = k0 / CK;
      int64_t cbase = (int64_t)chunk * CB;
      for (int i = 0; i < 256; ++i) {
        int q = (blk[16 + i / 4] >> (2 * (i % 4))) & 3;
        CodePos p = code_pos(FMT, (int)tr, k0 + i);
        int w = p.step / 2, ts = p.step % 2;
        int64_t word = cbase + p.lane * 32 + w * 4;
        int shift = (p.hi ? 16 : 0) + 8 * ts + 2 * p.reg;
        or_bits(tb, word, (uint32_t)q << shift);
      }
      int r = (int)(tr % 8), hi_row = tr >= 8 ? 1 : 0;
      int64_t sc = cbase + CODE + r * 32 + hi_row * 16;
      for (int g = 0; g < 16; g += 4) {
        uint32_t v = (uint32_t)blk[g] | ((uint32_t)blk[g + 1] << 8) | ((uint32_t)blk[g + 2] << 16) | ((uint32_t)blk[g + 3] << 24);
        or_bits(tb, sc + g, v);
      }
      int64_t dd = cbase + CODE + 256 + r * 8 + hi_row * 4;
      uint32_t v = (uint32_t)blk[80] | ((uint32_t)blk[81] << 8) | ((uint32_t)blk[82] << 16) | ((uint32_t)blk[83] << 24);
      or_bits(tb, dd, v);
    }
  }
}

// Debug: decode expert `e` of a packed matrix back to fp32 [nmat, rows, K].
template <int FMT>
__global__ void unpack_kernel(moe_matrix_t kind, int64_t H, int64_t I, const uint8_t* packed, int64_t e, float* out) {
  constexpr int CK = Fmt<FMT>::CK, CB = Fmt<FMT>::CB, CODE = Fmt<FMT>::CODE;
  const int64_t K = kind == MOE_MAT_GATE_UP ? H : I;
  const int64_t rows = kind == MOE_MAT_GATE_UP ? I : H;
  const int64_t nmat = kind == MOE_MAT_GATE_UP ? 2 : 1;
  const int64_t tbytes = (K / CK) * CB;
  const int64_t estride = kind == MOE_MAT_GATE_UP ? (I / 8) * tbytes : (H / 16) * tbytes;
  const int64_t total = nmat * rows * K;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    int64_t k = t % K, row = (t / K) % rows, mi = t / K / rows;
    int64_t tile, tr;
    if (kind == MOE_MAT_GATE_UP) { tile = row / 8; tr = row % 8 + 8 * mi; }
    else { tile = row / 16; tr = row % 16; }
    const uint8_t* tb = packed + e * estride + tile * tbytes;
    CodePos p = code_pos(FMT, (int)tr, (int)k);
    const uint8_t* cb = tb + (int64_t)p.chunk * CB;
    int r = (int)(tr % 8), hi_row = tr >= 8 ? 1 : 0;
    float v;
    if (FMT == MOE_FMT_MXFP4) {
      uint8_t byte = cb[p.lane * 16 + p.step * 4 + p.reg];
      int code = p.hi ? (byte >> 4) : (byte & 15);
      const float tab[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
      int blk = (int)((k % CK) / 32);
      uint8_t ex = cb[CODE + r * 4 + blk * 2 + hi_row];
      float s = ex == 255 ? __int_as_float(0x7fc00000) : __uint_as_float((uint32_t)ex << 23);
      float m = tab[code & 7] * s;
      v = (code & 8) ? -m : m;
    } else if (FMT == MOE_FMT_INT4G32) {
      uint32_t word = *(const uint32_t*)(cb + p.lane * 16 + p.step * 4);
      int n = (word >> ((p.hi ? 16 : 0) + 4 * p.reg)) & 15;
      int q = n >= 8 ? n - 16 : n;
      int blk = (int)((k % CK) / 32);
      uint16_t sb = *(const uint16_t*)(cb + CODE + r * 8 + (blk * 2 + hi_row) * 2);
      v = (float)q * __uint_as_float((uint32_t)sb << 16);
    } else if (FMT == MOE_FMT_Q8_0) {
      const int q = (int)(int8_t)cb[p.lane * 32 + p.step * 8 + 2 * p.reg + p.hi];
      int blk = (int)((k % CK) / 32);
      uint16_t db = *(const uint16_t*)(cb + CODE + r * 8 + (blk * 2 + hi_row) * 2);
      v = (float)q * __half2float(__ushort_as_half(db));
    } else {
      uint32_t word = *(const uint32_t*)(cb + p.lane * 32 + (p.step / 2) * 4);
      int q = (word >> ((p.hi ? 16 : 0) + 8 * (p.step % 2) + 2 * p.reg)) & 3;
      int g = (int)((k % CK) / 16);
      uint8_t scm = cb[CODE + r * 32 + hi_row * 16 + g];
      const uint16_t* dd = (const uint16_t*)(cb + CODE + 256 + r * 8 + hi_row * 4);
      float d = __half2float(__ushort_as_half(dd[0])), dmin = __half2float(__ushort_as_half(dd[1]));
      float a = __fmul_rn(d, (float)(scm & 15));
      float bq = __fmul_rn(a, (float)q);
      float c = __fmul_rn(dmin, (float)(scm >> 4));
      v = __fsub_rn(bq, c);
    }
    out[t] = v;
  }
}

// Tensor-core layout (MXFP4 only): one thread per canonical block writes its 16 code bytes (nibbles swapped to
// even-k-low) and its exponent; every byte of the destination is written exactly once.
__global__ void pack_tc_kernel(moe_src_t skind, moe_matrix_t kind, int64_t n_e, int64_t H, int64_t I,
                               const void* src_a, const void* src_b, uint8_t* dst) {
  const TcGeom g = tc_geom(kind, H, I);
  const int64_t K = g.K, rows = kind == MOE_MAT_GATE_UP ? I : H, nmat = kind == MOE_MAT_GATE_UP ? 2 : 1;
  const int64_t bpr = K / 32;
  const int64_t total = n_e * nmat * rows * bpr;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bk = t % bpr, row = (t / bpr) % rows, mi = (t / bpr / rows) % nmat, e = t / bpr / rows / nmat;
    uint8_t blk[17];
    get_block<MOE_FMT_MXFP4>(mi == 0 ? src_a : src_b, skind, (e * rows + row) * bpr + bk, blk);
    uint8_t* base = dst + e * g.stride;
    const int64_t r = tc_row(kind, (int)mi, row);
    uint32_t words[4];
    for (int w = 0; w < 4; ++w) {
      uint32_t v = 0;
      for (int b = 0; b < 4; ++b) {
        const uint32_t c = blk[1 + w * 4 + b];
        v |= (((c >> 4) | ((c & 15) << 4)) & 255u) << (8 * b);  // canonical: even k high -> here: even k low
      }
      words[w] = v;
    }
    *reinterpret_cast<uint4*>(base + tc_code_off(g, r, bk * 32)) = make_uint4(words[0], words[1], words[2], words[3]);
    base[tc_scale_off(g, r, bk * 32)] = blk[0];
  }
}

__global__ void unpack_tc_kernel(moe_matrix_t kind, int64_t H, int64_t I, const uint8_t* packed, int64_t e, float* out) {
  const TcGeom g = tc_geom(kind, H, I);
  const int64_t K = g.K, rows = kind == MOE_MAT_GATE_UP ? I : H, nmat = kind == MOE_MAT_GATE_UP ? 2 : 1;
  const int64_t total = nmat * rows * K;
  const uint8_t* base = packed + e * g.stride;
  const float tab[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k = t % K, row = (t / K) % rows, mi = t / K / rows;
    const int64_t r = tc_row(kind, (int)mi, row);
    const uint8_t byte = base[tc_code_off(g, r, k)];
    const int code = (k % 2 == 0) ? (byte & 15) : (byte >> 4);
    const uint8_t ex = base[tc_scale_off(g, r, k)];
    const float s = ex == 255 ? __int_as_float(0x7fc00000) : __uint_as_float((uint32_t)ex << 23);
    const float m = tab[code & 7] * s;
    out[t] = (code & 8) ? -m : m;
  }
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_canonical_bytes(moe_format_t fmt, int64_t rows, int64_t k) {
  if (fmt < MOE_FMT_MXFP4 || fmt > MOE_FMT_Q8_0 || rows < 0 || k < 0 || k % fmt_bs(fmt)) return 0;
  return (size_t)(rows * (k / fmt_bs(fmt)) * fmt_bb(fmt));
}

extern "C" size_t moe_packed_bytes(moe_format_t fmt, moe_layout_t layout, moe_matrix_t kind, int64_t n_e, int64_t H,
                                   int64_t I) {
  if (fmt < MOE_FMT_MXFP4 || fmt > MOE_FMT_Q8_0 || n_e < 0) return 0;
  if (!moe_internal::shape_ok(H, I)) return 0;
  if (layout == MOE_LAYOUT_PREFILL) {
    if (fmt != MOE_FMT_MXFP4 || (kind != MOE_MAT_GATE_UP && kind != MOE_MAT_DOWN)) return 0;
    return (size_t)(n_e * tc_geom(kind, H, I).stride);
  }
  if (layout != MOE_LAYOUT_DECODE) return 0;
  int64_t s = kind == MOE_MAT_GATE_UP ? gate_up_stride(fmt, H, I) : down_stride(fmt, H, I);
  return (size_t)(n_e * s);
}

static int grid_for(int64_t n, int threads) {
  int64_t g = (n + threads - 1) / threads;
  if (g > 152 * 64) g = 152 * 64;
  if (g < 1) g = 1;
  return (int)g;
}

extern "C" moe_status_t moe_encode_blocks(moe_format_t fmt, const float* src, int64_t rows, int64_t k, void* dst,
                                          void* stream) {
  MOE_NVTX("moe_encode_blocks");
  if (moe_internal::fault("encode")) return MOE_ERR_FAULT_INJECTED;
  if (fmt < MOE_FMT_MXFP4 || fmt > MOE_FMT_Q8_0) return MOE_ERR_UNSUPPORTED_FORMAT;
  if (!src || !dst || rows < 0 || k < 0) return MOE_ERR_INVALID_ARG;
  if (k % fmt_bs(fmt)) return MOE_ERR_SHAPE;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  int64_t nblk = rows * (k / fmt_bs(fmt));
  if (nblk == 0) return MOE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  int thr = 128;
  switch (fmt) {
    case MOE_FMT_MXFP4: encode_kernel<MOE_FMT_MXFP4><<<grid_for(nblk, thr), thr, 0, s>>>(src, nblk, (uint8_t*)dst); break;
    case MOE_FMT_INT4G32: encode_kernel<MOE_FMT_INT4G32><<<grid_for(nblk, thr), thr, 0, s>>>(src, nblk, (uint8_t*)dst); break;
    case MOE_FMT_Q8_0: encode_kernel<MOE_FMT_Q8_0><<<grid_for(nblk, thr), thr, 0, s>>>(src, nblk, (uint8_t*)dst); break;
    default: encode_kernel<MOE_FMT_Q2K><<<grid_for(nblk, thr), thr, 0, s>>>(src, nblk, (uint8_t*)dst); break;
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t moe_pack_weights(moe_format_t fmt, moe_src_t src_kind, moe_layout_t layout, moe_matrix_t kind,
                                         int64_t n_e, int64_t H, int64_t I, const void* src_a, const void* src_b,
                                         void* dst, size_t dst_bytes, void* stream) {
  MOE_NVTX("moe_pack_weights");
  if (moe_internal::fault("pack")) return MOE_ERR_FAULT_INJECTED;
  if (fmt < MOE_FMT_MXFP4 || fmt > MOE_FMT_Q8_0) return MOE_ERR_UNSUPPORTED_FORMAT;
  if (src_kind != MOE_SRC_BLOCKS && src_kind != MOE_SRC_F32) return MOE_ERR_INVALID_ARG;
  if (kind != MOE_MAT_GATE_UP && kind != MOE_MAT_DOWN) return MOE_ERR_INVALID_ARG;
  if (!src_a || !dst || (kind == MOE_MAT_GATE_UP && !src_b)) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)dst & 15) != 0) return MOE_ERR_INVALID_ARG;
  if (n_e < 1 || !moe_internal::shape_ok(H, I)) return MOE_ERR_SHAPE;
  if (layout != MOE_LAYOUT_DECODE && layout != MOE_LAYOUT_PREFILL) return MOE_ERR_INVALID_ARG;
  if (layout == MOE_LAYOUT_PREFILL && fmt != MOE_FMT_MXFP4) return MOE_ERR_UNSUPPORTED_FORMAT;
  size_t need = moe_packed_bytes(fmt, layout, kind, n_e, H, I);
  if (dst_bytes < need) return MOE_ERR_INVALID_ARG;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (layout == MOE_LAYOUT_PREFILL) {
    const int64_t nblk = n_e * (kind == MOE_MAT_GATE_UP ? 2 * I * (H / 32) : H * (I / 32));
    pack_tc_kernel<<<grid_for(nblk, 128), 128, 0, s>>>(src_kind, kind, n_e, H, I, src_a, src_b, (uint8_t*)dst);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (cudaMemsetAsync(dst, 0, need, s) != cudaSuccess) return MOE_ERR_CUDA;
  int64_t K = kind == MOE_MAT_GATE_UP ? H : I, rows = kind == MOE_MAT_GATE_UP ? I : H;
  int64_t nmat = kind == MOE_MAT_GATE_UP ? 2 : 1;
  int64_t nblk = n_e * nmat * rows * (K / fmt_bs(fmt));
  int thr = 128;
  switch (fmt) {
    case MOE_FMT_MXFP4:
      pack_kernel<MOE_FMT_MXFP4><<<grid_for(nblk, thr), thr, 0, s>>>(src_kind, kind, n_e, H, I, src_a, src_b, (uint8_t*)dst);
      break;
    case MOE_FMT_INT4G32:
      pack_kernel<MOE_FMT_INT4G32><<<grid_for(nblk, thr), thr, 0, s>>>(src_kind, kind, n_e, H, I, src_a, src_b, (uint8_t*)dst);
      break;
    case MOE_FMT_Q8_0:
      pack_kernel<MOE_FMT_Q8_0><<<grid_for(nblk, thr), thr, 0, s>>>(src_kind, kind, n_e, H, I, src_a, src_b, (uint8_t*)dst);
      break;
    default:
      pack_kernel<MOE_FMT_Q2K><<<grid_for(nblk, thr), thr, 0, s>>>(src_kind, kind, n_e, H, I, src_a, src_b, (uint8_t*)dst);
      break;
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t moe_debug_unpack(moe_format_t fmt, moe_layout_t layout, moe_matrix_t kind, const void* packed,
                                         int64_t H, int64_t I, int64_t expert, float* out, void* stream) {
  if (fmt < MOE_FMT_MXFP4 || fmt > MOE_FMT_Q8_0) return MOE_ERR_UNSUPPORTED_FORMAT;
  if (!packed || !out || expert < 0) return MOE_ERR_INVALID_ARG;
  if (!moe_internal::shape_ok(H, I)) return MOE_ERR_SHAPE;
  if (layout != MOE_LAYOUT_DECODE && layout != MOE_LAYOUT_PREFILL) return MOE_ERR_INVALID_ARG;
  if (layout == MOE_LAYOUT_PREFILL && fmt != MOE_FMT_MXFP4) return MOE_ERR_UNSUPPORTED_FORMAT;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  int64_t total = (kind == MOE_MAT_GATE_UP ? 2 * I * H : H * I);
  int thr = 256;
  if (layout == MOE_LAYOUT_PREFILL) {
    unpack_tc_kernel<<<grid_for(total, thr), thr, 0, s>>>(kind, H, I, (const uint8_t*)packed, expert, out);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  switch (fmt) {
    case MOE_FMT_MXFP4: unpack_kernel<MOE_FMT_MXFP4><<<grid_for(total, thr), thr, 0, s>>>(kind, H, I, (const uint8_t*)packed, expert, out); break;
    case MOE_FMT_INT4G32: unpack_kernel<MOE_FMT_INT4G32><<<grid_for(total, thr), thr, 0, s>>>(kind, H, I, (const uint8_t*)packed, expert, out); break;
    case MOE_FMT_Q8_0: unpack_kernel<MOE_FMT_Q8_0><<<grid_for(total, thr), thr, 0, s>>>(kind, H, I, (const uint8_t*)packed, expert, out); break;
    default: unpack_kernel<MOE_FMT_Q2K><<<grid_for(total, thr), thr, 0, s>>>(kind, H, I, (const uint8_t*)packed, expert, out); break;
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
