/*
 * oracle.c -- plain, slow CPU oracle for the routed-MoE low-bit decode path.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg
 * may load this library. It shares no code, header, table or constant with the CUDA library under
 * bit_moe_decode_gb300/, and the CUDA library never calls it.
 *
 * Every value here follows the written definition of the method as given by these pages:
 *   [P2] "Mixed-precision compression of DeepSeek-V4-Flash" (lumirain.cn): top-6 routing, F16 router,
 *        "What compression does not solve" (every token reads all active weights), "Width drift" (verify of
 *        width 1+K must equal width-1 decode).
 *   [P3] "quant surgery" (blog.meowhead.cn), section 4: hash routing of the first three layers (tid2eid).
 *   [P4] "DeepSeek-V4-Flash-0731-W4A16" model card (alphaneural.io), "FP4 -> INT4 conversion": E2M1 table,
 *        INT4 group-32 symmetric quantisation with the r-grid MSE search, amax clamp 1e-8.
 *   [P5] "quantization" glossary (ds4-learning.pages.dev): block_mxfp4 (1 E8M0 byte + 16 code bytes),
 *        E2M1 table, E8M0 = 2^(e-127) with e=0 as zero, Q2_K super-block (84 bytes: scales[16], qs[64],
 *        fp16 d, fp16 dmin), the "Metal MXFP4 -> half LUT" section (4096 exact products rounded once).
 *
 * Readings where the pages are silent or garbled:
 *   - MXFP4 nibble order: element 2j is the HIGH nibble of code byte j, element 2j+1 the LOW nibble
 *     (the only printed unpack, P4 step 1 "dequant_fp4", takes byte>>4 first).
 *   - E8M0: e=0 -> 0 (P5 comment "e=0 treated as zero"), e=255 -> NaN (P5 LUT section: the 0xff row
 *     stays on the arithmetic path, inf x 0 -> NaN).
 *   - INT4 block (18 bytes): 16 code bytes (same nibble order, 4-bit two's complement) then a bf16 scale,
 *     little endian.
 *   - Q2_K: the page's formula "(qs - dmin) x scales x d" is garbled; the value is w = d*sc*q - dmin*m with
 *     scales[g] = sc (low nibble) | m (high nibble), q of weight i = (qs[i/4] >> 2*(i%4)) & 3.
 *   - Q2_K encoder: not on the pages; a plain min/max spec (q2k_encode below).
 *   - MXFP4 / MXFP8 scale choice: smallest k with amax <= qmax * 2^k, e = clamp(k+127, 1, 254).
 *
 * Precision: decoded weights are exact (fp64), products and sums are fp64, sums are sequential in index
 * order. Build with -O2 -ffp-contract=off so no fused multiply-add changes a rounding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------------------
 * Scalar conversions, written from the IEEE 754 definitions (not from any library).
 * ------------------------------------------------------------------------------------------------ */

/* binary16 bits -> double (exact). */
double orc_f16_to_f64(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);                      /* subnormal: m * 2^-24 */
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp(1.0 + m / 1024.0, e - 15);
  return s ? -v : v;
}

/* bfloat16 bits -> double (exact). */
double orc_bf16_to_f64(uint16_t b) {
  int s = (b >> 15) & 1, e = (b >> 7) & 255, m = b & 127;
  double v;
  if (e == 0) v = ldexp((double)m, -133);                     /* subnormal: m * 2^-126 / 128 */
  else if (e == 255) v = m ? NAN : INFINITY;
  else v = ldexp(1.0 + m / 128.0, e - 127);
  return s ? -v : v;
}

/* Round a double to the nearest value with `p` significant bits, ties to even, with a minimum exponent
 * `emin` (values below 2^emin are represented with spacing 2^(emin-p+1), i.e. gradual underflow) and
 * overflow to +-inf above `maxfinite`. Used for fp32 / fp16 / bf16 rounding of exact values. */
static double round_to_format(double x, int p, int emin, double maxfinite) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  double a = fabs(x);
  int e;
  frexp(a, &e);               /* a = f * 2^e, f in [0.5, 1): leading bit weight 2^(e-1) */
  int lead = e - 1;
  if (lead < emin) lead = emin;
  double ulp = ldexp(1.0, lead - (p - 1));
  double q = a / ulp;         /* exact: division by a power of two */
  double fl = floor(q);
  double rem = q - fl;
  double r;
  if (rem > 0.5) r = fl + 1.0;
  else if (rem < 0.5) r = fl;
  else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
  double v = r * ulp;
  if (v > maxfinite) v = INFINITY;
  return x < 0 ? -v : v;
}

double orc_round_f32(double x) { return round_to_format(x, 24, -126, 3.4028234663852886e38); }
double orc_round_f16(double x) { return round_to_format(x, 11, -14, 65504.0); }
double orc_round_bf16(double x) { return round_to_format(x, 8, -126, 3.3895313892515355e38); }

/* exact double (already representable in binary16) -> bits */
uint16_t orc_f64_to_f16_bits(double v) {
  uint16_t s = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (isnan(v)) return 0x7E00;
  if (isinf(v)) return s | 0x7C00;
  if (a == 0.0) return s;
  int e;
  frexp(a, &e);
  int lead = e - 1;
  if (lead < -14) return s | (uint16_t)(a / ldexp(1.0, -24));          /* subnormal */
  uint16_t m = (uint16_t)((a / ldexp(1.0, lead) - 1.0) * 1024.0);
  return s | (uint16_t)((lead + 15) << 10) | m;
}

/* float (value) -> fp16 bits, RNE */
uint16_t orc_f32_to_f16_rne(float f) { return orc_f64_to_f16_bits(orc_round_f16((double)f)); }

/* ------------------------------------------------------------------------------------------------
 * MXFP4 [P5 "MXFP4", P4 step 1]
 * ------------------------------------------------------------------------------------------------ */

/* E2M1 code -> value: the printed 16-entry table (bit 3 is the sign; code 8 is -0). */
static const double E2M1[16] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                                -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0};

double orc_e2m1_value(int code) { return E2M1[code & 15]; }

/* E8M0 -> scale: 2^(e-127); e=0 -> 0; e=255 -> NaN. */
double orc_e8m0_scale(int e) {
  if (e == 0) return 0.0;
  if (e == 255) return NAN;
  return ldexp(1.0, e - 127);
}

/* Element j (0..31) of a 17-byte block: byte 0 = E8M0 exponent, bytes 1..16 = codes,
 * element 2i in the high nibble of byte 1+i, element 2i+1 in the low nibble. */
static int mxfp4_code(const uint8_t* blk, int j) {
  uint8_t b = blk[1 + j / 2];
  return (j % 2 == 0) ? (b >> 4) : (b & 15);
}

/* Decode to fp32 values (the format's decoded weight is T[code] * 2^(e-127), rounded to fp32 by IEEE
 * rules: exact except overflow to +-inf for e >= 253 with large codes). */
void orc_decode_mxfp4(const uint8_t* blocks, int64_t nblk, float* out) {
  for (int64_t b = 0; b < nblk; ++b) {
    const uint8_t* blk = blocks + b * 17;
    double s = orc_e8m0_scale(blk[0]);
    for (int j = 0; j < 32; ++j) out[b * 32 + j] = (float)(E2M1[mxfp4_code(blk, j)] * s);
  }
}

/* exact decoded value in double (no fp32 overflow) for the FFN */
static double mxfp4_weight(const uint8_t* blk, int j) { return E2M1[mxfp4_code(blk, j)] * orc_e8m0_scale(blk[0]); }

/* Nearest E2M1 code for a magnitude-scaled value v, ties to the even code, saturating at 6.
 * Written as a plain search over the 8 magnitudes. The sign bit is signbit(v). */
static int e2m1_nearest(double v) {
  double a = fabs(v);
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = fabs(a - E2M1[c]);
    if (d < bestd || (d == bestd && (c % 2) == 0)) { bestd = d; best = c; }
  }
  if (a > 6.0) best = 7;
  return best | (signbit(v) ? 8 : 0);
}

/* smallest integer k with amax <= qmax * 2^k (exact comparisons; amax > 0 finite) */
static int smallest_k(double amax, double qmax) {
  int e;
  frexp(amax / qmax, &e);     /* amax/qmax = f * 2^e, f in [0.5,1): 2^(e-1) <= ratio < 2^e */
  int k = e - 2;
  while (amax > qmax * ldexp(1.0, k)) ++k;   /* at most a few steps */
  while (amax <= qmax * ldexp(1.0, k - 1)) --k;
  return k;
}

static int mx_exponent(double amax, double qmax) {
  if (!(amax > 0.0)) return 1;                /* all zeros: k = -inf -> clamps to 1 */
  int k = smallest_k(amax, qmax);
  int e = k + 127;
  if (e < 1) e = 1;
  if (e > 254) e = 254;
  return e;
}

/* MXFP4 encoder (32-weight blocks, fp32 input). */
void orc_encode_mxfp4(const float* w, int64_t nblk, uint8_t* out) {
  /* blocks are independent; each block's arithmetic is sequential */
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblk; ++b) {
    const float* x = w + b * 32;
    uint8_t* blk = out + b * 17;
    double amax = 0.0;
    for (int j = 0; j < 32; ++j) if (fabs((double)x[j]) > amax) amax = fabs((double)x[j]);
    int e = mx_exponent(amax, 6.0);
    blk[0] = (uint8_t)e;
    memset(blk + 1, 0, 16);
    for (int j = 0; j < 32; ++j) {
      double v = (double)x[j] * ldexp(1.0, 127 - e);   /* exact */
      int c = e2m1_nearest(v);
      if (j % 2 == 0) blk[1 + j / 2] |= (uint8_t)(c << 4);
      else blk[1 + j / 2] |= (uint8_t)c;
    }
  }
}

/* The "MXFP4 -> half" table of P5: fp16 bits of RNE(2^(e-127) * E2M1[c]) for e in 0..255, c in 0..15.
 * Row 0 is zero (+-0 by the code's sign); row 255 is NaN (left on the arithmetic path by the page). */
void orc_mxfp4_half_lut(uint16_t* lut) {
  for (int e = 0; e < 256; ++e)
    for (int c = 0; c < 16; ++c) {
      double v = E2M1[c] * orc_e8m0_scale(e);
      lut[e * 16 + c] = orc_f64_to_f16_bits(orc_round_f16(v));
    }
}

/* ------------------------------------------------------------------------------------------------
 * INT4 group-32 [P4 "FP4 -> INT4 conversion", step 2]
 * ------------------------------------------------------------------------------------------------ */

static int int4_code(const uint8_t* blk, int j) {
  uint8_t b = blk[j / 2];
  int n = (j % 2 == 0) ? (b >> 4) : (b & 15);
  return n >= 8 ? n - 16 : n;   /* two's complement */
}

static double int4_scale(const uint8_t* blk) { return orc_bf16_to_f64((uint16_t)(blk[16] | (blk[17] << 8))); }

void orc_decode_int4(const uint8_t* blocks, int64_t nblk, float* out) {
  for (int64_t b = 0; b < nblk; ++b) {
    const uint8_t* blk = blocks + b * 18;
    double s = int4_scale(blk);
    for (int j = 0; j < 32; ++j) out[b * 32 + j] = (float)(int4_code(blk, j) * s);
  }
}

static double int4_weight(const uint8_t* blk, int j) { return int4_code(blk, j) * int4_scale(blk); }

/* fp32 round-half-even to integer */
static float rne_int(float v) {
  float f = floorf(v);
  float r = v - f;
  if (r > 0.5f) return f + 1.0f;
  if (r < 0.5f) return f;
  return (fmodf(f, 2.0f) == 0.0f) ? f : f + 1.0f;
}

/* INT4 encoder: for r in the six-entry grid, s = amax*r/7 (fp32), q = clamp(round_half_even(w/s), -8, 7),
 * mse = sum over the group of (w - q*s)^2 in fp32, sequential; keep the first r with the smallest mse.
 * amax is clamped to at least 1e-8. The stored scale is the bf16 rounding of the winning s. */
void orc_encode_int4(const float* w, int64_t nblk, uint8_t* out) {
  const float grid[6] = {6.0f / 7.0f, 0.9f, 0.95f, 1.0f, 1.05f, 1.1f};
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblk; ++b) {
    const float* x = w + b * 32;
    uint8_t* blk = out + b * 18;
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) { float a = fabsf(x[j]); if (a > amax) amax = a; }
    if (amax < 1e-8f) amax = 1e-8f;
    float best_mse = INFINITY, best_s = 0.0f;
    int best_q[32];
    for (int gi = 0; gi < 6; ++gi) {
      float t = amax * grid[gi];
      float s = t / 7.0f;
      int q[32];
      float mse = 0.0f;
      for (int j = 0; j < 32; ++j) {
        float qq = rne_int(x[j] / s);
        if (qq < -8.0f) qq = -8.0f;
        if (qq > 7.0f) qq = 7.0f;
        q[j] = (int)qq;
        float rec = qq * s;
        float d = x[j] - rec;
        float sq = d * d;
        mse = mse + sq;
      }
      /* the first candidate is the initial best; a later one replaces it only with a strictly smaller error
         (so a group whose errors all overflow to inf keeps r = 6/7) */
      if (gi == 0 || mse < best_mse) { best_mse = mse; best_s = s; memcpy(best_q, q, sizeof q); }
    }
    memset(blk, 0, 16);
    for (int j = 0; j < 32; ++j) {
      uint8_t n = (uint8_t)(best_q[j] & 15);
      if (j % 2 == 0) blk[j / 2] |= (uint8_t)(n << 4);
      else blk[j / 2] |= n;
    }
    double sb = orc_round_bf16((double)best_s);
    /* bits of the bf16 value: top 16 bits of its fp32 pattern (sb is exactly representable) */
    float sf = (float)sb;
    uint32_t u;
    memcpy(&u, &sf, 4);
    uint16_t bits = (uint16_t)(u >> 16);
    blk[16] = (uint8_t)(bits & 255);
    blk[17] = (uint8_t)(bits >> 8);
  }
}

/* ------------------------------------------------------------------------------------------------
 * Q2_K [P5 "core principle": 84 bytes = scales[16] + qs[64] + fp16 d + fp16 dmin, 256 weights]
 * ------------------------------------------------------------------------------------------------ */

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Decoded weight i of a super-block, in fp32: (d*sc)*q - (dmin*m), one rounding (the two products are
 * exact in fp32: 11+4(+2) significant bits). */
static float q2k_weight_f32(const uint8_t* blk, int i) {
  int g = i / 16;
  int sc = blk[g] & 15, m = blk[g] >> 4;
  int q = (blk[16 + i / 4] >> (2 * (i % 4))) & 3;
  float d = (float)orc_f16_to_f64(rd16(blk + 80));
  float dmin = (float)orc_f16_to_f64(rd16(blk + 82));
  float a = d * (float)sc;
  float bq = a * (float)q;
  float c = dmin * (float)m;
  return bq - c;
}

void orc_decode_q2k(const uint8_t* blocks, int64_t nblk, float* out) {
  for (int64_t b = 0; b < nblk; ++b)
    for (int i = 0; i < 256; ++i) out[b * 256 + i] = q2k_weight_f32(blocks + b * 84, i);
}

/* Q2_K encoder (our spec; the pages give none):
 *   per 16-weight group g: lo = min(0, min w), hi = max w, s_g = (hi - lo)/3, o_g = -lo
 *   d = fp16(max_g s_g / 15), dmin = fp16(max_g o_g / 15)
 *   sc_g = round_half_even(s_g / d) clamped to [0,15] (0 if d == 0); m_g likewise from o_g / dmin
 *   q_i = round_half_even((w_i + dmin*m_g) / (d*sc_g)) clamped to [0,3] (0 if d*sc_g == 0)
 * All arithmetic fp32 with RNE. */
void orc_encode_q2k(const float* w, int64_t nblk, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblk; ++b) {
    const float* x = w + b * 256;
    uint8_t* blk = out + b * 84;
    float s[16], o[16];
    float smax = 0.0f, omax = 0.0f;
    for (int g = 0; g < 16; ++g) {
      float lo = 0.0f, hi = -INFINITY;
      for (int j = 0; j < 16; ++j) {
        float v = x[g * 16 + j];
        if (v < lo) lo = v;
        if (v > hi) hi = v;
      }
      s[g] = (hi - lo) / 3.0f;
      o[g] = -lo;
      if (s[g] > smax) smax = s[g];
      if (o[g] > omax) omax = o[g];
    }
    uint16_t dbits = orc_f32_to_f16_rne(smax / 15.0f);
    uint16_t mbits = orc_f32_to_f16_rne(omax / 15.0f);
    float d = (float)orc_f16_to_f64(dbits), dmin = (float)orc_f16_to_f64(mbits);
    memset(blk, 0, 84);
    int sc[16], m[16];
    for (int g = 0; g < 16; ++g) {
      float a = d > 0.0f ? rne_int(s[g] / d) : 0.0f;
      float c = dmin > 0.0f ? rne_int(o[g] / dmin) : 0.0f;
      if (a < 0.0f) a = 0.0f;
      if (a > 15.0f) a = 15.0f;
      if (c < 0.0f) c = 0.0f;
      if (c > 15.0f) c = 15.0f;
      sc[g] = (int)a;
      m[g] = (int)c;
      blk[g] = (uint8_t)(sc[g] | (m[g] << 4));
    }
    for (int i = 0; i < 256; ++i) {
      int g = i / 16;
      float step = d * (float)sc[g];
      float off = dmin * (float)m[g];
      int q = 0;
      if (step > 0.0f) {
        float t = x[i] + off;
        float qq = rne_int(t / step);
        if (qq < 0.0f) qq = 0.0f;
        if (qq > 3.0f) qq = 3.0f;
        q = (int)qq;
      }
      blk[16 + i / 4] |= (uint8_t)(q << (2 * (i % 4)));
    }
    blk[80] = (uint8_t)(dbits & 255);
    blk[81] = (uint8_t)(dbits >> 8);
    blk[82] = (uint8_t)(mbits & 255);
    blk[83] = (uint8_t)(mbits >> 8);
  }
}

/* ------------------------------------------------------------------------------------------------
 * MXFP8 (E4M3 + E8M0 per 32) activation quantiser for the prefill path (E4M3 "fn": bias 7, no inf,
 * max 448, S.1111.111 = NaN).
 * ------------------------------------------------------------------------------------------------ */

double orc_e4m3_value(int code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = m * ldexp(1.0, -9);
  else v = ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

/* nearest finite E4M3 magnitude code (0..126) by plain search, ties to even code; saturates at 448 */
static int e4m3_nearest(double v) {
  double a = fabs(v);
  int best = 0;
  double bestd = INFINITY;
  for (int c = 0; c <= 126; ++c) {
    double d = fabs(a - orc_e4m3_value(c));
    if (d < bestd || (d == bestd && (c % 2) == 0)) { bestd = d; best = c; }
  }
  return best | (signbit(v) ? 0x80 : 0);
}

/* Quantise nblk blocks of 32 values (given as doubles that the caller has already put in the precision
 * the decision is taken in). codes[nblk*32], scales[nblk]. */
void orc_quant_mxfp8(const double* v, int64_t nblk, uint8_t* codes, uint8_t* scales) {
  for (int64_t b = 0; b < nblk; ++b) {
    double amax = 0.0;
    for (int j = 0; j < 32; ++j) if (fabs(v[b * 32 + j]) > amax) amax = fabs(v[b * 32 + j]);
    int e = mx_exponent(amax, 448.0);
    scales[b] = (uint8_t)e;
    for (int j = 0; j < 32; ++j) codes[b * 32 + j] = (uint8_t)e4m3_nearest(v[b * 32 + j] * ldexp(1.0, 127 - e));
  }
}

/* ------------------------------------------------------------------------------------------------
 * Router [P2 "The recipe": top-6, router in F16]; rule: logits = W_r x, top-k by logit with ties to
 * the lower expert index, weights = softmax over all experts restricted to the k chosen, renormalised
 * to sum 1 (= softmax over the k chosen logits).
 * ------------------------------------------------------------------------------------------------ */

/* logits[t*E+e] (fp64, sequential sum) and abs_l[t*E+e] = sum |W x| (for near-tie detection) */
void orc_router_logits(const uint16_t* wr, const uint16_t* x, int T, int H, int E, double* logits, double* abs_l) {
  for (int t = 0; t < T; ++t)
    for (int e = 0; e < E; ++e) {
      double s = 0.0, a = 0.0;
      for (int h = 0; h < H; ++h) {
        double p = orc_f16_to_f64(wr[(int64_t)e * H + h]) * orc_bf16_to_f64(x[(int64_t)t * H + h]);
        s += p;
        a += fabs(p);
      }
      logits[(int64_t)t * E + e] = s;
      if (abs_l) abs_l[(int64_t)t * E + e] = a;
    }
}

/* brute force: repeatedly take the largest remaining logit, lowest index on ties */
void orc_topk_from_logits(const double* logits, int T, int E, int k, int32_t* idx, float* w) {
  char* used = (char*)calloc((size_t)E, 1);
  double* sel = (double*)malloc(sizeof(double) * (size_t)k);
  for (int t = 0; t < T; ++t) {
    memset(used, 0, (size_t)E);
    const double* l = logits + (int64_t)t * E;
    for (int r = 0; r < k; ++r) {
      int best = -1;
      for (int e = 0; e < E; ++e) {
        if (used[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e;   /* strict: keeps the lower index on equal logits */
      }
      used[best] = 1;
      idx[(int64_t)t * k + r] = best;
      sel[r] = l[best];
    }
    double mx = sel[0], den = 0.0;
    for (int r = 0; r < k; ++r) den += exp(sel[r] - mx);
    for (int r = 0; r < k; ++r) w[(int64_t)t * k + r] = (float)(exp(sel[r] - mx) / den);
  }
  free(used);
  free(sel);
}

void orc_route_topk(const uint16_t* wr, const uint16_t* x, int T, int H, int E, int k, int32_t* idx, float* w,
                    double* logits_out, double* abs_out) {
  double* l = logits_out ? logits_out : (double*)malloc(sizeof(double) * (size_t)T * E);
  orc_router_logits(wr, x, T, H, E, l, abs_out);
  orc_topk_from_logits(l, T, E, k, idx, w);
  if (!logits_out) free(l);
}

/* hash routing [P3 section 4]: idx = tid2eid[token], equal weights 1/k */
void orc_route_hash(const int32_t* tok, const int32_t* tid2eid, int T, int k, int32_t* idx, float* w) {
  for (int t = 0; t < T; ++t)
    for (int r = 0; r < k; ++r) {
      idx[(int64_t)t * k + r] = tid2eid[(int64_t)tok[t] * k + r];
      w[(int64_t)t * k + r] = (float)(1.0 / k);
    }
}

/* RMS normalisation between the layers of a stack (the model normalises the hidden state before each MoE layer:
 * "Mixed-precision compression of DeepSeek-V4-Flash", "The recipe"); no learned gain. Exact values in fp64:
 * out[t, i] = y[t, i] / sqrt(mean_i y[t, i]^2 + eps). The library rounds them to bf16. */
void orc_rms_norm(const float* y, int T, int H, double eps, double* out) {
  for (int t = 0; t < T; ++t) {
    const float* yr = y + (int64_t)t * H;
    double ss = 0.0;
    for (int i = 0; i < H; ++i) ss += (double)yr[i] * (double)yr[i];
    const double r = 1.0 / sqrt(ss / H + eps);
    for (int i = 0; i < H; ++i) out[(int64_t)t * H + i] = (double)yr[i] * r;
  }
}

/* ------------------------------------------------------------------------------------------------
 * Q8_0: the shared expert's 8-bit format ("Mixed-precision compression of DeepSeek-V4-Flash", "The recipe"
 * names Q8 for it and gives no layout; the library's own definition): 34 bytes per 32 weights, bytes 0..1 a
 * binary16 scale d (little-endian), bytes 2..33 signed 8-bit codes q_j; w_j = d * q_j.
 * ------------------------------------------------------------------------------------------------ */

static double q8_scale(const uint8_t* blk) { return orc_f16_to_f64(rd16(blk)); }
static int q8_code(const uint8_t* blk, int j) { return (int)(int8_t)blk[2 + j]; }
static double q8_weight(const uint8_t* blk, int j) { return q8_code(blk, j) * q8_scale(blk); }

void orc_decode_q8_0(const uint8_t* blocks, int64_t nblk, float* out) {
  for (int64_t b = 0; b < nblk; ++b)
    for (int j = 0; j < 32; ++j) out[b * 32 + j] = (float)q8_weight(blocks + b * 34, j);
}

/* Q8_0 encoder: amax = max |w| (fp32); d = fp16 RNE of amax / 127 (fp32 division); q_j = round_half_even(w_j / d)
 * (fp32 division by the fp16 value of d) clamped to [-127, 127]; q = 0 when d = 0 and for NaN quotients. */
void orc_encode_q8_0(const float* w, int64_t nblk, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblk; ++b) {
    const float* x = w + b * 32;
    uint8_t* blk = out + b * 34;
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) { float a = fabsf(x[j]); if (a > amax) amax = a; }
    const uint16_t dbits = orc_f32_to_f16_rne(amax / 127.0f);
    const float d = (float)orc_f16_to_f64(dbits);
    blk[0] = (uint8_t)(dbits & 255);
    blk[1] = (uint8_t)(dbits >> 8);
    for (int j = 0; j < 32; ++j) {
      float qq = 0.0f;
      if (d != 0.0f) {
        qq = rne_int(x[j] / d);
        if (qq != qq) qq = 0.0f;
        if (qq < -127.0f) qq = -127.0f;
        if (qq > 127.0f) qq = 127.0f;
      }
      blk[2 + j] = (uint8_t)(int8_t)(int)qq;
    }
  }
}

/* ------------------------------------------------------------------------------------------------
 * Expert FFN, SwiGLU form [P5 "Q4_K routed experts" bullets: a fused gate+up mat-vec, then the down
 * projection accumulated into the output]:
 *   g = Gate x, u = Up x, h = SiLU(g) * u = g / (1 + exp(-g)) * u, d = Down h, y = sum_r w_r d_r.
 * fmt: 1 = MXFP4 (17-byte blocks of 32), 2 = INT4 g32 (18-byte blocks), 3 = Q2_K (84-byte blocks of 256),
 * 4 = Q8_0 (34-byte blocks of 32).
 * A matrix [rows, K] is rows * K/bs consecutive canonical blocks.
 * ------------------------------------------------------------------------------------------------ */

static int fmt_bs(int fmt) { return fmt == 3 ? 256 : 32; }
static int fmt_bytes(int fmt) { return fmt == 1 ? 17 : fmt == 2 ? 18 : fmt == 4 ? 34 : 84; }

/* decoded weight (row, col) of a [rows, K] matrix, exact, in double */
static double weight_at(int fmt, const uint8_t* mat, int K, int64_t row, int col) {
  int bs = fmt_bs(fmt), nb = fmt_bytes(fmt);
  const uint8_t* blk = mat + (row * (K / bs) + col / bs) * nb;
  int j = col % bs;
  if (fmt == 1) return mxfp4_weight(blk, j);
  if (fmt == 2) return int4_weight(blk, j);
  if (fmt == 4) return q8_weight(blk, j);
  return (double)q2k_weight_f32(blk, j);
}

/* Decode a whole [rows, K] matrix to doubles (helper for speed; same values as weight_at). */
static void decode_matrix(int fmt, const uint8_t* mat, int64_t rows, int K, double* out) {
  int bs = fmt_bs(fmt);
  int64_t nblk = rows * (K / bs);
  float* tmp = (float*)malloc(sizeof(float) * (size_t)bs);
  int nb = fmt_bytes(fmt);
  for (int64_t b = 0; b < nblk; ++b) {
    const uint8_t* blk = mat + b * nb;
    if (fmt == 1) {
      double s = orc_e8m0_scale(blk[0]);
      for (int j = 0; j < 32; ++j) out[b * 32 + j] = E2M1[mxfp4_code(blk, j)] * s;
    } else if (fmt == 2) {
      double s = int4_scale(blk);
      for (int j = 0; j < 32; ++j) out[b * 32 + j] = int4_code(blk, j) * s;
    } else if (fmt == 4) {
      for (int j = 0; j < 32; ++j) out[b * 32 + j] = q8_weight(blk, j);
    }
    else { orc_decode_q2k(blk, 1, tmp); for (int j = 0; j < 256; ++j) out[b * 256 + j] = (double)tmp[j]; }
  }
  free(tmp);
}

double orc_weight_at(int fmt, const uint8_t* mat, int K, int64_t row, int col) { return weight_at(fmt, mat, K, row, col); }

static double silu(double g) { return g / (1.0 + exp(-g)); }

/* One expert applied to one activation vector (x given as doubles).
 * g,u,h: [I] ; d: [H] ; dabs[j] = sum_i |Down[j,i] * h[i]|. Any output pointer may be NULL. */
void orc_expert_ffn(int fmt, int H, int I, const uint8_t* gate, const uint8_t* up, const uint8_t* down,
                    const double* x, double* g_out, double* u_out, double* h_out, double* d_out, double* dabs_out) {
  double* G = (double*)malloc(sizeof(double) * (size_t)I * H);
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  decode_matrix(fmt, gate, I, H, G);
  double* gv = (double*)malloc(sizeof(double) * (size_t)I);
  for (int i = 0; i < I; ++i) {
    double s = 0.0;
    for (int c = 0; c < H; ++c) s += G[(int64_t)i * H + c] * x[c];
    gv[i] = s;
  }
  decode_matrix(fmt, up, I, H, G);
  for (int i = 0; i < I; ++i) {
    double s = 0.0;
    for (int c = 0; c < H; ++c) s += G[(int64_t)i * H + c] * x[c];
    if (g_out) g_out[i] = gv[i];
    if (u_out) u_out[i] = s;
    h[i] = silu(gv[i]) * s;
    if (h_out) h_out[i] = h[i];
  }
  free(G);
  free(gv);
  double* D = (double*)malloc(sizeof(double) * (size_t)H * I);
  decode_matrix(fmt, down, H, I, D);
  for (int j = 0; j < H; ++j) {
    double s = 0.0, a = 0.0;
    for (int i = 0; i < I; ++i) {
      double p = D[(int64_t)j * I + i] * h[i];
      s += p;
      a += fabs(p);
    }
    if (d_out) d_out[j] = s;
    if (dabs_out) dabs_out[j] = a;
  }
  free(D);
  free(h);
}

/* MoE output for one token: experts[r] -> (gate, up, down) canonical block pointers of the expert at rank r.
 * y[j] = sum_r w[r] * d_r[j] (rank order); absterm[j] = sum_r |w[r]| * sum_i |Down_r[j,i] h_r[i]|. */
void orc_moe_token(int fmt, int H, int I, int k, const uint8_t* const* gate, const uint8_t* const* up,
                   const uint8_t* const* down, const float* w, const uint16_t* x_bf16, double* y, double* absterm) {
  double* x = (double*)malloc(sizeof(double) * (size_t)H);
  double* d = (double*)malloc(sizeof(double) * (size_t)H);
  double* da = (double*)malloc(sizeof(double) * (size_t)H);
  for (int c = 0; c < H; ++c) x[c] = orc_bf16_to_f64(x_bf16[c]);
  for (int j = 0; j < H; ++j) { y[j] = 0.0; if (absterm) absterm[j] = 0.0; }
  for (int r = 0; r < k; ++r) {
    orc_expert_ffn(fmt, H, I, gate[r], up[r], down[r], x, NULL, NULL, NULL, d, da);
    for (int j = 0; j < H; ++j) {
      y[j] += (double)w[r] * d[j];
      if (absterm) absterm[j] += fabs((double)w[r]) * da[j];
    }
  }
  free(x);
  free(d);
  free(da);
}

/* Batch over T tokens of one layer whose experts are stored contiguously:
 *   gate_all/up_all: E x [I, H] matrices, down_all: E x [H, I] matrices (canonical blocks).
 * Tokens run in parallel over `nthreads` OpenMP threads; each token's arithmetic is sequential. */
void orc_moe_batch(int fmt, int H, int I, int E, int k, const uint8_t* gate_all, const uint8_t* up_all,
                   const uint8_t* down_all, int T, const int32_t* idx, const float* w, const uint16_t* x_bf16,
                   double* y, double* absterm, int nthreads) {
  int bs = fmt_bs(fmt), nb = fmt_bytes(fmt);
  int64_t gu_bytes = (int64_t)I * (H / bs) * nb, dn_bytes = (int64_t)H * (I / bs) * nb;
  (void)E;
#ifdef _OPENMP
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int t = 0; t < T; ++t) {
    const uint8_t* g[64];
    const uint8_t* u[64];
    const uint8_t* d[64];
    for (int r = 0; r < k; ++r) {
      int e = idx[(int64_t)t * k + r];
      g[r] = gate_all + e * gu_bytes;
      u[r] = up_all + e * gu_bytes;
      d[r] = down_all + e * dn_bytes;
    }
    orc_moe_token(fmt, H, I, k, g, u, d, w + (int64_t)t * k, x_bf16 + (int64_t)t * H, y + (int64_t)t * H,
                  absterm ? absterm + (int64_t)t * H : NULL);
  }
}

/* ------------------------------------------------------------------------------------------------
 * Prefill grouped GEMM [P5 table "GPU compute": block-scaled MXFP4 tensor-core instructions; P5 "V4.1 Flash"
 * section: the E4M3 + per-32 E8M0 sibling of MXFP4]: x and h are quantised per 32 along K to MXFP8 (E4M3 +
 * E8M0) before the contractions; weights MXFP4. The h quantisation decision is taken on h rounded to
 * fp32 (the precision the GPU path holds h in).
 * One token; xq/hq_codes/scales outputs are optional (for stage-wise comparison).
 * ------------------------------------------------------------------------------------------------ */
void orc_prefill_token(int H, int I, int k, const uint8_t* const* gate, const uint8_t* const* up,
                       const uint8_t* const* down, const float* w, const uint16_t* x_bf16, double* y,
                       double* absterm, uint8_t* xq_codes, uint8_t* xq_scales, uint8_t* hq_codes,
                       uint8_t* hq_scales, double* h_out) {
  double* x = (double*)malloc(sizeof(double) * (size_t)H);
  double* xq = (double*)malloc(sizeof(double) * (size_t)H);
  uint8_t* xc = (uint8_t*)malloc((size_t)H);
  uint8_t* xs = (uint8_t*)malloc((size_t)H / 32);
  for (int c = 0; c < H; ++c) x[c] = orc_bf16_to_f64(x_bf16[c]);
  orc_quant_mxfp8(x, H / 32, xc, xs);
  for (int c = 0; c < H; ++c) xq[c] = orc_e4m3_value(xc[c]) * orc_e8m0_scale(xs[c / 32]);
  if (xq_codes) memcpy(xq_codes, xc, (size_t)H);
  if (xq_scales) memcpy(xq_scales, xs, (size_t)H / 32);
  double* h = (double*)malloc(sizeof(double) * (size_t)I);
  double* h32 = (double*)malloc(sizeof(double) * (size_t)I);
  double* hq = (double*)malloc(sizeof(double) * (size_t)I);
  uint8_t* hc = (uint8_t*)malloc((size_t)I);
  uint8_t* hs = (uint8_t*)malloc((size_t)I / 32);
  double* d = (double*)malloc(sizeof(double) * (size_t)H);
  double* da = (double*)malloc(sizeof(double) * (size_t)H);
  for (int j = 0; j < H; ++j) { y[j] = 0.0; if (absterm) absterm[j] = 0.0; }
  for (int r = 0; r < k; ++r) {
    orc_expert_ffn(1, H, I, gate[r], up[r], down[r], xq, NULL, NULL, h, NULL, NULL);
    for (int i = 0; i < I; ++i) h32[i] = orc_round_f32(h[i]);
    orc_quant_mxfp8(h32, I / 32, hc, hs);
    for (int i = 0; i < I; ++i) hq[i] = orc_e4m3_value(hc[i]) * orc_e8m0_scale(hs[i / 32]);
    if (hq_codes) memcpy(hq_codes + (size_t)r * I, hc, (size_t)I);
    if (hq_scales) memcpy(hq_scales + (size_t)r * (I / 32), hs, (size_t)I / 32);
    if (h_out) memcpy(h_out + (size_t)r * I, h, sizeof(double) * (size_t)I);
    for (int j = 0; j < H; ++j) {
      double s = 0.0, a = 0.0;
      for (int i = 0; i < I; ++i) {
        double p = weight_at(1, down[r], I, j, i) * hq[i];
        s += p;
        a += fabs(p);
      }
      d[j] = s;
      da[j] = a;
    }
    for (int j = 0; j < H; ++j) {
      y[j] += (double)w[r] * d[j];
      if (absterm) absterm[j] += fabs((double)w[r]) * da[j];
    }
  }
  free(x); free(xq); free(xc); free(xs); free(h); free(h32); free(hq); free(hc); free(hs); free(d); free(da);
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------- speculative acceptance
 * [P2] "What compression does not solve": a drafted token x is accepted with probability min(1, p(x) / q(x));
 * on a rejection the token is drawn from max(p - q, 0), normalised; this keeps the target's distribution exact.
 * The chain of K drafts is the usual reading: drafts are tested in order, the first rejection ends the chain
 * and is replaced by a draw from that position's residual; if all K are accepted, one more token is drawn
 * from the target's distribution after the last draft.
 *
 * Readings (the pages give the rule, not its arithmetic):
 *   - p, q, u are fp32; draft k is accepted when u[k] < p_k(d) / q_k(d), the quotient one fp32 division
 *     (q = 0 < p accepts; p = q = 0 rejects);
 *   - a draw from weights r(v) (r = p - q or p, clamped to [0, 1], NaN as 0) with the uniform u_s: the
 *     smallest v whose running sum exceeds u_s times the total, in exact integers: R(v) = floor(r(v) 2^40),
 *     U = floor(u_s 2^32) (u_s clamped to [0, 1), NaN as 0), threshold floor(U * sum R / 2^32); V <= 2^22 keeps the
 *     sums inside 64 bits;
 *   - a residual with no mass falls back to p of that position; a row with no mass gives token -1;
 *   - a draft id outside [0, V) gives n = -1 and token -1.
 * p [K+1][V], q [K][V], draft [K], u [K+1] (u[K] is the draw's uniform); out[0] = accepted drafts n,
 * out[1] = the token drawn after them. */
static uint64_t spec_weight(const float* p, const float* q, int v) {
  float r = q ? p[v] - q[v] : p[v];
  if (!(r > 0.0f)) r = 0.0f;  /* negative or NaN: no mass */
  if (r > 1.0f) r = 1.0f;     /* a probability is at most 1 */
  return (uint64_t)ldexp((double)r, 40);
}
static int64_t spec_draw(const float* p, const float* q, int V, float us) {
  uint64_t total = 0;
  for (int v = 0; v < V; ++v) total += spec_weight(p, q, v);
  if (total == 0) return -1;
  const double uc = us > 0.0f ? (double)us : 0.0;  /* negative or NaN: 0 */
  const uint64_t U = uc >= 1.0 ? 0xFFFFFFFFull : (uint64_t)ldexp(uc, 32);
  const uint64_t thr = (uint64_t)(((unsigned __int128)U * total) >> 32);
  uint64_t run = 0;
  for (int v = 0; v < V; ++v) {
    run += spec_weight(p, q, v);
    if (run > thr) return v;
  }
  return -1;
}

void orc_spec_accept(const float* p, const float* q, int K, int V, const int32_t* draft, const float* u,
                     int32_t* out) {
  for (int k = 0; k < K; ++k)
    if (draft[k] < 0 || draft[k] >= V) { out[0] = -1; out[1] = -1; return; }
  int n = 0;
  while (n < K) {
    const int d = draft[n];
    const float ratio = p[(int64_t)n * V + d] / q[(int64_t)n * V + d];
    if (!(u[n] < ratio)) break;
    ++n;
  }
  int64_t tok;
  if (n < K) {
    tok = spec_draw(p + (int64_t)n * V, q + (int64_t)n * V, V, u[K]);
    if (tok < 0) tok = spec_draw(p + (int64_t)n * V, NULL, V, u[K]);
  } else {
    tok = spec_draw(p + (int64_t)K * V, NULL, V, u[K]);
  }
  out[0] = n;
  out[1] = (int32_t)tok;
}
