// decode_tc.cu -- decode and verify (1..8 tokens) of MXFP4 experts in the tensor-core layout on tcgen05.
//
// The work is a mat-vec per expert, so the block-scaled MMA runs with the weights as the 128-row operand A and a
// handful of activation columns as operand B:
//   gate/up: B = x split into two E4M3 parts per 32-block (x ~= p0 * 2^(e0-127) + p1 * 2^(e1-127), exact for
//            bf16 x except far below the block's largest element), 2 columns per token, N = 16;
//   down:    B = h split into three E4M3 parts the same way (about 12 significant bits), 3 columns per
//            (expert, token), N = 32.
// A token's result is the sum of its part columns; the MMA computes every column independently, so a token's
// numbers do not depend on which other tokens share the sweep (verify row t == decode of token t).
//
// Work units (fixed for every T, so the arithmetic of a token never changes):
//   G unit (expert u, 128-row tile rt of [Gate;Up], K segment ks): fp32 partial g/u of the tile's 64 gate and 64
//     up rows over KS_G k-tiles, written to the workspace. The unit that completes the last segment of (u, rt)
//     sums the segments in order, forms h = SiLU(g) * u and writes the three E4M3 parts of h for the D units.
//   D unit (expert u, 128-row tile jt of Down, segment ks): fp32 partial of Down * h. The unit that completes the
//     last D unit of row tile jt (over all experts and segments) sums each (expert, token) in segment order and
//     combines y[t] = sum_r w[t, r] * d_r in rank order.
// Units are dealt round-robin to persistent CTAs (one per SM, cooperative launch), G units first (expert-major),
// then D units. Inside a CTA, four independent pipelines (a TMA-issuing lane, an MMA-issuing thread, a two-slot
// shared-memory ring and two TMEM accumulators each) take the CTA's units in turn, because one issuing thread
// sustains only about one wait-and-issue round per 330 ns (TMA) or one 4-MMA stage plus commit per ~600 cycles
// (tcgen05), while one SM must consume an 8.5 KB weight tile every ~180 ns to keep pace with HBM. Four epilogue
// warps drain the accumulators. Cross-CTA dependencies (x parts ready, h of an expert ready) are global counters
// with bounded waits; the last CTA to finish resets them.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "layout.cuh"
#include "tcgen05.cuh"
#include "api_internal.h"

namespace moe {
namespace dtc {

constexpr int NPIPE = 4;                 // pipelines per CTA
constexpr int RING = 2;                  // stage slots per pipeline
constexpr int NSLOT = NPIPE * RING;
constexpr int A_BYTES = 16384;           // 128 x 128 E2M1 weights as unpacked in shared memory
constexpr int A_TX = 8192;               // bytes the TMA engine reads for them
constexpr int B_BYTES = 4096;            // up to 32 rows x 128 E4M3 activation parts
constexpr int SLOT_BYTES = A_BYTES + B_BYTES + 1024;  // + two 512-byte exponent blocks; 21 KB
constexpr int MAX_T = 8, MAX_K = 8, MAX_U = MAX_T * MAX_K;
constexpr int XROWS = 16, HROWS = 32;    // B rows: 2 parts x 8 tokens; 3 parts x 8 tokens (padded)
constexpr int EPI_WARP0 = 5;             // warps 0: producers, 1..4: MMA issuers, 5..20: epilogue
constexpr int NGRP = NPIPE;              // epilogue groups of 4 warps; group j drains pipeline j
constexpr int QN = 4;                    // unit-id queue entries per pipeline
constexpr int THREADS = (EPI_WARP0 + 4 * NGRP) * 32;
constexpr uint32_t TMEM_COLS = 512;      // accumulators: pipeline j, buffer a at 64 j + 32 a; scales from 256
constexpr uint32_t SF_COL0 = 256;
constexpr int SMEM = NSLOT * SLOT_BYTES + 1024;

// ------------------------------------------------------------------ geometry of one call
struct Geo {
  int H, I, T, k, U;
  int RTG, KTG, KSG, SG;   // gate/up: row tiles, k-tiles, k-tiles per unit, segments
  int RTD, KTD, KSD, SD;   // down
  int nG, nD;              // units
};
__host__ __device__ inline int ks_for(int kt) { return kt % 8 == 0 ? 8 : (kt % 4 == 0 ? 4 : 2); }

// ------------------------------------------------------------------ workspace (byte offsets from the base)
// [0, 256)       WsHeader (status word)
// [256, 20736)   counters (uint32): x_ready, done, h_ready[64], g_cnt[64 * 64], d_cnt[32]
// then xb [16][H] E4M3, xsf [H/128][512], hb [Umax * 32][I], hsf [Umax][I/128][512],
//      gpart [Umax][2I/128][S_G][TS][128] fp32, dpart [Umax][H/128][S_D][TS][128] fp32
// with Umax = T_max * k union experts and TS = T_max token columns of the partial buffers.
constexpr int64_t kCnt = 256;
constexpr int C_XREADY = 0, C_DONE = 1, C_HREADY = 2, C_G = C_HREADY + MAX_U, C_D = C_G + MAX_U * 64;
constexpr int C_END = C_D + 32;
struct Ws {
  int64_t xb, xsf, hb, hsf, gpart, dpart, total;
};
inline int64_t al1k(int64_t v) { return (v + 1023) & ~(int64_t)1023; }
inline Ws ws_layout(int64_t H, int64_t I, int64_t Umax, int64_t TS) {
  Ws w;
  int64_t o = al1k(kCnt + (int64_t)C_END * 4);
  const int64_t RTG = 2 * I / 128, KTG = H / 128, RTD = H / 128, KTD = I / 128;
  const int64_t SG = KTG / ks_for((int)KTG), SD = KTD / ks_for((int)KTD);
  w.xb = o;    o = al1k(o + XROWS * H);
  w.xsf = o;   o = al1k(o + KTG * 512);
  w.hb = o;    o = al1k(o + Umax * HROWS * I);
  w.hsf = o;   o = al1k(o + Umax * KTD * 512);
  w.gpart = o; o = al1k(o + Umax * RTG * SG * TS * 128 * 4);
  w.dpart = o; o = al1k(o + Umax * RTD * SD * TS * 128 * 4);
  w.total = o;
  return w;
}

struct Args {
  const uint8_t* gu;          // gate/up weights (tensor-core layout)
  const uint8_t* dn;          // down weights
  int64_t gu_stride, dn_stride;
  const uint16_t* x;          // [T][H] bf16
  const int32_t* idx;         // [T][k]
  const float* w;             // [T][k]
  float* y;                   // [T][H]
  __nv_bfloat16* yb;          // [T][H] or NULL
  int accumulate;
  int E;
  uint8_t* ws;
  Ws L;
  int ts;                     // token stride of the partial buffers
  Geo g;
  long long wait_ns;
};

// ------------------------------------------------------------------ small helpers
__device__ __forceinline__ int mx8_exp(float amax) {
  const uint32_t ab = __float_as_uint(amax) & 0x7FFFFFFFu;
  const int ef = (int)(ab >> 23);
  if (ef == 0) return 1;
  const int e = ef - 8 + ((ab & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < 1 ? 1 : (e > 254 ? 254 : e);
}
__device__ __forceinline__ float pow2_127m(int e) {  // 2^(127 - e), e in [1, 254]
  return e <= 253 ? __uint_as_float((uint32_t)(254 - e) << 23) : __uint_as_float(0x00400000u);
}
__device__ __forceinline__ float pow2_m127(int e) {  // 2^(e - 127), e in [1, 254]
  return __uint_as_float((uint32_t)e << 23);
}
__device__ __forceinline__ uint32_t e4m3_code(float v) {  // round to nearest even, saturating
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(0.0f), "f"(v));
  return d & 0xFFu;
}
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  uint32_t h2;
  const uint16_t c = (uint16_t)code;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}
__device__ __forceinline__ float warp_amax(float v) {
  const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(v)));
  return __uint_as_float(m);
}
// Split v (one element per lane of a 32-block) into `np` E4M3 parts with per-block exponents. Lane writes its
// codes to codes[p]; returns nothing else (exponents in exps[p], identical across the warp).
__device__ __forceinline__ void split_parts(float v, int np, uint32_t* codes, int* exps) {
  float r = v;
  for (int p = 0; p < np; ++p) {
    const int e = mx8_exp(warp_amax(r));
    const uint32_t c = e4m3_code(r * pow2_127m(e));
    codes[p] = c;
    exps[p] = e;
    r = r - e4m3_value(c) * pow2_m127(e);
  }
}
__device__ __forceinline__ int sfb(int row, int kb) { return (row & 31) * 16 + (row >> 5) * 4 + kb; }

// Bounded wait on a global counter (acquire); gives up when `abort_flag` is set elsewhere or after lim ns.
__device__ __forceinline__ bool wait_ge(const uint32_t* p, uint32_t target, volatile int* abort_flag, long long lim) {
  if (ld_acquire_u32(p) >= target) return true;
  const long long t0 = globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_u32(p) >= target) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > lim) { *abort_flag = 1; return false; }
  }
}
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, long long lim) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > lim) { *abort_flag = 1; return false; }
  }
}

// Publish: every store this thread has performed -- and, through the preceding CTA barrier, the stores of the
// threads it synchronised with -- becomes visible before the increment (release at GPU scope).
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Count-and-check: release our stores, acquire the stores of every earlier incrementer.
__device__ __forceinline__ uint32_t atom_acq_rel_add(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

struct Unit {
  int d, u, rt, ks;
};
__device__ __forceinline__ Unit unit_of(int v, const Geo& g) {
  Unit r;
  if (v < g.nG) {
    const int per = g.RTG * g.SG;
    r.d = 0; r.u = v / per; r.rt = (v % per) / g.SG; r.ks = v % g.SG;
  } else {
    v -= g.nG;
    const int per = g.RTD * g.SD;
    r.d = 1; r.u = v / per; r.rt = (v % per) / g.SD; r.ks = v % g.SD;
  }
  return r;
}

// Tables every CTA builds from idx: the union of experts (first-appearance order over (t, r)), each expert's
// tokens (slot order = token order) and, per (t, r), the union index and the token's slot in that expert.
struct Tables {
  int32_t ue[MAX_U];         // union index -> expert id
  int8_t ntok[MAX_U];        // tokens of each union expert
  int8_t tok[MAX_U][MAX_T];  // union expert, slot -> token
  int8_t pu[MAX_T][MAX_K];   // (t, r) -> union index
  int8_t ps[MAX_T][MAX_K];   // (t, r) -> slot
  int U;
  int bad;
};

__device__ void build_tables(Tables& tb, const int32_t* idx, int T, int k, int E) {
  tb.U = 0;
  tb.bad = 0;
  for (int t = 0; t < T; ++t)
    for (int r = 0; r < k; ++r) {
      const int e = idx[t * k + r];
      if (e < 0 || e >= E) { tb.bad = 1; tb.pu[t][r] = 0; tb.ps[t][r] = 0; continue; }
      int u = 0;
      while (u < tb.U && tb.ue[u] != e) ++u;
      if (u == tb.U) { tb.ue[u] = e; tb.ntok[u] = 0; tb.U = u + 1; }
      int s = 0;
      while (s < tb.ntok[u] && tb.tok[u][s] != t) ++s;
      if (s == tb.ntok[u]) { tb.tok[u][s] = (int8_t)t; tb.ntok[u] = (int8_t)(s + 1); }
      tb.pu[t][r] = (int8_t)u;
      tb.ps[t][r] = (int8_t)s;
    }
}

// x of every token, k-tile kt, split into two E4M3 parts: B rows 2t + p, one exponent per (row, 32-block).
// Run by the 4 epilogue warps of CTA kt: warp w takes the (token, 32-block) pairs w, w + 4, ...
__device__ void split_x(const Args& a, const Geo& g, int kt, int ew) {
  const int lane = threadIdx.x & 31;
  uint8_t* xb = a.ws + a.L.xb;
  uint8_t* xsf = a.ws + a.L.xsf + kt * 512;
  for (int pr = ew; pr < 4 * g.T; pr += 4) {
    const int t = pr / 4, blk = pr % 4;
    const int i = kt * 128 + blk * 32 + lane;
    const float xv = __uint_as_float((uint32_t)a.x[(int64_t)t * g.H + i] << 16);
    uint32_t c[2];
    int ex[2];
    split_parts(xv, 2, c, ex);
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      xb[(int64_t)(2 * t + p) * g.H + i] = (uint8_t)c[p];
      if (lane == 0) xsf[sfb(2 * t + p, blk)] = (uint8_t)ex[p];
    }
  }
}

// All G segments of (expert u, row tile rt) are in: g, u of the 64 intermediate indices rt*64 .. +63 (tile rows
// 0..63 gate, 64..127 up), h = SiLU(g) * u, three E4M3 parts per 32-block into the D operand rows 3s + p of u.
// Threads et < 64 (two whole warps, one 32-block each) do the work.
__device__ void finalize_h(const Args& a, const Geo& g, const Tables& tb, int u, int rt, int et) {
  if (et >= 64) return;
  const float* gp = reinterpret_cast<const float*>(a.ws + a.L.gpart) + ((int64_t)u * g.RTG + rt) * g.SG * a.ts * 128;
  const int i = rt * 64 + et, kt = i / 128, kb = (i % 128) / 32;
  uint8_t* hb = a.ws + a.L.hb + (int64_t)u * HROWS * g.I;
  uint8_t* hsf = a.ws + a.L.hsf + ((int64_t)u * g.KTD + kt) * 512;
  const int nt = tb.ntok[u];
  for (int s = 0; s < nt; ++s) {
    const int t = tb.tok[u][s];
    float gv = 0.f, uv = 0.f;
    for (int k0 = 0; k0 < g.SG; k0 += 4) {  // segments in order, loads issued four at a time
      float gl[4], ul[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (k0 + q < g.SG) {
          gl[q] = __ldcg(gp + ((int64_t)(k0 + q) * a.ts + t) * 128 + et);
          ul[q] = __ldcg(gp + ((int64_t)(k0 + q) * a.ts + t) * 128 + 64 + et);
        }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (k0 + q < g.SG) { gv += gl[q]; uv += ul[q]; }
    }
    const float h = gv / (1.0f + expf(-gv)) * uv;
    uint32_t c[3];
    int ex[3];
    split_parts(h, 3, c, ex);
#pragma unroll
    for (int p = 0; p < 3; ++p) {
      hb[(int64_t)(3 * s + p) * g.I + i] = (uint8_t)c[p];
      if ((et & 31) == 0) hsf[sfb(3 * s + p, kb)] = (uint8_t)ex[p];
    }
  }
}

// All D units of row tile jt are in: y[t][jt*128 + et] = sum_r w[t, r] * (sum over segments of the partial of
// (expert of rank r, token t)), ranks in order.
__device__ void combine_rows(const Args& a, const Geo& g, const Tables& tb, int jt, int et) {
  const float* dp = reinterpret_cast<const float*>(a.ws + a.L.dpart);
  const int j = jt * 128 + et;
  for (int t = 0; t < g.T; ++t) {
    float acc = 0.f;
    for (int r = 0; r < g.k; ++r) {
      const int u = tb.pu[t][r], s = tb.ps[t][r];
      const float* p = dp + (((int64_t)u * g.RTD + jt) * g.SD * a.ts + s) * 128 + et;
      float sum = 0.f;
      for (int k0 = 0; k0 < g.SD; k0 += 4) {
        float pl[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (k0 + q < g.SD) pl[q] = __ldcg(p + (int64_t)(k0 + q) * a.ts * 128);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (k0 + q < g.SD) sum += pl[q];
      }
      acc = fmaf(a.w[t * g.k + r], sum, acc);
    }
    float* yp = a.y + (int64_t)t * g.H + j;
    const float out = a.accumulate ? *yp + acc : acc;
    *yp = out;
    if (a.yb) a.yb[(int64_t)t * g.H + j] = __float2bfloat16_rn(out);
  }
}

__device__ void epilogue(const Args& a, const Geo& g, const Tables& tb, uint32_t tbase, uint64_t (*acc_full)[2],
                         uint64_t (*acc_empty)[2], uint64_t (*uq_full)[QN], volatile int (*uq)[QN], uint32_t* cnt,
                         volatile int* s_last, volatile int* s_ok, volatile int* s_unit, volatile int* s_abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3;
  const int grp = (warp - EPI_WARP0) / 4;
  const int bar = 1 + grp;                                      // named barrier of the group
  const int et = threadIdx.x - (EPI_WARP0 + 4 * grp) * 32;       // 0..127 inside the group
  const int m = q * 32 + lane;                                   // TMEM lane = weight row of the tile
  const long long lim = a.wait_ns;
  if (grp == 0 && g.nG > 0 && (int)blockIdx.x < g.KTG) {
    split_x(a, g, blockIdx.x, warp - EPI_WARP0);
    named_bar(bar, 128);
    if (et == 0) red_release_add(cnt + C_XREADY, 1u);
  }
  float* gpart = reinterpret_cast<float*>(a.ws + a.L.gpart);
  float* dpart = reinterpret_cast<float*>(a.ws + a.L.dpart);
  // the units pipeline j = grp took, in order (each accumulator's phases in order)
  const int j = grp;
  for (int c = 0;; ++c) {
    const int ab = c & 1;
    // one thread waits; the verdict is shared so that the group's four warps leave (or stay) together
    if (et == 0) {
      int st = 0;
      if (bwait(&uq_full[j][c % QN], (uint32_t)((c / QN) & 1), s_abort, lim)) {
        const int i = uq[j][c % QN];
        if (i < 0) st = 2;
        else { s_unit[grp] = i; st = bwait(&acc_full[j][ab], (uint32_t)((c >> 1) & 1), s_abort, lim) ? 1 : 0; }
      }
      s_ok[grp] = st;
    }
    named_bar(bar, 128);
    if (s_ok[grp] != 1) break;
    tc_fence_after();
    const int i = s_unit[grp];
    const Unit un = unit_of((int)blockIdx.x + i * (int)gridDim.x, g);
    const uint32_t taddr = tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(64 * j + 32 * ab);
    uint32_t v0[16], v1[16];
    tc_ld16(taddr, v0);
    if (un.d) tc_ld16(taddr + 16, v1);
    tc_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&acc_empty[j][ab]);
    if (!un.d) {
      float* gp = gpart + (((int64_t)un.u * g.RTG + un.rt) * g.SG + un.ks) * a.ts * 128 + m;
#pragma unroll
      for (int t = 0; t < MAX_T; ++t)
        if (t < g.T) gp[t * 128] = __uint_as_float(v0[2 * t]) + __uint_as_float(v0[2 * t + 1]);
    } else {
      float* dp = dpart + (((int64_t)un.u * g.RTD + un.rt) * g.SD + un.ks) * a.ts * 128 + m;
      const int nt = tb.ntok[un.u];
#pragma unroll
      for (int s = 0; s < MAX_T; ++s) {
        if (s < nt) {
          const int c0 = 3 * s;
          const float p0 = __uint_as_float(c0 < 16 ? v0[c0] : v1[c0 - 16]);
          const float p1 = __uint_as_float(c0 + 1 < 16 ? v0[c0 + 1] : v1[c0 + 1 - 16]);
          const float p2 = __uint_as_float(c0 + 2 < 16 ? v0[c0 + 2] : v1[c0 + 2 - 16]);
          dp[s * 128] = (p0 + p1) + p2;
        }
      }
    }
    // count the unit; the one that completes a group of units does the group's follow-up work
    named_bar(bar, 128);
    if (et == 0) {
      uint32_t old, target;
      if (!un.d) { old = atom_acq_rel_add(cnt + C_G + un.u * g.RTG + un.rt, 1u); target = (uint32_t)g.SG; }
      else { old = atom_acq_rel_add(cnt + C_D + un.rt, 1u); target = (uint32_t)(g.U * g.SD); }
      s_last[grp] = (old == target - 1) ? 1 : 0;
    }
    named_bar(bar, 128);
    if (s_last[grp]) {
      if (!un.d) {
        finalize_h(a, g, tb, un.u, un.rt, et);
        named_bar(bar, 128);
        if (et == 0) red_release_add(cnt + C_HREADY + un.u, 1u);
      } else {
        combine_rows(a, g, tb, un.rt, et);
      }
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1) decode_kernel(const __grid_constant__ CUtensorMap tm_gu,
                                                            const __grid_constant__ CUtensorMap tm_dn,
                                                            const __grid_constant__ CUtensorMap tm_x,
                                                            const __grid_constant__ CUtensorMap tm_h, const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[NSLOT], empty[NSLOT], acc_full[NPIPE][2], acc_empty[NPIPE][2], drain[NPIPE];
  __shared__ __align__(8) uint64_t uq_full[NPIPE][QN];
  __shared__ volatile int uq[NPIPE][QN];
  __shared__ int s_next;
  __shared__ Tables tb;
  __shared__ uint32_t s_tmem;
  __shared__ int s_units;
  __shared__ volatile int s_abort, s_ok[NGRP], s_last[NGRP], s_unit[NGRP];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(a.ws + kCnt);
  Geo g = a.g;
  const long long lim = a.wait_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSLOT; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
    for (int j = 0; j < NPIPE; ++j) {
      mbar_init(&acc_full[j][0], 1); mbar_init(&acc_full[j][1], 1);
      mbar_init(&acc_empty[j][0], 4); mbar_init(&acc_empty[j][1], 4);  // the 4 warps of one epilogue group
      mbar_init(&drain[j], 1);
      for (int e = 0; e < QN; ++e) mbar_init(&uq_full[j][e], 1);
    }
    s_abort = 0;
    s_next = 0;
    fence_mbar_init();
    build_tables(tb, a.idx, g.T, g.k, a.E);
    if (tb.bad) { s_abort = 1; if (blockIdx.x == 0) record_error(&hdr->status, MOE_ERR_INVALID_ARG); }
    s_units = tb.bad ? 0 : tb.U * (g.RTG * g.SG + g.RTD * g.SD);
  }
  if (warp == 1) tc_alloc(&s_tmem, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;
  g.U = tb.U;
  g.nG = g.U * g.RTG * g.SG;
  g.nD = g.U * g.RTD * g.SD;
  const int nunits = s_units;
  if (nunits == 0) g.nG = g.nD = 0;
  // this CTA's units: v = blockIdx.x + i * gridDim.x, i = 0 .. my_units - 1 (G units first). Pipelines take the
  // next i from a shared counter when they start a unit, so a pipeline waiting for h does not hold up the rest;
  // each publishes the ids it took through its queue uq[j] to its MMA thread and epilogue group.
  const int my_units = nunits > (int)blockIdx.x ? (nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (warp == 0) {
    // ---------------- producers: lane j feeds pipeline j
    if (lane < NPIPE) {
      const int j = lane;
      int n = 0;  // stages issued by this pipeline
      bool ok = true, x_ok = false, partial = false;
      int h_ok_u = -1;
      for (int c = 0; ok; ++c) {
        const int i = atomicAdd(&s_next, 1);
        // entry c % QN was last read for unit c - QN, which its epilogue group started before this pipeline's
        // MMA could move past unit c - 2; the producer is at most RING stages ahead of the MMA
        uq[j][c % QN] = i < my_units ? i : -1;
        mbar_arrive(&uq_full[j][c % QN]);
        if (i >= my_units) break;
        const Unit un = unit_of((int)blockIdx.x + i * (int)gridDim.x, g);
        const int e = tb.ue[un.u];
        const int ks = un.d ? g.KSD : g.KSG;
        for (int kk = 0; kk < ks; ++kk, ++n) {
          const int slot = j * RING + (n % RING);
          const uint32_t ph = (uint32_t)((n / RING) & 1);
          if (!bwait(&empty[slot], ph ^ 1, &s_abort, lim)) { ok = false; break; }
          uint8_t* st = smem + slot * SLOT_BYTES;
          if (!un.d) {
            const int kt = un.ks * g.KSG + kk;
            const int tile = un.rt * g.KTG + kt;
            mbar_arrive_expect_tx(&full[slot], A_TX + XROWS * 128 + 1024);
            tma_load_4d(st, &tm_gu, 0, 0, tile, e, &full[slot]);
            bulk_g2s_plain(st + A_BYTES + B_BYTES, a.gu + (int64_t)e * a.gu_stride + (int64_t)tile * kTcTileBytes + 8192,
                           512, &full[slot]);
            if (!x_ok) {
              if (!wait_ge(cnt + C_XREADY, (uint32_t)g.KTG, &s_abort, lim)) { ok = false; partial = true; break; }
              asm volatile("fence.proxy.async.global;" ::: "memory");  // generic-proxy writes -> TMA reads
              x_ok = true;
            }
            tma_load_2d(st + A_BYTES, &tm_x, kt * 128, 0, &full[slot]);
            bulk_g2s_plain(st + A_BYTES + B_BYTES + 512, a.ws + a.L.xsf + kt * 512, 512, &full[slot]);
          } else {
            const int kt = un.ks * g.KSD + kk;
            const int tile = un.rt * g.KTD + kt;
            mbar_arrive_expect_tx(&full[slot], A_TX + HROWS * 128 + 1024);
            tma_load_4d(st, &tm_dn, 0, 0, tile, e, &full[slot]);
            bulk_g2s_plain(st + A_BYTES + B_BYTES, a.dn + (int64_t)e * a.dn_stride + (int64_t)tile * kTcTileBytes + 8192,
                           512, &full[slot]);
            if (h_ok_u != un.u) {
              if (!wait_ge(cnt + C_HREADY + un.u, (uint32_t)g.RTG, &s_abort, lim)) { ok = false; partial = true; break; }
              asm volatile("fence.proxy.async.global;" ::: "memory");
              h_ok_u = un.u;
            }
            tma_load_2d(st + A_BYTES, &tm_h, kt * 128, un.u * HROWS, &full[slot]);
            bulk_g2s_plain(st + A_BYTES + B_BYTES + 512, a.ws + a.L.hsf + ((int64_t)un.u * g.KTD + kt) * 512, 512,
                           &full[slot]);
          }
        }
      }
      if (!ok) {
        record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
        // the weight copies of a stage whose activation copy never came leave the barrier short: wait (bounded)
        // for what was issued so the shared memory is not released under a copy in flight
        for (int q = 0; q < RING; ++q) {
          const int m = n - 1 - q;
          if (m >= 0) mbar_wait(&full[j * RING + (m % RING)], (uint32_t)((m / RING) & 1), 50000000LL);
        }
        if (partial) {  // stage n got its weight copies only: its barrier never completes, so give them 1 ms
          const long long t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 1000000LL) __nanosleep(1000);
        }
      }
    }
    __syncwarp();
  } else if (warp <= NPIPE) {
    // ---------------- MMA issuers: warp 1 + j, lane 0, pipeline j
    const int j = warp - 1;
    if (lane == 0) {
      int n = 0, c = 0;
      bool ok = true;
      const uint32_t sfa_col = tbase + SF_COL0;
      for (;; ++c) {
        if (!bwait(&uq_full[j][c % QN], (uint32_t)((c / QN) & 1), &s_abort, lim)) { ok = false; break; }
        const int i = uq[j][c % QN];
        if (i < 0) break;
        const Unit un = unit_of((int)blockIdx.x + i * (int)gridDim.x, g);
        const int ab = c & 1;
        if (!bwait(&acc_empty[j][ab], ((c >> 1) & 1) ^ 1, &s_abort, lim)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tbase + (uint32_t)(64 * j + 32 * ab);
        const int ks = un.d ? g.KSD : g.KSG;
        const uint32_t N = un.d ? HROWS : XROWS;
        for (int kk = 0; kk < ks; ++kk, ++n) {
          const int slot = j * RING + (n % RING);
          if (!bwait(&full[slot], (uint32_t)((n / RING) & 1), &s_abort, lim)) { ok = false; break; }
          tc_fence_after();
          uint8_t* st = smem + slot * SLOT_BYTES;
          const uint32_t sfa = sfa_col + (uint32_t)(slot * 8), sfbc = sfa + 4;
          tc_cp_sf(sfa, umma_desc_sf(smem_u32(st + A_BYTES + B_BYTES)));
          tc_cp_sf(sfbc, umma_desc_sf(smem_u32(st + A_BYTES + B_BYTES + 512)));
          const uint64_t ad = umma_desc_sw128(smem_u32(st)), bd = umma_desc_sw128(smem_u32(st + A_BYTES));
#pragma unroll
          for (int kb = 0; kb < 4; ++kb)
            tc_mma_mxf8f6f4(d_tmem, ad + 2 * kb, bd + 2 * kb, idesc_mxf8f6f4(5, 0, 128, N, kb, kb), sfa, sfbc,
                            (kk | kb) != 0);
          tc_commit(&empty[slot]);
        }
        if (ok) tc_commit(&acc_full[j][ab]);
      }
      if (!ok) record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
      tc_commit(&drain[j]);
      mbar_wait(&drain[j], 0, 100000000LL);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps (see the second part of this file)
    epilogue(a, g, tb, tbase, acc_full, acc_empty, uq_full, uq, cnt, s_last, s_ok, s_unit, &s_abort);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tc_dealloc(tbase, TMEM_COLS);
  // the last CTA to finish resets the per-call counters
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(cnt + C_DONE, 1u);
    if (old == gridDim.x - 1) {
      __threadfence();
      cnt[C_XREADY] = 0;
      for (int u = 0; u < tb.U; ++u) cnt[C_HREADY + u] = 0;
      for (int q = 0; q < tb.U * g.RTG; ++q) cnt[C_G + q] = 0;
      for (int q = 0; q < g.RTD; ++q) cnt[C_D + q] = 0;
      __threadfence();
      cnt[C_DONE] = 0;
    }
  }
}

// ------------------------------------------------------------------ host side
inline int64_t umax_of(int T, int k) { return (int64_t)(T * k < MAX_U ? T * k : MAX_U); }

size_t workspace_bytes(const moe_layer_t* L, int T_max, int k) {
  return (size_t)ws_layout(L->H, L->I, umax_of(T_max, k), T_max).total;
}

// The caller (ffn.cu) has checked pointers, T in [1, 8], k in [1, 8], the shape and the device.
moe_status_t run(const moe_layer_t* L, const void* x, int T, const int32_t* idx, const float* w, int k, float* y,
                 void* y_bf16, int accumulate, void* ws, size_t ws_bytes, void* stream) {
  if (L->fmt != MOE_FMT_MXFP4) return MOE_ERR_UNSUPPORTED_FORMAT;
  if (((uintptr_t)x & 1) || ((uintptr_t)y & 3)) return MOE_ERR_INVALID_ARG;
  // the workspace is laid out for the T_max it was sized for; recover it from the size (largest T_max that fits)
  int tmax = 0;
  for (int tm = MAX_T; tm >= T; --tm)
    if (ws_bytes >= workspace_bytes(L, tm, k)) { tmax = tm; break; }
  if (!tmax) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!moe_internal::tmap_available()) return MOE_ERR_CUDA;
  if (moe_internal::num_sms() < L->H / 128) return MOE_ERR_UNSUPPORTED_ARCH;  // x is split by CTAs 0 .. H/128 - 1
  Args a;
  a.gu = (const uint8_t*)L->gate_up;
  a.dn = (const uint8_t*)L->down;
  a.gu_stride = tc_geom(MOE_MAT_GATE_UP, L->H, L->I).stride;
  a.dn_stride = tc_geom(MOE_MAT_DOWN, L->H, L->I).stride;
  a.x = (const uint16_t*)x;
  a.idx = idx;
  a.w = w;
  a.y = y;
  a.yb = (__nv_bfloat16*)y_bf16;
  a.accumulate = accumulate;
  a.E = L->E;
  a.ws = (uint8_t*)ws;
  const int64_t umax = umax_of(tmax, k);
  a.L = ws_layout(L->H, L->I, umax, tmax);
  a.ts = tmax;
  a.wait_ns = kDefaultWaitNs;
  Geo& g = a.g;
  g.H = L->H; g.I = L->I; g.T = T; g.k = k; g.U = 0;
  g.RTG = 2 * L->I / 128; g.KTG = L->H / 128; g.KSG = ks_for(g.KTG); g.SG = g.KTG / g.KSG;
  g.RTD = L->H / 128;     g.KTD = L->I / 128; g.KSD = ks_for(g.KTD); g.SD = g.KTD / g.KSD;
  g.nG = g.nD = 0;
  CUtensorMap mgu, mdn, mx, mh;
  const uint64_t xd[2] = {(uint64_t)L->H, (uint64_t)XROWS}, xs[1] = {(uint64_t)L->H};
  const uint64_t hd[2] = {(uint64_t)L->I, (uint64_t)(umax * HROWS)}, hs[1] = {(uint64_t)L->I};
  const uint32_t xbox[2] = {128, XROWS}, hbox[2] = {128, HROWS};
  if (!moe_internal::tmap_tc_weights(&mgu, L->gate_up, MOE_MAT_GATE_UP, L->H, L->I, L->E) ||
      !moe_internal::tmap_tc_weights(&mdn, L->down, MOE_MAT_DOWN, L->H, L->I, L->E) ||
      !moe_internal::tmap_u8(&mx, a.ws + a.L.xb, 2, xd, xs, xbox) ||
      !moe_internal::tmap_u8(&mh, a.ws + a.L.hb, 2, hd, hs, hbox))
    return MOE_ERR_CUDA;
  static std::once_flag once;
  static bool attr_ok = false;
  std::call_once(once, [] {
    attr_ok = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) == cudaSuccess;
  });
  if (!attr_ok) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(moe_internal::num_sms());
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_kernel, mgu, mdn, mx, mh, a) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace dtc
}  // namespace moe

namespace moe_internal {
size_t tc_decode_workspace_bytes(const moe_layer_t* L, int T_max, int k) {
  return moe::dtc::workspace_bytes(L, T_max, k);
}
moe_status_t tc_decode(const moe_layer_t* L, const void* x, int T, const int32_t* idx, const float* w, int k, float* y,
                       void* y_bf16, int accumulate, void* ws, size_t ws_bytes, void* stream) {
  return moe::dtc::run(L, x, T, idx, w, k, y, y_bf16, accumulate, ws, ws_bytes, stream);
}
}  // namespace moe_internal
