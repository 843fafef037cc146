// decode_tc.cu -- decode and verify (1..8 tokens) of MXFP4 experts in the tensor-core layout on tcgen05.
//
// The work is a mat-vec per expert, so the block-scaled MMA (kind::mxf4: E2M1 x E2M1, one UE8M0 exponent per 32,
// K = 64 per instruction) runs with the weights as the 128-row operand A, read as PACKED codes straight from the
// tensor-core tile layout (8 KB per 128 x 128 tile in shared memory, no unpacking), and a few activation columns as
// operand B: x (gate/up) and h (down) are each split into PARTS = 6 E2M1 parts per 32-block (split_parts_n: part p
// has exponent e0 - 2p and quantises what the earlier parts left; error below 1/3072 of the block's largest value).
// Column t * PARTS + p holds part p of token t; N = W = 16 ceil(6 T / 16) columns. A token's result is the sum of
// its part columns in part order; the MMA computes every column on its own (whatever N is), so a token's numbers
// do not depend on which other tokens share the sweep (verify row t == decode of token t).
//
// Work units (fixed for every T, so the arithmetic of a token never changes):
//   G unit (expert u, 128-row tile rt of [Gate;Up], K segment ks): fp32 partial g/u of the tile's 64 gate and 64
//     up rows over KS_G k-tiles, written to the workspace. The unit that completes the last segment of (u, rt)
//     sums the segments in order, forms h = SiLU(g) * u and writes the E2M1 parts of h for the D units.
//   D unit (expert u, 128-row tile jt of Down, segment ks): fp32 partial of Down * h. The unit that completes the
//     last D unit of row tile jt (over all experts and segments) sums each (expert, token) in segment order and
//     combines y[t] = sum_r w[t, r] * d_r in rank order.
// Units are dealt round-robin to persistent CTAs (one per SM, cooperative launch), G units first (expert-major),
// then D units; the grid is a multiple of the number of gate/up segments, so all G units of a CTA share one K
// segment. x is split into its parts once per call by the epilogue warps of the whole grid (an operand image in
// the workspace); each CTA then bulk-copies its segment's part tiles into shared memory and keeps them resident.
// With a router (moe_route_expert_ffn), warps 2..7 of every CTA first compute halves of the router logits, and
// every CTA then selects each token's experts itself (route.cuh, the same arithmetic as the standalone router).
// Inside a CTA, three independent pipelines take the CTA's units as they free up. A pipeline is a weight-issuing
// warp, an activation-issuing warp (h parts of D units, after their h is final), an MMA-issuing warp, a three-slot
// shared-memory ring, two to four TMEM accumulators and a group of four epilogue warps. One issuing thread
// sustains only about one wait-and-issue round per 330 ns (TMA) or one stage of MMAs plus commit per ~600 cycles
// (tcgen05), while one SM must consume an 8.5 KB weight tile every ~180 ns to keep pace with HBM. Cross-CTA
// dependencies (partials complete, h of an expert's K segment final) are global counters with bounded waits; the
// last CTA to finish resets them.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "layout.cuh"
#include "tcgen05.cuh"
#include "route.cuh"
#include "api_internal.h"

namespace moe {
namespace dtc {

constexpr int NPIPE = 3;                 // pipelines per CTA
constexpr int RING = 3;                  // stage slots per pipeline (more bytes in flight only lengthen the queues:
                                         // every dependent L2 round trip of the call then takes longer)
constexpr int NSLOT = NPIPE * RING;
constexpr int PARTS = 6;                 // E2M1 parts per activation value
constexpr int NB = 48;                   // B rows (MMA N): PARTS x 8 tokens
constexpr int A_BYTES = 8192;            // 128 rows x 64 B of packed E2M1 weight codes
constexpr int B_BYTES = NB * 64;         // 48 rows x 64 B of packed E2M1 activation parts
constexpr int SLOT_BYTES = A_BYTES + B_BYTES + 1024;  // + two 512-byte exponent blocks; 12 KB
constexpr int MAX_T = 8, MAX_K = 8, MAX_U = MAX_T * MAX_K;
constexpr int HROWS = NB;                // B rows of each expert's h parts
constexpr int EPI_WARP0 = 3 * NPIPE;     // warps: 2 NPIPE producers, NPIPE MMA issuers, then the epilogue groups
// (each issuing thread has a warp of its own: issuing lanes that share a warp diverge and run one after another)
constexpr int NGRP = NPIPE;              // epilogue groups of 4 warps; group j drains pipeline j
constexpr int QN = 16;                   // unit-id queue entries per pipeline
constexpr int ABUF_MAX = 4;              // accumulators per pipeline
constexpr int THREADS = (EPI_WARP0 + 4 * NGRP) * 32;
constexpr uint32_t TMEM_COLS = 512;      // accumulators: pipeline j, buffer a at W (j ABUF + a); scales from 384
constexpr uint32_t SF_COL0 = 384;
static_assert(128 * NPIPE <= (int)SF_COL0 && SF_COL0 + 8 * NSLOT <= TMEM_COLS, "TMEM budget");
// Every gate/up unit of CTA b covers the same K segment (b mod S_G: the grid is a multiple of S_G), so the CTA keeps
// that segment's x parts resident: 8 k-tiles x 48 rows x 64 B in the 64-byte-swizzled MMA layout, and their
// exponent blocks.
constexpr int XRES_TILE = NB * 64;       // 3 KB per k-tile
constexpr int XRES_BYTES = 8 * XRES_TILE + 8 * 512;
constexpr int SMEM = NSLOT * SLOT_BYTES + XRES_BYTES + 1024;

// ------------------------------------------------------------------ geometry of one call
struct Geo {
  int H, I, T, k, U;
  int RTG, KTG, KSG, SG;   // gate/up: row tiles, k-tiles, k-tiles per unit, segments
  int RTD, KTD, KSD, SD;   // down
  int nG, nD;              // units
  int W, ABUF;             // accumulator width = MMA N (16 ceil(6 T / 16): a column per part and token, in 16s;
                           // each column is computed on its own, whatever N is) and accumulators per pipeline
};
// k-tiles per unit: gate/up 8 (or 4, 2), down 4 (or 2) -- shorter down units shorten the tail after the last h
__host__ __device__ inline int ks_for_g(int kt) { return kt % 8 == 0 ? 8 : (kt % 4 == 0 ? 4 : 2); }
__host__ __device__ inline int ks_for_d(int kt) { return kt % 4 == 0 ? 4 : 2; }

// ------------------------------------------------------------------ workspace (byte offsets from the base)
// [0, 256)       WsHeader (status word)
// [256, ...)     counters (uint32): (unused), done, h_ready[64][16] (per expert and down K segment),
//                g_cnt[64 * 64] (per expert and gate/up row tile), d_cnt[32] (per down row tile)
// then hb [Umax * 48][I/2] packed E2M1 h parts, hsf [Umax][I/128][512] their exponents,
//      gpart [Umax][2I/128][S_G][TS][128] fp32, dpart [Umax][H/128][S_D][TS][128] fp32
// with Umax = T_max * k union experts and TS = T_max token columns of the partial buffers.
constexpr int64_t kCnt = 256;
constexpr int C_DONE = 1, C_HREADY = 2, C_G = C_HREADY + MAX_U * 16, C_D = C_G + MAX_U * 64;
constexpr int C_ROUTE = C_D + 32;      // experts whose logits are in (routing inside the kernel)
constexpr int C_XP = C_ROUTE + 1;        // 32-blocks of x split into the x-part image
constexpr int C_END = C_XP + 1;
struct Ws {
  int64_t hb, hsf, gpart, dpart, lg, xp, total;
};
inline int64_t al1k(int64_t v) { return (v + 1023) & ~(int64_t)1023; }
inline Ws ws_layout(int64_t H, int64_t I, int64_t Umax, int64_t TS) {
  Ws w;
  int64_t o = al1k(kCnt + (int64_t)C_END * 4);
  const int64_t RTG = 2 * I / 128, KTG = H / 128, RTD = H / 128, KTD = I / 128;
  const int64_t SG = KTG / ks_for_g((int)KTG), SD = KTD / ks_for_d((int)KTD);
  w.hb = o;    o = al1k(o + Umax * HROWS * I / 2);
  w.hsf = o;   o = al1k(o + Umax * KTD * 512);
  w.gpart = o; o = al1k(o + Umax * RTG * SG * TS * 128 * 4);
  w.dpart = o; o = al1k(o + Umax * RTD * SD * TS * 128 * 4);
  w.lg = o;    o = al1k(o + (int64_t)kRouteTPC * 2 * kRouteMaxE * 4);  // router logit halves [token][half][expert]
  w.xp = o;    o = al1k(o + (H / 128) * (XRES_TILE + 512));      // x parts: [k-tile][48 rows][64 B], then exponents
  w.total = o;
  return w;
}

struct Args {
  const uint8_t* gu;          // gate/up weights (tensor-core layout)
  const uint8_t* dn;          // down weights
  int64_t gu_stride, dn_stride;
  const uint16_t* x;          // [T][H] bf16
  const int32_t* idx;         // [T][k] (routing given), or
  const float* w;             // [T][k]
  const uint16_t* wr;         // [E][H] fp16 router: route inside the kernel, writing idx_out / w_out
  int32_t* idx_out;
  float* w_out;
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
// Exponent of an E2M1 block: e = clamp(k + 127, 1, 254), k the smallest integer with amax <= 6 * 2^k.
__device__ __forceinline__ int mx4_exp(float amax) {
  const uint32_t ab = __float_as_uint(amax) & 0x7FFFFFFFu;
  const int ef = (int)(ab >> 23);
  if (ef == 0) return 1;
  const int e = ef - 2 + ((ab & 0x7FFFFFu) > 0x400000u ? 1 : 0);
  return e < 1 ? 1 : (e > 254 ? 254 : e);
}
__device__ __forceinline__ float pow2_127m(int e) {  // 2^(127 - e), e in [1, 254]
  return e <= 253 ? __uint_as_float((uint32_t)(254 - e) << 23) : __uint_as_float(0x00400000u);
}
__device__ __forceinline__ float pow2_m127(int e) {  // 2^(e - 127), e in [1, 254]
  return __uint_as_float((uint32_t)e << 23);
}
// E2M1 code of v (round to nearest even, saturating to +-6) in the low nibble
__device__ __forceinline__ uint32_t e2m1_code(float v) {
  uint16_t d;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}" : "=h"(d) : "f"(0.0f), "f"(v));
  return d & 15u;
}
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const float mag = (c & 4) ? ((c & 2) ? ((c & 1) ? 6.f : 4.f) : ((c & 1) ? 3.f : 2.f))
                            : (float)(c & 3) * 0.5f;
  return (c & 8) ? -mag : mag;
}
__device__ __forceinline__ float warp_amax(float v) {
  const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(v)));
  return __uint_as_float(m);
}
// Split v (lane l holds element l of a 32-block) into PARTS E2M1 parts: part 0 uses the block exponent e0 (largest
// magnitude <= 6 * 2^(e0 - 127)); part p uses e0 - 2p (clamped at 1) and quantises what parts 0 .. p-1 left. After
// a part the remainder is at most half an E2M1 step, <= 1 unit of its scale = 4 units of the next part's, so no
// part saturates and each adds at least 2 bits: the final error is below 2^-10 of part 0's scale, i.e. below
// 1/3072 of the block's largest magnitude. Only e0 needs a warp reduction. Even lanes get the packed byte of
// elements (l, l + 1) of each part in bytes[p] (element l in the low nibble). A block holding NaN or infinity has
// no E2M1 encoding: every part gets the E8M0 NaN exponent (255), which the block-scaled MMA turns into NaN.
// live[q] must be the same for every lane of the warp (the parts of a dead block are skipped by all lanes).
template <int NV>
__device__ __forceinline__ void split_parts_n(const float (&v)[NV], const bool (&live)[NV], uint32_t (&bytes)[NV][PARTS],
                                              int (&exps)[NV][PARTS]) {
  const int lane = threadIdx.x & 31;
  float r[NV], am[NV];
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    r[q] = v[q];
    const float m = warp_amax(live[q] ? v[q] : 0.f);  // every lane takes part in the reduction
    am[q] = live[q] ? m : 0.f;
  }
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    if (!live[q]) continue;
    const bool nonfinite = !(am[q] <= 3.4028235e38f);
    const int e0 = mx4_exp(am[q]);
#pragma unroll
    for (int p = 0; p < PARTS; ++p) {
      const int e = nonfinite ? 255 : (e0 - 2 * p > 1 ? e0 - 2 * p : 1);
      const uint32_t c = nonfinite ? 0u : e2m1_code(r[q] * pow2_127m(e));
      const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, c, 1);
      bytes[q][p] = (lane & 1) ? 0u : (c | (hi << 4));
      exps[q][p] = e;
      if (!nonfinite) r[q] = r[q] - e2m1_value(c) * pow2_m127(e);
    }
  }
}
__device__ __forceinline__ void split_parts(float v, uint32_t (&bytes)[PARTS], int (&exps)[PARTS]) {
  const float vv[1] = {v};
  const bool live[1] = {true};
  uint32_t b[1][PARTS];
  int e[1][PARTS];
  split_parts_n<1>(vv, live, b, e);
#pragma unroll
  for (int p = 0; p < PARTS; ++p) { bytes[p] = b[0][p]; exps[p] = e[0][p]; }
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
// Spinning threads back off briefly between polls so that warps doing arithmetic on the same SM keep their issue
// slots.
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, long long lim) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = globaltimer_ns();
  while (true) {
    __nanosleep(20);
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
// Global order of the work: blocks of units G(u) (all row tiles and segments of expert u's gate/up) and D(u); D(u)
// is placed after G(u + LAG). With LAG = MAX_U every G block comes first (G0 .. G(U-1) D0 .. D(U-1)), which measured
// best: a D block placed earlier waits for h of its expert while holding a pipeline.
constexpr int LAG = MAX_U;
struct Order {
  int n;                       // blocks
  int start[2 * MAX_U + 1];    // first unit of each block; start[n] = total units
  int8_t d[2 * MAX_U], u[2 * MAX_U];
};
// Blocks of the global unit order: G(0) .. G(U-1) then D(0) .. D(U-1) (every gate/up unit first: a down block
// placed earlier waits for h of its expert while holding a pipeline). Built by one warp, a block per lane.
static_assert(LAG == MAX_U, "the unit order puts every gate/up block first");
__device__ void build_order_warp(Order& o, const Geo& g, int U) {
  const int lane = threadIdx.x & 31;
  const int nGu = g.RTG * g.SG, nDu = g.RTD * g.SD;
  for (int b = lane; b < 2 * U; b += 32) {
    const bool d = b >= U;
    o.start[b] = d ? U * nGu + (b - U) * nDu : b * nGu;
    o.d[b] = (int8_t)d;
    o.u[b] = (int8_t)(d ? b - U : b);
  }
  if (lane == 0) {
    o.start[2 * U] = U * (nGu + nDu);
    o.n = 2 * U;
  }
}
__device__ __forceinline__ Unit unit_of(int v, const Geo& g, const Order& o) {
  int lo = 0, hi = o.n - 1;  // last block with start <= v
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (o.start[mid] <= v) lo = mid; else hi = mid - 1;
  }
  Unit r;
  r.d = o.d[lo];
  r.u = o.u[lo];
  const int rr = v - o.start[lo], S = r.d ? g.SD : g.SG;
  r.rt = rr / S;
  r.ks = rr % S;
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
  float w[MAX_T][MAX_K];     // routing weights
  int U;
  int bad;
};

// Built in two steps so that the weight stream starts as early as possible.
// (1) build_union_warp, one warp: the union of the experts in first-appearance order over (t, r) and whether any id
//     is out of range (match_any / ballot over the T k <= 64 entries, two per lane; no dependent memory chains).
__device__ void build_union_warp(Tables& tb, const int32_t (*idx)[MAX_K], int T, int k, int E) {
  const int lane = threadIdx.x & 31;
  const int n = T * k;
  const bool v0 = lane < n, v1 = lane + 32 < n;
  const int e0 = v0 ? idx[lane / k][lane % k] : 0, e1 = v1 ? idx[(lane + 32) / k][(lane + 32) % k] : 0;
  const bool bad = __any_sync(0xFFFFFFFFu, (v0 && (e0 < 0 || e0 >= E)) || (v1 && (e1 < 0 || e1 >= E)));
  const int key0 = v0 ? e0 : -1 - lane, key1 = v1 ? e1 : -33 - lane;  // absent entries never match
  const uint32_t lt = (1u << lane) - 1u;
  // every lane takes part in each warp-wide operation (none sits inside a short-circuit or a branch)
  const uint32_t m0 = __match_any_sync(0xFFFFFFFFu, key0), m1 = __match_any_sync(0xFFFFFFFFu, key1);
  bool in0 = false;  // entry lane + 32 already appeared among entries 0 .. 31
  for (int q = 0; q < 32; ++q) in0 |= __shfl_sync(0xFFFFFFFFu, key0, q) == key1;
  const bool first0 = v0 && (m0 & lt) == 0;
  const bool first1 = v1 && !in0 && (m1 & lt) == 0;
  const uint32_t b0 = __ballot_sync(0xFFFFFFFFu, first0), b1 = __ballot_sync(0xFFFFFFFFu, first1);
  if (first0) tb.ue[__popc(b0 & lt)] = e0;
  if (first1) tb.ue[__popc(b0) + __popc(b1 & lt)] = e1;
  if (lane == 0) {
    tb.U = __popc(b0) + __popc(b1);
    tb.bad = bad ? 1 : 0;
  }
}
// (2) build_slots, one thread, while the first weight tiles are in flight: the routing weights, each union expert's
//     tokens (slot order = token order) and, per (t, r), the union index and the token's slot in that expert.
__device__ void build_slots(Tables& tb, const int32_t (*idx)[MAX_K], const float (*w)[MAX_K], int T, int k) {
  for (int u = 0; u < tb.U; ++u) tb.ntok[u] = 0;
  for (int t = 0; t < T; ++t)
    for (int r = 0; r < k; ++r) {
      tb.w[t][r] = w[t][r];
      const int e = idx[t][r];
      int u = 0;
      while (u < tb.U && tb.ue[u] != e) ++u;
      if (u == tb.U) { tb.pu[t][r] = 0; tb.ps[t][r] = 0; continue; }  // an invalid id (no units run)
      int s = 0;
      while (s < tb.ntok[u] && tb.tok[u][s] != t) ++s;
      if (s == tb.ntok[u]) { tb.tok[u][s] = (int8_t)t; tb.ntok[u] = (int8_t)(s + 1); }
      tb.pu[t][r] = (int8_t)u;
      tb.ps[t][r] = (int8_t)s;
    }
}

// The x parts, split once per call: 32-block j = (token t, k-tile kt, block kb) of x goes to warp j of the grid's
// epilogue warps (warp ew of CTA b is number 12 b + ew), which splits it into PARTS E2M1 parts (split_parts_n) and
// writes them into the x-part image in the workspace: k-tile kt at xp + kt * XRES_TILE, row PARTS * t + p, 64 bytes
// a row, 16-byte chunks in the 64-byte TMA swizzle (chunk c of row r at chunk c ^ ((r >> 1) & 3)) -- the resident
// B operand as it sits in shared memory -- and the exponents into the permuted blocks at xp + KTG XRES_TILE + 512 kt.
// Each CTA then copies its K segment's tiles in with two bulk copies.
__device__ __forceinline__ float load_x_block(const Args& a, const Geo& g, int j) {
  const int lane = threadIdx.x & 31;
  if (j >= g.T * g.KTG * 4) return 0.f;
  const int t = j / (g.KTG * 4), rem = j % (g.KTG * 4);
  return __uint_as_float((uint32_t)a.x[(int64_t)t * g.H + rem * 32 + lane] << 16);
}
__device__ void split_x_global(const Args& a, const Geo& g, int gw, int nwarps, float xfirst) {
  const int lane = threadIdx.x & 31;
  const int nblk = g.T * g.KTG * 4;
  uint8_t* xp = a.ws + a.L.xp;
  uint8_t* xpsf = xp + (int64_t)g.KTG * XRES_TILE;
  for (int j = gw; j < nblk; j += nwarps) {
    float r = j == gw ? xfirst : load_x_block(a, g, j);
    const int t = j / (g.KTG * 4), rem = j % (g.KTG * 4), kt = rem / 4, kb = rem % 4;
    const float am = warp_amax(r);
    const bool nonfinite = !(am <= 3.4028235e38f);
    const int e0 = mx4_exp(am);
#pragma unroll
    for (int p = 0; p < PARTS; ++p) {
      const int e = nonfinite ? 255 : (e0 - 2 * p > 1 ? e0 - 2 * p : 1);
      const uint32_t c = nonfinite ? 0u : e2m1_code(r * pow2_127m(e));
      const uint32_t byte = c | (__shfl_down_sync(0xFFFFFFFFu, c, 1) << 4);  // elements (l, l + 1), even l
      if (!nonfinite) r = r - e2m1_value(c) * pow2_m127(e);
      // the 16 bytes of the part gathered into four words: word w from the even lanes 8 w .. 8 w + 6
      uint32_t word = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) word |= (__shfl_sync(0xFFFFFFFFu, byte, (lane & ~7) + 2 * i) & 0xFFu) << (8 * i);
      const int n = PARTS * t + p;
      if ((lane & 7) == 0)
        *reinterpret_cast<uint32_t*>(xp + (int64_t)kt * XRES_TILE + n * 64 + ((kb ^ ((n >> 1) & 3)) << 4) + (lane >> 1)) = word;
      if (lane == 0) xpsf[kt * 512 + sfb(n, kb)] = (uint8_t)e;
    }
    __syncwarp();
    if (lane == 0) red_release_add(reinterpret_cast<uint32_t*>(a.ws + kCnt) + C_XP, 1u);
  }
}

// All G segments of (expert u, row tile rt) are in: g, u of the 64 intermediate indices rt*64 .. +63 (tile rows
// 0..63 gate, 64..127 up), h = SiLU(g) * u, PARTS E2M1 parts per 32-block into the D operand rows PARTS * s + p.
// The group's 128 threads take the token slots two at a time.
__device__ void finalize_h(const Args& a, const Geo& g, const Tables& tb, int u, int rt, int et) {
  // thread et: row et % 64 of the tile (a warp = one 32-block), token slots et / 64, et / 64 + 2, ...
  const int row = et & 63, lane = threadIdx.x & 31;
  const float* gp = reinterpret_cast<const float*>(a.ws + a.L.gpart) + ((int64_t)u * g.RTG + rt) * g.SG * a.ts * 128;
  const int i = rt * 64 + row, kt = i / 128, kb = (i % 128) / 32;
  uint8_t* hb = a.ws + a.L.hb + (int64_t)u * HROWS * (g.I / 2);
  uint8_t* hsf = a.ws + a.L.hsf + ((int64_t)u * g.KTD + kt) * 512;
  const int nt = tb.ntok[u];
  for (int s = et >> 6; s < nt; s += 2) {
    const int t = tb.tok[u][s];
    float gv = 0.f, uv = 0.f;
    for (int k0 = 0; k0 < g.SG; k0 += 4) {  // segments in order, loads issued four at a time
      float gl[4], ul[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (k0 + q < g.SG) {
          gl[q] = __ldcg(gp + ((int64_t)(k0 + q) * a.ts + t) * 128 + row);
          ul[q] = __ldcg(gp + ((int64_t)(k0 + q) * a.ts + t) * 128 + 64 + row);
        }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (k0 + q < g.SG) { gv += gl[q]; uv += ul[q]; }
    }
    const float h = gv / (1.0f + expf(-gv)) * uv;
    uint32_t c[PARTS];
    int ex[PARTS];
    split_parts(h, c, ex);
#pragma unroll
    for (int p = 0; p < PARTS; ++p) {
      if (!(lane & 1)) hb[(int64_t)(PARTS * s + p) * (g.I / 2) + i / 2] = (uint8_t)c[p];
      if (lane == 0) hsf[sfb(PARTS * s + p, kb)] = (uint8_t)ex[p];
    }
  }
}

// All D units of row tile jt are in: y[t][jt*128 + et] = sum_r w[t, r] * (sum over segments of the partial of
// (expert of rank r, token t)), ranks in order.
__device__ void combine_rows(const Args& a, const Geo& g, const Tables& tb, int jt, int et) {
  const float* dp = reinterpret_cast<const float*>(a.ws + a.L.dpart);
  const int j = jt * 128 + et;
  for (int t = 0; t < g.T; ++t) {
    // the partials of every (rank, segment) of the token are loaded before the sums (segments in order per rank,
    // then ranks in order), four segments at a time
    float sum[MAX_K];
#pragma unroll
    for (int r = 0; r < MAX_K; ++r) sum[r] = 0.f;
    for (int k0 = 0; k0 < g.SD; k0 += 4) {
      float pl[MAX_K][4];
#pragma unroll
      for (int r = 0; r < MAX_K; ++r) {
        if (r < g.k) {
          const float* p = dp + (((int64_t)tb.pu[t][r] * g.RTD + jt) * g.SD * a.ts + tb.ps[t][r]) * 128 + et;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (k0 + q < g.SD) pl[r][q] = __ldcg(p + (int64_t)(k0 + q) * a.ts * 128);
        }
      }
#pragma unroll
      for (int r = 0; r < MAX_K; ++r)
        if (r < g.k)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (k0 + q < g.SD) sum[r] += pl[r][q];
    }
    float acc = 0.f;
#pragma unroll
    for (int r = 0; r < MAX_K; ++r)
      if (r < g.k) acc = fmaf(tb.w[t][r], sum[r], acc);
    float* yp = a.y + (int64_t)t * g.H + j;
    const float out = a.accumulate ? *yp + acc : acc;
    *yp = out;
    if (a.yb) a.yb[(int64_t)t * g.H + j] = __float2bfloat16_rn(out);
  }
}

__device__ void epilogue(const Args& a, const Geo& g, const Tables& tb, const Order& ord, uint32_t tbase,
                         uint64_t (*acc_full)[ABUF_MAX], uint64_t (*acc_empty)[ABUF_MAX], uint64_t (*uq_full)[QN], volatile int (*uq)[QN], uint32_t* cnt,
                         volatile int* s_last, volatile int* s_ok, volatile int* s_unit, volatile int* s_abort) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, q = warp & 3;
  const int grp = (warp - EPI_WARP0) / 4;
  const int bar = 1 + grp;                                      // named barrier of the group
  const int et = threadIdx.x - (EPI_WARP0 + 4 * grp) * 32;       // 0..127 inside the group
  const int m = q * 32 + lane;                                   // TMEM lane = weight row of the tile
  const long long lim = a.wait_ns;
  float* gpart = reinterpret_cast<float*>(a.ws + a.L.gpart);
  float* dpart = reinterpret_cast<float*>(a.ws + a.L.dpart);
  // the units pipeline j = grp took, in order (each accumulator's phases in order)
  const int j = grp;
  for (int c = 0;; ++c) {
    const int ab = c % g.ABUF;
    // one thread waits; the verdict is shared so that the group's four warps leave (or stay) together
    if (et == 0) {
      int st = 0;
      if (bwait(&uq_full[j][c % QN], (uint32_t)((c / QN) & 1), s_abort, lim)) {
        const int i = uq[j][c % QN];
        if (i < 0) st = 2;
        else { s_unit[grp] = i; st = bwait(&acc_full[j][ab], (uint32_t)((c / g.ABUF) & 1), s_abort, lim) ? 1 : 0; }
      }
      s_ok[grp] = st;
    }
    named_bar(bar, 128);
    if (s_ok[grp] != 1) break;
    tc_fence_after();
    const int i = s_unit[grp];
    const Unit un = unit_of((int)blockIdx.x + i * (int)gridDim.x, g, ord);
    const uint32_t taddr = tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(g.W * (j * g.ABUF + ab));
    // column t * PARTS + p = part p of token (or slot) t; sum the parts of each column group in part order
    float acc[MAX_T];
#pragma unroll
    for (int t = 0; t < MAX_T; ++t) acc[t] = 0.f;
#pragma unroll
    for (int cb = 0; cb < NB / 16; ++cb) {
      if (16 * cb >= g.W) break;
      uint32_t v[16];
      tc_ld16(taddr + 16 * cb, v);
      tc_wait_ld();
#pragma unroll
      for (int c = 0; c < 16; ++c) acc[(16 * cb + c) / PARTS] += __uint_as_float(v[c]);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_relaxed(&acc_empty[j][ab]);  // TMEM read; no wait for the earlier global stores
    if (!un.d) {
      float* gp = gpart + (((int64_t)un.u * g.RTG + un.rt) * g.SG + un.ks) * a.ts * 128 + m;
#pragma unroll
      for (int t = 0; t < MAX_T; ++t)
        if (t < g.T) gp[t * 128] = acc[t];
    } else {
      float* dp = dpart + (((int64_t)un.u * g.RTD + un.rt) * g.SD + un.ks) * a.ts * 128 + m;
      const int nt = tb.ntok[un.u];
#pragma unroll
      for (int s = 0; s < MAX_T; ++s)
        if (s < nt) dp[s * 128] = acc[s];
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
        if (et == 0) red_release_add(cnt + C_HREADY + un.u * 16 + (un.rt * 64) / (128 * g.KSD), 1u);
      } else {
        combine_rows(a, g, tb, un.rt, et);
      }
    }
  }
}

__global__ void __launch_bounds__(THREADS, 1) decode_kernel(const __grid_constant__ CUtensorMap tm_gu,
                                                            const __grid_constant__ CUtensorMap tm_dn,
                                                            const __grid_constant__ CUtensorMap tm_h, const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ __align__(8) uint64_t full[NSLOT], empty[NSLOT], acc_full[NPIPE][ABUF_MAX],
      acc_empty[NPIPE][ABUF_MAX], drain[NPIPE];
  __shared__ __align__(8) uint64_t uq_full[NPIPE][QN], xres_full, tab_full, tab2_full;
  uint8_t* xres = smem + NSLOT * SLOT_BYTES;    // resident x parts of this CTA's gate/up K segment
  uint8_t* xres_sf = xres + 8 * XRES_TILE;
  __shared__ volatile int uq[NPIPE][QN];
  __shared__ int s_next;
  __shared__ Tables tb;
  __shared__ Order ord;
  __shared__ uint32_t s_tmem;
  __shared__ int s_units;
  __shared__ volatile int s_abort, s_ok[NGRP], s_last[NGRP], s_unit[NGRP];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(a.ws + kCnt);
  Geo g = a.g;
  const long long lim = a.wait_ns;
  const int xwarp = (int)blockIdx.x * (4 * NGRP) + (warp - EPI_WARP0), nxwarps = (int)gridDim.x * (4 * NGRP);
  const float xfirst = warp >= EPI_WARP0 ? load_x_block(a, g, xwarp) : 0.f;  // before the weight stream starts

  float* lgw = reinterpret_cast<float*>(a.ws + a.L.lg);  // router logit halves [token][half][expert]
  if (a.wr && warp >= 2 && warp < 2 + 2 * NPIPE) {
    // routing, phase 1 (at entry, while thread 0 and warp 1 set the CTA up): the logit halves (expert e, half c),
    // task q = blockIdx.x + gridDim.x * (w + 2 NPIPE i), e = q / 2, c = q % 2, w = warp - 2, spread over the grid
    for (int q = (int)blockIdx.x + (int)gridDim.x * (warp - 2); q < 2 * a.E; q += (int)gridDim.x * 2 * NPIPE) {
      const int e = q >> 1, c = q & 1;
      float acc[kRouteTPC];
      route_half_logits<8>(a.wr + (size_t)e * g.H, g.H, g.T, [&](int t) { return a.x + (size_t)t * g.H; }, c, acc);
      if (lane == 0)
        for (int t = 0; t < g.T; ++t) __stcg(lgw + (t * 2 + c) * a.E + e, acc[t]);
      __syncwarp();
      if (lane == 0) red_release_add(cnt + C_ROUTE, 1u);
    }
  }
  __shared__ int32_t s_idx[MAX_T][MAX_K];
  __shared__ float s_wt[MAX_T][MAX_K];
  if (threadIdx.x == 0) {
    for (int s = 0; s < NSLOT; ++s) { mbar_init(&full[s], 2); mbar_init(&empty[s], 1); }  // full: both producers arrive
    for (int j = 0; j < NPIPE; ++j) {
      for (int b = 0; b < ABUF_MAX; ++b) {
        mbar_init(&acc_full[j][b], 1);
        mbar_init(&acc_empty[j][b], 4);  // the 4 warps of one epilogue group
      }
      mbar_init(&drain[j], 1);
      for (int e = 0; e < QN; ++e) mbar_init(&uq_full[j][e], 1);
    }
    mbar_init(&xres_full, 1);
    mbar_init(&tab_full, 1);
    mbar_init(&tab2_full, 1);
    s_abort = 0;
    s_next = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc_alloc(&s_tmem, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = s_tmem;
  if (warp >= EPI_WARP0) {
    // this CTA's share of the x parts (independent of the routing), while the other warps route and build the
    // tables; once every share is in, one thread copies the CTA's K segment of the image into the resident
    // operand; then wait for the tables
    split_x_global(a, g, xwarp, nxwarps, xfirst);
    if (warp == EPI_WARP0) {  // (the other lanes wait at the warp barrier, not spinning beside lane 0)
      if (lane == 0) {
        if (wait_ge(cnt + C_XP, (uint32_t)(g.T * g.KTG * 4), &s_abort, lim)) {
          asm volatile("fence.proxy.async.global;" ::: "memory");  // generic-proxy writes -> bulk-copy reads
          const int ks0 = (int)blockIdx.x % g.SG;
          const uint8_t* xp = a.ws + a.L.xp;
          mbar_arrive_expect_tx(&xres_full, (uint32_t)(g.KSG * (XRES_TILE + 512)));
          bulk_g2s_plain(xres, xp + (int64_t)ks0 * g.KSG * XRES_TILE, (uint32_t)(g.KSG * XRES_TILE), &xres_full);
          bulk_g2s_plain(xres_sf, xp + (int64_t)g.KTG * XRES_TILE + ks0 * g.KSG * 512, (uint32_t)(g.KSG * 512),
                         &xres_full);
        } else {
          record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
        }
      }
      __syncwarp();
    }
    if (!bwait(&tab_full, 0, &s_abort, lim) && threadIdx.x == EPI_WARP0 * 32) record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
    if (warp == EPI_WARP0) {  // the token tables the epilogues need, while the first tiles stream in
      if (lane == 0) {
        build_slots(tb, s_idx, s_wt, g.T, g.k);
        mbar_arrive(&tab2_full);
      }
      __syncwarp();
    }
    if (!bwait(&tab2_full, 0, &s_abort, lim) && threadIdx.x == EPI_WARP0 * 32) record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
  } else {
    if (a.wr) {
      // routing, phase 2: every CTA selects each token's experts from all the logits (one warp per token)
      if (warp < g.T) {
        bool ok = true;
        if (lane == 0) ok = wait_ge(cnt + C_ROUTE, (uint32_t)(2 * a.E), &s_abort, lim);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        int sid[8];
        float sw[8];
        if (ok) {
          const float* row = lgw + warp * 2 * a.E;  // half 0, then half 1, of every expert's logit
          route_topk_warp<kRouteMaxE / 32 / 4>([&](int e) { return __ldcg(row + e) + __ldcg(row + a.E + e); }, a.E, g.k,
                                               sid, sw);
        }
        if (lane == 0)
          for (int r = 0; r < g.k; ++r) {
            s_idx[warp][r] = ok ? sid[r] : -1;
            s_wt[warp][r] = ok ? sw[r] : 0.f;
            if (blockIdx.x == 0 && ok) {
              a.idx_out[warp * g.k + r] = sid[r];
              a.w_out[warp * g.k + r] = sw[r];
            }
          }
      }
    } else if (threadIdx.x < g.T * g.k) {
      s_idx[threadIdx.x / g.k][threadIdx.x % g.k] = a.idx[threadIdx.x];
      s_wt[threadIdx.x / g.k][threadIdx.x % g.k] = a.w[threadIdx.x];
    }
    named_bar(2 + NGRP, EPI_WARP0 * 32);
    if (warp == 0) {
      build_union_warp(tb, s_idx, g.T, g.k, a.E);
      __syncwarp();
      const int U = tb.bad ? 0 : tb.U;
      build_order_warp(ord, g, U);
      __syncwarp();
      if (lane == 0) {
        // an expert id out of range: no units (every role finds an empty queue), status MOE_ERR_INVALID_ARG
        if (tb.bad && blockIdx.x == 0) record_error(&hdr->status, MOE_ERR_INVALID_ARG);
        s_units = U * (g.RTG * g.SG + g.RTD * g.SD);
        mbar_arrive(&tab_full);
      }
    }
    named_bar(2 + NGRP, EPI_WARP0 * 32);
  }
  g.U = tb.U;
  g.nG = g.U * g.RTG * g.SG;
  g.nD = g.U * g.RTD * g.SD;
  const int nunits = s_units;
  if (nunits == 0) g.nG = g.nD = 0;
  // this CTA's units: v = blockIdx.x + i * gridDim.x, i = 0 .. my_units - 1 (G units first). Pipelines take the
  // next i from a shared counter when they start a unit, so a pipeline waiting for h does not hold up the rest;
  // each publishes the ids it took through its queue uq[j] to its MMA thread and epilogue group.
  const int my_units = nunits > (int)blockIdx.x ? (nunits - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;

  if (warp < 2 * NPIPE) {
    // ---------------- producers, two warps per pipeline j (lane 0 issues): warp j streams the weight tiles of
    // every stage (no dependency, so weights keep flowing while activations are not ready), warp NPIPE + j adds
    // the activation parts of each stage once they exist (x split done; h of the expert finalised). Each posts its
    // own byte count on the stage's barrier.
    const bool wprod = warp < NPIPE;
    const int j = wprod ? warp : warp - NPIPE;
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int n = 0;  // stages of this pipeline
      bool ok = true;
      int h_ok_u = -1;
      for (int c = 0; ok; ++c) {
        int i;
        if (wprod) {
          i = atomicAdd(&s_next, 1);
          // entry c % QN was last read for unit c - QN: the weight producer is at most RING stages ahead of the
          // MMA, so (units having at least 2 stages) the MMA has started unit c - 3 and the epilogue group has
          // finished unit c - 3 - ABUF >= c - 7 > c - QN; the activation producer is ahead of the MMA
          uq[j][c % QN] = i < my_units ? i : -1;
          mbar_arrive(&uq_full[j][c % QN]);
        } else {
          if (!bwait(&uq_full[j][c % QN], (uint32_t)((c / QN) & 1), &s_abort, lim)) { ok = false; break; }
          i = uq[j][c % QN];
        }
        if (i < 0 || i >= my_units) break;
        const Unit un = unit_of((int)blockIdx.x + i * (int)gridDim.x, g, ord);
        const int e = tb.ue[un.u];
        const int ks = un.d ? g.KSD : g.KSG;
        const int KT = un.d ? g.KTD : g.KTG;
        if (!wprod && un.d && h_ok_u != un.u * 16 + un.ks) {  // down: wait once for h of its K segment
          const uint32_t* dep_cnt = cnt + C_HREADY + un.u * 16 + un.ks;
          if (!wait_ge(dep_cnt, (uint32_t)(2 * g.KSD), &s_abort, lim)) { ok = false; break; }
          asm volatile("fence.proxy.async.global;" ::: "memory");  // generic-proxy writes -> TMA reads
          h_ok_u = un.u * 16 + un.ks;
        }
        for (int kk = 0; kk < ks; ++kk, ++n) {
          const int slot = j * RING + (n % RING);
          const uint32_t ph = (uint32_t)((n / RING) & 1);
          if (!bwait(&empty[slot], ph ^ 1, &s_abort, lim)) { ok = false; break; }
          uint8_t* st = smem + slot * SLOT_BYTES;
          const int kt = un.ks * ks + kk;
          if (wprod) {
            const int tile = un.rt * KT + kt;
            const uint8_t* wbase = un.d ? a.dn + (int64_t)e * a.dn_stride : a.gu + (int64_t)e * a.gu_stride;
            // weights are read once per call: evict-first keeps them from displacing the instructions, partial
            // sums and activation parts that the dependent steps read back through L2
            mbar_arrive_expect_tx(&full[slot], A_BYTES + 512);
            tma_load_4d_hint(st, un.d ? &tm_dn : &tm_gu, 0, 0, tile, e, &full[slot], pol);
            bulk_g2s(st + A_BYTES + B_BYTES, wbase + (int64_t)tile * kTcTileBytes + 8192, 512, &full[slot], pol);
          } else if (!un.d) {
            mbar_arrive(&full[slot]);  // gate/up: the x parts are resident; nothing to copy
          } else {
            mbar_arrive_expect_tx(&full[slot], B_BYTES + 512);
            tma_load_2d(st + A_BYTES, &tm_h, kt * 64, un.u * HROWS, &full[slot]);
            bulk_g2s_plain(st + A_BYTES + B_BYTES + 512, a.ws + a.L.hsf + ((int64_t)un.u * g.KTD + kt) * 512, 512,
                           &full[slot]);
          }
        }
      }
      if (!ok) {
        record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
        // a stage may hold the copies of one producer only, so its barrier never completes: give the copies this
        // warp issued 1 ms to land before the CTA's shared memory is released
        const long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000LL) __nanosleep(1000);
      }
    }
    __syncwarp();
  } else if (warp < 3 * NPIPE) {
    // ---------------- MMA issuers: lane 0 of warp 2 NPIPE + j, pipeline j
    const int j = warp - 2 * NPIPE;
    if (lane == 0) {
      int n = 0, c = 0;
      bool ok = true, xres_ok = false;
      const uint32_t sfa_col = tbase + SF_COL0;
      for (;; ++c) {
        if (!bwait(&uq_full[j][c % QN], (uint32_t)((c / QN) & 1), &s_abort, lim)) { ok = false; break; }
        const int i = uq[j][c % QN];
        if (i < 0) break;
        const Unit un = unit_of((int)blockIdx.x + i * (int)gridDim.x, g, ord);
        const int ab = c % g.ABUF;
        if (!bwait(&acc_empty[j][ab], ((c / g.ABUF) & 1) ^ 1, &s_abort, lim)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tbase + (uint32_t)(g.W * (j * g.ABUF + ab));
        const int ks = un.d ? g.KSD : g.KSG;
        if (!un.d && !xres_ok) {  // the resident x parts (built by the epilogue warps at start)
          if (!bwait(&xres_full, 0, &s_abort, lim)) { ok = false; break; }
          xres_ok = true;
        }
        for (int kk = 0; kk < ks; ++kk, ++n) {
          const int slot = j * RING + (n % RING);
          if (!bwait(&full[slot], (uint32_t)((n / RING) & 1), &s_abort, lim)) { ok = false; break; }
          tc_fence_after();
          uint8_t* st = smem + slot * SLOT_BYTES;
          const uint32_t sfa = sfa_col + (uint32_t)(slot * 8), sfbc = sfa + 4;
          // B: gate/up from the resident x parts (k-tile kk of the CTA's segment), down from the stage
          const uint8_t* bsrc = un.d ? st + A_BYTES : xres + kk * XRES_TILE;
          const uint8_t* bsf = un.d ? st + A_BYTES + B_BYTES + 512 : xres_sf + kk * 512;
          tc_cp_sf(sfa, umma_desc_sf(smem_u32(st + A_BYTES + B_BYTES)));
          tc_cp_sf(sfbc, umma_desc_sf(smem_u32(bsf)));
          const uint64_t ad = umma_desc_sw64(smem_u32(st)), bd = umma_desc_sw64(smem_u32(bsrc));
#pragma unroll
          for (int kh = 0; kh < 2; ++kh)  // two K = 64 halves of the 128-column tile, scale bytes 2kh, 2kh + 1
            tc_mma_mxf4(d_tmem, ad + 2 * kh, bd + 2 * kh, idesc_mxf4(128, (uint32_t)g.W, 2 * kh), sfa, sfbc, (kk | kh) != 0);
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
    // ---------------- epilogue warps (the resident x parts are done)
    epilogue(a, g, tb, ord, tbase, acc_full, acc_empty, uq_full, uq, cnt, s_last, s_ok, s_unit, &s_abort);
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
      for (int q = 0; q < tb.U * 16; ++q) cnt[C_HREADY + q] = 0;
      for (int q = 0; q < tb.U * g.RTG; ++q) cnt[C_G + q] = 0;
      for (int q = 0; q < g.RTD; ++q) cnt[C_D + q] = 0;
      cnt[C_ROUTE] = 0;
      cnt[C_XP] = 0;
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
                 void* y_bf16, int accumulate, void* ws, size_t ws_bytes, void* stream, const void* router_w,
                 int32_t* idx_out, float* w_out) {
  if (L->fmt != MOE_FMT_MXFP4) return MOE_ERR_UNSUPPORTED_FORMAT;
  if (((uintptr_t)x & 1) || ((uintptr_t)y & 3)) return MOE_ERR_INVALID_ARG;
  // the workspace is laid out for the T_max it was sized for; recover it from the size (largest T_max that fits)
  int tmax = 0;
  for (int tm = MAX_T; tm >= T; --tm)
    if (ws_bytes >= workspace_bytes(L, tm, k)) { tmax = tm; break; }
  if (!tmax) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!moe_internal::tmap_available()) return MOE_ERR_CUDA;
  Args a;
  a.gu = (const uint8_t*)L->gate_up;
  a.dn = (const uint8_t*)L->down;
  a.gu_stride = tc_geom(MOE_MAT_GATE_UP, L->H, L->I).stride;
  a.dn_stride = tc_geom(MOE_MAT_DOWN, L->H, L->I).stride;
  a.x = (const uint16_t*)x;
  a.idx = idx;
  a.w = w;
  a.wr = (const uint16_t*)router_w;
  a.idx_out = idx_out;
  a.w_out = w_out;
  if (router_w && (L->E > kRouteMaxE / 4 || k > L->E || ((uintptr_t)x & 15) || ((uintptr_t)router_w & 15)))
    return router_w && L->E > kRouteMaxE / 4 ? MOE_ERR_SHAPE : MOE_ERR_INVALID_ARG;
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
  g.RTG = 2 * L->I / 128; g.KTG = L->H / 128; g.KSG = ks_for_g(g.KTG); g.SG = g.KTG / g.KSG;
  g.RTD = L->H / 128;     g.KTD = L->I / 128; g.KSD = ks_for_d(g.KTD); g.SD = g.KTD / g.KSD;
  g.nG = g.nD = 0;
  g.W = 16 * ((PARTS * T + 15) / 16);
  g.ABUF = g.W <= 32 ? 4 : 2;
  if (NPIPE * g.ABUF * g.W > (int)SF_COL0) return MOE_ERR_SHAPE;
  CUtensorMap mgu, mdn, mh;
  const uint64_t hd[2] = {(uint64_t)L->I / 2, (uint64_t)(umax * HROWS)}, hs[1] = {(uint64_t)L->I / 2};
  const uint32_t hbox[2] = {64, HROWS};
  if (!moe_internal::tmap_tc_weights_packed(&mgu, L->gate_up, MOE_MAT_GATE_UP, L->H, L->I, L->E) ||
      !moe_internal::tmap_tc_weights_packed(&mdn, L->down, MOE_MAT_DOWN, L->H, L->I, L->E) ||
      !moe_internal::tmap_u8(&mh, a.ws + a.L.hb, 2, hd, hs, hbox, 64))
    return MOE_ERR_CUDA;
  static std::once_flag once;
  static bool attr_ok = false;
  std::call_once(once, [] {
    attr_ok = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) == cudaSuccess;
  });
  if (!attr_ok) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  const int nsm = moe_internal::num_sms();
  cfg.gridDim = dim3(nsm - nsm % g.SG);  // a multiple of S_G: every gate/up unit of a CTA has the same K segment
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = SMEM;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, decode_kernel, mgu, mdn, mh, a) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

}  // namespace dtc
}  // namespace moe

namespace moe_internal {
size_t tc_decode_workspace_bytes(const moe_layer_t* L, int T_max, int k) {
  return moe::dtc::workspace_bytes(L, T_max, k);
}
moe_status_t tc_decode(const moe_layer_t* L, const void* x, int T, const int32_t* idx, const float* w, int k, float* y,
                       void* y_bf16, int accumulate, void* ws, size_t ws_bytes, void* stream, const void* router_w,
                       int32_t* idx_out, float* w_out) {
  return moe::dtc::run(L, x, T, idx, w, k, y, y_bf16, accumulate, ws, ws_bytes, stream, router_w, idx_out, w_out);
}
}  // namespace moe_internal
