// decode_tc.cu -- decode and verify (1..8 tokens) of MXFP4 experts in the tensor-core layout on tcgen05.
//
// What it computes: y_t = sum_r w[t,r] * Down_e( SiLU(Gate_e x_t) * (Up_e x_t) ), e = idx[t,r] ("quantization"
// glossary, "Q4_K routed experts": gate and up fused in one pass, the down projection accumulated into the output;
// "Mixed-precision compression of DeepSeek-V4-Flash", "What compression does not solve": one decode step reads every
// active expert weight once, so the step is bound by HBM bandwidth).
//
// Arithmetic. The block-scaled MMA (kind::mxf4: E2M1 x E2M1, one UE8M0 exponent per 32, K = 64 per instruction) has
// the weights as the 128-row operand A, read as PACKED codes straight from the layout, and a few activation columns
// as operand B: x (gate/up) and h (down) are each split into PARTS = 6 E2M1 parts per 32-block (part p has exponent
// e0 - 2p and quantises what the earlier parts left; the error is below 1/3072 of the block's largest value).
// Column 6 t + p holds part p of token t; N = W = 16 ceil(6 T / 16). A token's value is the sum of its part
// columns in part order, and every column is computed on its own, so a token's numbers do not depend on which
// other tokens share the sweep (verify row t == decode of token t, "Width drift").
//
// Decomposition. A SLICE is 64 intermediate indices of one expert: one 128-row gate/up tile row (64 gate + 64 up
// rows) over all of H, and the 64 matching columns of Down (the DOWN layout stores them as chunks of 256 rows x 64
// columns). The arithmetic of a slice never changes:
//   g, u of the slice = sum over SG segments (KSG k-tiles each, accumulated in TMEM) in segment order;
//   h = SiLU(g) * u in fp32, split into E2M1 parts;
//   one MMA (K = 64) per 128 rows of Down gives the slice's partial of those rows of the expert output;
//   y[t] = sum_r w[t, r] * (sum over the expert's slices, in slice order, of the partials), ranks in order.
// Only WHICH CTA does which slice depends on the call. Every CTA owns nw = floor(slices / CTAs) WHOLE slices: it
// runs all their segments, forms h in its own shared memory and runs their down chunks, with no global hand-off.
// The remaining R < CTAs slices are SPLIT: their segments (exports) are spread over the CTAs and run early; their
// partials go to global memory and are counted. Their down chunks (imports) are dealt in contiguous runs, so a CTA
// imports from one or two split slices and runs the chunks last; the runs are sized so that every CTA streams the
// same number of weight bytes to within one tile. Up to two tokens, every importer forms the h of its slices from
// the counted partials; with more, the slice's exporters each form a share of its h blocks once, into an image in
// global memory that the importers copy. Each
// CTA's order: the exports, the whole slices (W0 W1 D0 W2 D1 ..: forming h of a slice overlaps the next slice's
// stream), the imports. A grid barrier then lets every CTA sum the down partials of its share of the outputs (one
// warp per (token, 32 rows, rank): a lane per row, the slices in order).
//
// Inside a CTA, three independent pipelines take the CTA's units as they free up: a copy-issuing warp, an
// MMA-issuing warp, a shared-memory ring of three or four stage slots, TMEM accumulators and a group of four
// epilogue warps. Two helper warps do the work that waits on global memory (storing and counting export partials,
// forming the split slices' h) so that no epilogue group stalls on it. One issuing thread
// sustains only about one wait-and-issue round per 330 ns (TMA) or one
// stage of MMAs plus commit per ~600 cycles (tcgen05), while one SM must consume an 8.5 KB weight tile every
// ~180 ns to keep pace with HBM. Every wait is bounded; on a timeout the kernel records MOE_ERR_DEVICE_TIMEOUT, lets
// its own copies land, frees TMEM and returns. With a router (moe_route_expert_ffn), warps 2..7 of every CTA first
// compute halves of the router logits, and every CTA then selects each token's experts itself (route.cuh, the same
// arithmetic as the standalone router).
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
constexpr int RING_MAX = 4;              // stage slots per pipeline at most (as many as shared memory allows, >= 3;
                                         // five measured no faster: deeper rings lengthen every copy's latency)
constexpr int NSLOT = NPIPE * RING_MAX;
constexpr int NC_MAX = 2;                // down chunks per local down unit at most
constexpr int PARTS = 6;                 // E2M1 parts per activation value
constexpr int MAX_T = 8, MAX_K = 8, MAX_U = MAX_T * MAX_K;
constexpr int WMAX = 48;                 // B rows (MMA N) at most: PARTS x 8 tokens
// a stage slot: [0, 8192) weight codes (gate/up tile 128 rows x 64 B, 64-byte swizzle; down chunk 256 rows x 32 B,
// 32-byte swizzle), [8192, 8704) weight exponents (a down chunk is one 8704-byte copy); [8704, 9216) activation
// exponents, [9216, 9216 + 64 W) activation codes (x parts W x 64 B, swizzled like the weights)
constexpr int SL_SFA = 8192, SL_SFB = 8704;  // activation codes at SL_SFB + 512
// bytes of a stage slot for W activation rows, a multiple of 1024 (10 KB for W = 16, 12 KB for W = 48)
__host__ __device__ inline int slot_bytes(int W) { return ((SL_SFB + 512 + 64 * W + 1023) / 1024) * 1024; }
// activation images: [512 B exponent block][W rows of codes, pre-arranged in the MMA's swizzle], so one bulk copy
// (x, from global memory) or none (h, formed in shared memory) gives a stage its whole activation operand
constexpr int XIMG = 512 + WMAX * 64;    // per gate/up k-tile (x parts), in the workspace
constexpr int HIMG = 2048;               // per slice (h parts: 512 + WMAX * 32), in shared memory
constexpr int NHB = 2;                   // h buffers of whole slices in flight per CTA
constexpr int NIB = 4;                   // h buffers of imported slices
constexpr int NXB = 4;                   // staging buffers of export partials
constexpr int MAX_SG = 8;                // segments per slice at most
constexpr int RMAX = 256;                // split slices at most (fewer than the CTAs)
constexpr int EPI_WARP0 = 2 * NPIPE;     // warps: NPIPE producers, NPIPE MMA issuers (each issuing thread has a warp
constexpr int NGRP = NPIPE;              // of its own: issuing lanes of one warp run one after another), then the epilogue
constexpr int QN = 32;                   // groups of 4 warps (group j drains pipeline j), then the helper warps;
constexpr int HELPER = EPI_WARP0 + 4 * NGRP;  // unit-queue entries per pipeline
constexpr int NHELP = 2;                 // helper warps (20 warps in all: 96 registers a thread)
constexpr int THREADS = (HELPER + NHELP) * 32;
// named barriers: 0 the CTA, 1..NGRP the epilogue groups, NB_ROUTE warps 0..EPI_WARP0-1 (routing), NB_TAB / NB_TAB2
// the routing tables handed from warp 0 to the other warps, NB_HELP the helper warps
constexpr int NB_ROUTE = 2 + NGRP, NB_TAB = NB_ROUTE + 1, NB_TAB2 = NB_ROUTE + 2, NB_HELP = NB_ROUTE + 3;
constexpr uint32_t TMEM_COLS = 512;      // accumulators below SF_COL0, 8 scale columns per slot from there
constexpr uint32_t SF_COL0 = TMEM_COLS - 8 * NSLOT;
static_assert(SF_COL0 + 8 * NSLOT <= TMEM_COLS, "TMEM budget");

// unit types
enum { U_EXPORT = 0, U_LOCAL = 1, U_DLOCAL = 2, U_DIMPORT = 3 };

// ------------------------------------------------------------------ geometry and schedule of one call
struct Geo {
  int H, I, T, k, E, W, RING, SLOT;  // ..., stage slots per pipeline, bytes per slot
  int RC, UREG;                 // TMEM columns of one unit's accumulator region, regions per pipeline
  int NC, NDL;                  // down chunks per local down unit, local down units per slice
  int NS, NQ, KTG, KSG, SG;     // slices per expert, row pairs of Down, k-tiles of gate/up, k-tiles per segment, segments
  int G;                        // CTAs
  // schedule (depends on U, set on the device once the routing is known)
  int U, Z, nw, Zw, R, ne_lo, X, A, A1;
  int F1, Rm1, F2, Rm2;         // import counts: CTA c gets F + (1 if its index < Rm) of each dealing round
};
// Segments of a gate/up slice: the largest divisor SG of the k-tile count with SG <= MAX_SG and at least two k-tiles
// per segment (one k-tile when there are only two); a function of H alone, so every call sums the same segments.
__host__ __device__ inline int sg_for(int ktg) {
  for (int sg = MAX_SG; sg > 1; --sg)
    if (ktg % sg == 0 && ktg / sg >= 2) return sg;
  return 1;
}

__host__ __device__ inline void make_schedule(Geo& g, int U) {
  g.U = U;
  g.Z = U * g.NS;
  g.nw = g.Z / g.G;
  g.Zw = g.nw * g.G;
  g.R = g.Z - g.Zw;
  const int ne = g.R * g.SG;                     // export segments
  g.ne_lo = ne / g.G;
  g.X = ne % g.G;                                // CTAs with one export segment more
  g.A = g.R * g.NQ;                              // import chunks
  // the CTAs without the extra segment first get up to KSG chunks each (a segment is KSG tiles), then the rest goes
  // round-robin over all CTAs: every CTA streams the same number of tiles to within one
  const int a1 = (g.G - g.X) * g.KSG;
  g.A1 = g.A < a1 ? g.A : a1;
  g.F1 = g.A1 / (g.G - g.X);
  g.Rm1 = g.A1 % (g.G - g.X);
  g.F2 = (g.A - g.A1) / g.G;
  g.Rm2 = (g.A - g.A1) % g.G;
}

struct Unit {
  int type, u, s, x, li, ib;  // x: segment (gate/up) or first row pair q (down); li: local slice ordinal or split
};                            // index; ib: ordinal of the import slice in this CTA
// packed form of a unit for the table in shared memory
__device__ __forceinline__ uint64_t pack_unit(const Unit& r) {
  return (uint64_t)(r.type & 255) | ((uint64_t)(r.x & 255) << 8) | ((uint64_t)(r.u & 255) << 16) |
         ((uint64_t)(r.s & 255) << 24) | ((uint64_t)(r.li & 0xFFFF) << 32) | ((uint64_t)(r.ib & 255) << 48);
}
__device__ __forceinline__ Unit unpack_unit(uint64_t v) {
  Unit r;
  r.type = (int)(v & 255); r.x = (int)((v >> 8) & 255); r.u = (int)((v >> 16) & 255); r.s = (int)((v >> 24) & 255);
  r.li = (int)((v >> 32) & 0xFFFF); r.ib = (int)((v >> 48) & 255);
  return r;
}
struct Mine {                 // this CTA's share: export segments, whole-slice units, imports (a contiguous run of
  int ne, nloc, nimp, n;      // the import chunks, numbered split slice * NQ + row pair, from a0)
  int a0, nis;                // first import chunk, import slices
};
__host__ __device__ inline int mn(int a, int b) { return a < b ? a : b; }
__host__ __device__ inline Mine my_share(const Geo& g, int c) {
  Mine m;
  m.ne = g.ne_lo + (c < g.X ? 1 : 0);
  m.nloc = g.nw * (g.SG + g.NDL);
  const int n1 = c < g.X ? 0 : g.F1 + (c - g.X < g.Rm1 ? 1 : 0);
  const int n2 = g.F2 + (c < g.Rm2 ? 1 : 0);
  const int p1 = c <= g.X ? 0 : g.F1 * (c - g.X) + mn(c - g.X, g.Rm1);
  const int p2 = g.F2 * c + mn(c, g.Rm2);
  m.nimp = n1 + n2;
  m.a0 = p1 + p2;
  m.nis = m.nimp > 0 ? (m.a0 + m.nimp - 1) / g.NQ - m.a0 / g.NQ + 1 : 0;
  m.n = m.ne + m.nloc + m.nimp;
  return m;
}
// A CTA's order: its export segments first (their partials travel through global memory to the importing CTAs, so
// they get the most time), then the whole slices as W0 W1 D0 W2 D1 .. W(nw-1) D(nw-2) D(nw-1) (forming h of a slice
// overlaps the stream of the next slice's segments; the stage ring covers the last one), then the imports.
__host__ __device__ inline int export_pos(const Geo& g, int xo) { return xo; }
__device__ inline Unit unit_at(const Geo& g, const Mine& mi, int c, int i) {
  Unit r;
  r.ib = 0;
  const int e0 = export_pos(g, 0);
  if (i >= e0 && i < e0 + mi.ne) {                  // export segment
    const int j = c + g.G * (i - e0);
    const int z = g.Zw + j / g.SG;
    r.type = U_EXPORT; r.u = z / g.NS; r.s = z % g.NS; r.x = j % g.SG; r.li = z - g.Zw;
    return r;
  }
  if (i >= e0) i -= mi.ne;
  if (i < mi.nloc) {                                // whole slices
    int m, isd, x;
    if (i < g.SG) { m = 0; isd = 0; x = i; }
    else {
      const int ip = i - g.SG, blk = g.SG + g.NDL;
      const int b = ip / blk + 1, rr = ip % blk;
      if (b < g.nw && rr < g.SG) { m = b; isd = 0; x = rr; }
      else if (b < g.nw) { m = b - 1; isd = 1; x = rr - g.SG; }
      else { m = g.nw - 1; isd = 1; x = rr; }
    }
    const int z = c * g.nw + m;
    r.type = isd ? U_DLOCAL : U_LOCAL; r.u = z / g.NS; r.s = z % g.NS; r.x = isd ? x * g.NC : x; r.li = m;
    return r;
  }
  i -= mi.nloc;                                     // import chunk
  const int a = mi.a0 + i;
  const int z = g.Zw + a / g.NQ;
  r.type = U_DIMPORT; r.u = z / g.NS; r.s = z % g.NS; r.x = a % g.NQ; r.li = z - g.Zw;
  r.ib = a / g.NQ - mi.a0 / g.NQ;
  return r;
}

// ------------------------------------------------------------------ workspace (byte offsets from the base)
// [0, 256)   WsHeader (status word, done, grid barrier)
// [256, ..)  counters (uint32): x parts done, router logits done, then per split slice: its segments stored, then
//            per split slice: its segments' exporters done writing their blocks of its h image
// then gpart [RMAX * MAX_SG][TS][128] fp32 (split slices' segment partials, by token), himg [RMAX][HIMG] (split
//      slices' h images), ximg [KTG][XIMG] (x parts), dpart [cols][H / 32][NS][32] fp32 (down partials: a column
//      per (expert, token) pair of the call), lg [tokens][2][E] router logit halves.
constexpr int64_t kCnt = 256;
constexpr int C_XP = 0, C_ROUTE = 1, C_SPLIT = 2, C_HREADY = C_SPLIT + RMAX, C_END = C_HREADY + RMAX;
struct Ws {
  int64_t gpart, himg, ximg, dpart, lg, total;
};
inline int64_t al1k(int64_t v) { return (v + 1023) & ~(int64_t)1023; }
inline Ws ws_layout(int64_t H, int64_t I, int64_t cols, int64_t TS) {
  Ws w;
  int64_t o = al1k(kCnt + (int64_t)C_END * 4);
  w.gpart = o; o = al1k(o + (int64_t)RMAX * MAX_SG * TS * 128 * 4);
  w.himg = o;  o = al1k(o + (int64_t)RMAX * HIMG);
  w.ximg = o;  o = al1k(o + (H / 128) * XIMG);
  w.dpart = o; o = al1k(o + cols * H * (I / 64) * 4);
  w.lg = o;    o = al1k(o + (int64_t)kRouteTPC * 2 * kRouteMaxE * 4);
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
  uint8_t* ws;
  Ws L;
  int ts;                     // token stride of the segment partials
  Geo g;
  long long wait_ns;
};

// ------------------------------------------------------------------ E2M1 parts
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
// value of E2M1 code c, built from its bits: exponent field f = (c >> 1) & 3 and mantissa bit m = c & 1 give
// 2^(f - 1) (1 + m / 2) for f > 0 and m / 2 for f = 0; bit 3 is the sign
__device__ __forceinline__ float e2m1_value(uint32_t c) {
  const uint32_t f = (c >> 1) & 3u, m = c & 1u;
  const uint32_t mag = f ? ((126u + f) << 23) | (m << 22) : (m ? 0x3F000000u : 0u);
  return __uint_as_float(mag | ((c & 8u) << 28));
}
__device__ __forceinline__ float warp_amax(float v) {
  const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(v)));
  return __uint_as_float(m);
}
// Split v (lane l holds element l of a 32-block) into PARTS E2M1 parts: part 0 uses the block exponent e0 (largest
// magnitude <= 6 * 2^(e0 - 127)); part p uses e0 - 2p (clamped at 1) and quantises what parts 0 .. p-1 left. After
// a part the remainder is at most half an E2M1 step, <= 1 unit of its scale = 4 units of the next part's, so no
// part saturates and each adds at least 2 bits: the final error is below 2^-10 of part 0's scale, i.e. below
// 1/3072 of the block's largest magnitude. A block holding NaN or infinity has no E2M1 encoding: every part gets
// the E8M0 NaN exponent (255), which the block-scaled MMA turns into NaN. Even lanes get the packed byte of elements
// (l, l + 1) of part p in bytes[p] (element l in the low nibble), every lane the exponents. Every lane of the warp
// must call it.
__device__ __forceinline__ void split_parts(float v, uint32_t (&bytes)[PARTS], int (&exps)[PARTS]) {
  const float am = warp_amax(v);
  const bool nonfinite = !(am <= 3.4028235e38f);
  const int e0 = mx4_exp(am);
  float r = nonfinite ? 0.f : v;
  uint32_t cs[PARTS];
#pragma unroll
  for (int p = 0; p < PARTS; ++p) {  // the remainder chain first (the value times a power of two is exact)
    const int e = e0 - 2 * p > 1 ? e0 - 2 * p : 1;
    cs[p] = e2m1_code(r * pow2_127m(e));
    r = fmaf(-e2m1_value(cs[p]), pow2_m127(e), r);
  }
#pragma unroll
  for (int p = 0; p < PARTS; ++p) {
    bytes[p] = cs[p] | (__shfl_down_sync(0xFFFFFFFFu, cs[p], 1) << 4);
    exps[p] = nonfinite ? 255 : (e0 - 2 * p > 1 ? e0 - 2 * p : 1);
  }
}
// byte of the permuted 512-byte exponent block that holds (operand row n, 32-block b)
__device__ __forceinline__ int sfb(int n, int b) { return (n & 31) * 16 + (n >> 5) * 4 + b; }

// ------------------------------------------------------------------ waits and counters
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
// Bounded wait on an mbarrier phase by one thread: non-blocking tests with short sleeps in between. A thread parked
// in mbarrier.try_wait was measured to slow the shuffles of the other warps on its SM several-fold, so no thread of
// this kernel waits that way.
__device__ __forceinline__ bool bwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, long long lim) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = globaltimer_ns();
  while (true) {
    __nanosleep(32);  // 128 and 512 ns measured slower
    if (mbar_test_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > lim) { *abort_flag = 1; return false; }
  }
}
// K-major operand with 32-byte rows and the 32-byte swizzle (8-row atoms of 256 bytes)
__device__ __forceinline__ uint64_t umma_desc_sw32(uint32_t saddr) { return umma_desc(saddr, 16, 256, 6); }
// kind::mxf4 instruction descriptor with separate scale-byte selectors for A and B (0 or 2)
__device__ __forceinline__ uint32_t idesc_mxf4_ab(uint32_t N, uint32_t a_sf, uint32_t b_sf) {
  return (b_sf << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | (1u << 23) | ((128u >> 4) << 24) | (a_sf << 29);
}

// ------------------------------------------------------------------ routing tables
// Tables every CTA builds from idx: the union of experts (first-appearance order over (t, r)), each expert's
// tokens (slot order = token order), per (t, r) the union index and the token's slot, and the first down-partial
// column of each union expert (its tokens' columns follow in slot order).
struct Tables {
  int32_t ue[MAX_U];
  int8_t ntok[MAX_U];
  int8_t tok[MAX_U][MAX_T];
  int8_t pu[MAX_T][MAX_K];
  int8_t ps[MAX_T][MAX_K];
  int16_t col0[MAX_U];
  uint32_t tmask[MAX_U];   // bit t: token t routes to union expert u
  float w[MAX_T][MAX_K];
  int U;
  int bad;
};
// (1) one warp: the union in first-appearance order over (t, r) and whether any id is out of range
__device__ void build_union_warp(Tables& tb, const int32_t (*idx)[MAX_K], int T, int k, int E) {
  const int lane = threadIdx.x & 31;
  const int n = T * k;
  const bool v0 = lane < n, v1 = lane + 32 < n;
  const int e0 = v0 ? idx[lane / k][lane % k] : 0, e1 = v1 ? idx[(lane + 32) / k][(lane + 32) % k] : 0;
  const bool bad = __any_sync(0xFFFFFFFFu, (v0 && (e0 < 0 || e0 >= E)) || (v1 && (e1 < 0 || e1 >= E)));
  const int key0 = v0 ? e0 : -1 - lane, key1 = v1 ? e1 : -33 - lane;  // absent entries never match
  const uint32_t lt = (1u << lane) - 1u;
  const uint32_t m0 = __match_any_sync(0xFFFFFFFFu, key0), m1 = __match_any_sync(0xFFFFFFFFu, key1);
  bool in0 = false;  // entry lane + 32 already appeared among entries 0 .. 31 (only when there are more than 32)
  if (n > 32)
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
// (2) one warp: weights, each union expert's tokens, per (t, r) the union index and slot, the column bases. A lane
// per (t, r) entry (two when T k > 32): its union index by search, the union experts' token sets as bit masks, a
// token's slot = the number of earlier tokens in its expert's set (slot order = token order).
__device__ void build_slots_warp(Tables& tb, const int32_t (*idx)[MAX_K], const float (*w)[MAX_K], int T, int k) {
  const int lane = threadIdx.x & 31;
  const int n = T * k, U = tb.U;
  for (int u = lane; u < MAX_U; u += 32) tb.tmask[u] = 0u;
  __syncwarp();
  int uu[2] = {0, 0};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = lane + 32 * h;
    if (i >= n) continue;
    const int t = i / k, r = i % k, e = idx[t][r];
    int u = 0;
    while (u < U && tb.ue[u] != e) ++u;
    uu[h] = u;
    tb.w[t][r] = w[t][r];
    if (u < U) atomicOr(&tb.tmask[u], 1u << t);
  }
  __syncwarp();
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int i = lane + 32 * h;
    if (i >= n) continue;
    const int t = i / k, r = i % k, u = uu[h];
    const bool valid = u < U;  // an invalid id: no units run
    tb.pu[t][r] = (int8_t)(valid ? u : 0);
    tb.ps[t][r] = (int8_t)(valid ? __popc(tb.tmask[u] & ((1u << t) - 1u)) : 0);
  }
  // per union expert: its token count and tokens; the column bases are the exclusive prefix sums of the counts
  int cnt[2] = {0, 0};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int u = lane + 32 * h;
    if (u >= U) continue;
    uint32_t m = tb.tmask[u];
    cnt[h] = __popc(m);
    tb.ntok[u] = (int8_t)cnt[h];
    for (int s = 0; m; ++s, m &= m - 1u) tb.tok[u][s] = (int8_t)(__ffs(m) - 1);
  }
  int x0 = cnt[0], x1 = cnt[1];  // inclusive scans of the two halves
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y0 = __shfl_up_sync(0xFFFFFFFFu, x0, o), y1 = __shfl_up_sync(0xFFFFFFFFu, x1, o);
    if (lane >= o) { x0 += y0; x1 += y1; }
  }
  const int total0 = __shfl_sync(0xFFFFFFFFu, x0, 31);
  if (lane < U) tb.col0[lane] = (int16_t)(x0 - cnt[0]);
  if (lane + 32 < U) tb.col0[lane + 32] = (int16_t)(total0 + x1 - cnt[1]);
}

// ------------------------------------------------------------------ x parts
// 32-block j = (token t, k-tile kt, block kb) of x goes to warp j of the grid's epilogue warps, which splits it into
// PARTS parts and writes them into the x image: k-tile kt at ximg + kt * XIMG = [512 B exponents][W rows x 64 B],
// row 6 t + p, 16-byte chunk kb at chunk kb ^ ((row >> 1) & 3) (the MMA's 64-byte swizzle). The warp of the last
// token also clears the padding rows 6T .. W-1 of (kt, kb) (zero codes, exponent 127).
__device__ __forceinline__ float load_x_block(const Args& a, const Geo& g, int j) {
  const int lane = threadIdx.x & 31;
  if (j >= g.T * g.KTG * 4) return 0.f;
  const int t = j / (g.KTG * 4), rem = j % (g.KTG * 4);
  return __uint_as_float((uint32_t)a.x[(int64_t)t * g.H + rem * 32 + lane] << 16);
}
__device__ void split_x_global(const Args& a, const Geo& g, int gw, int nwarps, float xfirst, uint32_t* cnt) {
  const int lane = threadIdx.x & 31;
  const int nblk = g.T * g.KTG * 4;
  for (int j = gw; j < nblk; j += nwarps) {
    const float v = j == gw ? xfirst : load_x_block(a, g, j);
    const int t = j / (g.KTG * 4), rem = j % (g.KTG * 4), kt = rem / 4, kb = rem % 4;
    uint8_t* img = a.ws + a.L.ximg + (int64_t)kt * XIMG;
    uint32_t by[PARTS];
    int ex[PARTS];
    split_parts(v, by, ex);
#pragma unroll
    for (int p = 0; p < PARTS; ++p) {
      const int n = PARTS * t + p;
      if (!(lane & 1)) img[512 + n * 64 + ((kb ^ ((n >> 1) & 3)) << 4) + (lane >> 1)] = (uint8_t)by[p];
      if (lane == 0) img[sfb(n, kb)] = (uint8_t)ex[p];
    }
    if (t == g.T - 1) {
      for (int n = PARTS * g.T + lane; n < g.W; n += 32) {
        *reinterpret_cast<uint4*>(img + 512 + n * 64 + ((kb ^ ((n >> 1) & 3)) << 4)) = make_uint4(0, 0, 0, 0);
        img[sfb(n, kb)] = 127;
      }
    }
    __syncwarp();
    if (lane == 0) red_release_add(cnt + C_XP, 1u);
  }
}

// ------------------------------------------------------------------ h of a slice
// The slice's segment partials are in: g and u of its 64 intermediate indices (partial rows 0..63 gate, 64..127
// up) summed over the SG segments in order, h = SiLU(g) * u, split into PARTS parts per 32-block into an h image
// [512 B exponents][W rows x 32 B] (row 6 s + p for token slot s, 16-byte half b at half b ^ ((row >> 2) & 1): the
// MMA's 32-byte swizzle). Rows 6 ntok .. W-1 are padding (zero codes, exponent 127). The partial of (segment sg,
// token t, row m) is at part[sg * seg_stride + t * 128 + m]; slot s holds token tok[s]. One warp forms one
// 32-block (block b of slot s, lane = index in the block).
// h = SiLU(g) * u of one 32-block (lane = index in the block) -> the PARTS rows of slot s in an h image
__device__ __forceinline__ void h_emit(float gv, float uv, int s, int b, uint8_t* img) {
  const int lane = threadIdx.x & 31;
  const float h = __fdividef(gv * uv, 1.0f + __expf(-gv));  // SiLU(g) * u
  uint32_t by[PARTS];
  int ex[PARTS];
  split_parts(h, by, ex);
#pragma unroll
  for (int q = 0; q < PARTS; ++q) {
    const int n = PARTS * s + q;
    if (!(lane & 1)) img[512 + n * 32 + ((b ^ ((n >> 2) & 1)) << 4) + (lane >> 1)] = (uint8_t)by[q];
    if (lane == 0) img[sfb(n, b)] = (uint8_t)ex[q];
  }
}
// padding rows 6 ntok .. W-1 of an h image, by `nthr` threads numbered from th
__device__ __forceinline__ void h_padding(uint8_t* img, int ntok, int W, int th, int nthr) {
  for (int q = th; q < 2 * (W - PARTS * ntok); q += nthr) {
    const int n = PARTS * ntok + (q >> 1), c = q & 1;
    *reinterpret_cast<uint4*>(img + 512 + n * 32 + (c << 4)) = make_uint4(0, 0, 0, 0);
    img[sfb(n, c)] = 127;
  }
}
// whole slice, by an epilogue group (thread et of 128: warp et / 32 takes blocks (slot, b) = (w / 2, w % 2), then
// every fourth), partials in shared memory, summed over the segments in order
__device__ void finalize_local(const float* part, int64_t seg_stride, int SG, int ntok, const int8_t* tok, int W,
                               uint8_t* img, int et) {
  const int lane = threadIdx.x & 31;
  for (int k = et >> 5; k < 2 * ntok; k += 4) {
    const int s = k >> 1, b = k & 1;
    const float* p = part + tok[s] * 128 + 32 * b + lane;
    float gl[MAX_SG], ul[MAX_SG];
#pragma unroll
    for (int sg = 0; sg < MAX_SG; ++sg)
      if (sg < SG) { gl[sg] = p[sg * seg_stride]; ul[sg] = p[sg * seg_stride + 64]; }
    float gv = 0.f, uv = 0.f;
#pragma unroll
    for (int sg = 0; sg < MAX_SG; ++sg)
      if (sg < SG) { gv += gl[sg]; uv += ul[sg]; }
    h_emit(gv, uv, s, b, img);
  }
  h_padding(img, ntok, W, et, 128);
}
// imported slice, by the helper warps (helper hw of NHELP takes the 32-blocks q = 2 slot + half with q = hw mod
// NHELP), partials in global memory
__device__ void finalize_import(const float* part, int64_t seg_stride, int SG, int ntok, const int8_t* tok, int W,
                                uint8_t* img, int hw) {
  const int lane = threadIdx.x & 31;
  for (int q = hw; q < 2 * ntok; q += NHELP) {
    const int s = q >> 1, b = q & 1;
    const float* p = part + tok[s] * 128 + 32 * b + lane;
    float gl[MAX_SG], ul[MAX_SG];
#pragma unroll
    for (int sg = 0; sg < MAX_SG; ++sg)
      if (sg < SG) { gl[sg] = __ldcg(p + sg * seg_stride); ul[sg] = __ldcg(p + sg * seg_stride + 64); }
    float gv = 0.f, uv = 0.f;
#pragma unroll
    for (int sg = 0; sg < MAX_SG; ++sg)
      if (sg < SG) { gv += gl[sg]; uv += ul[sg]; }
    h_emit(gv, uv, s, b, img);
  }
  h_padding(img, ntok, W, lane + 32 * hw, 32 * NHELP);
}

// The blocks of a split slice's h that the exporter of segment x forms (q = 2 slot + half, q = x mod SG; helper hw
// of NHELP takes every NHELP-th of them), from all the segments' partials in global memory, written straight into
// the slice's h image in global memory; exporter 0 also writes the padding rows.
__device__ void form_blocks(const float* part, int64_t seg_stride, int SG, int x, int ntok, const int8_t* tok, int W,
                            uint8_t* img, int hw) {
  const int lane = threadIdx.x & 31;
  for (int q = x + SG * hw; q < 2 * ntok; q += SG * NHELP) {
    const int s = q >> 1, b = q & 1;
    const float* p = part + tok[s] * 128 + 32 * b + lane;
    float gl[MAX_SG], ul[MAX_SG];
#pragma unroll
    for (int sg = 0; sg < MAX_SG; ++sg)
      if (sg < SG) { gl[sg] = __ldcg(p + sg * seg_stride); ul[sg] = __ldcg(p + sg * seg_stride + 64); }
    float gv = 0.f, uv = 0.f;
#pragma unroll
    for (int sg = 0; sg < MAX_SG; ++sg)
      if (sg < SG) { gv += gl[sg]; uv += ul[sg]; }
    h_emit(gv, uv, s, b, img);
  }
  if (x == 0) h_padding(img, ntok, W, lane + 32 * hw, 32 * NHELP);
}

// ------------------------------------------------------------------ the kernel
struct Smem {                   // static shared state (the stage ring, h buffers and partials are dynamic)
  uint64_t full[NSLOT], empty[NSLOT];
  uint64_t ucomp[NPIPE][8], acc_empty[NPIPE][8];   // unit c of a pipeline done (slot c % 8) / its region drained
  uint64_t uq_full[NPIPE][QN];
  uint64_t hready[NHB], hfree[NHB];     // whole slices: h formed / its down chunks done reading it
  uint64_t iready[NIB], ifree[NIB];     // imported slices: the same
  uint64_t xstaged[NXB], xfree[NXB];    // export partials staged / copied out
  uint64_t drain[NPIPE];
  int uq[NPIPE][QN];                    // unit index, and the unit itself (packed), per queue entry
  uint64_t uqu[NPIPE][QN];
  int lcnt[NHB];
  Tables tb;
  int32_t idx[MAX_T][MAX_K];
  float wt[MAX_T][MAX_K];
  uint32_t tmem;
  int next;
  int abort;
  int ok[NGRP][2], last[NGRP], unit[NGRP];
  int hok[NHELP];
  int gok;
};
// dynamic shared memory: the stage ring, then h images of whole and imported slices, export staging, and the
// segment partials of whole slices
inline size_t smem_bytes(int T, int SG, int ring, int slot) {
  return 1024 + (size_t)NPIPE * ring * slot + (NHB + NIB) * HIMG + (size_t)NXB * T * 128 * 4 +
         (size_t)NHB * SG * T * 128 * 4;
}

// TT: the most tokens this instance serves (2: decode and 2-token verify, W = 16; 8: the rest). Only the size of the
// per-thread arrays differs; the arithmetic of every token is the same in both.
template <int TT>
__global__ void __launch_bounds__(THREADS, 1) decode_kernel(const __grid_constant__ CUtensorMap tm_gu, const Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  __shared__ Smem S;
  volatile int* s_abort = &S.abort;
  const Geo& ga = a.g;
  uint8_t* hbuf = smem + NPIPE * ga.RING * ga.SLOT;                   // [NHB][HIMG] whole slices' h
  uint8_t* ibuf = hbuf + NHB * HIMG;                                    // [NIB][HIMG] imported slices' h
  float* xstage = reinterpret_cast<float*>(ibuf + NIB * HIMG);          // [NXB][T][128] export partials
  float* spart = xstage + NXB * ga.T * 128;                             // [NHB][SG][T][128] whole slices' partials

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = reinterpret_cast<WsHeader*>(a.ws);
  uint32_t* cnt = reinterpret_cast<uint32_t*>(a.ws + kCnt);
  Geo g = a.g;
  const long long lim = a.wait_ns;
  const int xwarp = (int)blockIdx.x * (4 * NGRP) + (warp - EPI_WARP0), nxwarps = (int)gridDim.x * (4 * NGRP);
  const bool epi = warp >= EPI_WARP0 && warp < HELPER;
  const float xfirst = epi ? load_x_block(a, g, xwarp) : 0.f;  // before the weight stream starts
  int32_t pre_idx = 0;                                          // a given routing, fetched before the set-up
  float pre_w = 0.f;
  if (!a.wr && threadIdx.x < g.T * g.k) { pre_idx = a.idx[threadIdx.x]; pre_w = a.w[threadIdx.x]; }
  if (warp < NPIPE && lane == 0) asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_gu) : "memory");

  float* lgw = reinterpret_cast<float*>(a.ws + a.L.lg);  // router logit halves [token][half][expert]
  if (a.wr && warp >= 2 && warp < 2 + 2 * NPIPE) {
    // routing, phase 1 (at entry, while thread 0 and warp 1 set the CTA up): the logit halves (expert e, half c),
    // task q = blockIdx.x + gridDim.x * (w + 2 NPIPE i), e = q / 2, c = q % 2, w = warp - 2, spread over the grid
    for (int q = (int)blockIdx.x + (int)gridDim.x * (warp - 2); q < 2 * g.E; q += (int)gridDim.x * 2 * NPIPE) {
      const int e = q >> 1, c = q & 1;
      float acc[TT];
      route_half_logits<8, TT>(a.wr + (size_t)e * g.H, g.H, g.T, [&](int t) { return a.x + (size_t)t * g.H; }, c, acc);
      if (lane == 0)
#pragma unroll
        for (int t = 0; t < TT; ++t)
          if (t < g.T) __stcg(lgw + (t * 2 + c) * g.E + e, acc[t]);
      __syncwarp();
      if (lane == 0) red_release_add(cnt + C_ROUTE, 1u);
    }
  }
  if (warp == 0) {  // barriers, initialised by the lanes of warp 0 in parallel
    for (int s = lane; s < NSLOT; s += 32) { mbar_init(&S.full[s], 1); mbar_init(&S.empty[s], 1); }
    for (int q = lane; q < NPIPE * 8; q += 32) {
      mbar_init(&S.ucomp[q / 8][q % 8], 1);
      mbar_init(&S.acc_empty[q / 8][q % 8], 4);  // the 4 warps of one epilogue group
    }
    for (int q = lane; q < NPIPE * QN; q += 32) mbar_init(&S.uq_full[q / QN][q % QN], 1);
    __syncwarp();  // before lane 0's fence below
  }
  if (threadIdx.x == 0) {
    for (int j = 0; j < NPIPE; ++j) mbar_init(&S.drain[j], 1);
    for (int b = 0; b < NHB; ++b) {
      mbar_init(&S.hready[b], 1);
      mbar_init(&S.hfree[b], g.NDL);       // one commit per local down unit of the slice
      S.lcnt[b] = 0;
    }
    // ifree: one commit per down chunk of the slice (the helper arrives for the chunks other CTAs hold)
    for (int b = 0; b < NIB; ++b) { mbar_init(&S.iready[b], 1); mbar_init(&S.ifree[b], g.NQ); }
    for (int b = 0; b < NXB; ++b) { mbar_init(&S.xstaged[b], 1); mbar_init(&S.xfree[b], 1); }
    S.abort = 0;
    S.next = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc_alloc(&S.tmem, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = S.tmem;
  Tables& tb = S.tb;

  if (warp >= EPI_WARP0) {
    // this CTA's share of the x parts (independent of the routing) while the other warps route and build the
    // tables, then the token tables the epilogues need
    if (epi) split_x_global(a, g, xwarp, nxwarps, xfirst, cnt);
    // hardware barriers: warp 0 arrives once the union is built, then the first epilogue warp builds the slots
    named_bar(NB_TAB, 32 + THREADS - EPI_WARP0 * 32);
    if (warp == EPI_WARP0) build_slots_warp(tb, S.idx, S.wt, g.T, g.k);
    named_bar(NB_TAB2, THREADS - EPI_WARP0 * 32);
  } else {
    if (a.wr) {
      // routing, phase 2: every CTA selects each token's experts from all the logits (a warp per token)
      for (int t = warp; t < g.T; t += EPI_WARP0) {
        bool ok = true;
        if (lane == 0) ok = wait_ge(cnt + C_ROUTE, (uint32_t)(2 * g.E), s_abort, lim);
        ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
        int sid[8];
        float sw[8];
        if (ok) {
          const float* row = lgw + t * 2 * g.E;  // half 0, then half 1, of every expert's logit
          route_topk_warp<kRouteMaxE / 32 / 4>([&](int e) { return __ldcg(row + e) + __ldcg(row + g.E + e); }, g.E, g.k,
                                               sid, sw);
        }
        if (lane == 0)
#pragma unroll
          for (int r = 0; r < MAX_K; ++r) {
            if (r >= g.k) break;
            S.idx[t][r] = ok ? sid[r] : -1;
            S.wt[t][r] = ok ? sw[r] : 0.f;
            if (blockIdx.x == 0 && ok) {
              a.idx_out[t * g.k + r] = sid[r];
              a.w_out[t * g.k + r] = sw[r];
            }
          }
      }
    } else if (threadIdx.x < g.T * g.k) {
      S.idx[threadIdx.x / g.k][threadIdx.x % g.k] = pre_idx;
      S.wt[threadIdx.x / g.k][threadIdx.x % g.k] = pre_w;
    }
    named_bar(NB_ROUTE, EPI_WARP0 * 32);
    if (warp == 0) {
      build_union_warp(tb, S.idx, g.T, g.k, g.E);
      __syncwarp();
      if (lane == 0) {
        // an expert id out of range: no units (every role finds an empty queue), status MOE_ERR_INVALID_ARG
        if (tb.bad && blockIdx.x == 0) record_error(&hdr->status, MOE_ERR_INVALID_ARG);
        if (tb.bad) tb.U = 0;
      }
      __syncwarp();
      named_bar_arrive(NB_TAB, 32 + THREADS - EPI_WARP0 * 32);
    }
    named_bar(NB_ROUTE, EPI_WARP0 * 32);
  }
  make_schedule(g, tb.U);
  const Mine mine = my_share(g, (int)blockIdx.x);
  const int nunits = tb.U > 0 ? mine.n : 0;

  if (warp < NPIPE) {
    // ---------------- producer of pipeline j = warp (lane 0 issues): the weights of every stage and, for gate/up
    // stages, the stage's x parts, all counted on the stage's barrier
    const int j = warp;
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int n = 0;  // stages of this pipeline
      bool ok = true, x_ok = false;
      for (int c = 0; ok; ++c) {
        const int i = atomicAdd(&S.next, 1);
        const Unit un = unit_at(g, mine, (int)blockIdx.x, i < nunits ? i : 0);
        // entry c % QN was last read for unit c - QN, long consumed (the producer runs at most RING stages ahead of
        // the MMA, the MMA at most UREG units ahead of the epilogue)
        S.uq[j][c % QN] = i < nunits ? i : -1;
        S.uqu[j][c % QN] = pack_unit(un);
        mbar_arrive(&S.uq_full[j][c % QN]);
        if (i >= nunits) break;
        const int e = tb.ue[un.u];
        const bool d = un.type >= U_DLOCAL;
        const int nst = d ? (un.type == U_DLOCAL ? g.NC : 1) : g.KSG;
        for (int kk = 0; kk < nst; ++kk, ++n) {
          const int slot = j * g.RING + (n % g.RING);
          const uint32_t ph = (uint32_t)((n / g.RING) & 1);
          if (!bwait(&S.empty[slot], ph ^ 1, s_abort, lim)) { ok = false; break; }
          uint8_t* st = smem + slot * g.SLOT;
          const uint32_t xbytes = d ? 0u : (uint32_t)(512 + 64 * g.W);
          mbar_arrive_expect_tx(&S.full[slot], (uint32_t)kTcTileBytes + xbytes);
          // weights are read once per call: evict-first keeps them from displacing what the dependent steps read
          // back through L2
          if (!d) {
            const int tile = un.s * g.KTG + un.x * g.KSG + kk;
            tma_load_4d_hint(st, &tm_gu, 0, 0, tile, e, &S.full[slot], pol);
            bulk_g2s(st + SL_SFA, a.gu + (int64_t)e * a.gu_stride + (int64_t)tile * kTcTileBytes + 8192, 512,
                     &S.full[slot], pol);
            if (!x_ok) {  // the x image, built by the epilogue warps of the whole grid at entry
              if (!wait_ge(cnt + C_XP, (uint32_t)(g.T * g.KTG * 4), s_abort, lim)) { ok = false; break; }
              asm volatile("fence.proxy.async.global;" ::: "memory");  // generic-proxy writes -> bulk-copy reads
              x_ok = true;
            }
            bulk_g2s_plain(st + SL_SFB, a.ws + a.L.ximg + (int64_t)(un.x * g.KSG + kk) * XIMG, xbytes, &S.full[slot]);
          } else {  // a down chunk: codes (stored in the operand's swizzle) and exponents in one copy; its h is in
                    // this CTA's shared memory
            const int64_t ch = ((int64_t)e * g.NS + un.s) * g.NQ + un.x + kk;
            bulk_g2s(st, a.dn + ch * kTcTileBytes, (uint32_t)kTcTileBytes, &S.full[slot], pol);
          }
        }
      }
      if (!ok) {
        record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
        // a stage may hold only the weight copy, so its barrier never completes: give the copies this warp issued
        // 1 ms to land before the CTA's shared memory is released
        const long long t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 1000000LL) __nanosleep(1000);
      }
    }
    __syncwarp();
  } else if (warp < 2 * NPIPE) {
    // ---------------- MMA issuers: lane 0 of warp NPIPE + j, pipeline j
    const int j = warp - NPIPE;
    if (lane == 0) {
      int n = 0;
      bool ok = true;
      for (int c = 0; ok; ++c) {
        if (!bwait(&S.uq_full[j][c % QN], (uint32_t)((c / QN) & 1), s_abort, lim)) { ok = false; break; }
        const int i = S.uq[j][c % QN];
        if (i < 0) break;
        const Unit un = unpack_unit(S.uqu[j][c % QN]);
        const bool d = un.type >= U_DLOCAL;
        const int nst = d ? (un.type == U_DLOCAL ? g.NC : 1) : g.KSG;
        // the unit's accumulators: region c % UREG of the pipeline, W columns per accumulator (a down chunk has
        // two: its two 128-row halves)
        const int rg = c % g.UREG;
        if (!bwait(&S.acc_empty[j][rg], (uint32_t)(((c / g.UREG) & 1) ^ 1), s_abort, lim)) { ok = false; break; }
        const uint32_t acc0 = tbase + (uint32_t)(g.RC * (j * g.UREG + rg));
        const int hb = un.li % NHB, ib = un.ib, kb = ib % NIB;
        if (un.type == U_DLOCAL && !bwait(&S.hready[hb], (uint32_t)((un.li / NHB) & 1), s_abort, lim)) { ok = false; break; }
        if (un.type == U_DIMPORT && !bwait(&S.iready[kb], (uint32_t)((ib / NIB) & 1), s_abort, lim)) { ok = false; break; }
        tc_fence_after();
        uint32_t sfb_unit = 0;  // down units: the h exponents, copied into the first stage's columns once
        for (int kk = 0; kk < nst; ++kk, ++n) {
          const int slot = j * g.RING + (n % g.RING);
          if (!bwait(&S.full[slot], (uint32_t)((n / g.RING) & 1), s_abort, lim)) { ok = false; break; }
          tc_fence_after();
          uint8_t* st = smem + slot * g.SLOT;
          const uint32_t sfa = tbase + SF_COL0 + (uint32_t)(slot * 8);
          uint32_t sfbc = sfa + 4;
          // activation image [512 B exponents][codes]: x in the stage, h of the slice in this CTA's buffers
          const uint8_t* bimg = un.type == U_DLOCAL ? hbuf + hb * HIMG : (un.type == U_DIMPORT ? ibuf + kb * HIMG : st + SL_SFB);
          tc_cp_sf(sfa, umma_desc_sf(smem_u32(st + SL_SFA)));
          if (!d || kk == 0) {
            tc_cp_sf(sfbc, umma_desc_sf(smem_u32(bimg)));
            sfb_unit = sfbc;
          } else {
            sfbc = sfb_unit;  // that stage's slot is reused only RING >= 3 stages later
          }
          if (!d) {
            // gate/up tile: two K = 64 halves, scale bytes (0, 1) and (2, 3) of A and B
            const uint64_t ad = umma_desc_sw64(smem_u32(st)), bd = umma_desc_sw64(smem_u32(bimg + 512));
#pragma unroll
            for (int kh = 0; kh < 2; ++kh)
              tc_mma_mxf4(acc0, ad + 2 * kh, bd + 2 * kh, idesc_mxf4_ab((uint32_t)g.W, 2 * kh, 2 * kh), sfa, sfbc,
                          (kk | kh) != 0);
          } else {
            // down chunk: rows 0..127 and 128..255 (A scale bytes (0, 1) and (2, 3)) times the slice's h (K = 64)
            const uint64_t bd = umma_desc_sw32(smem_u32(bimg + 512));
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tc_mma_mxf4(acc0 + (uint32_t)(g.W * (2 * kk + h)), umma_desc_sw32(smem_u32(st + 4096 * h)), bd,
                          idesc_mxf4_ab((uint32_t)g.W, 2 * h, 0), sfa, sfbc, 0);
          }
          tc_commit(&S.empty[slot]);
        }
        if (!ok) break;
        // one completion per unit (a commit costs its issuing thread a few hundred cycles): the epilogue drains all
        // the unit's accumulators on it. An h buffer that a later slice reuses is released once every chunk that
        // reads it has been multiplied.
        tc_commit(&S.ucomp[j][c % 8]);
        if (un.type == U_DLOCAL && un.li + NHB < g.nw) tc_commit(&S.hfree[hb]);
        if (un.type == U_DIMPORT && ib + NIB < mine.nis) tc_commit(&S.ifree[kb]);
      }
      if (!ok) record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
      tc_commit(&S.drain[j]);
      // every MMA of this pipeline has completed before TMEM is released (bounded: 100 ms)
      const long long t0 = globaltimer_ns();
      while (!mbar_test_wait(&S.drain[j], 0) && globaltimer_ns() - t0 < 100000000LL) __nanosleep(64);
    }
    __syncwarp();
  } else if (warp >= HELPER) {
    // ---------------- helpers. Helper 0 stores the export partials staged by the epilogue groups and counts them
    // per split slice (the store, fence and count wait on global memory, so they are kept off the epilogue groups).
    // Then the h of the slices this CTA imports. Up to two tokens (at most 4 blocks a slice) both helpers form it
    // from the counted partials into the import buffers. With more tokens, for each of this CTA's exports, once the
    // slice's segments are all counted, both helpers form that exporter's share of the slice's blocks straight into
    // the slice's h image in global memory and count that; helper 0 then copies the finished image of each slice
    // this CTA imports (one bulk copy, counted on the buffer's ready barrier).
    const int hw = warp - HELPER;
    float* gpart = reinterpret_cast<float*>(a.ws + a.L.gpart);
    uint8_t* himg = a.ws + a.L.himg;
    bool ok = true;
    for (int i = 0; i < (nunits && hw == 0 ? mine.ne : 0) && ok; ++i) {
      const int k = i % NXB;
      int w = 1;
      if (lane == 0) w = bwait(&S.xstaged[k], (uint32_t)((i / NXB) & 1), s_abort, lim) ? 1 : 0;
      if (!__shfl_sync(0xFFFFFFFFu, w, 0)) { ok = false; break; }
      const Unit un = unit_at(g, mine, (int)blockIdx.x, export_pos(g, i));
      const float* src = xstage + k * g.T * 128;
      float* dst = gpart + ((int64_t)un.li * g.SG + un.x) * a.ts * 128;
      for (int t = 0; t < g.T; ++t)
        reinterpret_cast<float4*>(dst + t * 128)[lane] = reinterpret_cast<const float4*>(src + t * 128)[lane];
      // __syncwarp orders the lanes' stores before lane 0's release, which publishes them with the count (a
      // release costs one store round trip; a full fence here measured several times that while the weights stream)
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.xfree[k]);
        red_release_add(cnt + C_SPLIT + un.li, 1u);
      }
    }
    if constexpr (TT <= 2) {
      // up to two tokens: an imported slice has at most 4 h blocks, so every importer forms them itself
      for (int ib = 0; ib < (nunits ? mine.nis : 0); ++ib) {
        const int kb = ib % NIB;
        const int li = mine.a0 / g.NQ + ib, z = g.Zw + li, u = z / g.NS;
        int w = ok ? 1 : 0;
        if (lane == 0) {
          // the buffer's previous slice must be done with it, and every segment of this one stored
          if (w && ib >= NIB) w = bwait(&S.ifree[kb], (uint32_t)(((ib / NIB) - 1) & 1), s_abort, lim) ? 1 : 0;
          if (w) w = wait_ge(cnt + C_SPLIT + li, (uint32_t)g.SG, s_abort, lim) ? 1 : 0;
          S.hok[hw] = w;
        }
        named_bar(NB_HELP, 32 * NHELP);
        bool all = true;
#pragma unroll
        for (int h = 0; h < NHELP; ++h) all = all && S.hok[h] != 0;
        if (!all) { ok = false; break; }  // both helpers leave together
        // lane 0's acquire (and the barrier) -> the lanes' loads of the partials
        finalize_import(gpart + (int64_t)li * g.SG * a.ts * 128, (int64_t)a.ts * 128, g.SG, tb.ntok[u], tb.tok[u], g.W,
                        ibuf + kb * HIMG, hw);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> the MMA's reads
        named_bar(NB_HELP, 32 * NHELP);
        if (hw == 0 && lane == 0) {
          mbar_arrive(&S.iready[kb]);
          const int lo = mine.a0 > li * g.NQ ? mine.a0 : li * g.NQ;
          const int hi = mine.a0 + mine.nimp < (li + 1) * g.NQ ? mine.a0 + mine.nimp : (li + 1) * g.NQ;
          if (ib + NIB < mine.nis && g.NQ - (hi - lo) > 0) mbar_arrive_n(&S.ifree[kb], (uint32_t)(g.NQ - (hi - lo)));
        }
      }
    } else {
      // more tokens: each exporter forms its share of the slice's blocks once, the importers copy the image
      for (int i = 0; i < (nunits ? mine.ne : 0); ++i) {
        const Unit un = unit_at(g, mine, (int)blockIdx.x, export_pos(g, i));
        const int z = g.Zw + un.li, u = z / g.NS;
        int w = ok ? 1 : 0;
        if (lane == 0) {
          if (w) w = wait_ge(cnt + C_SPLIT + un.li, (uint32_t)g.SG, s_abort, lim) ? 1 : 0;
          S.hok[hw] = w;
        }
        named_bar(NB_HELP, 32 * NHELP);  // also orders helper 0's exports before helper 1 goes on
        bool all = true;
#pragma unroll
        for (int h = 0; h < NHELP; ++h) all = all && S.hok[h] != 0;
        if (!all) { ok = false; break; }  // both helpers leave together
        form_blocks(gpart + (int64_t)un.li * g.SG * a.ts * 128, (int64_t)a.ts * 128, g.SG, un.x, tb.ntok[u], tb.tok[u],
                    g.W, himg + (int64_t)un.li * HIMG, hw);
        named_bar(NB_HELP, 32 * NHELP);  // every store of the block before the count's release
        if (hw == 0 && lane == 0) red_release_add(cnt + C_HREADY + un.li, 1u);
      }
      for (int ib = 0; ib < (nunits && hw == 0 && ok ? mine.nis : 0); ++ib) {
        const int kb = ib % NIB;
        const int li = mine.a0 / g.NQ + ib;
        int w = 1;
        if (lane == 0) {
          // the buffer's previous slice must be done with it, and every exporter of this one done with its h blocks
          if (ib >= NIB) w = bwait(&S.ifree[kb], (uint32_t)(((ib / NIB) - 1) & 1), s_abort, lim) ? 1 : 0;
          if (w) w = wait_ge(cnt + C_HREADY + li, (uint32_t)g.SG, s_abort, lim) ? 1 : 0;
          if (w) {
            asm volatile("fence.proxy.async.global;" ::: "memory");  // the acquire -> the bulk copy's reads
            const uint32_t nbytes = (uint32_t)(512 + 32 * g.W);     // exponent block + W rows of 32 B
            mbar_arrive_expect_tx(&S.iready[kb], nbytes);
            bulk_g2s_plain(ibuf + kb * HIMG, himg + (int64_t)li * HIMG, nbytes, &S.iready[kb]);
            const int lo = mine.a0 > li * g.NQ ? mine.a0 : li * g.NQ;
            const int hi = mine.a0 + mine.nimp < (li + 1) * g.NQ ? mine.a0 + mine.nimp : (li + 1) * g.NQ;
            if (ib + NIB < mine.nis && g.NQ - (hi - lo) > 0) mbar_arrive_n(&S.ifree[kb], (uint32_t)(g.NQ - (hi - lo)));
          }
        }
        if (!__shfl_sync(0xFFFFFFFFu, w, 0)) { ok = false; break; }
      }
    }
    if (!ok && lane == 0) record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
  } else {
    // ---------------- epilogue group j (warps EPI_WARP0 + 4 j ..): drains pipeline j's accumulators in order
    const int q = warp & 3;
    const int grp = (warp - EPI_WARP0) / 4, j = grp;
    const int bar = 1 + grp;                                   // named barrier of the group
    const int et = threadIdx.x - (EPI_WARP0 + 4 * grp) * 32;    // 0..127 inside the group
    const int m = q * 32 + lane;                                // TMEM lane = weight row of the tile
    float* dpart = reinterpret_cast<float*>(a.ws + a.L.dpart);
    int bc = 0;
    // thread et == 0 waits and shares the verdict with its group: two flag slots used in turn, so a slot is
    // rewritten only after every thread has passed the barrier that follows its last read
    auto shared_ok = [&](int v) -> int {
      const int sl = bc++ & 1;
      if (et == 0) S.ok[grp][sl] = v;
      named_bar(bar, 128);
      return S.ok[grp][sl];
    };
    for (int c = 0;; ++c) {
      int st = 0;
      if (et == 0 && bwait(&S.uq_full[j][c % QN], (uint32_t)((c / QN) & 1), s_abort, lim)) {
        const int i = S.uq[j][c % QN];
        st = i < 0 ? 2 : 1;
        S.unit[grp] = i;
      }
      if (shared_ok(st) != 1) break;
      const int ui = S.unit[grp];
      const Unit un = unpack_unit(S.uqu[j][c % QN]);
      const bool d = un.type >= U_DLOCAL;
      const int nt = tb.ntok[un.u];
      const int nuse = d ? 2 * (un.type == U_DLOCAL ? g.NC : 1) : 1;
      bool good = true;
      if (!shared_ok(et != 0 || bwait(&S.ucomp[j][c % 8], (uint32_t)((c / 8) & 1), s_abort, lim))) break;
      tc_fence_after();
      const uint32_t rbase = tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(g.RC * (j * g.UREG + c % g.UREG));
      // what accumulator h of the unit goes to (its token or slot values acc[]); false if a wait gave up
      auto put = [&](int h, const float (&acc)[TT]) -> bool {
        if (un.type == U_EXPORT) {  // staged by token for helper 0, which stores and counts it
          const int xo = ui - export_pos(g, 0), k = xo % NXB;
          if (xo >= NXB && !shared_ok(et != 0 || bwait(&S.xfree[k], (uint32_t)(((xo / NXB) - 1) & 1), s_abort, lim)))
            return false;
          float* xp = xstage + k * g.T * 128 + m;
#pragma unroll
          for (int t = 0; t < TT; ++t)
            if (t < g.T) xp[t * 128] = acc[t];
          named_bar(bar, 128);
          if (et == 0) mbar_arrive(&S.xstaged[k]);
        } else if (un.type == U_LOCAL) {
          const int hb = un.li % NHB;
          // the buffer's previous slice must be finished with it (normally long since)
          if (un.li >= NHB &&
              !shared_ok(et != 0 || bwait(&S.hready[hb], (uint32_t)(((un.li / NHB) - 1) & 1), s_abort, lim)))
            return false;
          float* sp = spart + ((int64_t)hb * g.SG + un.x) * g.T * 128 + m;
#pragma unroll
          for (int t = 0; t < TT; ++t)
            if (t < g.T) sp[t * 128] = acc[t];
        } else {
          // chunk un.x + h / 2, rows 256 q + 128 (h % 2) + m; the partial goes to column (expert, slot), 32-row
          // group, slice, row in the group
          const int row = 256 * (un.x + (h >> 1)) + 128 * (h & 1) + m;
          float* dp = dpart + ((((int64_t)tb.col0[un.u]) * (g.H / 32) + row / 32) * g.NS + un.s) * 32 + (row & 31);
#pragma unroll
          for (int s = 0; s < TT; ++s)
            if (s < nt) dp[(int64_t)s * (g.H / 32) * g.NS * 32] = acc[s];
        }
        return true;
      };
      // drain the unit's accumulators (W columns each; column 6 t + p = part p of token or slot t, summed in part
      // order): two at a time with one wait when W = 16; the region is handed back after its last load
      const int hstep = TT <= 2 ? 2 : 1;  // accumulators drained per TMEM-load wait
      for (int h0 = 0; h0 < nuse && good; h0 += hstep) {
        const int nh = nuse - h0 < hstep ? nuse - h0 : hstep;
        float acc0[TT], acc1[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) { acc0[t] = 0.f; acc1[t] = 0.f; }
        if constexpr (TT <= 2) {
          // W = 16 and columns 0..11 at most hold parts (T <= 2): 8 + 4 columns per accumulator, the padding is
          // not read
          uint32_t a0[8], b0[4], a1[8], b1[4];
          tc_ld8(rbase + 16 * h0, a0);
          if (g.T == 2) tc_ld4(rbase + 16 * h0 + 8, b0);
          if (nh == 2) {
            tc_ld8(rbase + 16 * h0 + 16, a1);
            if (g.T == 2) tc_ld4(rbase + 16 * h0 + 24, b1);
          }
          tc_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 12; ++cc)  // part order, as for the wider accumulators
            if (cc / PARTS < TT && (cc < 6 || g.T == 2))
              acc0[cc / PARTS] += __uint_as_float(cc < 8 ? a0[cc & 7] : b0[cc & 3]);
          if (nh == 2)
#pragma unroll
            for (int cc = 0; cc < 12; ++cc)
              if (cc / PARTS < TT && (cc < 6 || g.T == 2))
                acc1[cc / PARTS] += __uint_as_float(cc < 8 ? a1[cc & 7] : b1[cc & 3]);
        } else {
#pragma unroll
          for (int cb = 0; cb < WMAX / 16; ++cb) {
            if (16 * cb >= g.W) break;
            uint32_t v[16];
            tc_ld16(rbase + g.W * h0 + 16 * cb, v);
            tc_wait_ld();
#pragma unroll
            for (int cc = 0; cc < 16; ++cc)
              if ((16 * cb + cc) / PARTS < TT) acc0[(16 * cb + cc) / PARTS] += __uint_as_float(v[cc]);
          }
        }
        if (h0 + nh == nuse) {  // TMEM reads done; no wait for earlier global stores
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_relaxed(&S.acc_empty[j][c % g.UREG]);
        }
        if (!put(h0, acc0)) good = false;
        else if (nh == 2 && !put(h0 + 1, acc1)) good = false;
      }
      if (!good) break;
      if (un.type == U_LOCAL) {
        // count the segment; the one completing the slice forms its h in this CTA's shared memory
        const int hb = un.li % NHB;
        __threadfence_block();
        named_bar(bar, 128);
        if (et == 0) {
          const int old = atomicAdd(&S.lcnt[hb], 1);
          __threadfence_block();
          S.last[grp] = old == g.SG - 1 ? 1 : 0;
        }
        named_bar(bar, 128);
        if (S.last[grp]) {
          // the previous slice of this buffer: its down MMAs must be done reading it
          if (un.li >= NHB &&
              !shared_ok(et != 0 || bwait(&S.hfree[hb], (uint32_t)(((un.li / NHB) - 1) & 1), s_abort, lim)))
            break;
          finalize_local(spart + (int64_t)hb * g.SG * g.T * 128, (int64_t)g.T * 128, g.SG, nt, tb.tok[un.u], g.W,
                         hbuf + hb * HIMG, et);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> the MMA's reads
          named_bar(bar, 128);
          if (et == 0) { S.lcnt[hb] = 0; mbar_arrive(&S.hready[hb]); }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tc_dealloc(tbase, TMEM_COLS);

  // ---------------- grid barrier, then this CTA's share of the outputs: y[t][32 jb + l] = sum_r w[t, r] *
  // (sum over the slices of expert pu[t][r], in order, of the partial), ranks in order. One warp per
  // (t, jb, r) task (lane l = row), the rank sums meet in shared memory.
  if (tb.U > 0) {
    if (threadIdx.x == 0) {
      // the CTA barrier above orders every thread's down partials before this release (cumulative at gpu scope)
      red_release_add(&hdr->gbar, 1u);
      S.gok = wait_ge(&hdr->gbar, gridDim.x, s_abort, lim) ? 1 : 0;
      if (!S.gok) record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
    }
    __syncthreads();
    if (S.gok && !*s_abort) {
      const int nb32 = g.H / 32, ntask = g.T * nb32;
      const int nmine = ntask > (int)blockIdx.x ? (ntask - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
      float* sd = reinterpret_cast<float*>(smem);  // [nmine][k][32] (the stage ring is idle now)
      const float* dpart = reinterpret_cast<const float*>(a.ws + a.L.dpart);
      for (int tk = warp; tk < nmine * g.k; tk += THREADS / 32) {
        const int ln = tk / g.k, r = tk % g.k, task = (int)blockIdx.x + ln * (int)gridDim.x;
        const int t = task / nb32, jb = task % nb32;
        const int u = tb.pu[t][r];
        const int col = tb.col0[u] + tb.ps[t][r];
        const float* p = dpart + (((int64_t)col * nb32 + jb) * g.NS) * 32 + lane;
        float sum = 0.f;
        for (int s0 = 0; s0 < g.NS; s0 += 32) {  // slices in order, loads issued 32 at a time
          float v[32];
#pragma unroll
          for (int qq = 0; qq < 32; ++qq) v[qq] = s0 + qq < g.NS ? __ldcg(p + (int64_t)(s0 + qq) * 32) : 0.f;
#pragma unroll
          for (int qq = 0; qq < 32; ++qq)
            if (s0 + qq < g.NS) sum += v[qq];
        }
        sd[(ln * MAX_K + r) * 32 + lane] = sum;
      }
      __syncthreads();
      for (int o = threadIdx.x; o < nmine * 32; o += THREADS) {
        const int ln = o >> 5, l = o & 31, task = (int)blockIdx.x + ln * (int)gridDim.x;
        const int t = task / nb32, jb = task % nb32;
        float acc = 0.f;
        for (int r = 0; r < g.k; ++r) acc = fmaf(tb.w[t][r], sd[(ln * MAX_K + r) * 32 + l], acc);
        const int64_t yi = (int64_t)t * g.H + 32 * jb + l;
        const float out = a.accumulate ? a.y[yi] + acc : acc;
        a.y[yi] = out;
        if (a.yb) a.yb[yi] = __float2bfloat16_rn(out);
      }
    }
  }
  // the last CTA to finish resets the per-call counters
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t old = atomicAdd(&hdr->done, 1u);
    if (old == gridDim.x - 1) {
      __threadfence();
      for (int r = 0; r < g.R; ++r) { cnt[C_SPLIT + r] = 0; cnt[C_HREADY + r] = 0; }
      cnt[C_XP] = 0;
      cnt[C_ROUTE] = 0;
      hdr->gbar = 0;
      __threadfence();
      hdr->done = 0;
    }
  }
}

// ------------------------------------------------------------------ host side
inline int64_t cols_of(int T, int k) { return (int64_t)(T * k < MAX_U ? T * k : MAX_U); }

size_t workspace_bytes(const moe_layer_t* L, int T_max, int k) {
  return (size_t)ws_layout(L->H, L->I, cols_of(T_max, k), T_max).total;
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
  if (router_w && (L->E > kRouteMaxE / 4 || k > L->E || ((uintptr_t)x & 15) || ((uintptr_t)router_w & 15)))
    return router_w && L->E > kRouteMaxE / 4 ? MOE_ERR_SHAPE : MOE_ERR_INVALID_ARG;
  const int nsm = moe_internal::num_sms();
  if (nsm <= 0 || nsm > RMAX) return MOE_ERR_CUDA;
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
  a.y = y;
  a.yb = (__nv_bfloat16*)y_bf16;
  a.accumulate = accumulate;
  a.ws = (uint8_t*)ws;
  a.L = ws_layout(L->H, L->I, cols_of(tmax, k), tmax);
  a.ts = tmax;
  a.wait_ns = kDefaultWaitNs;
  Geo& g = a.g;
  g = Geo{};
  g.H = L->H; g.I = L->I; g.T = T; g.k = k; g.E = L->E;
  g.W = 16 * ((PARTS * T + 15) / 16);
  g.NS = L->I / 64; g.NQ = L->H / 256; g.KTG = L->H / 128; g.SG = sg_for(g.KTG); g.KSG = g.KTG / g.SG;
  // TMEM: every unit of a pipeline takes one accumulator region; a local down unit of NC chunks needs 2 NC
  // accumulators of W columns. Two chunks per unit when two such regions still fit in a pipeline's share.
  const int share = (int)SF_COL0 / NPIPE;
  g.NC = (share >= 2 * (2 * NC_MAX * g.W) && g.NQ % NC_MAX == 0) ? NC_MAX : 1;
  g.NDL = g.NQ / g.NC;
  g.RC = 2 * g.NC * g.W;
  g.UREG = share / g.RC < 8 ? share / g.RC : 8;
  g.G = nsm;
  if (g.SG > MAX_SG || g.UREG < 1) return MOE_ERR_SHAPE;
  static int smem_max = 0, static_smem = 0;
  if (!smem_max) {
    int dev = 0, v = 0;
    cudaFuncAttributes fa2, fa8;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
        cudaFuncGetAttributes(&fa2, decode_kernel<2>) != cudaSuccess || cudaFuncGetAttributes(&fa8, decode_kernel<8>) != cudaSuccess)
      return MOE_ERR_CUDA;
    static_smem = (int)(fa2.sharedSizeBytes > fa8.sharedSizeBytes ? fa2.sharedSizeBytes : fa8.sharedSizeBytes);
    smem_max = v;
  }
  g.SLOT = slot_bytes(g.W);
  g.RING = RING_MAX;  // the deepest ring that fits
  while (g.RING > 3 && (int)smem_bytes(T, g.SG, g.RING, g.SLOT) + static_smem > smem_max) --g.RING;
  if ((int)smem_bytes(T, g.SG, g.RING, g.SLOT) + static_smem > smem_max) return MOE_ERR_SHAPE;
  CUtensorMap mgu;
  if (!moe_internal::tmap_tc_weights_packed(&mgu, L->gate_up, MOE_MAT_GATE_UP, L->H, L->I, L->E)) return MOE_ERR_CUDA;
  const size_t smem = smem_bytes(T, g.SG, g.RING, g.SLOT);
  static std::once_flag once;
  static bool attr_ok = false;
  std::call_once(once, [] {
    attr_ok = cudaFuncSetAttribute(decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   smem_max - static_smem) == cudaSuccess &&
              cudaFuncSetAttribute(decode_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   smem_max - static_smem) == cudaSuccess;
  });
  if (!attr_ok) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nsm);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = T <= 2 ? cudaLaunchKernelEx(&cfg, decode_kernel<2>, mgu, a) : cudaLaunchKernelEx(&cfg, decode_kernel<8>, mgu, a);
  if (le != cudaSuccess) return MOE_ERR_CUDA;
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
