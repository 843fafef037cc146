// prefill.cu -- prefill grouped GEMM: the routed experts applied to many tokens at once, as dense contractions on
// the 5th-generation tensor cores (block-scaled MXFP4 weights x MXFP8 activations, fp32 accumulation in TMEM).
//
// Steps (one call, all on the caller's stream):
//   1. bucket_hist / bucket_scan / bucket_place: a stable counting sort of the (token, rank) pairs by expert.
//      Each expert's pairs occupy whole 128-row tiles of the activation buffers (the last tile of an expert is
//      partly filled); pair order inside an expert is (token, rank) order.
//   2. quant_x: every pair's token row x (bf16) is quantised to MXFP8 (E4M3 codes, one E8M0 exponent per 32
//      along H) into its row of the sorted activation buffer; the exponents go straight into the permuted
//      512-byte blocks that tcgen05.cp loads into TMEM.
//   3. gemm<GATE_UP>: per (tile, 64 intermediate indices) unit, G|U = X_tile * [Gate;Up]^T over K = H; the
//      epilogue forms h = SiLU(g) * u in fp32 and quantises it to MXFP8 (per 32 along I) for the next GEMM.
//   4. gemm<DOWN>: per (tile, 128 hidden indices) unit, D = H_tile * Down^T over K = I, fp32 rows per pair.
//   5. combine: y[t] = sum_r w[t, r] * D[pair (t, r)] in rank order, fp32 and/or bf16 (round to nearest even).
// The GEMM kernel is persistent (one CTA per SM) and warp-specialised: warps 0..2 issue TMA tensor copies into a
// 6-stage shared-memory ring (one issuing thread per warp: issuing lanes of one warp serialise), warp 3 issues
// tcgen05.cp (scale factors) and tcgen05.mma into one of two TMEM accumulators, warps 4..7 drain the other
// accumulator with tcgen05.ld. Every wait is bounded (timeout ->
// device status MOE_ERR_DEVICE_TIMEOUT, the CTA drains its own copies and frees TMEM).
#include <mutex>

#include "common.cuh"
#include "layout.cuh"
#include "tcgen05.cuh"
#include "api_internal.h"

namespace moe {
namespace pf {

constexpr int BM = 128;       // tokens per tile: MMA M, TMEM lanes
constexpr int BN = 128;       // weight rows per unit: MMA N, accumulator columns
constexpr int BK = 128;       // K per pipeline stage (4 MMAs of K = 32)
constexpr int A_BYTES = BM * BK;          // E4M3 activations, 16 KB
constexpr int B_BYTES = BN * BK;          // E2M1 weights as unpacked into shared memory (one byte per code)
constexpr int B_TX = BN * BK / 2;         // bytes the TMA engine reads for them
constexpr int SF_BYTES = 512;
// A stage: codes of A and B, then the exponent blocks of A and of B. Gate/up: B is one 128 x 128 weight tile, loaded
// by the TMA engine's 16U4 unpacking. Down: the stage's 128 columns are two 64-column chunks of the DOWN layout
// (each with its own exponent block); their packed codes are bulk-copied into a staging area and expanded by four
// converter warps into the same padded, 128-byte-swizzled operand (the unpacking TMA only takes 128-code boxes).
constexpr int SF_OFF = A_BYTES + B_BYTES;            // exponents: A, B (chunk 0), B (chunk 1)
constexpr int STAGING_OFF = SF_OFF + 4 * SF_BYTES;   // down only: the two chunks' packed codes, 2 x 4 KB
template <int PHASE> struct StageCfg;
template <> struct StageCfg<0> { static constexpr int STAGES = 6, BYTES = SF_OFF + 2 * SF_BYTES; };   // 33 KB
template <> struct StageCfg<1> { static constexpr int STAGES = 5, BYTES = STAGING_OFF + 8192; };     // 42 KB
constexpr int MAX_STAGES = 6;
constexpr uint32_t GU_TX = A_BYTES + B_TX + 2 * SF_BYTES;
constexpr uint32_t DN_TX = A_BYTES + 3 * SF_BYTES;    // the packed codes count on their own barrier
constexpr int PRODUCERS = 3;             // TMA-issuing warps (lane 0 of warps 0 .. PRODUCERS - 1)
constexpr int W_MMA = PRODUCERS;         // the MMA-issuing warp
constexpr int W_EPI = 4;                 // epilogue warps 4 .. 7 (TMEM lanes 32 (warp % 4) ..)
constexpr int W_CVT = 8;                 // converter warps 8 .. 11 (down only)
constexpr int THREADS = (W_CVT + 4) * 32;
static_assert(W_MMA < W_EPI, "warp roles");
constexpr uint32_t TMEM_COLS = 512;       // accumulators at columns 0 and 128, scale columns from 256 (12 per stage)
constexpr uint32_t SF_COL0 = 256;
static_assert(SF_COL0 + 12 * MAX_STAGES <= TMEM_COLS, "TMEM budget");
template <int PHASE> constexpr int smem_of() { return StageCfg<PHASE>::STAGES * StageCfg<PHASE>::BYTES + 1024 + 512; }
static_assert(StageCfg<0>::BYTES % 1024 == 0 && StageCfg<1>::BYTES % 1024 == 0, "stage alignment");
constexpr int ACT_TILE = A_BYTES + SF_BYTES;  // one 128-row x 128-column activation tile: codes, then exponents
constexpr int PLACE_CHUNK = 256;          // pairs per CTA of the counting sort
constexpr int MAX_E = 1024;

enum { GATE_UP = 0, DOWN = 1 };

// ------------------------------------------------------------------ workspace layout (byte offsets)
struct Plan {
  int64_t npairs, tiles_max, rows_max, nchunks;
  int64_t o_cnt, o_tstart, o_chist, o_tile_e, o_tile_n, o_tile_c0, o_pslot, o_xq, o_hq, o_dout, total;
};
// header (status word) 0..255; n_tiles at byte 256
constexpr int64_t kNTilesOff = 256;

inline int64_t al(int64_t v) { return (v + 1023) & ~(int64_t)1023; }

inline Plan make_plan(int64_t T, int64_t k, int64_t E, int64_t H, int64_t I) {
  Plan p;
  p.npairs = T * k;
  p.tiles_max = (p.npairs + BM - 1) / BM + (E < p.npairs ? E : p.npairs);
  p.rows_max = p.tiles_max * BM;
  p.nchunks = (p.npairs + PLACE_CHUNK - 1) / PLACE_CHUNK;
  int64_t o = 1024;
  p.o_cnt = o;    o = al(o + E * 4);
  p.o_tstart = o; o = al(o + (E + 1) * 4);
  p.o_chist = o;  o = al(o + p.nchunks * E * 4);
  p.o_tile_e = o; o = al(o + p.tiles_max * 4);
  p.o_tile_n = o; o = al(o + p.tiles_max * 4);
  p.o_tile_c0 = o; o = al(o + p.tiles_max * 4);
  p.o_pslot = o;  o = al(o + p.npairs * 4);
  p.o_xq = o;     o = al(o + p.tiles_max * (H / 128) * ACT_TILE);
  p.o_hq = o;     o = al(o + p.tiles_max * (I / 128) * ACT_TILE);
  p.o_dout = o;   o = al(o + p.npairs * H * 4);
  p.total = o;
  return p;
}

// ------------------------------------------------------------------ MXFP8 quantiser
// Exponent of a block whose largest magnitude is amax: e = clamp(k + 127, 1, 254) with k the smallest integer
// such that amax <= 448 * 2^k (448 = 1.75 * 2^8 is the largest E4M3 value).
__device__ __forceinline__ int mx8_exponent(float amax) {
  const uint32_t ab = __float_as_uint(amax) & 0x7FFFFFFFu;
  const int ef = (int)(ab >> 23);
  if (ef == 0) return 1;                      // zero or subnormal amax: k + 127 < 1
  int e = ef - 8 + ((ab & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return e < 1 ? 1 : (e > 254 ? 254 : e);
}
// 2^(127 - e) as fp32 for e in [1, 254]
__device__ __forceinline__ float mx8_inv_scale(int e) {
  return e <= 253 ? __uint_as_float((uint32_t)(254 - e) << 23) : __uint_as_float(0x00400000u);
}
// two fp32 -> two E4M3 codes, round to nearest even, saturating to +-448; `lo` lands in the low byte
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}
// Quantise 32 fp32 values: returns the exponent, writes 32 codes as 8 words (element j in byte j).
__device__ __forceinline__ int quant_block32(const float (&v)[32], uint32_t (&codes)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  const int e = mx8_exponent(amax);
  const float s = mx8_inv_scale(e);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t a = e4m3x2(v[4 * w] * s, v[4 * w + 1] * s);
    const uint32_t b = e4m3x2(v[4 * w + 2] * s, v[4 * w + 3] * s);
    codes[w] = a | (b << 16);
  }
  return e;
}
// byte offset of (tile row r, 32-block kb of a 128-column group) inside a permuted 512-byte scale block
__device__ __forceinline__ int sf_byte(int r, int kb) { return (r & 31) * 16 + (r >> 5) * 4 + kb; }
// Sorted activation buffers (x, then h) are tile-major like the weights: tile (row tile, 128-column group) is
// 16 KB of E4M3 codes [128 rows][128] followed by its 512-byte permuted exponent block.
__device__ __forceinline__ int64_t act_tile(int64_t tile, int KG, int kg) { return (tile * KG + kg) * (int64_t)ACT_TILE; }

// ------------------------------------------------------------------ 1. counting sort of (token, rank) pairs
__global__ void bucket_hist(const int32_t* idx, int64_t npairs, int E, int32_t* chist, int32_t* status) {
  __shared__ int32_t h[MAX_E];
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const int64_t p = (int64_t)blockIdx.x * PLACE_CHUNK + threadIdx.x;
  if (p < npairs) {
    const int e = idx[p];
    if (e >= 0 && e < E) atomicAdd(&h[e], 1);
    else record_error(status, MOE_ERR_INVALID_ARG);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chist[(int64_t)blockIdx.x * E + e] = h[e];
}

// One CTA of 1024 threads: per-expert totals, tile and pair prefix sums, per-chunk offsets, the tile table.
__global__ void __launch_bounds__(1024) bucket_scan(int E, int64_t nchunks, int32_t* chist, int32_t* cnt,
                                                    int32_t* tstart, int32_t* tile_e, int32_t* tile_n,
                                                    int32_t* tile_c0, uint32_t* n_tiles) {
  __shared__ int32_t s_t[MAX_E], s_p[MAX_E];
  const int e = threadIdx.x;
  int32_t c = 0;
  if (e < E) {
    for (int64_t ch = 0; ch < nchunks; ++ch) {
      const int32_t v = chist[ch * E + e];
      chist[ch * E + e] = c;  // offset of this chunk's pairs inside the expert
      c += v;
    }
    cnt[e] = c;
  }
  s_t[e] = e < E ? (c + BM - 1) / BM : 0;
  s_p[e] = e < E ? c : 0;
  __syncthreads();
  // inclusive scans (Hillis-Steele over 1024 entries)
  for (int d = 1; d < MAX_E; d <<= 1) {
    const int32_t a = e >= d ? s_t[e - d] : 0, b = e >= d ? s_p[e - d] : 0;
    __syncthreads();
    s_t[e] += a;
    s_p[e] += b;
    __syncthreads();
  }
  if (e < E) {
    const int32_t t1 = s_t[e], t0 = t1 - (c + BM - 1) / BM, p0 = s_p[e] - c;
    tstart[e] = t0;
    if (e == E - 1) { tstart[E] = t1; *n_tiles = (uint32_t)t1; }
    for (int32_t j = 0; t0 + j < t1; ++j) {
      tile_e[t0 + j] = e;
      tile_n[t0 + j] = min(BM, c - j * BM);
      tile_c0[t0 + j] = p0 + j * BM;
    }
  }
}

// Rows of the pairs of one chunk: row = 128 * tstart[e] + (offset of the chunk in e) + (rank inside the chunk).
__global__ void bucket_place(const int32_t* idx, int64_t npairs, int E, const int32_t* chist, const int32_t* tstart,
                             int32_t* pslot) {
  constexpr int NW = PLACE_CHUNK / 32;
  __shared__ int32_t wh[NW][MAX_E];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < NW * E; i += blockDim.x) wh[i / E][i % E] = 0;
  __syncthreads();
  const int64_t p = (int64_t)blockIdx.x * PLACE_CHUNK + threadIdx.x;
  int e = p < npairs ? idx[p] : -1;
  if (e >= E) e = -1;
  const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
  const int rank = __popc(peers & ((1u << lane) - 1));
  if (e >= 0 && rank == 0) wh[warp][e] = __popc(peers);
  __syncthreads();
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int32_t run = chist[(int64_t)blockIdx.x * E + x];
    for (int w = 0; w < NW; ++w) {
      const int32_t v = wh[w][x];
      wh[w][x] = run;
      run += v;
    }
  }
  __syncthreads();
  if (p < npairs) pslot[p] = e >= 0 ? tstart[e] * BM + wh[warp][e] + rank : -1;
}

// ------------------------------------------------------------------ 2. MXFP8 activations of every pair
// One warp per pair; lane j quantises 32-blocks j, j+32, ...
__global__ void quant_x(const uint16_t* x, int k, int64_t npairs, int H, const int32_t* pslot, uint8_t* xq) {
  const int64_t p = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (p >= npairs) return;
  const int32_t row = pslot[p];
  if (row < 0) return;
  const int64_t t = p / k;
  const int tile = row / BM, r = row % BM, KG = H / 128;
  for (int b = lane; b < H / 32; b += 32) {
    const uint4* src = reinterpret_cast<const uint4*>(x + t * H + b * 32);
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = src[q];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[q * 8 + 2 * i] = __uint_as_float(w[i] << 16);
        v[q * 8 + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
    uint32_t c[8];
    const int e = quant_block32(v, c);
    uint8_t* at = xq + act_tile(tile, KG, b / 4);
    uint4* dst = reinterpret_cast<uint4*>(at + r * 128 + (b % 4) * 32);
    dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
    dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
    at[A_BYTES + sf_byte(r, b % 4)] = (uint8_t)e;
  }
}

// ------------------------------------------------------------------ 3, 4. the grouped GEMM
struct GemmArgs {
  const uint8_t* w;           // packed weights of the layer (tensor-core layout)
  int64_t wstride;            // bytes per expert
  int K, NB;                  // reduction size; 128-row weight blocks per expert
  const uint8_t* act;         // sorted activations, tile-major with exponent blocks
  const int32_t* tile_e;
  const int32_t* tile_n;
  const int32_t* tile_c0;
  const uint32_t* n_tiles;
  uint8_t* hq;                // GATE_UP: MXFP8 h, tile-major like the activations
  float* gu_dump;             // GATE_UP, tests only: fp32 g and u [rows][2I] (NULL in the product path)
  int I;
  float* dout;                // DOWN: fp32 rows [pairs][H] (compact pair order)
  int H;
  int32_t* status;
  long long wait_ns;
};

// Bounded mbarrier wait that also gives up when another role of the CTA has given up.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, long long lim) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > lim) { *abort_flag = 1; return false; }
  }
}

template <int PHASE>
__global__ void __launch_bounds__(THREADS, 1) gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                                                          const __grid_constant__ CUtensorMap tmB, const GemmArgs a) {
  constexpr int STAGES = StageCfg<PHASE>::STAGES, STAGE_BYTES = StageCfg<PHASE>::BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* full = bars;                 // [STAGES] TMA (and, down, the converters) -> MMA
  uint64_t* empty = bars + STAGES;       // [STAGES] MMA -> TMA
  uint64_t* acc_full = bars + 2 * STAGES;       // [2] MMA -> epilogue
  uint64_t* acc_empty = bars + 2 * STAGES + 2;  // [2] epilogue -> MMA
  uint64_t* drain = bars + 2 * STAGES + 4;
  uint64_t* packed = bars + 2 * STAGES + 5;     // [STAGES] down: packed codes landed -> converters
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 5);
  volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // full: the producer's arrival with its byte count (down: also one arrival per converter warp)
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], PHASE == DOWN ? 5 : 1);
      mbar_init(&empty[s], 1);
      mbar_init(&packed[s], 1);
    }
    for (int s = 0; s < 2; ++s) { mbar_init(&acc_full[s], 1); mbar_init(&acc_empty[s], 4); }
    mbar_init(drain, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == W_MMA) tc_alloc(s_tmem, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *s_tmem;
  const int KG = a.K / BK;
  const int64_t n_units = (int64_t)(*a.n_tiles) * a.NB;
  const long long lim = a.wait_ns;

  if (warp < PRODUCERS) {
    // ---------------- TMA producers. One issuing thread completes about one wait-and-issue round per 330 ns on
    // GB300 however many bytes it moves, so PRODUCERS warps take turns: warp w issues all four copies of stages
    // w, w + PRODUCERS, ... of this CTA's sequence of (unit, k-group) stages.
    if (lane == 0) {
      int issued_slot = -1;
      uint32_t issued_ph = 0;
      bool ok = true;
      for (int64_t g = warp;; g += PRODUCERS) {
        const int64_t u = blockIdx.x + (g / KG) * gridDim.x;
        if (u >= n_units) break;
        const int kg = (int)(g % KG), s = (int)(g % STAGES);
        const uint32_t ph = (uint32_t)((g / STAGES) & 1);
        if (!pf_wait(&empty[s], ph ^ 1, s_abort, lim)) { ok = false; break; }
        const int tile = (int)(u / a.NB), nb = (int)(u % a.NB);
        const int e = a.tile_e[tile];
        uint8_t* st = smem + s * STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], PHASE == DOWN ? DN_TX : GU_TX);
        tma_load_3d(st, &tmA, 0, 0, tile * KG + kg, &full[s]);
        bulk_g2s_plain(st + SF_OFF, a.act + act_tile(tile, KG, kg) + A_BYTES, SF_BYTES, &full[s]);
        if (PHASE == GATE_UP) {
          const uint8_t* wt = a.w + (int64_t)e * a.wstride + ((int64_t)nb * KG + kg) * kTcTileBytes;
          tma_load_4d(st + A_BYTES, &tmB, 0, 0, nb * KG + kg, e, &full[s]);
          bulk_g2s_plain(st + SF_OFF + SF_BYTES, wt + 8192, SF_BYTES, &full[s]);
        } else {
          // down: weight rows 128 nb .. +127 are half nb % 2 of row pair nb / 2 in the chunks of slices 2 kg and
          // 2 kg + 1 (64 columns each): 128 rows x 32 B of packed codes, contiguous in each chunk
          const int NQ = a.H / 256, NS = a.I / 64;
          mbar_arrive_expect_tx(&packed[s], 8192);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint8_t* ch = a.w + (((int64_t)e * NS + 2 * kg + h) * NQ + nb / 2) * kTcTileBytes;
            bulk_g2s_plain(st + STAGING_OFF + 4096 * h, ch + 4096 * (nb & 1), 4096, &packed[s]);
            bulk_g2s_plain(st + SF_OFF + (1 + h) * SF_BYTES, ch + 8192, SF_BYTES, &full[s]);
          }
        }
        issued_slot = s;
        issued_ph = ph;
      }
      if (!ok) {
        record_error(a.status, MOE_ERR_DEVICE_TIMEOUT);
        // let the last stage this lane issued land before the CTA's shared memory is released
        if (issued_slot >= 0) mbar_wait(&full[issued_slot], issued_ph, 100000000LL);
      }
    }
    __syncwarp();
  } else if (warp == W_MMA) {
    // ---------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t ph = 0;
      bool ok = true;
      int j = 0;
      for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++j) {
        const int acc = j & 1;
        const uint32_t use = (uint32_t)(j >> 1);
        if (!pf_wait(&acc_empty[acc], (use & 1) ^ 1, s_abort, lim)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tbase + (uint32_t)(acc * BN);
        for (int kg = 0; kg < KG; ++kg) {
          if (!pf_wait(&full[stage], ph, s_abort, lim)) { ok = false; break; }
          tc_fence_after();
          uint8_t* st = smem + stage * STAGE_BYTES;
          const uint32_t sfa = tbase + SF_COL0 + (uint32_t)(stage * 12), sfb = sfa + 4;
          tc_cp_sf(sfa, umma_desc_sf(smem_u32(st + SF_OFF)));
          tc_cp_sf(sfb, umma_desc_sf(smem_u32(st + SF_OFF + SF_BYTES)));
          const uint64_t ad = umma_desc_sw128(smem_u32(st)), bd = umma_desc_sw128(smem_u32(st + A_BYTES));
          if (PHASE == GATE_UP) {
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)
              tc_mma_mxf8f6f4(d_tmem, ad + 2 * kb, bd + 2 * kb, idesc_mxf8f6f4(0, 5, BM, BN, kb, kb), sfa, sfb,
                              (kg | kb) != 0);
          } else {
            // K-blocks 0, 1 come from chunk 0 and 2, 3 from chunk 1, each chunk with its own exponent block; the
            // weight rows are half nb % 2 of their chunks' row pair, so they read scale bytes 2 (nb % 2) + (0, 1)
            tc_cp_sf(sfb + 4, umma_desc_sf(smem_u32(st + SF_OFF + 2 * SF_BYTES)));
            const int nb = (int)(u % a.NB);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb)
              tc_mma_mxf8f6f4(d_tmem, ad + 2 * kb, bd + 2 * kb,
                              idesc_mxf8f6f4(0, 5, BM, BN, kb, (uint32_t)(2 * (nb & 1) + (kb & 1))), sfa,
                              sfb + 4 * (kb >> 1), (kg | kb) != 0);
          }
          tc_commit(&empty[stage]);  // the stage is free once these MMAs have read it
          if (++stage == STAGES) { stage = 0; ph ^= 1; }
        }
        if (ok) tc_commit(&acc_full[acc]);
      }
      if (!ok) record_error(a.status, MOE_ERR_DEVICE_TIMEOUT);
      tc_commit(drain);  // completes when every tcgen05 operation issued above has finished
      mbar_wait(drain, 0, 100000000LL);
    }
    __syncwarp();
  } else if (warp >= W_CVT) {
    // ---------------- down converters: expand each stage's packed codes into the padded operand the MMA reads
    // (what the TMA engine's 16U4_ALIGN16B type writes: every 8 packed bytes followed by 8 bytes of gap, 128-byte
    // rows, 16-byte chunk c of row r at chunk c ^ (r % 8)). Chunk c of weight row r holds codes 16c .. 16c + 15 of the
    // stage's 128 columns: from the staged chunk c / 4, bytes 8 (c % 4) .. +7 of the row's 32 (stored in the layout's
    // 32-byte swizzle: 16-byte half (c % 4) / 2 of row r sits at half ((c % 4) / 2) ^ ((r >> 2) & 1)).
    if (PHASE == DOWN) {
      const int ct = threadIdx.x - W_CVT * 32;
      int64_t g = 0;
      bool ok = true;
      for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x)
        for (int kg = 0; kg < KG; ++kg, ++g) {
          const int s = (int)(g % STAGES);
          uint8_t* st = smem + s * STAGE_BYTES;
          int w = 1;
          if (lane == 0) w = pf_wait(&packed[s], (uint32_t)((g / STAGES) & 1), s_abort, lim) ? 1 : 0;
          if (!__shfl_sync(0xFFFFFFFFu, w, 0)) { ok = false; break; }
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int idx = ct + 128 * it, r = idx >> 3, c = idx & 7;
            const int hh = ((c & 3) >> 1) ^ ((r >> 2) & 1);
            const uint2 v = *reinterpret_cast<const uint2*>(st + STAGING_OFF + 4096 * (c >> 2) + r * 32 + hh * 16 + (c & 1) * 8);
            *reinterpret_cast<uint4*>(st + A_BYTES + r * 128 + ((c ^ (r & 7)) << 4)) = make_uint4(v.x, v.y, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> the MMA's reads
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[s]);
        }
      if (!ok) record_error(a.status, MOE_ERR_DEVICE_TIMEOUT);
    }
  } else {
    // ---------------- epilogue: warps 4..7 own TMEM lanes 32*(warp % 4) .. +31
    const int q = warp & 3;
    const int r = q * 32 + lane;  // tile row = token slot inside the tile
    int j = 0;
    for (int64_t u = blockIdx.x; u < n_units; u += gridDim.x, ++j) {
      const int acc = j & 1;
      const uint32_t use = (uint32_t)(j >> 1);
      int ok = 1;
      if (lane == 0) ok = pf_wait(&acc_full[acc], use & 1, s_abort, lim) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int tile = (int)(u / a.NB), nb = (int)(u % a.NB);
      const bool valid = r < a.tile_n[tile];
      const uint32_t taddr = tbase + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      if (PHASE == GATE_UP) {
        const int64_t row = (int64_t)tile * BM + r;
#pragma unroll 1
        for (int hb = 0; hb < 2; ++hb) {
          uint32_t g0[16], g1[16], u0[16], u1[16];
          tc_ld16(taddr + 32 * hb, g0);
          tc_ld16(taddr + 32 * hb + 16, g1);
          tc_ld16(taddr + 64 + 32 * hb, u0);
          tc_ld16(taddr + 64 + 32 * hb + 16, u1);
          tc_wait_ld();
          float h[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float g = __uint_as_float(c < 16 ? g0[c] : g1[c - 16]);
            const float uu = __uint_as_float(c < 16 ? u0[c] : u1[c - 16]);
            h[c] = g / (1.0f + expf(-g)) * uu;
          }
          uint32_t codes[8];
          const int e = quant_block32(h, codes);
          if (valid) {
            const int i0 = nb * 64 + hb * 32;
            uint8_t* at = a.hq + act_tile(tile, a.I / 128, i0 / 128);
            uint4* dst = reinterpret_cast<uint4*>(at + r * 128 + i0 % 128);
            dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
            dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
            at[A_BYTES + sf_byte(r, (i0 % 128) / 32)] = (uint8_t)e;
            if (a.gu_dump) {
              float* gd = a.gu_dump + row * 2 * a.I;
              for (int c = 0; c < 32; ++c) {
                gd[i0 + c] = __uint_as_float(c < 16 ? g0[c] : g1[c - 16]);
                gd[a.I + i0 + c] = __uint_as_float(c < 16 ? u0[c] : u1[c - 16]);
              }
            }
          }
        }
      } else {
        float* dst = a.dout + ((int64_t)a.tile_c0[tile] + r) * a.H + nb * BN;
#pragma unroll 1
        for (int cb = 0; cb < BN / 16; ++cb) {
          uint32_t v[16];
          tc_ld16(taddr + 16 * cb, v);
          tc_wait_ld();
          if (valid) {
            float4* d4 = reinterpret_cast<float4*>(dst + 16 * cb);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                  __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == W_MMA) tc_dealloc(tbase, TMEM_COLS);
}

// ------------------------------------------------------------------ 5. weighted combine in rank order
__global__ void combine(const float* dout, const int32_t* pslot, const int32_t* tile_c0, const float* wts, int k, int H,
                        float* y, __nv_bfloat16* yb) {
  const int64_t t = blockIdx.x;
  const int j = (blockIdx.y * blockDim.x + threadIdx.x) * 4;
  if (j >= H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int r = 0; r < k; ++r) {
    const int32_t row = pslot[t * k + r];
    if (row < 0) continue;
    const float w = wts[t * k + r];
    const float4 d = *reinterpret_cast<const float4*>(dout + ((int64_t)tile_c0[row / BM] + row % BM) * H + j);
    acc.x = fmaf(w, d.x, acc.x);
    acc.y = fmaf(w, d.y, acc.y);
    acc.z = fmaf(w, d.z, acc.z);
    acc.w = fmaf(w, d.w, acc.w);
  }
  if (y) *reinterpret_cast<float4*>(y + t * H + j) = acc;
  if (yb) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    __nv_bfloat162* d = reinterpret_cast<__nv_bfloat162*>(yb + t * H + j);
    d[0] = lo;
    d[1] = hi;
  }
}

// ------------------------------------------------------------------ host side
// 3-D map over tile-major E4M3 activations: [n tiles][128 rows][128 B], tile stride ACT_TILE
bool map_act(CUtensorMap* m, const void* base, int64_t ntiles) {
  const uint64_t dims[3] = {128, 128, (uint64_t)ntiles}, strides[2] = {128, (uint64_t)ACT_TILE};
  const uint32_t box[3] = {BK, BM, 1};
  return moe_internal::tmap_u8(m, base, 3, dims, strides, box);
}

bool check_layer(const moe_layer_t* L) {
  return L && L->fmt == MOE_FMT_MXFP4 && L->layout == MOE_LAYOUT_PREFILL && L->E >= 1 && L->E <= MAX_E &&
         moe_internal::shape_ok(L->H, L->I) && L->gate_up && L->down && ((uintptr_t)L->gate_up & 15) == 0 &&
         ((uintptr_t)L->down & 15) == 0;
}

moe_status_t run(const moe_layer_t* L, const void* x_bf16, int32_t T, const int32_t* idx, const float* w, int32_t k,
                 float* y, void* y_bf16, void* ws, size_t ws_bytes, float* gu_dump, void* stream) {
  if (moe_internal::fault("prefill")) return MOE_ERR_FAULT_INJECTED;
  if (!L || !x_bf16 || !idx || !w || !ws || (!y && !y_bf16)) return MOE_ERR_INVALID_ARG;
  if (L->fmt != MOE_FMT_MXFP4 || L->layout != MOE_LAYOUT_PREFILL) return MOE_ERR_UNSUPPORTED_FORMAT;
  if (!check_layer(L)) return L->E > MAX_E || !moe_internal::shape_ok(L->H, L->I) ? MOE_ERR_SHAPE : MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || k > 8 || k > L->E) return MOE_ERR_SHAPE;
  if (((uintptr_t)x_bf16 & 15) || ((uintptr_t)ws & 255) || ((uintptr_t)y & 15) || ((uintptr_t)y_bf16 & 7) ||
      ((uintptr_t)idx & 3) || ((uintptr_t)w & 3))
    return MOE_ERR_INVALID_ARG;
  const Plan P = make_plan(T, k, L->E, L->H, L->I);
  if (ws_bytes < (size_t)P.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  if (!moe_internal::tmap_available()) return MOE_ERR_CUDA;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* B = (uint8_t*)ws;
  int32_t* status = reinterpret_cast<int32_t*>(B);
  uint32_t* n_tiles = reinterpret_cast<uint32_t*>(B + kNTilesOff);
  int32_t* cnt = reinterpret_cast<int32_t*>(B + P.o_cnt);
  int32_t* tstart = reinterpret_cast<int32_t*>(B + P.o_tstart);
  int32_t* chist = reinterpret_cast<int32_t*>(B + P.o_chist);
  int32_t* tile_e = reinterpret_cast<int32_t*>(B + P.o_tile_e);
  int32_t* tile_n = reinterpret_cast<int32_t*>(B + P.o_tile_n);
  int32_t* tile_c0 = reinterpret_cast<int32_t*>(B + P.o_tile_c0);
  int32_t* pslot = reinterpret_cast<int32_t*>(B + P.o_pslot);
  const int H = L->H, I = L->I, E = L->E;

  // tensor maps (host encodes; they travel as __grid_constant__ kernel parameters)
  const TcGeom ggu = tc_geom(MOE_MAT_GATE_UP, H, I), gdn = tc_geom(MOE_MAT_DOWN, H, I);
  CUtensorMap mx, mgu, mh, mdn = {};  // mdn: unused by the down GEMM, which bulk-copies its packed chunks
  if (!map_act(&mx, B + P.o_xq, P.tiles_max * (H / 128)) || !moe_internal::tmap_tc_weights(&mgu, L->gate_up, MOE_MAT_GATE_UP, H, I, E) ||
      !map_act(&mh, B + P.o_hq, P.tiles_max * (I / 128)))
    return MOE_ERR_CUDA;

  static std::once_flag attr_once;
  static bool attr_ok = false;
  std::call_once(attr_once, [] {
    attr_ok = cudaFuncSetAttribute(gemm_kernel<GATE_UP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   smem_of<GATE_UP>()) == cudaSuccess &&
              cudaFuncSetAttribute(gemm_kernel<DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   smem_of<DOWN>()) == cudaSuccess;
  });
  if (!attr_ok) return MOE_ERR_CUDA;

  const int nch = (int)P.nchunks;
  bucket_hist<<<nch, PLACE_CHUNK, 0, s>>>(idx, P.npairs, E, chist, status);
  bucket_scan<<<1, 1024, 0, s>>>(E, P.nchunks, chist, cnt, tstart, tile_e, tile_n, tile_c0, n_tiles);
  bucket_place<<<nch, PLACE_CHUNK, 0, s>>>(idx, P.npairs, E, chist, tstart, pslot);
  quant_x<<<(int)((P.npairs * 32 + 255) / 256), 256, 0, s>>>((const uint16_t*)x_bf16, k, P.npairs, H, pslot,
                                                             B + P.o_xq);
  const int grid = moe_internal::num_sms();
  GemmArgs ga{};
  ga.w = (const uint8_t*)L->gate_up;
  ga.wstride = ggu.stride;
  ga.K = H;
  ga.NB = (int)(ggu.R / BN);
  ga.act = B + P.o_xq;
  ga.tile_e = tile_e;
  ga.tile_n = tile_n;
  ga.tile_c0 = tile_c0;
  ga.n_tiles = n_tiles;
  ga.hq = B + P.o_hq;
  ga.gu_dump = gu_dump;
  ga.I = I;
  ga.dout = reinterpret_cast<float*>(B + P.o_dout);
  ga.H = H;
  ga.status = status;
  ga.wait_ns = kDefaultWaitNs;
  gemm_kernel<GATE_UP><<<grid, THREADS, smem_of<GATE_UP>(), s>>>(mx, mgu, ga);
  GemmArgs gd = ga;
  gd.w = (const uint8_t*)L->down;
  gd.wstride = gdn.stride;
  gd.K = I;
  gd.NB = (int)(gdn.R / BN);
  gd.act = B + P.o_hq;
  gd.gu_dump = nullptr;
  gemm_kernel<DOWN><<<grid, THREADS, smem_of<DOWN>(), s>>>(mh, mdn, gd);
  dim3 cg(T, (H / 4 + 255) / 256);
  combine<<<cg, 256, 0, s>>>(ga.dout, pslot, tile_c0, w, k, H, y, (__nv_bfloat16*)y_bf16);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace pf
}  // namespace moe

using namespace moe;

extern "C" size_t moe_prefill_workspace_bytes(const moe_layer_t* L, int32_t T_max, int32_t k) {
  if (!L || L->E < 1 || L->E > pf::MAX_E || !moe_internal::shape_ok(L->H, L->I) || T_max < 1 || k < 1 || k > 8)
    return 0;
  return (size_t)pf::make_plan(T_max, k, L->E, L->H, L->I).total;
}

extern "C" moe_status_t moe_expert_grouped_gemm_prefill(const moe_layer_t* layer, const void* x_bf16, int32_t T,
                                                        const int32_t* idx, const float* w, int32_t k, float* y,
                                                        void* y_bf16, void* ws, size_t ws_bytes, void* stream) {
  MOE_NVTX("moe_expert_grouped_gemm_prefill");
  return pf::run(layer, x_bf16, T, idx, w, k, y, y_bf16, ws, ws_bytes, nullptr, stream);
}

extern "C" moe_status_t moe_debug_prefill(const moe_layer_t* layer, const void* x_bf16, int32_t T, const int32_t* idx,
                                          const float* w, int32_t k, float* y, void* y_bf16, void* ws, size_t ws_bytes,
                                          float* gu_dump, int64_t* offsets, void* stream) {
  if (offsets) {
    if (!layer || T < 1 || k < 1) return MOE_ERR_INVALID_ARG;
    const pf::Plan P = pf::make_plan(T, k, layer->E, layer->H, layer->I);
    const int64_t o[8] = {P.rows_max, P.tiles_max, pf::kNTilesOff, P.o_tile_c0, P.o_pslot, P.o_xq, P.o_hq, P.o_dout};
    for (int i = 0; i < 8; ++i) offsets[i] = o[i];
  }
  return pf::run(layer, x_bf16, T, idx, w, k, y, y_bf16, ws, ws_bytes, gu_dump, stream);
}
