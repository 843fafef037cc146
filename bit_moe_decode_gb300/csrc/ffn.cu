// ffn.cu -- fused routed-expert FFN for decode (T = 1) and speculative verify (T <= 8) in one persistent kernel.
//
// What it computes: y_t = sum_r w[t,r] * Down_e( SiLU(Gate_e x_t) * (Up_e x_t) ), e = idx[t,r]
//   ("quantization" glossary, ds4-learning.pages.dev, "Q4_K routed experts": fused gate+up mat-vec, then the down
//   projection accumulated into the output; "Mixed-precision compression of DeepSeek-V4-Flash" (lumirain.cn),
//   "What compression does not solve": decode is bound by one read of the active expert weights per token;
//   "Width drift" / "Why this is not a host-side patch": a verify of width 1+K must read each weight once while
//   reproducing width-1 arithmetic bit for bit).
//
// Design (one CTA per SM, cooperative launch so all CTAs are co-resident):
//   * The union of the experts of the T tokens is formed on the device (sorted, deduplicated); each expert in it
//     is read exactly once per call, whatever T is.
//   * Work units are 16-row tiles: phase G (gate/up tiles of each union expert) then phase D (down tiles). Each
//     CTA owns a contiguous range of G units and of D units.
//   * A producer warp streams tiles from HBM into an 8-13 stage shared-memory ring with 1-D bulk copies
//     (cp.async.bulk, mbarrier completion, L2 evict-first); 8 consumer warps split K of every tile, run the
//     tensor-core mat-vec (mma.m16n8k16, weights as A decoded in registers, the T tokens as the 8 B columns) and
//     reduce across warps in a fixed order through shared memory.
//   * Numerics: weights are decoded exactly to fp16; x is rescaled per token by 2^sigma into fp16; block scales
//     multiply fp32 partial sums; h = SiLU(g)*u in fp32 is rescaled per (expert, token) into fp16 for the down
//     projection; the combine sums the ranks in rank order with fp32 FMAs.
//   * Width-1 exactness: a token's column goes through the same instructions whatever T is (column-independent
//     MMA, per-token rescale, fixed warp and rank orders), so verify row t equals decode of token t bitwise.
//   * Handoff G -> D: per-expert counters, published with release adds and read with acquire loads (a full
//     fence before a relaxed atomic costs microseconds under load); D units wait (bounded) for all G tiles of
//     their expert. Then a grid barrier and each CTA combines its share of the output rows in a fixed order, so no
//     floating-point atomics are used anywhere. When every token has a single expert (a shared expert, k = 1) the
//     owner of a down tile writes y directly with the same arithmetic and the grid barrier is skipped. The last
//     CTA to finish clears the counters.
#include <mutex>

#include "common.cuh"
#include "layout.cuh"
#include "api_internal.h"

namespace moe {

constexpr int kMaxCW = 16;             // consumer warps (tensor-core mat-vec), at most
constexpr int kNR = 4;                 // reduction slots between consumers and the epilogue warp
constexpr int kMaxT = 8;
constexpr int kMaxK = 8;
constexpr int kMaxU = kMaxT * kMaxK;   // 64

// workspace: [header 256][cnt_g 64 u32][amax_h 64*8 u32] -> 4096 bytes, then h [U, 8, I] and d [U, H, 8] fp32
constexpr size_t kWsCounters = 4096;
constexpr size_t kOffCntG = 256, kOffAmax = kOffCntG + kMaxU * 4;
static_assert(kOffAmax + kMaxU * kMaxT * 4 <= kWsCounters, "counter area");

struct FfnArgs {
  const uint8_t* gate_up;
  const uint8_t* down;
  const uint16_t* x;   // [T, H] bf16
  const int32_t* idx;  // [T, k]
  const float* w;      // [T, k]
  float* y;            // [T, H]
  uint16_t* y_bf16;    // [T, H] or null
  int accumulate;
  int H, I, E, T, k;
  WsHeader* hdr;
  uint32_t* cnt_g;     // [kMaxU]
  uint32_t* amax_h;    // [kMaxU * 8]
  float* hbuf;         // [U, 8, I]
  float* dbuf;         // [U, H, 8]
  long long wait_ns;
};

template <int FMT> struct Cfg {
  using F = Fmt<FMT>;
  // Warp roles: CW consumer warps (each owns a K slice of every tile), one producer warp (bulk copies), one
  // epilogue warp (cross-warp sums, outputs, signals, combine).
  static constexpr int CW = FMT == MOE_FMT_Q2K ? 8 : 16;
  static constexpr int PROD = CW, EPI = CW + 1, THREADS = (CW + 2) * 32;
  static constexpr int SB = F::CPS * F::CB;                                // stage bytes (2048 columns)
  static constexpr int NS = FMT == MOE_FMT_Q2K ? 13 : FMT == MOE_FMT_Q8_0 ? 10 : 8;   // ring stages
  static constexpr int NCH = 4096 / F::CK / CW;                            // max chunks per warp per tile
  static constexpr int NPS = F::CPS / CW;                                  // chunks per warp per stage
  static constexpr int SXF = 0;
  static constexpr int RED = kNR * CW * 32 * 4;                            // reduction slots (floats)
  static constexpr size_t SMEM = (size_t)NS * SB + (size_t)(RED + SXF) * 4;
};

// Every instance fits a CTA's 227 KB of shared memory (the kernel's static arrays add ~6.5 KB), splits each stage
// evenly over its consumer warps, and moves chunks whose size the 1-D bulk copy accepts (multiples of 16 bytes).
template <int FMT> constexpr bool cfg_ok() {
  return Cfg<FMT>::SMEM + 8192 <= 232448 && Fmt<FMT>::CPS % Cfg<FMT>::CW == 0 && Fmt<FMT>::CB % 16 == 0 &&
         4096 % (Fmt<FMT>::CK * Cfg<FMT>::CW) == 0;
}
static_assert(cfg_ok<MOE_FMT_MXFP4>() && cfg_ok<MOE_FMT_INT4G32>() && cfg_ok<MOE_FMT_Q2K>() && cfg_ok<MOE_FMT_Q8_0>(),
              "mat-vec kernel configuration");

__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  return e == 255u ? __uint_as_float(0x7fc00000u) : __uint_as_float(e << 23);
}
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }
__device__ __forceinline__ float h16_to_f32(uint32_t b) { return __half2float(__ushort_as_half((unsigned short)b)); }

// Process one chunk: acc += (A . B) with the format's block scaling. bx: the warp's B fragments for this chunk.
template <int FMT>
__device__ __forceinline__ void chunk_mma(const uint8_t* cp, int lane, const uint32_t (&bx)[Fmt<FMT>::STEPS][2],
                                          const float* sx /* Q2_K group sums [STEPS][8] or null */, float (&acc)[4]) {
  const float zero[4] = {0.f, 0.f, 0.f, 0.f};
  if constexpr (FMT == MOE_FMT_MXFP4) {
    const uint4 cw = *reinterpret_cast<const uint4*>(cp + lane * 16);
    const uint32_t sw = *reinterpret_cast<const uint32_t*>(cp + 512 + (lane >> 2) * 4);
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      float c[4];
      const uint32_t w0 = words[2 * blk], w1 = words[2 * blk + 1];
      mma_f16(c, e2m1x2_to_f16x2(w0, 0), e2m1x2_to_f16x2(w0, 1), e2m1x2_to_f16x2(w0, 2), e2m1x2_to_f16x2(w0, 3),
              bx[2 * blk][0], bx[2 * blk][1], zero);
      mma_f16(c, e2m1x2_to_f16x2(w1, 0), e2m1x2_to_f16x2(w1, 1), e2m1x2_to_f16x2(w1, 2), e2m1x2_to_f16x2(w1, 3),
              bx[2 * blk + 1][0], bx[2 * blk + 1][1], c);
      const float sr = e8m0_to_f32((sw >> (16 * blk)) & 255u), sr8 = e8m0_to_f32((sw >> (16 * blk + 8)) & 255u);
      acc[0] = fmaf(c[0], sr, acc[0]);
      acc[1] = fmaf(c[1], sr, acc[1]);
      acc[2] = fmaf(c[2], sr8, acc[2]);
      acc[3] = fmaf(c[3], sr8, acc[3]);
    }
  } else if constexpr (FMT == MOE_FMT_INT4G32) {
    const uint4 cw = *reinterpret_cast<const uint4*>(cp + lane * 16);
    const uint2 sc = *reinterpret_cast<const uint2*>(cp + 512 + (lane >> 2) * 8);
    const uint32_t words[4] = {cw.x, cw.y, cw.z, cw.w};
    // nibble n (two's complement) -> fp16 1024 + (n^8) [low nibble slot] or 1024 + 16 (n^8) [high nibble slot],
    // then an exact fma maps it to n.
    const uint32_t one = 0x3C003C00u, m1032 = 0xE408E408u, sixteenth = 0x2C002C00u, m72 = 0xD480D480u;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      float c[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t W = words[2 * blk + h], W8 = W >> 8;
        const uint32_t a0 = hfma2(lop3_and_xor(W, 0x000F000Fu, 0x64086408u), one, m1032);
        const uint32_t a1 = hfma2(lop3_and_xor(W, 0x00F000F0u, 0x64806480u), sixteenth, m72);
        const uint32_t a2 = hfma2(lop3_and_xor(W8, 0x000F000Fu, 0x64086408u), one, m1032);
        const uint32_t a3 = hfma2(lop3_and_xor(W8, 0x00F000F0u, 0x64806480u), sixteenth, m72);
        if (h == 0) mma_f16(c, a0, a1, a2, a3, bx[2 * blk][0], bx[2 * blk][1], zero);
        else mma_f16(c, a0, a1, a2, a3, bx[2 * blk + 1][0], bx[2 * blk + 1][1], c);
      }
      const uint32_t sv = blk == 0 ? sc.x : sc.y;
      const float sr = bf16_bits_to_f32(sv & 0xFFFFu), sr8 = bf16_bits_to_f32(sv >> 16);
      acc[0] = fmaf(c[0], sr, acc[0]);
      acc[1] = fmaf(c[1], sr, acc[1]);
      acc[2] = fmaf(c[2], sr8, acc[2]);
      acc[3] = fmaf(c[3], sr8, acc[3]);
    }
  } else if constexpr (FMT == MOE_FMT_Q8_0) {
    // Each 32-bit word holds registers 2i, 2i+1 of a step (4 codes). A code q (two's complement) becomes the fp16
    // 1024 + (q ^ 0x80) = 1152 + q once the byte sits under the exponent byte 0x64; an exact fma subtracts 1152.
    // |q| <= 128 is exact in fp16 and so is every product with an fp16 x in the fp32 sums; d scales each 32-block.
    const uint4 c0 = *reinterpret_cast<const uint4*>(cp + lane * 32);
    const uint4 c1 = *reinterpret_cast<const uint4*>(cp + lane * 32 + 16);
    const uint2 sc = *reinterpret_cast<const uint2*>(cp + 1024 + (lane >> 2) * 8);
    const uint32_t flip = 0x80808080u;
    const uint32_t words[8] = {c0.x ^ flip, c0.y ^ flip, c0.z ^ flip, c0.w ^ flip,
                               c1.x ^ flip, c1.y ^ flip, c1.z ^ flip, c1.w ^ flip};
    const uint32_t one = 0x3C003C00u, m1152 = 0xE480E480u, e64 = 0x64646464u;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
      float c[4];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int st = 2 * blk + h;
        uint32_t a[4];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t v;
          asm("prmt.b32 %0, %1, %2, %3;" : "=r"(v) : "r"(words[2 * st + (b >> 1)]), "r"(e64),
              "r"((b & 1) ? 0x4342u : 0x4140u));
          a[b] = hfma2(v, one, m1152);
        }
        if (h == 0) mma_f16(c, a[0], a[1], a[2], a[3], bx[st][0], bx[st][1], zero);
        else mma_f16(c, a[0], a[1], a[2], a[3], bx[st][0], bx[st][1], c);
      }
      const uint32_t sv = blk == 0 ? sc.x : sc.y;
      const float sr = h16_to_f32(sv & 0xFFFFu), sr8 = h16_to_f32(sv >> 16);
      acc[0] = fmaf(c[0], sr, acc[0]);
      acc[1] = fmaf(c[1], sr, acc[1]);
      acc[2] = fmaf(c[2], sr8, acc[2]);
      acc[3] = fmaf(c[3], sr8, acc[3]);
    }
  } else {  // Q2_K: one chunk = one 256-weight super-block per row, 16 groups of 16 = 16 mma steps
    // w = d sc q - dmin m per group: the MMA sums (sc q) . x and m . x over the super-block (sc q <= 45 and m <= 15
    // are exact in fp16, every product exact in fp32), then d and dmin scale the two sums once per chunk
    const uint4 cw0 = *reinterpret_cast<const uint4*>(cp + lane * 32);
    const uint4 cw1 = *reinterpret_cast<const uint4*>(cp + lane * 32 + 16);
    const uint32_t words[8] = {cw0.x, cw0.y, cw0.z, cw0.w, cw1.x, cw1.y, cw1.z, cw1.w};
    const int r = lane >> 2;
    const uint4 sr4 = *reinterpret_cast<const uint4*>(cp + 1024 + r * 32);
    const uint4 sr84 = *reinterpret_cast<const uint4*>(cp + 1024 + r * 32 + 16);
    const uint2 dd = *reinterpret_cast<const uint2*>(cp + 1280 + r * 8);
    const float d_r = h16_to_f32(dd.x & 0xFFFFu), dm_r = h16_to_f32(dd.x >> 16);
    const float d_r8 = h16_to_f32(dd.y & 0xFFFFu), dm_r8 = h16_to_f32(dd.y >> 16);
    const uint32_t s_r[4] = {sr4.x, sr4.y, sr4.z, sr4.w}, s_r8[4] = {sr84.x, sr84.y, sr84.z, sr84.w};
    // 2-bit code at bit 2b of a half's low byte -> fp16 1024 + 4^b q -> exact fma -> q
    const uint32_t mul[4] = {0x3C003C00u, 0x34003400u, 0x2C002C00u, 0x24002400u};
    const uint32_t add[4] = {0xE400E400u, 0xDC00DC00u, 0xD400D400u, 0xCC00CC00u};
    const uint32_t k1024 = 0x64006400u, sixteenth = 0x2C002C00u, m64 = 0xD400D400u, one = 0x3C003C00u;
    const float zero[4] = {0.f, 0.f, 0.f, 0.f};
    float cq[4] = {0.f, 0.f, 0.f, 0.f}, cm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      const uint32_t W = (s & 1) ? (words[s >> 1] >> 8) : words[s >> 1];
      // the group's scale byte of rows r and r + 8 in both halves of a word: sc = low nibble, m = high nibble
      const uint32_t sel = (uint32_t)(s & 3) | 0x4040u | ((uint32_t)(s & 3) << 8);
      uint32_t br, br8;
      asm("prmt.b32 %0, %1, 0, %2;" : "=r"(br) : "r"(s_r[s >> 2]), "r"(sel));
      asm("prmt.b32 %0, %1, 0, %2;" : "=r"(br8) : "r"(s_r8[s >> 2]), "r"(sel));
      const uint32_t sc_r = hfma2(lop3_and_xor(br, 0x000F000Fu, k1024), one, 0xE400E400u);      // sc, exact
      const uint32_t sc_r8 = hfma2(lop3_and_xor(br8, 0x000F000Fu, k1024), one, 0xE400E400u);
      const uint32_t m_r = hfma2(lop3_and_xor(br, 0x00F000F0u, k1024), sixteenth, m64);         // m, exact
      const uint32_t m_r8 = hfma2(lop3_and_xor(br8, 0x00F000F0u, k1024), sixteenth, m64);
      uint32_t a[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) a[b] = hfma2(lop3_and_xor(W, 0x00030003u << (2 * b), 0x64006400u), mul[b], add[b]);
      // registers 0, 2: row r; 1, 3: row r + 8
      const uint32_t z = 0u;
      mma_f16(cq, hfma2(a[0], sc_r, z), hfma2(a[1], sc_r8, z), hfma2(a[2], sc_r, z), hfma2(a[3], sc_r8, z),
              bx[s][0], bx[s][1], cq);
      mma_f16(cm, m_r, m_r8, m_r, m_r8, bx[s][0], bx[s][1], cm);
    }
    (void)zero;
    (void)sx;
    acc[0] = fmaf(-dm_r, cm[0], fmaf(cq[0], d_r, acc[0]));
    acc[1] = fmaf(-dm_r, cm[1], fmaf(cq[1], d_r, acc[1]));
    acc[2] = fmaf(-dm_r8, cm[2], fmaf(cq[2], d_r8, acc[2]));
    acc[3] = fmaf(-dm_r8, cm[3], fmaf(cq[3], d_r8, acc[3]));
  }
}

// Consumer side of one tile (G or D): waits the tile's stages, runs the warp's chunks, releases the stages.
// Returns false on a timeout (the caller marks the CTA aborted).
template <int FMT>
__device__ __forceinline__ bool consume_tile(uint8_t* ring, uint64_t* full, uint64_t* empty, uint32_t& it, int nchunks,
                                             int warp, int lane, const uint32_t (&b)[Cfg<FMT>::NCH][Fmt<FMT>::STEPS][2],
                                             const float* sxw, float (&acc)[4], long long wait_ns, volatile int* abort) {
  using C = Cfg<FMT>;
  using F = Fmt<FMT>;
  const int nst = (nchunks + F::CPS - 1) / F::CPS;
  bool ok = true;
  int slot = 0;
#pragma unroll
  for (int n = 0; n < C::NCH; ++n) {
    const int s = n / C::NPS;
    if (n % C::NPS == 0 && s < nst) {
      slot = (int)((it + s) % C::NS);
      const uint32_t par = ((it + s) / C::NS) & 1;
      if (*abort || !mbar_wait(&full[slot], par, wait_ns)) ok = false;
    }
    const int c = warp + C::CW * n;
    if (ok && c < nchunks) {
      const uint8_t* cp = ring + (size_t)slot * C::SB + (size_t)(c - s * F::CPS) * F::CB;
      chunk_mma<FMT>(cp, lane, b[n], sxw ? sxw + n * F::STEPS * kMaxT : nullptr, acc);
    }
    if (((n + 1) % C::NPS == 0) && s < nst) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }
  }
  it += nst;
  return ok;
}

// Loads the warp's B fragments of expert u's h (rescaled per token into fp16) after its G tiles are all done.
template <int FMT>
__device__ __forceinline__ void load_h_fragments(const FfnArgs& a, int u, int ncd, int warp, int lane,
                                                 uint32_t (&bh)[Cfg<FMT>::NCH][Fmt<FMT>::STEPS][2], float* sxw) {
  using C = Cfg<FMT>;
  using F = Fmt<FMT>;
  const int col = lane >> 2, q = lane & 3, T = a.T, I = a.I;
  const float am = col < T ? __uint_as_float(__ldcg(&a.amax_h[u * kMaxT + col])) : 0.f;
  const float sc = exp2i(rescale_exponent(am));
#pragma unroll
  for (int n = 0; n < C::NCH; ++n) {
    const int c = warp + C::CW * n;
#pragma unroll
    for (int j = 0; j < F::STEPS; ++j) {
      uint32_t v[2] = {0u, 0u};
      if (c < ncd && col < T) {
        const float* hr = a.hbuf + ((size_t)u * kMaxT + col) * I + c * F::CK + 16 * j + 2 * q;
        const float2 p0 = __ldcg(reinterpret_cast<const float2*>(hr));
        const float2 p1 = __ldcg(reinterpret_cast<const float2*>(hr + 8));
        const __half2 h0 = __floats2half2_rn(p0.x * sc, p0.y * sc);
        const __half2 h1 = __floats2half2_rn(p1.x * sc, p1.y * sc);
        v[0] = *reinterpret_cast<const uint32_t*>(&h0);
        v[1] = *reinterpret_cast<const uint32_t*>(&h1);
      }
      bh[n][j][0] = v[0];
      bh[n][j][1] = v[1];
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(Cfg<FMT>::THREADS, 1) ffn_kernel(const FfnArgs a) {
  using C = Cfg<FMT>;
  using F = Fmt<FMT>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float* red = reinterpret_cast<float*>(smem + (size_t)C::NS * C::SB);   // [kNR][C::CW warps][32 lanes][4]
  float* sx = red + C::RED;
  __shared__ __align__(8) uint64_t full[C::NS], empty[C::NS], redfull[kNR], redempty[kNR];
  __shared__ int s_val[kMaxU], s_first[kMaxU], s_slot[kMaxU], s_union[kMaxU];
  __shared__ int s_routed[kMaxT][kMaxU];        // per token: does it route to this union expert
  __shared__ float s_wsum[kMaxT][kMaxU];        // per token: summed router weight of each union expert
  __shared__ int s_nu[kMaxT];                   // per token: its union experts in ascending order ...
  __shared__ int s_ulist[kMaxT][kMaxK];
  __shared__ float s_uw[kMaxT][kMaxK];          // ... and their summed weights
  __shared__ int s_U, s_last, s_direct;
  __shared__ volatile int s_abort;
  __shared__ int s_sig[kMaxT];
  __shared__ float s_colmax[kMaxCW][kMaxT];
  __shared__ float s_hinv[kMaxT];               // epilogue warp: 2^-sigma of the current D expert, per token

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int T = a.T, k = a.k, H = a.H, I = a.I;
  const int n_ent = T * k;

  // ---------------- prologue
  // Consumers start fetching their x fragments at once (they do not depend on the routing); the producer warp
  // forms the union of the tokens' experts (sorted, deduplicated) and the per-token weight sums meanwhile.
  uint32_t bx[C::NCH][F::STEPS][2];
  float xmax = 0.f;
  if (warp < C::CW) {
    const int col = lane >> 2, q = lane & 3, ncg0 = H / F::CK;
#pragma unroll
    for (int n = 0; n < C::NCH; ++n) {
      const int c = warp + C::CW * n;
#pragma unroll
      for (int j = 0; j < F::STEPS; ++j) {
        uint32_t v0 = 0, v1 = 0;
        if (c < ncg0 && col < T) {
          const int k0 = c * F::CK + 16 * j + 2 * q;
          const uint16_t* xr = a.x + (size_t)col * H;
          v0 = __ldg(reinterpret_cast<const uint32_t*>(xr + k0));
          v1 = __ldg(reinterpret_cast<const uint32_t*>(xr + k0 + 8));
        }
        bx[n][j][0] = v0;
        bx[n][j][1] = v1;
      }
    }
  }
  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], C::CW); }
    for (int s = 0; s < kNR; ++s) { mbar_init(&redfull[s], C::CW); mbar_init(&redempty[s], 1); }
    fence_mbar_init();
    s_abort = 0;
  }
  if (warp == C::PROD) {
    int bad = 0;
    for (int i = lane; i < n_ent; i += 32) {
      const int v = a.idx[i];
      s_val[i] = v;
      bad |= (v < 0 || v >= a.E);
    }
    for (int i = lane; i < T * kMaxU; i += 32) {
      (&s_wsum[0][0])[i] = 0.f;
      (&s_routed[0][0])[i] = 0;
    }
    bad = __any_sync(0xffffffffu, bad);
    __syncwarp();
    for (int i = lane; i < n_ent; i += 32) {
      const int v = s_val[i];
      int first = 1;
      for (int j = 0; j < i; ++j) first &= (s_val[j] != v);
      s_first[i] = first;
    }
    __syncwarp();
    int nfirst = 0;
    for (int i = lane; i < n_ent; i += 32) {
      const int v = s_val[i];
      int rank = 0;
      for (int j = 0; j < n_ent; ++j) rank += (s_first[j] && s_val[j] < v) ? 1 : 0;
      s_slot[i] = rank;
      if (s_first[i]) s_union[rank] = v;
      nfirst += s_first[i];
    }
    nfirst = __reduce_add_sync(0xffffffffu, nfirst);
    __syncwarp();
    if (lane < T) {  // rank order, so a token's weight sums do not depend on the other tokens
      for (int r = 0; r < k; ++r) {
        const int u = s_slot[lane * k + r];
        s_wsum[lane][u] += __ldg(&a.w[lane * k + r]);
        s_routed[lane][u] = 1;
      }
      int n = 0;
      for (int u = 0; u < nfirst; ++u)
        if (s_routed[lane][u]) { s_ulist[lane][n] = u; s_uw[lane][n] = s_wsum[lane][u]; ++n; }
      s_nu[lane] = n;
    }
    const int nu_lane = lane < T ? s_nu[lane] : 1;
    const int direct = __all_sync(0xffffffffu, nu_lane == 1);
    if (lane == 0) {
      s_U = nfirst;
      s_direct = direct;
      if (bad) { s_abort = 1; if (blockIdx.x == 0) record_error(&a.hdr->status, MOE_ERR_INVALID_ARG); }
    }
  }
  __syncthreads();
  const int U = s_U;
  const int G = gridDim.x, bid = blockIdx.x;
  const int gt = I / 8, dt = H / 16;  // tiles per expert
  // 32-bit unit arithmetic (U * gt <= 64 * 512 units): a 64-bit division is a long software sequence on the path
  // from the prologue to the first weight copy
  const uint32_t NG = (uint32_t)(U * gt), ND = (uint32_t)(U * dt), uG = (uint32_t)G, ub = (uint32_t)bid;
  const int g0 = (int)(NG * ub / uG), g1 = (int)(NG * (ub + 1) / uG);
  const int d0 = (int)(ND * ub / uG), d1 = (int)(ND * (ub + 1) / uG);
  const int m0 = (int)((uint32_t)dt * ub / uG), m1 = (int)((uint32_t)dt * (ub + 1) / uG);
  const int ncg = H / F::CK, ncd = I / F::CK;                       // chunks per G / D tile
  const int64_t tbg = tile_bytes(FMT, H), tbd = tile_bytes(FMT, I);
  const int64_t sgu = gate_up_stride(FMT, H, I), sdn = down_stride(FMT, H, I);

  if (warp == C::PROD) {
    // ================= producer: G tiles of the CTA's range, then its D tiles (expert-major)
    if (lane == 0 && !s_abort) {
      const uint64_t pol = policy_evict_first();
      uint32_t it = 0;
      bool ok = true;
      auto issue_tile = [&](const uint8_t* base, int nchunks) {
        for (int c0 = 0; c0 < nchunks && ok; c0 += F::CPS) {
          const int nc = min(F::CPS, nchunks - c0);
          const int slot = (int)(it % C::NS);
          if (it >= (uint32_t)C::NS) {
            if (s_abort || !mbar_wait(&empty[slot], ((it / C::NS) - 1) & 1, a.wait_ns)) { ok = false; break; }
          }
          mbar_arrive_expect_tx(&full[slot], (uint32_t)(nc * F::CB));
          bulk_g2s(ring + (size_t)slot * C::SB, base + (size_t)c0 * F::CB, (uint32_t)(nc * F::CB), &full[slot], pol);
          ++it;
        }
      };
      for (int gu = g0; gu < g1 && ok; ++gu) {
        const int u = gu / gt, j = gu % gt;
        issue_tile(a.gate_up + (size_t)s_union[u] * sgu + (size_t)j * tbg, ncg);
      }
      for (int du = d0; du < d1 && ok; ++du) {
        const int u = du / dt, m = du % dt;
        issue_tile(a.down + (size_t)s_union[u] * sdn + (size_t)m * tbd, ncd);
      }
      if (!ok) {
        record_error(&a.hdr->status, MOE_ERR_DEVICE_TIMEOUT);
        s_abort = 1;
        // let the copies already in flight land before the CTA can exit
        const uint32_t lo = it > (uint32_t)C::NS ? it - C::NS : 0;
        for (uint32_t i = lo; i < it; ++i) mbar_wait(&full[i % C::NS], (i / C::NS) & 1, a.wait_ns);
      }
    }
  } else if (warp == C::EPI) {
    // ================= epilogue warp: per unit, sum the 8 warps' partials in warp order, then
    //   G: h = SiLU(g) * u -> h buffer (fp32) and the per-(expert, token) max |h|
    //   D: d = down partial of the unit's expert -> d buffer
    // then the grid barrier and the combine of the CTA's output rows.
    uint32_t ri = 0;
    auto wait_red = [&](uint32_t r) -> const float* {
      const int slot = (int)(r % kNR);
      if (s_abort || !mbar_wait(&redfull[slot], (r / kNR) & 1, a.wait_ns)) {
        record_error(&a.hdr->status, MOE_ERR_DEVICE_TIMEOUT);
        s_abort = 1;
      }
      return red + (size_t)slot * (C::CW * 32 * 4);
    };
    auto release_red = [&](uint32_t r) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&redempty[r % kNR]);
    };
    int pend_u = -1, pend_n = 0;  // G tiles done but not yet published, for one expert
    for (int gu = g0; gu < g1; ++gu, ++ri) {
      const int u = gu / gt, jt = gu % gt;
      const float* rb = wait_red(ri);
      uint32_t hmax[2] = {0u, 0u};
      int htc[2] = {-1, -1};
#pragma unroll
      for (int pp = 0; pp < 2; ++pp) {
        // output pair p -> fragment lane fl, column slot cc: g from c[cc] (row fl/4), u from c[cc+2] (row fl/4+8)
        const int p = lane + 32 * pp, fl = p >> 1, cc = p & 1;
        const int r = fl >> 2, tc = 2 * (fl & 3) + cc;
        if (tc < T) {
          float gs = 0.f, us = 0.f;
#pragma unroll
          for (int w = 0; w < C::CW; ++w) {
            gs += rb[(w * 32 + fl) * 4 + cc];
            us += rb[(w * 32 + fl) * 4 + cc + 2];
          }
          const float inv = exp2i_neg(s_sig[tc]);
          const float g = gs * inv, uu = us * inv;
          const float h = g * __frcp_rn(1.0f + __expf(-g)) * uu;   // SiLU(g) * u
          a.hbuf[((size_t)u * kMaxT + tc) * I + (size_t)jt * 8 + r] = h;
          hmax[pp] = __float_as_uint(fabsf(h));
          htc[pp] = tc;
        }
      }
      // max |h| per token: the warp's largest first (non-negative floats, NaN included, order like their bit
      // patterns), then one atomic per token instead of one per lane
      for (int t = 0; t < T; ++t) {
        const uint32_t v = __reduce_max_sync(0xffffffffu, max(htc[0] == t ? hmax[0] : 0u, htc[1] == t ? hmax[1] : 0u));
        if (lane == 0) atomicMax(&a.amax_h[u * kMaxT + t], v);
      }
      release_red(ri);   // its __syncwarp orders every lane's h writes before lane 0's release below
      // publish per expert: when the expert changes and after the CTA's last G tile
      if (pend_u != u) {
        if (pend_u >= 0 && lane == 0) red_release_add(&a.cnt_g[pend_u], (uint32_t)pend_n);
        pend_u = u;
        pend_n = 0;
      }
      ++pend_n;
    }
    if (pend_u >= 0 && lane == 0) red_release_add(&a.cnt_g[pend_u], (uint32_t)pend_n);
    // With one expert per token (a shared expert, or k = 1) the owner of a down tile is the only contributor to its
    // output rows: it writes y itself, with the combine's arithmetic, and no grid barrier is needed.
    const bool direct = s_direct != 0;
    int hu = -1;
    for (int du = d0; du < d1; ++du, ++ri) {
      const int u = du / dt, m = du % dt;
      const float* rb = wait_red(ri);
      if (u != hu) {  // the consumers waited for this expert's G tiles before handing over this unit
        if (lane < T) s_hinv[lane] = exp2i_neg(rescale_exponent(__uint_as_float(__ldcg(&a.amax_h[u * kMaxT + lane]))));
        __syncwarp();
        hu = u;
      }
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const int p = lane + 32 * pp, fl = p >> 2, cc = p & 3;
        const int row = (fl >> 2) + 8 * (cc >> 1), tc = 2 * (fl & 3) + (cc & 1);
        if (tc < T && s_routed[tc][u]) {
          float ds = 0.f;
#pragma unroll
          for (int w = 0; w < C::CW; ++w) ds += rb[(w * 32 + fl) * 4 + cc];
          const float dv = ds * s_hinv[tc];
          if (direct) {
            const size_t yi = (size_t)tc * H + (size_t)m * 16 + row;
            const float acc2 = fmaf(s_uw[tc][0], dv, 0.f);
            const float yv = a.accumulate ? a.y[yi] + acc2 : acc2;
            a.y[yi] = yv;
            if (a.y_bf16) a.y_bf16[yi] = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
          } else {
            a.dbuf[((size_t)u * H + (size_t)m * 16 + row) * kMaxT + tc] = dv;
          }
        }
      }
      release_red(ri);
    }
    // ---- grid-wide barrier, then the CTA combines its output rows: y_t = sum over the token's own experts, in
    //      ascending expert id, of w * d (fp32 fma), so the result does not depend on the other tokens
    __syncwarp();
    if (lane == 0 && !direct) {
      red_release_add(&a.hdr->gbar, 1u);   // after the __syncwarp: every lane's down partials before it
      if (!s_abort && !wait_counter(&a.hdr->gbar, (uint32_t)G, a.wait_ns)) {
        record_error(&a.hdr->status, MOE_ERR_DEVICE_TIMEOUT);
        s_abort = 1;
      }
    }
    __syncwarp();
    for (int i = lane; i < (direct ? 0 : (m1 - m0) * 16 * T); i += 32) {
      const int tok = i % T, row = (i / T) % 16, mi = i / T / 16;
      const size_t hrow = (size_t)(m0 + mi) * 16 + row;
      const int nu = s_nu[tok];
      float acc2 = 0.f;
      for (int j = 0; j < nu; ++j)
        acc2 = fmaf(s_uw[tok][j], __ldcg(&a.dbuf[((size_t)s_ulist[tok][j] * H + hrow) * kMaxT + tok]), acc2);
      const size_t yi = (size_t)tok * H + hrow;
      const float yv = a.accumulate ? a.y[yi] + acc2 : acc2;
      a.y[yi] = yv;
      if (a.y_bf16) a.y_bf16[yi] = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
    }
  } else {
    // ================= consumers (warps 0..7): tensor-core mat-vec over their K slices
    uint32_t it = 0, ri = 0;
    const int col = lane >> 2, q = lane & 3;
    float* sxw = nullptr;  // no format needs per-group sums of the activations
    auto hand_over = [&](const float (&acc)[4]) {
      const int slot = (int)(ri % kNR);
      if (ri >= (uint32_t)kNR) {
        if (s_abort || !mbar_wait(&redempty[slot], ((ri / kNR) - 1) & 1, a.wait_ns)) {
          record_error(&a.hdr->status, MOE_ERR_DEVICE_TIMEOUT);
          s_abort = 1;
        }
      }
      float* rb = red + (size_t)slot * (C::CW * 32 * 4);
      *reinterpret_cast<float4*>(rb + (warp * 32 + lane) * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&redfull[slot]);
      ++ri;
    };

    // ---- phase G: B fragments = x of the T tokens (fetched in the prologue), rescaled per token into fp16
    {
      float mx = xmax;
#pragma unroll
      for (int n = 0; n < C::NCH; ++n)
#pragma unroll
        for (int j = 0; j < F::STEPS; ++j) {
          const uint32_t v0 = bx[n][j][0], v1 = bx[n][j][1];
          mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16_bits_to_f32(v0 & 0xFFFFu)), fabsf(bf16_bits_to_f32(v0 >> 16))),
                               fmaxf(fabsf(bf16_bits_to_f32(v1 & 0xFFFFu)), fabsf(bf16_bits_to_f32(v1 >> 16)))));
        }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      if (q == 0) s_colmax[warp][col] = mx;
      named_bar(1, C::CW * 32);
      float cm = 0.f;
#pragma unroll
      for (int w = 0; w < C::CW; ++w) cm = fmaxf(cm, s_colmax[w][col]);
      const int sig = rescale_exponent(cm);
      if (warp == 0 && q == 0) s_sig[col] = sig;   // read by the epilogue warp after the first hand-over
      const float sc = exp2i(sig);
#pragma unroll
      for (int n = 0; n < C::NCH; ++n)
#pragma unroll
        for (int j = 0; j < F::STEPS; ++j)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t v = bx[n][j][h];
            const __half2 hv = __floats2half2_rn(bf16_bits_to_f32(v & 0xFFFFu) * sc, bf16_bits_to_f32(v >> 16) * sc);
            bx[n][j][h] = *reinterpret_cast<const uint32_t*>(&hv);
          }

      for (int gu = g0; gu < g1; ++gu) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (!consume_tile<FMT>(ring, full, empty, it, ncg, warp, lane, bx, sxw, acc, a.wait_ns, &s_abort)) {
          record_error(&a.hdr->status, MOE_ERR_DEVICE_TIMEOUT);
          s_abort = 1;
        }
        hand_over(acc);
      }
    }

    // ---- phase D: the CTA's range of down tiles (expert-major, so it loads the h of one or two experts)
    {
      uint32_t bh[C::NCH][F::STEPS][2];
      int loaded = -1;
      for (int du = d0; du < d1; ++du) {
        const int u = du / dt;
        if (u != loaded) {
          // one thread per CTA polls the expert's counter (a poller per warp, grid-wide, crowded the counter's L2
          // line and delayed both the publishing adds and the observation); its acquire and the barrier order the
          // other warps' reads of h after it. Every consumer warp walks the same units, so all reach the barrier.
          if (warp == 0 && lane == 0 && !s_abort) {
            if (!wait_counter(&a.cnt_g[u], (uint32_t)gt, a.wait_ns)) {
              record_error(&a.hdr->status, MOE_ERR_DEVICE_TIMEOUT);
              s_abort = 1;
            }
          }
          named_bar(2, C::CW * 32);
          load_h_fragments<FMT>(a, u, ncd, warp, lane, bh, sxw);
          loaded = u;
        }
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (!consume_tile<FMT>(ring, full, empty, it, ncd, warp, lane, bh, sxw, acc, a.wait_ns, &s_abort)) {
          record_error(&a.hdr->status, MOE_ERR_DEVICE_TIMEOUT);
          s_abort = 1;
        }
        hand_over(acc);
      }
    }
  }

  // ---------------- epilogue: the last CTA to finish clears the per-call counters
  __syncthreads();
  if (tid == 0) {
    // acq_rel: releases this CTA's reads of the counters (ordered before it by the barrier); the last CTA's acquire
    // then orders its clears after every CTA's reads
    const uint32_t prev = atom_acq_rel_add(&a.hdr->done, 1u);
    s_last = (prev == (uint32_t)(G - 1));
  }
  __syncthreads();
  if (s_last) {
    for (int i = tid; i < U; i += blockDim.x) a.cnt_g[i] = 0u;
    for (int i = tid; i < U * kMaxT; i += blockDim.x) a.amax_h[i] = 0u;
    if (tid == 0) { a.hdr->gbar = 0u; a.hdr->done = 0u; }
  }
}

}  // namespace moe

using namespace moe;

static size_t ws_needed(const moe_layer_t* L, int T, int k) {
  const size_t U = (size_t)T * k;
  return kWsCounters + U * kMaxT * L->I * sizeof(float) + U * L->H * kMaxT * sizeof(float);
}

extern "C" size_t moe_workspace_bytes(const moe_layer_t* L, int32_t T_max, int32_t k) {
  if (!L || T_max < 1 || T_max > kMaxT || k < 1 || k > kMaxK) return 0;
  if (!moe_internal::shape_ok(L->H, L->I)) return 0;
  if (L->layout == MOE_LAYOUT_TC) return L->fmt == MOE_FMT_MXFP4 ? moe_internal::tc_decode_workspace_bytes(L, T_max, k) : 0;
  return ws_needed(L, T_max, k);
}

template <int FMT>
static moe_status_t launch_ffn(const FfnArgs& a, cudaStream_t s) {
  using C = Cfg<FMT>;
  static int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(ffn_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM) != cudaSuccess)
      return MOE_ERR_CUDA;
    configured[dev] = 1;
  }
  const int nsm = moe_internal::num_sms();
  if (nsm <= 0) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nsm);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, ffn_kernel<FMT>, a) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

static moe_status_t ffn_common(const char* site, const moe_layer_t* L, const void* x, int32_t T, const int32_t* idx,
                               const float* w, int32_t k, float* y, void* y_bf16, int32_t accumulate, void* ws,
                               size_t ws_bytes, void* stream) {
  if (site && moe_internal::fault(site)) return MOE_ERR_FAULT_INJECTED;
  if (!L || !x || !idx || !w || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (L->fmt < MOE_FMT_MXFP4 || L->fmt > MOE_FMT_Q8_0) return MOE_ERR_UNSUPPORTED_FORMAT;
  if (L->layout != MOE_LAYOUT_DECODE && L->layout != MOE_LAYOUT_TC) return MOE_ERR_UNSUPPORTED_FORMAT;
  if (!L->gate_up || !L->down || ((uintptr_t)L->gate_up & 15) || ((uintptr_t)L->down & 15)) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)x & 3) || ((uintptr_t)ws & 255) || ((uintptr_t)y & 3)) return MOE_ERR_INVALID_ARG;
  if (y_bf16 && ((uintptr_t)y_bf16 & 1)) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > kMaxT || k < 1 || k > kMaxK || L->E < 1) return MOE_ERR_SHAPE;
  if (!moe_internal::shape_ok(L->H, L->I)) return MOE_ERR_SHAPE;
  if (L->layout == MOE_LAYOUT_TC) {
    if (L->fmt != MOE_FMT_MXFP4) return MOE_ERR_UNSUPPORTED_FORMAT;
    moe_status_t st = moe_check_device();
    if (st != MOE_OK) return st;
    return moe_internal::tc_decode(L, x, T, idx, w, k, y, y_bf16, accumulate, ws, ws_bytes, stream);
  }
  if (ws_bytes < ws_needed(L, T, k)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  FfnArgs a;
  a.gate_up = (const uint8_t*)L->gate_up;
  a.down = (const uint8_t*)L->down;
  a.x = (const uint16_t*)x;
  a.idx = idx;
  a.w = w;
  a.y = y;
  a.y_bf16 = (uint16_t*)y_bf16;
  a.accumulate = accumulate;
  a.H = L->H; a.I = L->I; a.E = L->E; a.T = T; a.k = k;
  uint8_t* base = (uint8_t*)ws;
  a.hdr = (WsHeader*)base;
  a.cnt_g = (uint32_t*)(base + kOffCntG);
  a.amax_h = (uint32_t*)(base + kOffAmax);
  a.hbuf = (float*)(base + kWsCounters);
  a.dbuf = a.hbuf + (size_t)T * k * kMaxT * L->I;
  a.wait_ns = kDefaultWaitNs;
  cudaStream_t s = (cudaStream_t)stream;
  switch (L->fmt) {
    case MOE_FMT_MXFP4: return launch_ffn<MOE_FMT_MXFP4>(a, s);
    case MOE_FMT_INT4G32: return launch_ffn<MOE_FMT_INT4G32>(a, s);
    case MOE_FMT_Q8_0: return launch_ffn<MOE_FMT_Q8_0>(a, s);
    default: return launch_ffn<MOE_FMT_Q2K>(a, s);
  }
}

extern "C" moe_status_t moe_expert_ffn_decode(const moe_layer_t* L, const void* x_bf16, const int32_t* idx,
                                              const float* w, int32_t k, float* y, void* y_bf16, int32_t accumulate,
                                              void* ws, size_t ws_bytes, void* stream) {
  MOE_NVTX("moe_expert_ffn_decode");
  return ffn_common("decode", L, x_bf16, 1, idx, w, k, y, y_bf16, accumulate, ws, ws_bytes, stream);
}

// Router and expert FFN in one launch (tensor-core layout, MXFP4): the decode kernel computes the router logits
// across the grid first, every CTA selects the experts, CTA 0 writes idx / w, then the FFN proceeds as in
// moe_expert_ffn_verify. The routing equals moe_route_topk's bit for bit (same arithmetic, route.cuh).
extern "C" moe_status_t moe_route_expert_ffn(const moe_layer_t* L, const void* router_w_f16, const void* x_bf16, int32_t T,
                                            int32_t k, int32_t* idx, float* w, float* y, void* y_bf16,
                                            int32_t accumulate, void* ws, size_t ws_bytes, void* stream) {
  MOE_NVTX("moe_route_expert_ffn");
  if (moe_internal::fault("route_ffn")) return MOE_ERR_FAULT_INJECTED;
  if (!L || !router_w_f16 || !x_bf16 || !idx || !w || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (L->layout != MOE_LAYOUT_TC || L->fmt != MOE_FMT_MXFP4) return MOE_ERR_UNSUPPORTED_FORMAT;
  if (!L->gate_up || !L->down || ((uintptr_t)L->gate_up & 15) || ((uintptr_t)L->down & 15)) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)x_bf16 & 15) || ((uintptr_t)router_w_f16 & 15) || ((uintptr_t)ws & 255) || ((uintptr_t)y & 3) ||
      ((uintptr_t)idx & 3) || ((uintptr_t)w & 3))
    return MOE_ERR_INVALID_ARG;
  if (y_bf16 && ((uintptr_t)y_bf16 & 1)) return MOE_ERR_INVALID_ARG;
  if (T < 1 || T > kMaxT || k < 1 || k > kMaxK || L->E < k || L->E > 256) return MOE_ERR_SHAPE;
  if (!moe_internal::shape_ok(L->H, L->I)) return MOE_ERR_SHAPE;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  return moe_internal::tc_decode(L, x_bf16, T, nullptr, nullptr, k, y, y_bf16, accumulate, ws, ws_bytes, stream,
                                 router_w_f16, idx, w);
}

extern "C" moe_status_t moe_expert_ffn_verify(const moe_layer_t* L, const void* x_bf16, int32_t T, const int32_t* idx,
                                              const float* w, int32_t k, float* y, void* y_bf16, int32_t accumulate,
                                              void* ws, size_t ws_bytes, void* stream) {
  MOE_NVTX("moe_expert_ffn_verify");
  return ffn_common("verify", L, x_bf16, T, idx, w, k, y, y_bf16, accumulate, ws, ws_bytes, stream);
}

// ------------------------------------------------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory: a plugin whose host hands it only the input and output buffers, code
// that runs under a device-memory budget owned by another allocator, or code that must not allocate while a stream
// is being captured. For them moe_expert_ffn_decode_static() runs the same decode kernel with its scratch in the
// file-scope array below instead of a workspace. The array is sized for one token with k <= 8 and H, I <= 4096:
// kStaticScratchBytes = 4096 (counters) + 8 * 8 * 4096 * 4 (h) + 8 * 4096 * 8 * 4 (d) = 2,101,248 bytes, held by
// every GPU that loads this library until the process exits.
// ------------------------------------------------------------------------------------------------------------------
namespace {
constexpr size_t kStaticScratchBytes = kWsCounters + (size_t)kMaxK * kMaxT * 4096 * 4 + (size_t)kMaxK * 4096 * kMaxT * 4;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
std::mutex g_static_mu;
// Device address of g_static_scratch, per device ordinal, looked up by the first call on that device (with the
// device current). cudaDeviceReset() unloads the module, so the cached address is stale after it: a process that
// resets a device must not call moe_expert_ffn_decode_static() on that device again.
void* g_static_ptr[64];

moe_status_t static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    // host code only sees a stand-in for the symbol; the kernel needs its device address
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return MOE_OK;
}
}  // namespace

extern "C" moe_status_t moe_expert_ffn_decode_static(const moe_layer_t* L, const void* x_bf16, const int32_t* idx,
                                                     const float* w, int32_t k, float* y, void* y_bf16,
                                                     int32_t accumulate, void* stream) {
  MOE_NVTX("moe_expert_ffn_decode_static");
  if (moe_internal::fault("decode")) return MOE_ERR_FAULT_INJECTED;
  if (!L || !x_bf16 || !idx || !w || !y) return MOE_ERR_INVALID_ARG;
  if (k < 1 || k > kMaxK || !moe_internal::shape_ok(L->H, L->I)) return MOE_ERR_SHAPE;
  if (L->layout != MOE_LAYOUT_DECODE) return MOE_ERR_UNSUPPORTED_FORMAT;  // the fixed scratch serves this layout
  if (ws_needed(L, 1, k) > kStaticScratchBytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  void* scratch = nullptr;
  st = static_scratch(&scratch);
  if (st != MOE_OK) return st;
  // every call shares the array: clear the counters and status word the kernel expects to start at zero
  if (cudaMemsetAsync(scratch, 0, kWsCounters, (cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
  return ffn_common(nullptr, L, x_bf16, 1, idx, w, k, y, y_bf16, accumulate, scratch, kStaticScratchBytes, stream);
}

// Device status word of the most recent moe_expert_ffn_decode_static() call on the current device (the first word of
// the static scratch): synchronises `stream`, then copies it out. The next static call clears it.
extern "C" moe_status_t moe_static_device_status(void* stream) {
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  int32_t v = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyFromSymbolAsync(&v, g_static_scratch, sizeof(v), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return (moe_status_t)v;
}
