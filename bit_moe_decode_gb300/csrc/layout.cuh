// layout.cuh -- the packed device layouts of expert weights.
//
// ---- MOE_LAYOUT_DECODE (all four formats; the mat-vec kernels of ffn.cu)
//
// A matrix is cut into TILES of 16 rows x K and each tile into CHUNKS of 16 rows x CK columns along K.
//   Gate/Up: tile j holds gate rows 8j..8j+7 (tile rows 0..7) and up rows 8j..8j+7 (tile rows 8..15), so one
//            tensor-core tile yields g and u of the same 8 intermediate indices (gate+up fused in one pass).
//   Down:    tile m holds rows 16m..16m+15.
// A chunk is [codes][scales] and holds exactly the canonical bytes of its 16 x CK weights (same bits per weight):
//   MXFP4   CK = 64,  512 B codes + 32 B E8M0            = 544 B
//   INT4    CK = 64,  512 B codes + 64 B bf16 scales     = 576 B
//   Q2_K    CK = 256, 1024 B codes + 256 B sc|m + 64 B d,dmin = 1344 B
//   Q8_0    CK = 64,  1024 B codes + 64 B fp16 scales     = 1088 B
// Codes are in mma.m16n8k16 A-fragment order: lane l owns (CK/64) x 16 consecutive bytes; its rows are l/4 and
// l/4 + 8 and its k offsets inside a 16-wide step are 2(l%4), 2(l%4)+1, +8, +9 (Q8_0: lane l owns 32 bytes).
//   MXFP4: byte (l*16 + j*4 + b) = codes of (row l/4 + 8*(b&1), k = 16j + 2(l%4) + 8*(b>>1) + {0: low nibble,
//          1: high nibble}) -- the byte feeds cvt.rn.f16x2.e2m1x2 directly.
//   INT4:  32-bit word (l*16 + j*4): register b's lower-k nibble at bits 4b..4b+3, its higher-k nibble at bits
//          16+4b..16+4b+3 (two's complement codes), decoded with an exponent-bias trick into exact fp16.
//   Q2_K:  32-bit word (l*32 + w*4) holds steps 2w and 2w+1; step s = 2w + t, register b: lower-k 2-bit code at
//          bits 8t + 2b, higher-k code at bits 16 + 8t + 2b.
//   Q8_0:  byte (l*32 + j*8 + 2b + h) = the two's-complement code of (row l/4 + 8*(b&1), k = 16j + 2(l%4) +
//          8*(b>>1) + h): register b of step j is one 32-bit half of an 8-byte word.
// Scales: MXFP4 word r (r < 8) = {e[r][blk0], e[r+8][blk0], e[r][blk1], e[r+8][blk1]};
//         INT4  8 bytes per r  = bf16 {s[r][blk0], s[r+8][blk0], s[r][blk1], s[r+8][blk1]};
//         Q2_K  32 bytes per r = scales[16] of row r then of row r+8; then 8 bytes per r = fp16 {d[r], dmin[r],
//               d[r+8], dmin[r+8]};
//         Q8_0  8 bytes per r  = fp16 {d[r][blk0], d[r+8][blk0], d[r][blk1], d[r+8][blk1]}.
#pragma once
#include <cstdint>

namespace moe {

template <int FMT> struct Fmt;
template <> struct Fmt<MOE_FMT_MXFP4> {
  static constexpr int BS = 32, BB = 17;           // canonical block: weights, bytes
  static constexpr int CK = 64, CODE = 512, CB = 544, STEPS = 4, CPS = 32;
};
template <> struct Fmt<MOE_FMT_INT4G32> {
  static constexpr int BS = 32, BB = 18;
  static constexpr int CK = 64, CODE = 512, CB = 576, STEPS = 4, CPS = 32;
};
template <> struct Fmt<MOE_FMT_Q2K> {
  static constexpr int BS = 256, BB = 84;
  static constexpr int CK = 256, CODE = 1024, CB = 1344, STEPS = 16, CPS = 8;
};
template <> struct Fmt<MOE_FMT_Q8_0> {
  static constexpr int BS = 32, BB = 34;
  static constexpr int CK = 64, CODE = 1024, CB = 1088, STEPS = 4, CPS = 16;
};
// CPS = chunks per pipeline stage: a stage covers 2048 columns of K (1024 for Q8_0, whose chunks are twice as big).

__host__ __device__ inline int fmt_ck(int fmt) { return fmt == MOE_FMT_Q2K ? 256 : 64; }
__host__ __device__ inline int fmt_cb(int fmt) {
  return fmt == MOE_FMT_MXFP4 ? 544 : fmt == MOE_FMT_INT4G32 ? 576 : fmt == MOE_FMT_Q2K ? 1344 : 1088;
}
__host__ __device__ inline int fmt_bs(int fmt) { return fmt == MOE_FMT_Q2K ? 256 : 32; }
__host__ __device__ inline int fmt_bb(int fmt) {
  return fmt == MOE_FMT_MXFP4 ? 17 : fmt == MOE_FMT_INT4G32 ? 18 : fmt == MOE_FMT_Q2K ? 84 : 34;
}

// bytes of one tile (16 rows x K)
__host__ __device__ inline int64_t tile_bytes(int fmt, int64_t K) { return (K / fmt_ck(fmt)) * fmt_cb(fmt); }
// per-expert strides of the packed matrices
__host__ __device__ inline int64_t gate_up_stride(int fmt, int64_t H, int64_t I) { return (I / 8) * tile_bytes(fmt, H); }
__host__ __device__ inline int64_t down_stride(int fmt, int64_t H, int64_t I) { return (H / 16) * tile_bytes(fmt, I); }

// Location of weight (tile row tr, column k) of a tile: chunk index, lane, and position inside the lane's codes.
struct CodePos {
  int chunk, lane, step, reg, hi;  // hi: 0 = lower k of the register's pair, 1 = higher k
};
__host__ __device__ inline CodePos code_pos(int fmt, int tr, int k) {
  CodePos p;
  int ck = fmt_ck(fmt);
  p.chunk = k / ck;
  int kc = k % ck;
  p.step = kc / 16;
  int ks = kc % 16;
  int q = (ks % 8) / 2;
  p.hi = ks % 2;
  p.reg = (tr >= 8 ? 1 : 0) + (ks >= 8 ? 2 : 0);
  p.lane = (tr % 8) * 4 + q;
  return p;
}

// ---- MOE_LAYOUT_TC (MXFP4; operands of the block-scaled tcgen05 MMA, used by prefill, decode and verify)
// Codes hold element k of a row in byte k/2 of the row's run, even k in the LOW nibble (the order in which the TMA
// engine's 16U4_ALIGN16B type unpacks E2M1 codes into the MMA's shared-memory operand, and the order kind::mxf4
// reads packed codes in). Every storage unit is one contiguous run of 8704 bytes: 8192 bytes of codes, then a
// 512-byte block of E8M0 exponents permuted for tcgen05.cp .32x128b.warpx4 (byte l*16 + c*4 + b feeds TMEM lane l,
// column c, byte b; the MMA reads row m of a 128-row operand from lane m % 32, column m / 32).
//   GATE_UP (R = 2I rows, K = H): 128 x 128 TILES in (row tile rt, column tile kt) order. Tile rows are 64 gate
//            rows 64rt..64rt+63 followed by the same 64 up rows, so one accumulator holds g and u of the same 64
//            intermediate indices (a SLICE). Codes [128 rows][64 B]; exponent byte b = 32-block b of the tile.
//   DOWN     (R = H rows, K = I): CHUNKS of 256 rows x 64 columns in (slice s = k / 64, row pair q = r / 256)
//            order: the 64 columns of a chunk are exactly the intermediate indices of one gate/up slice, so the
//            down projection of a slice reads whole chunks. Codes [256 rows][32 B], stored already in the
//            32-byte swizzle of the MMA's shared-memory operand (16-byte half h of row r at half h ^ ((r >> 2) & 1)),
//            so one plain bulk copy of the whole 8704-byte chunk lands a ready operand; exponent byte b holds row
//            tile (256q + 128(b / 2) + ..) and 32-block b % 2 of the slice: the two 128-row halves of a chunk are two
//            MMAs that select scale bytes (0, 1) and (2, 3).
// The per-expert stride R*K*17/32 equals the canonical size (same bits per weight).
constexpr int64_t kTcTileBytes = 8704;
struct TcGeom {
  int64_t R, K, RT, KT, stride;  // rows, columns, row tiles (128 rows), column tiles (128 columns), bytes per expert
  int kind;
};
__host__ __device__ inline TcGeom tc_geom(int kind, int64_t H, int64_t I) {
  TcGeom g;
  g.kind = kind;
  g.R = kind == MOE_MAT_GATE_UP ? 2 * I : H;
  g.K = kind == MOE_MAT_GATE_UP ? H : I;
  g.RT = g.R / 128;
  g.KT = g.K / 128;
  g.stride = g.RT * g.KT * kTcTileBytes;
  return g;
}
// storage row of canonical row `row` of matrix mi (0 = gate / down, 1 = up)
__host__ __device__ inline int64_t tc_row(int kind, int mi, int64_t row) {
  if (kind != MOE_MAT_GATE_UP) return row;
  return (row / 64) * 128 + mi * 64 + row % 64;
}
// byte offset (inside one expert) of the run holding storage row r, column k
__host__ __device__ inline int64_t tc_tile_off(const TcGeom& g, int64_t r, int64_t k) {
  if (g.kind == MOE_MAT_DOWN) return ((k / 64) * (g.R / 256) + r / 256) * kTcTileBytes;
  return ((r / 128) * g.KT + k / 128) * kTcTileBytes;
}
// byte offset of the code byte of (storage row r, column k) and of the exponent of (r, 32-block of k)
__host__ __device__ inline int64_t tc_code_off(const TcGeom& g, int64_t r, int64_t k) {
  if (g.kind == MOE_MAT_DOWN)
    return tc_tile_off(g, r, k) + (r % 256) * 32 + ((((k % 64) / 32) ^ ((r >> 2) & 1)) << 4) + (k % 32) / 2;
  return tc_tile_off(g, r, k) + (r % 128) * 64 + (k % 128) / 2;
}
__host__ __device__ inline int64_t tc_scale_off(const TcGeom& g, int64_t r, int64_t k) {
  const int64_t rr = r % 128;
  const int64_t b = g.kind == MOE_MAT_DOWN ? 2 * ((r % 256) / 128) + (k % 64) / 32 : (k % 128) / 32;
  return tc_tile_off(g, r, k) + 8192 + (rr % 32) * 16 + (rr / 32) * 4 + b;
}

}  // namespace moe
