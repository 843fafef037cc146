// spec.cu -- acceptance of K drafted tokens after a verify sweep ("Mixed-precision compression of DeepSeek-V4-Flash"
// (lumirain.cn), "What compression does not solve": a draft x is kept with probability min(1, p(x) / q(x)); on a
// rejection the token is drawn from max(p - q, 0), normalised, which leaves the target's distribution unchanged).
//
// Drafts are tested in order; the first rejection ends the chain and is replaced by a draw from that position's
// residual; when all K are kept, one more token is drawn from the target row after the last draft. The
// arithmetic is fixed so that every run gives the same tokens:
//   - decision: u[k] < p_k(d) / q_k(d), one IEEE fp32 division (q = 0 < p keeps the draft, p = q = 0 rejects);
//   - draw: weights r = p - q (or p) clamped to [0, 1] (NaN as 0) become integers R = floor(r 2^40); the token is
//     the smallest v whose running sum of R exceeds floor(U S / 2^32), U = floor(u_s 2^32) (u_s clamped to
//     [0, 1)), S the sum of R. Integer sums do not depend on the order of addition, so the parallel scan here
//     and a sequential loop choose the same token;
//   - a residual without mass falls back to p of that position; a row without mass gives token -1.
// One CTA of 1024 threads: warp 0 decides the K drafts with one ballot; the draw sums pieces of 512 values
// (coalesced float4 loads), scans the piece sums, and walks the piece that holds the threshold.
#include "common.cuh"
#include "api_internal.h"

namespace moe {
namespace spec {

constexpr int THREADS = 1024;
constexpr int MAX_K = 8;
constexpr int MAX_V = 1 << 22;  // keeps V * 2^40 inside 64 bits

// floor(r * 2^40) of r clamped to [0, 1] (NaN as 0), in two 32-bit parts: with s = r 2^16 (exact: a change of
// exponent), hi = floor(s) <= 2^16 and lo = floor((s - hi) 2^24) < 2^24 (s - hi is exact, and so is the scaling),
// floor(r 2^40) = hi 2^24 + lo. Sums of the parts stay in 32 bits for up to 256 values.
__device__ __forceinline__ void weight_parts(float r, uint32_t& hi, uint32_t& lo) {
  const float sv = fminf(fmaxf(r, 0.f), 1.f) * 65536.0f;
  const float h = floorf(sv);
  hi = __float2uint_rz(h);
  lo = __float2uint_rz((sv - h) * 16777216.0f);
}
__device__ __forceinline__ uint64_t weight_fx(float r) {
  uint32_t hi, lo;
  weight_parts(r, hi, lo);
  return ((uint64_t)hi << 24) + lo;
}
// floor(u * 2^32) of u clamped to [0, 1) (NaN as 0), exact for the same reason
__device__ __forceinline__ uint64_t uniform_fx(float u) {
  return u >= 1.f ? 0xFFFFFFFFull : __float2ull_rz(fmaxf(u, 0.f) * 4294967296.0f);
}

__device__ __forceinline__ uint64_t weight_at(const float* pr, const float* qr, int v) {
  return weight_fx(qr ? __ldg(pr + v) - __ldg(qr + v) : __ldg(pr + v));
}
__device__ __forceinline__ void add_weight(float r, uint32_t& hs, uint32_t& ls) {
  uint32_t hi, lo;
  weight_parts(r, hi, lo);
  hs += hi;
  ls += lo;
}
__device__ __forceinline__ void weight4(const float4 a, const float4 b, bool minus, uint32_t& hs, uint32_t& ls) {
  add_weight(minus ? a.x - b.x : a.x, hs, ls);
  add_weight(minus ? a.y - b.y : a.y, hs, ls);
  add_weight(minus ? a.z - b.z : a.z, hs, ls);
  add_weight(minus ? a.w - b.w : a.w, hs, ls);
}

// Inclusive scan of one value per thread over the block; returns the thread's inclusive sum, *total the block's.
__device__ __forceinline__ uint64_t block_scan(uint64_t x, uint64_t* s_warp, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint64_t w = s_warp[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  *total = s_warp[31];
  const uint64_t r = x + (warp ? s_warp[warp - 1] : 0ull);
  __syncthreads();  // s_warp is reused by the next scan
  return r;
}

constexpr int PIECE = 512;                      // values per piece: 32 lanes x 16
constexpr int MAX_PIECES = MAX_V / PIECE;       // 8192: 64 KB of piece sums in shared memory

struct DrawShared {
  uint64_t warp[32];
  uint64_t cbase;   // running sum before the piece that crosses the threshold
  int cpiece;       // that piece
  int tok;
};

// Block-wide draw from the weights of row pr (minus qr if given); every thread gets the token (-1: no mass).
//   1. the row is cut into pieces of 512 consecutive values; warp w sums pieces w, w + 32, ... (each lane reads
//      16 values, coalesced: float4 loads for 16-byte aligned rows) and stores each piece's sum in shared memory;
//   2. a block scan over the piece sums gives the total, the threshold and the piece that crosses it;
//   3. the block walks that piece, one value per thread, with one more block scan.
__device__ int block_draw(const float* pr, const float* qr, int V, float us, DrawShared& sh, uint64_t* psum) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int np = (V + PIECE - 1) / PIECE;
  const bool vec = (((uintptr_t)pr | (uintptr_t)qr) & 15) == 0 && (V & 3) == 0;
  for (int pc = warp; pc < np; pc += THREADS / 32) {
    const int base = pc * PIECE;
    uint64_t sum = 0;
    if (vec) {
      const float4* p4 = reinterpret_cast<const float4*>(pr);
      const float4* q4 = reinterpret_cast<const float4*>(qr);
      float4 a[4], b[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int v = base + 4 * (lane + 32 * k);
        const bool in = v < V;  // V is a multiple of 4: a float4 is wholly in or out
        a[k] = in ? __ldg(p4 + v / 4) : make_float4(0.f, 0.f, 0.f, 0.f);
        b[k] = (in && qr) ? __ldg(q4 + v / 4) : a[k];
      }
      uint32_t hs = 0, ls = 0;  // 16 values: at most 2^20 and 2^28
#pragma unroll
      for (int k = 0; k < 4; ++k) weight4(a[k], b[k], qr != nullptr, hs, ls);
      sum = ((uint64_t)hs << 24) + ls;
    } else {
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int v = base + lane + 32 * k;
        if (v < V) sum += weight_at(pr, qr, v);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane == 0) psum[pc] = sum;
  }
  if (tid == 0) sh.tok = -1;
  __syncthreads();
  // scan of the piece sums: thread t takes pieces [t m, t m + m)
  const int m = (np + THREADS - 1) / THREADS;
  const int p0 = min(np, tid * m), p1 = min(np, p0 + m);
  uint64_t own = 0;
  for (int pc = p0; pc < p1; ++pc) own += psum[pc];
  uint64_t total;
  const uint64_t incl = block_scan(own, sh.warp, &total);
  if (total == 0) return -1;  // the same for every thread
  const uint64_t U = uniform_fx(us);
  const uint64_t lo = U * total, hi = __umul64hi(U, total);
  const uint64_t thr = (hi << 32) | (lo >> 32);  // floor(U total / 2^32) < total
  uint64_t run = incl - own;
  if (run <= thr && thr < incl) {  // exactly one thread: the one whose pieces cross the threshold
    int pc = p0;
    while (run + psum[pc] <= thr) run += psum[pc++];
    sh.cbase = run;
    sh.cpiece = pc;
  }
  __syncthreads();
  // walk the crossing piece: thread t < 512 takes its value t
  const int vv = sh.cpiece * PIECE + tid;
  const uint64_t w = (tid < PIECE && vv < V) ? weight_at(pr, qr, vv) : 0ull;
  uint64_t step;
  const uint64_t r = sh.cbase + block_scan(w, sh.warp, &step);
  if (w != 0 && r - w <= thr && thr < r) sh.tok = vv;  // the first value whose running sum passes thr
  __syncthreads();
  const int tok = sh.tok;
  __syncthreads();  // the shared fields are reused by a second draw
  return tok;
}

__global__ void __launch_bounds__(THREADS, 1) spec_accept_kernel(const float* __restrict__ p, const float* __restrict__ q,
                                                                int K, int V, const int32_t* __restrict__ draft,
                                                                const float* __restrict__ u, int32_t* __restrict__ out) {
  __shared__ DrawShared sh;
  __shared__ int s_n;
  extern __shared__ uint64_t psum[];  // one sum per piece of 512 values
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid < 32) {
    bool bad = false, keep = true;
    if (lane < K) {
      const int d = draft[lane];
      bad = d < 0 || d >= V;
      if (!bad) keep = u[lane] < __ldg(p + (size_t)lane * V + d) / __ldg(q + (size_t)lane * V + d);
    }
    const bool any_bad = __any_sync(0xFFFFFFFFu, bad);
    const uint32_t rejected = __ballot_sync(0xFFFFFFFFu, lane < K && !keep);
    if (lane == 0) s_n = any_bad ? -1 : (rejected ? __ffs(rejected) - 1 : K);
  }
  __syncthreads();
  const int n = s_n;
  if (n < 0) {
    if (tid == 0) { out[0] = -1; out[1] = -1; }
    return;
  }
  const float us = u[K];
  int tok;
  if (n < K) {
    tok = block_draw(p + (size_t)n * V, q + (size_t)n * V, V, us, sh, psum);
    if (tok < 0) tok = block_draw(p + (size_t)n * V, nullptr, V, us, sh, psum);
  } else {
    tok = block_draw(p + (size_t)K * V, nullptr, V, us, sh, psum);
  }
  if (tid == 0) { out[0] = n; out[1] = tok; }
}

}  // namespace spec
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_spec_accept(const float* p, const float* q, int32_t K, int32_t V, const int32_t* draft,
                                        const float* u, int32_t* result, void* stream) {
  MOE_NVTX("moe_spec_accept");
  if (moe_internal::fault("spec")) return MOE_ERR_FAULT_INJECTED;
  if (!p || !u || !result || (K > 0 && (!q || !draft))) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)p & 3) || ((uintptr_t)q & 3) || ((uintptr_t)u & 3) || ((uintptr_t)draft & 3) ||
      ((uintptr_t)result & 3))
    return MOE_ERR_INVALID_ARG;
  if (K < 0 || K > spec::MAX_K || V < 1 || V > spec::MAX_V) return MOE_ERR_SHAPE;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  static int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(spec::spec_accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(spec::MAX_PIECES * sizeof(uint64_t))) != cudaSuccess)
      return MOE_ERR_CUDA;
    configured[dev] = 1;
  }
  const size_t smem = (size_t)((V + spec::PIECE - 1) / spec::PIECE) * sizeof(uint64_t);
  spec::spec_accept_kernel<<<1, spec::THREADS, smem, (cudaStream_t)stream>>>(p, q, K, V, draft, u, result);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
