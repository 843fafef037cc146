// route.cuh -- the router arithmetic shared by the standalone router (route.cu) and the decode kernel that routes
// in its first phase (decode_tc.cu), so that both give the same bits ("Mixed-precision compression of
// DeepSeek-V4-Flash" (lumirain.cn), "The recipe": F16 router, top-6 of 256 routed experts, softmax weights).
//
// Logit of expert e for token t: sum over h of W_r[e, h] * x[t, h] (fp16 x bf16 products are exact in fp32), as two
// halves over h, each a lane-strided ordered sum and a fixed butterfly (route_half_logits), added. Top-k: k rounds of a warp arg-max with ties to the
// lower expert index; weights exp(l_r - l_0) / sum_j exp(l_j - l_0) in rank order.
#pragma once
#include <cstdint>
#include <cuda_fp16.h>

namespace moe {

constexpr int kRouteTPC = 8;    // tokens per pass
constexpr int kRouteMaxE = 1024;

// Half c (0 or 1) of the logits of one expert row for tokens 0 .. nt-1: lane l sums, in order, the 8-element
// pieces at h = 8 l + 256 i for i in [c P2, min(P, (c + 1) P2)), P = H / 256, P2 = ceil(P / 2), with fused
// multiply-adds; then a fixed butterfly (xor 16, 8, 4, 2, 1) adds the lanes. The logit is half 0 + half 1, so the
// two halves can be computed by different warps. xrow(t) points at token t's x (shared or global memory); BATCH
// pieces per lane are loaded before they are used (it changes when the loads are issued, not the sums). NT is the
// most tokens a caller passes (nt <= NT): it only sizes the unrolled code, not any token's sum.
template <int BATCH, int NT, typename XRow>
__device__ __forceinline__ void route_half_logits(const uint16_t* __restrict__ row, int H, int nt, XRow xrow, int c,
                                                  float (&acc)[NT]) {
  const int lane = threadIdx.x & 31;
  const int P = H / 256, P2 = (P + 1) / 2, i_beg = c * P2, i_end = min(P, (c + 1) * P2);
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.f;
  for (int i0 = i_beg; i0 < i_end; i0 += BATCH) {
    uint4 wv[BATCH];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      const int h = lane * 8 + 256 * (i0 + b);
      wv[b] = i0 + b < i_end ? __ldg(reinterpret_cast<const uint4*>(row + h)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      if (i0 + b >= i_end) break;
      const int h = lane * 8 + 256 * (i0 + b);
      const uint32_t ww[4] = {wv[b].x, wv[b].y, wv[b].z, wv[b].w};
      float wf[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        wf[2 * j] = __half2float(__ushort_as_half((unsigned short)(ww[j] & 0xFFFFu)));
        wf[2 * j + 1] = __half2float(__ushort_as_half((unsigned short)(ww[j] >> 16)));
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (t < nt) {
          const uint4 xv = *reinterpret_cast<const uint4*>(xrow(t) + h);
          const uint32_t xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[t] = fmaf(wf[2 * j], __uint_as_float(xx[j] << 16), acc[t]);
            acc[t] = fmaf(wf[2 * j + 1], __uint_as_float(xx[j] & 0xFFFF0000u), acc[t]);
          }
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    float v = acc[t];
    v += __shfl_xor_sync(0xffffffffu, v, 16);
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    acc[t] = v;
  }
}
// The whole logit: half 0 + half 1.
template <int BATCH, typename XRow>
__device__ __forceinline__ void route_row_logits(const uint16_t* __restrict__ row, int H, int nt, XRow xrow,
                                                 float (&acc)[kRouteTPC]) {
  float h1[kRouteTPC];
  route_half_logits<BATCH, kRouteTPC>(row, H, nt, xrow, 0, acc);
  route_half_logits<BATCH, kRouteTPC>(row, H, nt, xrow, 1, h1);
#pragma unroll
  for (int t = 0; t < kRouteTPC; ++t) acc[t] = acc[t] + h1[t];
}

// Top-k of one token by the whole warp; logit(e) gives expert e's logit (e < E <= 32 * NE). Lane 0 gets the experts
// in rank order in sid[] and their weights in sw[].
template <int NE, typename Logit>
__device__ __forceinline__ void route_topk_warp(Logit logit, int E, int k, int (&sid)[8], float (&sw)[8]) {
  const int lane = threadIdx.x & 31;
  // every logit as an order-preserving key, computed once: larger key = larger logit; NaN, -inf and absent
  // experts get key 0 and are never chosen (as with comparisons), -0 gets the key of +0
  uint32_t key[NE];
#pragma unroll
  for (int j = 0; j < NE; ++j) {
    const int e = lane + 32 * j;
    const float v = e < E ? logit(e) : -__int_as_float(0x7f800000);
    const uint32_t u = __float_as_uint(v) == 0x80000000u ? 0u : __float_as_uint(v);
    key[j] = v > -__int_as_float(0x7f800000) ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;
  }
  // the rounds are unrolled to the largest k so that sel, sid and sw stay in registers (a dynamically indexed
  // array would live in local memory, whose round trips are slow while the weights stream). A round is two warp
  // reductions: the largest key, then the lowest expert index among the lanes holding it (ties to the lower index).
  float sel[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    sel[r] = 0.f;
    sid[r] = 0;
    if (r >= k) continue;
    uint32_t bk = 0u;  // this lane's best key and its expert (the lowest j among equal keys)
    int be = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < NE; ++j)
      if (key[j] > bk) { bk = key[j]; be = lane + 32 * j; }
    const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
    const int bi = mk ? (int)__reduce_min_sync(0xffffffffu, bk == mk ? (uint32_t)be : 0xffffffffu) : 0x7fffffff;
    sel[r] = mk ? __uint_as_float((mk & 0x80000000u) ? (mk & 0x7fffffffu) : ~mk) : -__int_as_float(0x7f800000);
    sid[r] = bi;
#pragma unroll
    for (int j = 0; j < NE; ++j)  // remove the winner
      if (lane + 32 * j == bi) key[j] = 0u;
  }
  float den = 0.f;
#pragma unroll
  for (int r = 0; r < 8; ++r)
    if (r < k) den += expf(sel[r] - sel[0]);
#pragma unroll
  for (int r = 0; r < 8; ++r) sw[r] = r < k ? expf(sel[r] - sel[0]) / den : 0.f;
}

}  // namespace moe
