// norm.cu -- RMS normalisation of a layer's fp32 output into the next layer's bf16 input, for stacks of layers.
//
// The model the pages describe normalises the hidden state before each MoE layer ("Mixed-precision compression of
// DeepSeek-V4-Flash", "The recipe": 43 transformer layers, each with its MoE FFN). A stack of routed-expert layers
// that passes y_L on unnormalised drifts: with random weights the FFN maps an activation of rms r to roughly c r^2,
// so the chain collapses to zero (routing then degenerates to ties) or overflows. This call restores unit scale:
//   x[t, i] = bf16_rne( y[t, i] * r ),  r = fp32( 1 / sqrt(mean_i y[t, i]^2 + eps) )   (no learned gain)
// The row is first scaled by the power of two 2^-E (E the exponent of its largest |y|: exact), so the fp32 sum of
// squares neither overflows nor loses the small rows; r is formed from it in fp64 (one operation per token), the
// product y * r in fp32. One CTA per token, both reductions in a fixed order (strided per thread, then a fixed
// tree): a token's result does not depend on the other tokens.
#include "common.cuh"
#include "api_internal.h"

namespace moe {

constexpr int kNormThreads = 512;

// block-wide reduction in a fixed order: a warp tree, then the warps' results in warp order (all threads get it)
template <typename Op>
__device__ __forceinline__ float block_reduce(float v, float* part, Op op) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();   // part may still be read by the previous reduction
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = part[0];
#pragma unroll
  for (int w = 1; w < kNormThreads / 32; ++w) t = op(t, part[w]);
  return t;
}

__global__ void __launch_bounds__(kNormThreads) rms_norm_kernel(const float* y, int H, float eps, uint16_t* out) {
  __shared__ float part[kNormThreads / 32];
  const float* yr = y + (size_t)blockIdx.x * H;
  uint16_t* xr = out + (size_t)blockIdx.x * H;
  float m = 0.f;   // largest |y| (NaN ignored here; it reaches the sum below)
  for (int i = threadIdx.x; i < H; i += kNormThreads) m = fmaxf(m, fabsf(yr[i]));
  m = block_reduce(m, part, [](float a, float b) { return fmaxf(a, b); });
  const uint32_t eb = (__float_as_uint(m) >> 23) & 255u;          // biased exponent of max |y|
  // 2^(127 - eb) puts max |y| in [1, 2); for eb >= 253 the normal 2^-126 (max |y| in [1, 4)); 1 for a zero,
  // subnormal, infinite or all-NaN row (eps then dominates, or the non-finite value propagates)
  const float sc = (eb == 0u || eb == 255u) ? 1.0f : __uint_as_float((eb >= 253u ? 1u : 254u - eb) << 23);
  float s = 0.f;
  for (int i = threadIdx.x; i < H; i += kNormThreads) { const float v = yr[i] * sc; s = fmaf(v, v, s); }
  s = block_reduce(s, part, [](float a, float b) { return a + b; });
  // mean(y^2) = s / (H sc^2): r = sc / sqrt(s / H + eps sc^2), in fp64 (IEEE division and square root)
  const double scd = (double)sc;
  const float r = (float)(scd / sqrt((double)s / (double)H + (double)eps * scd * scd));
  for (int i = threadIdx.x; i < H; i += kNormThreads)
    xr[i] = __bfloat16_as_ushort(__float2bfloat16_rn(yr[i] * r));
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_rms_norm_bf16(const float* y, int32_t T, int32_t H, float eps, void* x_bf16,
                                          void* stream) {
  MOE_NVTX("moe_rms_norm_bf16");
  if (moe_internal::fault("norm")) return MOE_ERR_FAULT_INJECTED;
  if (!y || !x_bf16 || ((uintptr_t)y & 3) || ((uintptr_t)x_bf16 & 1)) return MOE_ERR_INVALID_ARG;
  if (T < 1 || H < 1 || H > (1 << 20) || !(eps >= 0.f)) return MOE_ERR_SHAPE;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  rms_norm_kernel<<<T, kNormThreads, 0, (cudaStream_t)stream>>>(y, H, eps, (uint16_t*)x_bf16);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
