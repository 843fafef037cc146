// norm.cu -- RMS normalisation of a layer's fp32 output into the next layer's bf16 input, for stacks of layers.
//
// The model the pages describe normalises the hidden state before each MoE layer ("Mixed-precision compression of
// DeepSeek-V4-Flash", "The recipe": 43 transformer layers, each with its MoE FFN). A stack of routed-expert layers
// that passes y_L on unnormalised drifts: with random weights the FFN maps an activation of rms r to roughly c r^2,
// so the chain collapses to zero (routing then degenerates to ties) or overflows. This call restores unit scale:
//   x[t, i] = bf16_rne( y[t, i] * r ),  r = fp32( 1 / sqrt(mean_i y[t, i]^2 + eps) )   (no learned gain)
// The sum of squares and r are formed in fp64, so neither overflows nor loses the small rows (a few fp64
// operations per element: negligible even at the GPU's fp64 rate); the product is fp32. One CTA per token, the sum
// in a fixed order (strided per thread, then a fixed tree): a token's result does not depend on the other tokens.
#include "common.cuh"
#include "api_internal.h"

namespace moe {

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads) rms_norm_kernel(const float* y, int H, float eps, uint16_t* out) {
  __shared__ double part[kNormThreads / 32];
  const float* yr = y + (size_t)blockIdx.x * H;
  uint16_t* xr = out + (size_t)blockIdx.x * H;
  double s = 0.0;
  for (int i = threadIdx.x; i < H; i += kNormThreads) s = fma((double)yr[i], (double)yr[i], s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
  __syncthreads();
  double tot = 0.0;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += part[w];
  const float r = (float)(1.0 / sqrt(tot / (double)H + (double)eps));   // IEEE fp64 division and square root
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
