// route.cu -- router top-k ("Mixed-precision compression of DeepSeek-V4-Flash" (lumirain.cn), "The recipe": F16
// router, top-6 of 256 routed experts) and hash routing ("quant surgery" (blog.meowhead.cn), section 4: the first
// layers map a token id to fixed experts through a tid2eid table).
//
// Softmax mode (arithmetic in route.cuh): one thread-block cluster of 16 CTAs handles up to 8 tokens. Each of its 256 warps computes the
// logits of its experts (fp16 x bf16 products are exact in fp32; each lane sums its strided slice in order, then a
// fixed butterfly reduces the lanes), keeps them in its CTA's shared memory, and CTA 0 gathers all logits through
// distributed shared memory and selects the top k per token (one warp per token): k rounds of a warp arg-max with
// ties to the lower expert index, then weights = exp(l_r - l_0) / sum_j exp(l_j - l_0) in rank order.
// A token's arithmetic does not depend on the other tokens of its cluster, so routing T tokens together gives
// the same result as routing each alone.
#include <cooperative_groups.h>

#include "common.cuh"
#include "route.cuh"
#include "api_internal.h"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kRouteCluster = 16;
constexpr int kRouteWarps = 16;
constexpr int kRouteSlots = kRouteMaxE / (kRouteCluster * kRouteWarps);  // experts per warp (max 4)

__global__ void __launch_bounds__(kRouteWarps * 32, 1)
route_kernel(const uint16_t* __restrict__ wr, const uint16_t* __restrict__ x, int T, int H, int E, int k,
             int32_t* __restrict__ idx_out, float* __restrict__ w_out) {
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(16) uint8_t smem[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);               // [kRouteTPC][H] bf16
  __shared__ float lg[kRouteSlots * kRouteWarps][kRouteTPC];      // this CTA's logits
  const int cr = (int)cluster.block_rank();
  const int cl = blockIdx.x / kRouteCluster;
  const int t0 = cl * kRouteTPC;
  const int nt = min(kRouteTPC, T - t0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // stage the cluster's tokens (16-byte copies)
  const int per_tok = H / 8;
  for (int i = threadIdx.x; i < nt * per_tok; i += blockDim.x) {
    const int t = i / per_tok, c = i % per_tok;
    reinterpret_cast<uint4*>(xs + (size_t)t * H)[c] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + t) * H) + c);
  }
  __syncthreads();

  const int gw = cr * kRouteWarps + warp;
#pragma unroll 1
  for (int sl = 0; sl < kRouteSlots; ++sl) {
    const int e = gw + sl * kRouteCluster * kRouteWarps;
    if (e >= E) break;
    float acc[kRouteTPC];
    route_row_logits<16>(wr + (size_t)e * H, H, nt, [&](int t) { return xs + (size_t)t * H; }, acc);
    if (lane == 0)
#pragma unroll
      for (int t = 0; t < kRouteTPC; ++t) lg[sl * kRouteWarps + warp][t] = acc[t];
  }
  cluster.sync();

  if (cr == 0 && warp < nt) {
    const int t = warp;
    // gather: expert e lives in CTA (e % 256) / 16, warp e % 16, slot e / 256
    int sid[8];
    float sw[8];
    route_topk_warp<kRouteMaxE / 32>(
        [&](int e) {
          const int owner = (e % (kRouteCluster * kRouteWarps)) / kRouteWarps;
          const int slot = (e / (kRouteCluster * kRouteWarps)) * kRouteWarps + e % kRouteWarps;
          const float* remote = cluster.map_shared_rank(&lg[0][0], owner);
          return remote[slot * kRouteTPC + t];
        },
        E, k, sid, sw);
    if (lane == 0)
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < k) {
          idx_out[(size_t)(t0 + t) * k + r] = sid[r];
          w_out[(size_t)(t0 + t) * k + r] = sw[r];
        }
  }
  cluster.sync();  // keep every CTA's logits alive until CTA 0 has read them
}

__global__ void hash_route_kernel(const int32_t* tok, const int32_t* tid2eid, int T, int k, int V, int32_t* idx,
                                  float* w, int32_t* status) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= T * k) return;
  const int t = i / k, r = i % k;
  const int id = tok[t];
  if (id < 0 || id >= V) {  // out-of-range token id: report and write a harmless routing
    if (status) atomicCAS(status, 0, (int)MOE_ERR_INVALID_ARG);
    idx[i] = 0;
    w[i] = 0.f;
    return;
  }
  idx[i] = tid2eid[(size_t)id * k + r];
  w[i] = 1.0f / (float)k;
}

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_route_topk(const void* router_w_f16, const void* x_bf16, int32_t T, int32_t H, int32_t E,
                                       int32_t k, const int32_t* token_ids, const int32_t* tid2eid, int32_t V,
                                       int32_t* idx, float* weights, void* stream) {
  MOE_NVTX("moe_route_topk");
  if (moe_internal::fault("route")) return MOE_ERR_FAULT_INJECTED;
  if (!idx || !weights) return MOE_ERR_INVALID_ARG;
  if (T < 1 || k < 1 || k > 8) return MOE_ERR_SHAPE;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (token_ids) {
    if (!tid2eid || V < 1) return MOE_ERR_INVALID_ARG;
    const int n = T * k;
    hash_route_kernel<<<(n + 127) / 128, 128, 0, s>>>(token_ids, tid2eid, T, k, V, idx, weights, nullptr);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (!router_w_f16 || !x_bf16) return MOE_ERR_INVALID_ARG;
  if (E < k || E > kRouteMaxE || H < 256 || H % 256 || H > 8192) return MOE_ERR_SHAPE;
  if (((uintptr_t)router_w_f16 & 15) || ((uintptr_t)x_bf16 & 15)) return MOE_ERR_INVALID_ARG;
  const size_t smem = (size_t)kRouteTPC * H * 2;
  static int configured[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(route_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kRouteTPC * 8192 * 2)) != cudaSuccess)
      return MOE_ERR_CUDA;
    configured[dev] = 1;
  }
  const int nclusters = (T + kRouteTPC - 1) / kRouteTPC;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nclusters * kRouteCluster);
  cfg.blockDim = dim3(kRouteWarps * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kRouteCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, route_kernel, (const uint16_t*)router_w_f16, (const uint16_t*)x_bf16, (int)T, (int)H,
                         (int)E, (int)k, idx, weights) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
