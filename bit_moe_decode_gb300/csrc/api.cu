// api.cu -- status strings, device check, fault injection, workspace helpers and the bounded-wait probe.
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "layout.cuh"
#include "api_internal.h"

namespace moe_internal {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool tmap_available() { return encode_fn() != nullptr; }

bool tmap_tc_weights(CUtensorMap* m, const void* base, int kind, int64_t H, int64_t I, int64_t E) {
  if (!encode_fn()) return false;
  const moe::TcGeom g = moe::tc_geom(kind, H, I);
  cuuint64_t dims[4] = {128, 128, (cuuint64_t)(g.RT * g.KT), (cuuint64_t)E};
  cuuint64_t strides[3] = {64, (cuuint64_t)moe::kTcTileBytes, (cuuint64_t)g.stride};
  cuuint32_t box[4] = {128, 128, 1, 1}, es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tmap_tc_weights_packed(CUtensorMap* m, const void* base, int kind, int64_t H, int64_t I, int64_t E) {
  if (!encode_fn()) return false;
  const moe::TcGeom g = moe::tc_geom(kind, H, I);
  cuuint64_t dims[4] = {64, 128, (cuuint64_t)(g.RT * g.KT), (cuuint64_t)E};
  cuuint64_t strides[3] = {64, (cuuint64_t)moe::kTcTileBytes, (cuuint64_t)g.stride};
  cuuint32_t box[4] = {64, 128, 1, 1}, es[4] = {1, 1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tmap_u8(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
             const uint32_t* box, int swizzle_bytes) {
  if (!encode_fn() || rank < 2 || rank > 3) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
  for (int i = 0; i < rank - 1; ++i) st[i] = strides[i];
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), d, st, b, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool fault(const char* site) {
  const char* f = std::getenv("MOE_FAULT");
  if (!f || !*f) return false;
  // comma-separated list of call names
  size_t n = std::strlen(site);
  const char* p = f;
  while (*p) {
    const char* q = std::strchr(p, ',');
    size_t len = q ? (size_t)(q - p) : std::strlen(p);
    if (len == n && std::strncmp(p, site, n) == 0) return true;
    if (!q) break;
    p = q + 1;
  }
  return false;
}

bool shape_ok(int64_t H, int64_t I) {
  return H >= 256 && I >= 256 && H <= 4096 && I <= 4096 && H % 256 == 0 && I % 256 == 0;
}

static std::mutex g_mu;
static int g_sms[64];
static int g_arch_ok[64];  // 0 unknown, 1 ok, 2 bad

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

}  // namespace moe_internal

extern "C" const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_SHAPE: return "unsupported shape";
    case MOE_ERR_UNSUPPORTED_FORMAT: return "unsupported weight format for this call";
    case MOE_ERR_UNSUPPORTED_ARCH: return "device is not compute capability 10.3 (GB300, sm_103a)";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "a device-side wait ran out of time";
    case MOE_ERR_FAULT_INJECTED: return "fault injected (MOE_FAULT)";
  }
  return "unknown status";
}

extern "C" int32_t moe_version(void) { return 100; }

extern "C" moe_status_t moe_check_device(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(moe_internal::g_mu);
    if (moe_internal::g_arch_ok[dev] == 1) return MOE_OK;
    if (moe_internal::g_arch_ok[dev] == 2) return MOE_ERR_UNSUPPORTED_ARCH;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return MOE_ERR_CUDA;
  bool ok = (major == 10 && minor == 3);
  std::lock_guard<std::mutex> lk(moe_internal::g_mu);
  moe_internal::g_arch_ok[dev] = ok ? 1 : 2;
  return ok ? MOE_OK : MOE_ERR_UNSUPPORTED_ARCH;
}

extern "C" moe_status_t moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!ws || ws_bytes < sizeof(moe::WsHeader)) return MOE_ERR_INVALID_ARG;
  if (((uintptr_t)ws & 255) != 0) return MOE_ERR_INVALID_ARG;
  return cudaMemsetAsync(ws, 0, ws_bytes, (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t moe_get_device_status(void* ws, void* stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  int32_t st = 0;
  cudaStream_t s = (cudaStream_t)stream;
  if (cudaMemcpyAsync(&st, ws, sizeof(st), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (st != 0) {
    int32_t z = 0;
    if (cudaMemcpyAsync(ws, &z, sizeof(z), cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  }
  return (moe_status_t)st;
}

// One CTA waits on a workspace flag that nothing sets, gives up after limit_us, records the timeout.
__global__ void timeout_probe_kernel(moe::WsHeader* hdr, long long limit_ns) {
  if (threadIdx.x != 0) return;
  volatile uint32_t* flag = &hdr->pad[0];
  long long t0;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (*flag == 0) {
    long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 > limit_ns) {
      moe::record_error(&hdr->status, MOE_ERR_DEVICE_TIMEOUT);
      return;
    }
    __nanosleep(1000);
  }
}

extern "C" moe_status_t moe_debug_timeout_probe(void* ws, size_t ws_bytes, int32_t limit_us, void* stream) {
  if (!ws || ws_bytes < sizeof(moe::WsHeader) || limit_us < 1 || limit_us > 2000000) return MOE_ERR_INVALID_ARG;
  moe_status_t st = moe_check_device();
  if (st != MOE_OK) return st;
  timeout_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((moe::WsHeader*)ws, (long long)limit_us * 1000);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
