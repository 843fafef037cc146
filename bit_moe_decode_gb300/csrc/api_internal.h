// api_internal.h -- host-side helpers shared by the translation units of libmoe.so (not part of the C ABI).
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/moe.h"

// An NVTX range named after the API call around its host-side body (launches included), for timeline tools; with
// no tool attached a push / pop costs a function-pointer test.
struct MoeNvtxRange {
  explicit MoeNvtxRange(const char* name) { nvtxRangePushA(name); }
  ~MoeNvtxRange() { nvtxRangePop(); }
};
#define MOE_NVTX(name) MoeNvtxRange moe_nvtx_range_(name)

namespace moe_internal {

// true if the environment variable MOE_FAULT names `site` (host-side fault injection for tests)
bool fault(const char* site);
// H, I multiples of 256 within [256, 4096]
bool shape_ok(int64_t H, int64_t I);
// number of SMs of the current device (cached per device)
int num_sms();

// decode / verify of MXFP4 experts in MOE_LAYOUT_TC on tcgen05 (decode_tc.cu); arguments checked by the caller
size_t tc_decode_workspace_bytes(const moe_layer_t* L, int T_max, int k);
// router_w != NULL: route inside the kernel (fp16 router [E][H], E <= 256), writing idx_out / w_out ([T][k]);
// idx / w are then unused
moe_status_t tc_decode(const moe_layer_t* L, const void* x, int T, const int32_t* idx, const float* w, int k, float* y,
                       void* y_bf16, int accumulate, void* ws, size_t ws_bytes, void* stream,
                       const void* router_w = nullptr, int32_t* idx_out = nullptr, float* w_out = nullptr);

// TMA tensor maps (host-side encoding through the runtime's driver entry point; false if it is unavailable or
// rejects the arguments). tmap_tc_weights: the E2M1 code tiles of a MOE_LAYOUT_TC matrix as a 4-D map
// [E][row tiles * column tiles][128 rows][64 B] with a 128 x 128 box (16U4_ALIGN16B, 128-byte swizzle).
// tmap_u8: a rank-2 or rank-3 byte tensor (dims innermost first, strides in bytes for dims 1..), 128- or 64-byte
// swizzle.
bool tmap_available();
bool tmap_tc_weights(CUtensorMap* m, const void* base, int kind, int64_t H, int64_t I, int64_t E);
// the same tiles as packed bytes ([E][tiles][128 rows][64 B], box 64 x 128, 64-byte swizzle) for kind::mxf4
bool tmap_tc_weights_packed(CUtensorMap* m, const void* base, int kind, int64_t H, int64_t I, int64_t E);
bool tmap_u8(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
             const uint32_t* box, int swizzle_bytes = 128);

}  // namespace moe_internal
