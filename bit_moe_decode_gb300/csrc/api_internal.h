// api_internal.h -- host-side helpers shared by the translation units of libmoe.so (not part of the C ABI).
#pragma once
#include <cstddef>
#include <cstdint>

#include "../../include/moe.h"

namespace moe_internal {

// true if the environment variable MOE_FAULT names `site` (host-side fault injection for tests)
bool fault(const char* site);
// H, I multiples of 256 within [256, 4096]
bool shape_ok(int64_t H, int64_t I);
// number of SMs of the current device (cached per device)
int num_sms();

// prefill layout (grouped GEMM); implemented in prefill.cu
size_t prefill_packed_bytes(moe_format_t fmt, moe_matrix_t kind, int64_t n_e, int64_t H, int64_t I);
moe_status_t pack_prefill(moe_format_t fmt, moe_src_t src_kind, moe_matrix_t kind, int64_t n_e, int64_t H, int64_t I,
                          const void* src_a, const void* src_b, void* dst, size_t dst_bytes, void* stream);
moe_status_t unpack_prefill(moe_format_t fmt, moe_matrix_t kind, const void* packed, int64_t H, int64_t I,
                            int64_t expert, float* out, void* stream);

}  // namespace moe_internal
