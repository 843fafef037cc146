// prefill.cu -- prefill grouped GEMM layout and kernels (block-scaled MXFP4 x MXFP8 on tcgen05).
#include "common.cuh"
#include "api_internal.h"

namespace moe_internal {

size_t prefill_packed_bytes(moe_format_t, moe_matrix_t, int64_t, int64_t, int64_t) { return 0; }

moe_status_t pack_prefill(moe_format_t, moe_src_t, moe_matrix_t, int64_t, int64_t, int64_t, const void*, const void*,
                          void*, size_t, void*) {
  return MOE_ERR_UNSUPPORTED_FORMAT;
}

moe_status_t unpack_prefill(moe_format_t, moe_matrix_t, const void*, int64_t, int64_t, int64_t, float*, void*) {
  return MOE_ERR_UNSUPPORTED_FORMAT;
}

}  // namespace moe_internal
