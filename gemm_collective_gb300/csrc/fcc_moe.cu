// fcc_moe.cu -- MoE route, dispatch (all-to-all) and grouped expert GEMM.
#include <cuda_runtime.h>

#include "fcc.h"
#include "fcc_internal.h"

extern "C" {

fcc_status fcc_moe_dispatch_gemm(int, const void* const*, const float* const*, const void* const*,
                                 int64_t, int64_t, int64_t, int, int, void* const*, void* const*,
                                 int64_t, int32_t* const*, float* const*, int32_t*, int32_t*,
                                 int32_t* const*, fcc_dtype, fcc_dtype, const fcc_opts*,
                                 fcc_stream_t) {
  return FCC_ERR_UNSUPPORTED;
}

size_t fcc_moe_workspace_size(int, int64_t, int64_t, int64_t, int, int, int64_t, const fcc_opts*) {
  return 0;
}

}  // extern "C"
