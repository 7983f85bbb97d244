// Block-scaled FP8 GEMM (1x128 activation/gradient tiles, 128x128 weight
// tiles): placeholder until the promotion kernel lands.
#include "common.cuh"
#include "kernels.h"

namespace fp8 {

cudaError_t launch_gemm_block(const uint8_t *, const uint8_t *, int64_t, int64_t, int64_t,
                              const float *, int64_t, const float *, int64_t, int64_t, int,
                              uint16_t *, cudaStream_t, const char **why) {
    *why = "block-scaled GEMM not available yet";
    return cudaErrorNotSupported;
}

}  // namespace fp8
