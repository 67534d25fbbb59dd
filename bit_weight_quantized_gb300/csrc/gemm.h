// gemm.h -- host interface of the tiled (M >= 17) kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/qmm.h"
#include "gemv.h"

namespace qmm {

// Widths the tiled kernel dequantizes.
bool gemm_supports_bits(int bits);

qmm_status gemm_dispatch(const void *x, bool x_bf16, const uint8_t *packed, int bits, int group,
                         const void *scales, const uint8_t *zeros, int zero_const, void *y, int M,
                         int N, int K, int *status, int num_sms, int smem_optin,
                         cudaStream_t stream);

}  // namespace qmm
