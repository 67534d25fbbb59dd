// w4a8.h -- host interface of the integer-native W4A8 / W8A8 paths.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qmm.h"

namespace qmm {

// Signed `bits`-bit weights (4 or 8) x int8 activations on the skinny kernel.
qmm_status wxa8_dispatch(int bits, const int8_t *xq, const void *sa, const uint8_t *w, const void *ws,
                         int group, void *y, int32_t *acc_out, int M, int N, int K, int *status,
                         int num_sms, int smem_optin, int smem_pair, cudaStream_t stream);

}  // namespace qmm
