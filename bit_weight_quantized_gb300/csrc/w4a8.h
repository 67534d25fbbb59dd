// w4a8.h -- host interface of the integer-native W4A8 path.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qmm.h"

namespace qmm {

qmm_status w4a8_dispatch(const int8_t *xq, const void *sa, const uint8_t *w4, const void *ws,
                         int group, void *y, int32_t *acc_out, int M, int N, int K, int *status,
                         int num_sms, int smem_optin, int smem_pair, cudaStream_t stream);

}  // namespace qmm
