// w4a8.h -- host interface of the integer-native W4A8 / W8A8 paths.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qmm.h"

namespace qmm {

// Signed `bits`-bit weights (4 or 8) x int8 activations: the tcgen05 kernel
// from the batch sizes below, else the decode kernel's exact-integer mode
// where it takes the shape (and allow_decode), else the skinny kernel.
qmm_status wxa8_dispatch(int bits, const int8_t *xq, const void *sa, const uint8_t *w, const void *ws,
                         int group, void *y, int32_t *acc_out, int M, int N, int K, int *status,
                         int num_sms, int smem_optin, int smem_pair, bool allow_decode, cudaStream_t stream);

// The tcgen05 path (wxa8_tc.cu): whether it takes the shape, and its launch.
// Below these batch sizes the skinny kernel is faster (measured: W4A8 up to
// M = 4, W8A8 at M = 1).  Where the decode kernel's exact-integer mode takes
// the shape it is faster than tcgen05 up to kWxa8DecodeMaxM tokens (measured,
// K = N = 4096, group 128: W4A8 M = 8 7.9 against 9.1 us, M = 12 9.9 against
// 9.2 us; W8A8 M = 8 8.5 against 9.0 us).
constexpr int kW4a8TcMinM = 6;
constexpr int kW8a8TcMinM = 2;
constexpr int kWxa8DecodeMaxM = 8;
bool wxa8_tc_takes(int bits, int M, int N, int K, int group, const void *xq, const void *w);
qmm_status wxa8_tc_dispatch(int bits, const int8_t *xq, const void *sa, const uint8_t *w, const void *ws,
                            int group, void *y, int32_t *acc_out, int M, int N, int K, int *status,
                            int smem_optin, cudaStream_t stream);

}  // namespace qmm
