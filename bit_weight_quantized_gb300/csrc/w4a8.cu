// w4a8.cu -- integer-native W4A8 path (placeholder until the kernel lands).
#include "common.cuh"
#include "w4a8.h"

namespace qmm {

qmm_status w4a8_dispatch(const int8_t *, const void *, const uint8_t *, const void *, int, void *,
                         int32_t *, int, int, int, int *, int, int, cudaStream_t)
{
    return QMM_ERR_UNSUPPORTED;
}

}  // namespace qmm
