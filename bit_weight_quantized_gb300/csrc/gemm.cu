// gemm.cu -- tiled tcgen05 path (placeholder until the kernel lands).
#include "common.cuh"
#include "gemm.h"

namespace qmm {

qmm_status gemm_dispatch(const void *, bool, const uint8_t *, int, int, const void *,
                         const uint8_t *, int, void *, int, int, int, int *, int, int,
                         cudaStream_t)
{
    return QMM_ERR_UNSUPPORTED;
}

}  // namespace qmm
