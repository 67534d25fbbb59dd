// gemv_w7.cu -- the skinny kernel instantiated for 7-bit weights.
#include "skinny.cuh"

namespace qmm {

cudaError_t gemv_launch_w7(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    return launch_skinny_width<7, 0>(p, grid, smem, stream);
}

}  // namespace qmm
