// gemv_w4.cu -- the skinny kernel instantiated for 4-bit weights.
#include "skinny.cuh"

namespace qmm {

cudaError_t gemv_launch_w4(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    return launch_skinny_width<4, 0>(p, grid, smem, stream);
}

}  // namespace qmm
