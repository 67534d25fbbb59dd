// gemv_w1.cu -- the skinny kernel instantiated for 1-bit weights.
#include "skinny.cuh"

namespace qmm {

cudaError_t gemv_launch_w1(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    return launch_skinny_width<1, 0>(p, grid, smem, stream);
}

}  // namespace qmm
