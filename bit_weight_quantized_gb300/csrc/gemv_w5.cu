// gemv_w5.cu -- the skinny kernel instantiated for 5-bit weights.
#include "skinny.cuh"

namespace qmm {

cudaError_t gemv_launch_w5(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    return launch_skinny_width<5, 0>(p, grid, smem, stream);
}

}  // namespace qmm
