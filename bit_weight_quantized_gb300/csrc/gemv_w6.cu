// gemv_w6.cu -- the skinny kernel instantiated for 6-bit weights.
#include "skinny.cuh"

namespace qmm {

cudaError_t gemv_launch_w6(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    return launch_skinny_width<6, 0>(p, grid, smem, stream);
}

}  // namespace qmm
