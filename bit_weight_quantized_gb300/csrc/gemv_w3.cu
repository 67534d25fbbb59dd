// gemv_w3.cu -- the skinny kernel instantiated for 3-bit weights.
#include "skinny.cuh"

namespace qmm {

cudaError_t gemv_launch_w3(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    return launch_skinny_width<3, 0>(p, grid, smem, stream);
}

}  // namespace qmm
