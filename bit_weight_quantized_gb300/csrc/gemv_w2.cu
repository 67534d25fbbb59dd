// gemv_w2.cu -- the skinny kernel instantiated for 2-bit weights.
#include "skinny.cuh"

namespace qmm {

cudaError_t gemv_launch_w2(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    return launch_skinny_width<2, 0>(p, grid, smem, stream);
}

}  // namespace qmm
