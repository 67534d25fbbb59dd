// gemv_w8.cu -- the skinny kernel instantiated for 8-bit weights.
#include "skinny.cuh"

namespace qmm {

cudaError_t gemv_launch_w8(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    return launch_skinny_width<8, 0>(p, grid, smem, stream);
}

}  // namespace qmm
