// w8a8.cu -- integer-native W8A8 (BitLLM, Experiment Setup: 8-bit weights and
// activations with group-wise scaling) on the skinny kernel: the W4A8 scheme
// of w4a8.cu with signed int8 weights.  c is read as u = c xor 128 in
// [0, 255], so w = u - 128; D = sum u*x stays an integer below 2^24 for groups
// of at most 128 (|D| <= 128 * 255 * 128), and acc = D - 128 * sum x is the
// exact int32 accumulator.  Its own translation unit, so that the 8-bit
// instantiations compile in parallel with the rest.
#include "gemv.h"
#include "skinny.cuh"

namespace qmm {

cudaError_t w8a8_launch(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    return launch_skinny_width<8, 1>(p, grid, smem, stream);
}

}  // namespace qmm
