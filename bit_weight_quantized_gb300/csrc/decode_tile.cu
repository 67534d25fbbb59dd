// decode_tile.cu -- the staged decode kernel for weights in the
// fragment-ordered (tile16) layout (decode.cuh; one translation unit per
// layout so that the two compile in parallel).
#include "decode.cuh"

namespace qmm {

cudaError_t launch_decode_tile16(const DecodeParams &p, int bits, cudaStream_t stream)
{
    return launch_decode_layout<true>(p, bits, stream);
}

}  // namespace qmm
