// decode_float_hi.cu -- the decode kernel on float weight codes of 6..8 bits
// (see decode_float.cu).
#include "decode.cuh"

namespace qmm {

cudaError_t launch_decode_float_hi(const DecodeParams &p, int bits, cudaStream_t stream)
{
    switch (bits) {
    case 6: return launch_decode_float_width<6>(p, stream);
    case 7: return launch_decode_float_width<7>(p, stream);
    case 8: return launch_decode_float_width<8>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
