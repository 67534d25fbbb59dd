// decode_float.cu -- the decode kernel on float weight codes (qmm_gemv_float
// with 4- or 8-bit codes of at most 4 exponent bits); its own translation unit
// so that it compiles beside the integer widths.
#include "decode.cuh"

namespace qmm {

cudaError_t launch_decode_float(const DecodeParams &p, int bits, cudaStream_t stream)
{
    return launch_decode_float_layout(p, bits, stream);
}

}  // namespace qmm
