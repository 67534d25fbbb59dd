// decode_float.cu -- the decode kernel on float weight codes (qmm_gemv_float
// with codes of at most 4 exponent bits), widths 2..5; widths 6..8 are in
// decode_float_hi.cu, so that the two compile in parallel.
#include "decode.cuh"

namespace qmm {

cudaError_t launch_decode_float_hi(const DecodeParams &p, int bits, cudaStream_t stream);

cudaError_t launch_decode_float(const DecodeParams &p, int bits, cudaStream_t stream)
{
    switch (bits) {
    case 2: return launch_decode_float_width<2>(p, stream);
    case 3: return launch_decode_float_width<3>(p, stream);
    case 4: return launch_decode_float_width<4>(p, stream);
    case 5: return launch_decode_float_width<5>(p, stream);
    default: return launch_decode_float_hi(p, bits, stream);
    }
}

}  // namespace qmm
