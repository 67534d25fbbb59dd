// decode_int.cu -- the decode kernel in its exact-integer mode (qmm_w4a8 /
// qmm_w8a8 at small batches: int8 activations staged as exact fp16, signed
// weights read as offset-binary codes with the plan's 2^E offset taken off
// before the MMA, so that every product and group sum is an exact integer in
// fp32), and the canonical ring's tensor map.
#include "decode.cuh"
#include "gemv.h"

namespace qmm {

cudaError_t launch_decode_int(const DecodeParams &p, int bits, cudaStream_t stream)
{
    switch (bits) {
    case 4: return launch_decode_int_width<4>(p, stream);
    case 8: return launch_decode_int_width<8>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

void decode_set_tma(DecodeParams &p)
{
    p.tma = 0;
    if (decode_tma_fits(p.pl, p.row_bytes) &&
        encode_u64_tmap(&p.tmw, p.packed, p.row_bytes / 8, p.N, p.pl.pitch / 8, decode_tma_rows(p.pl)))
        p.tma = 1;
}

}  // namespace qmm
