// w4a8.cu -- integer-native W4A8 (BitLLM sec. 4.3-4.4) on the skinny kernel.
//
// Signed int4 weights c (two's complement nibbles, the 4-bit bitstream) are
// read as u = c xor 8 in [0, 15], so w = u - 8; int8 activations are staged as
// exact fp16.  Per group the kernel forms D = sum u*x on fp16 tensor cores --
// every product and partial sum is an integer below 2^24, so fp32 accumulation
// is exact -- and acc = D - 8 * sum x, the exact int32 accumulator.  The
// epilogue applies the per-group weight scale and per-token activation scale:
// y = sa[m] * sum_g ws[n][g] * acc.  The host dispatch here also serves W8A8
// (signed int8 weights, w8a8.cu).
#include <cstring>

#include "decode.h"
#include "gemv.h"
#include "skinny.cuh"
#include "w4a8.h"

namespace qmm {

cudaError_t w4a8_launch(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    return launch_skinny_width<4, 1>(p, grid, smem, stream);
}

qmm_status wxa8_dispatch(int bits, const int8_t *xq, const void *sa, const uint8_t *w, const void *ws,
                         int group, void *y, int32_t *acc_out, int M, int N, int K, int *status,
                         int num_sms, int smem_optin, int smem_pair, bool allow_decode, cudaStream_t stream)
{
    DecodePlan plan;
    const bool decode = allow_decode && M <= kWxa8DecodeMaxM && reinterpret_cast<uintptr_t>(w) % 16 == 0 &&
                        reinterpret_cast<uintptr_t>(xq) % 16 == 0 &&
                        decode_plan(M, N, K, group, bits, false, false, num_sms, smem_pair, smem_optin, &plan);
    const int tc_min = decode ? kWxa8DecodeMaxM + 1 : bits == 8 ? kW8a8TcMinM : kW4a8TcMinM;
    if (M >= tc_min && wxa8_tc_takes(bits, M, N, K, group, xq, w))
        return wxa8_tc_dispatch(bits, xq, sa, w, ws, group, y, acc_out, M, N, K, status, smem_optin, stream);
    if (decode) {
        // the decode kernel's exact-integer mode: weights staged before the
        // dependency wait, codes as exact small integers on the tensor cores
        DecodeParams d;
        std::memset(&d, 0, sizeof(d));
        d.x = reinterpret_cast<const uint16_t *>(xq);
        d.packed = w;
        d.scales = static_cast<const uint16_t *>(ws);
        d.zeros = nullptr;
        d.y = y;
        d.status = status;
        d.row_bytes = static_cast<long long>(K) * bits / 8;
        d.M = M;
        d.N = N;
        d.K = K;
        d.group_log2 = group == 64 ? 6 : 7;
        d.zero_const = 1 << (bits - 1);
        d.vec_sz = reinterpret_cast<uintptr_t>(ws) % 16 == 0;
        d.sa = static_cast<const uint16_t *>(sa);
        d.acc_out = acc_out;
        d.pl = plan;
        decode_set_tma(d);
        return launch_decode_int(d, bits, stream) == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
    }
    GemvParams p;
    std::memset(&p, 0, sizeof(p));
    p.xq = xq;
    p.sa = static_cast<const uint16_t *>(sa);
    p.acc_out = acc_out;
    p.packed = w;
    p.scales = static_cast<const uint16_t *>(ws);
    p.zeros = nullptr;
    p.zero_const = 1 << (bits - 1);
    p.y = y;
    p.status = status;
    p.row_bytes = static_cast<long long>(K) * bits / 8;
    p.M = M;
    p.N = N;
    p.K = K;
    p.group = group;
    p.ng = K / group;
    p.y_bf16 = 0;
    int grid = 0, smem = 0;
    qmm_status st = skinny_plan(p, bits, num_sms, smem_optin, smem_pair, &grid, &smem);
    if (st != QMM_OK)
        return st;
    p.use_bulk = (reinterpret_cast<uintptr_t>(w) % 16 == 0) && (p.row_bytes % 16 == 0);
    skinny_set_tma(p);
    const cudaError_t e = bits == 8 ? w8a8_launch(p, grid, smem, stream) : w4a8_launch(p, grid, smem, stream);
    return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

}  // namespace qmm
