// gemm.cu -- host dispatch of the tiled kernel (gemm.cuh): tensor maps,
// parameters, and the per-width launchers in gemm_w1.cu .. gemm_w8.cu.
#include <cstring>

#include "common.cuh"
#include "gemm.h"

namespace qmm {

bool gemm_supports_bits(int bits) { return bits >= 1 && bits <= 8; }

qmm_status gemm_dispatch(const void *x, bool x_bf16, const uint8_t *packed, int bits, int group,
                         const void *scales, const uint8_t *zeros, int zero_const, void *y, int M,
                         int N, int K, int *status, int num_sms, int smem_optin,
                         cudaStream_t stream)
{
    if (!gemm_supports_bits(bits))
        return QMM_ERR_BITS;
    if (group != 32 && group != 64 && group != 128)
        return QMM_ERR_SHAPE;
    const long long row_bytes = static_cast<long long>(K) * bits / 8;
    if (reinterpret_cast<uintptr_t>(packed) % 16 || row_bytes % 16 ||
        reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(y) % 16)
        return QMM_ERR_ALIGN;
    CUtensorMap tmx, tmw;
    std::memset(&tmx, 0, sizeof(tmx));
    std::memset(&tmw, 0, sizeof(tmw));
    if (!encode_u16_tmap(&tmx, x, K, M, kGemmBK, kGemmBM))
        return QMM_ERR_CUDA;
    const bool pow2 = bits == 1 || bits == 2 || bits == 4 || bits == 8;
    const int box = (pow2 ? 16 / bits : 2) * 8 * bits;   // bytes per row of a packed-weight stage
    if (!encode_byte_tmap(&tmw, packed, row_bytes, N, box, kGemmBN, pow2))
        return QMM_ERR_CUDA;
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.scales = static_cast<const uint16_t *>(scales);
    p.zeros = zeros;
    p.y = static_cast<uint16_t *>(y);
    p.status = status;
    p.M = M;
    p.N = N;
    p.K = K;
    p.group = group;
    p.ng = K / group;
    p.zero_const = zeros ? 0 : zero_const;
    p.bf16 = x_bf16 ? 1 : 0;
    p.zsplit = x_bf16 && (zeros || zero_const > 128) ? 1 : 0;
    p.group_log2 = group == 32 ? 5 : group == 64 ? 6 : 7;
    p.vec_scales = reinterpret_cast<uintptr_t>(scales) % 16 == 0 && p.ng % 8 == 0 &&
                   (!zeros || reinterpret_cast<uintptr_t>(zeros) % 8 == 0);
    p.tiles_n = (N + kGemmBN - 1) / kGemmBN;
    p.mtiles = (M + kGemmBM - 1) / kGemmBM;
    p.ksteps = (K + kGemmBK - 1) / kGemmBK;
    const int grid = p.tiles_n < num_sms ? p.tiles_n : num_sms;
    switch (bits) {
    case 1: return gemm_launch_w1(tmx, tmw, p, grid, smem_optin, stream);
    case 2: return gemm_launch_w2(tmx, tmw, p, grid, smem_optin, stream);
    case 3: return gemm_launch_w3(tmx, tmw, p, grid, smem_optin, stream);
    case 4: return gemm_launch_w4(tmx, tmw, p, grid, smem_optin, stream);
    case 5: return gemm_launch_w5(tmx, tmw, p, grid, smem_optin, stream);
    case 6: return gemm_launch_w6(tmx, tmw, p, grid, smem_optin, stream);
    case 7: return gemm_launch_w7(tmx, tmw, p, grid, smem_optin, stream);
    default: return gemm_launch_w8(tmx, tmw, p, grid, smem_optin, stream);
    }
}

}  // namespace qmm
