// gemm.h -- host interface of the tiled (M >= 17) kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/qmm.h"
#include "gemv.h"

namespace qmm {

// Tile shape of the tiled kernel: output columns per tile (the MMA's N),
// tokens per M tile (the MMA's M), K per step.
constexpr int kGemmBN = 192;
constexpr int kGemmBM = 128;
constexpr int kGemmBK = 64;

struct GemmParams {
    const uint16_t *scales;   // fp16 [N][K/G]
    const uint8_t *zeros;     // uint8 [N][K/G] or nullptr
    uint16_t *y;              // [M][N]
    int *status;
    int M, N, K, group, ng, zero_const, bf16;
    int group_log2;           // G = 1 << group_log2
    int vec_scales;           // scale rows 16-byte aligned and ng % 8 == 0 (zeros 8-byte aligned)
    int zsplit;               // bf16 with zeros that may exceed 128: subtract z in two exact steps
    int tiles_n, mtiles, passes, ksteps;
};

// Per-width launchers (gemm_w1.cu .. gemm_w8.cu).
#define QMM_GEMM_DECL(W)                                                                                     \
    qmm_status gemm_launch_w##W(const CUtensorMap &tmx, const CUtensorMap &tmw, const GemmParams &p, int grid, \
                                int smem_optin, cudaStream_t stream);
QMM_GEMM_DECL(1)
QMM_GEMM_DECL(2)
QMM_GEMM_DECL(3)
QMM_GEMM_DECL(4)
QMM_GEMM_DECL(5)
QMM_GEMM_DECL(6)
QMM_GEMM_DECL(7)
QMM_GEMM_DECL(8)
#undef QMM_GEMM_DECL

// Widths the tiled kernel dequantizes.
bool gemm_supports_bits(int bits);

qmm_status gemm_dispatch(const void *x, bool x_bf16, const uint8_t *packed, int bits, int group,
                         const void *scales, const uint8_t *zeros, int zero_const, void *y, int M,
                         int N, int K, int *status, int num_sms, int smem_optin,
                         cudaStream_t stream);

}  // namespace qmm
