// decode.h -- the staging-free decode kernel (decode.cu): 1 <= M <= 8, groups of
// 64 or 128, K a multiple of 8 groups, at most 32 output columns per CTA.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qmm {

struct DecodeParams {
    const uint16_t *x;        // fp16 [M][K], 16-byte aligned
    const uint8_t *packed;    // [N][K*b/8], 16-byte aligned
    const uint16_t *scales;   // fp16 [N][K/G]
    const uint8_t *zeros;     // uint8 [N][K/G] or nullptr (then zero_const)
    void *y;                  // fp16 or bf16 [M][N]
    int M, N, K, group_log2, zero_const, y_bf16;
    int rows_base, rows_rem;  // set by launch_decode: CTA c owns rows_base + (c < rows_rem) rows
};

// True when the shape is one the kernel takes (with a grid of min(N, num_sms) CTAs).
bool decode_supports(int M, int N, int K, int group, int num_sms);

// Launches the kernel for b = bits (1..8) with programmatic dependent launch.
cudaError_t launch_decode(DecodeParams p, int bits, int num_sms, cudaStream_t stream);

}  // namespace qmm
