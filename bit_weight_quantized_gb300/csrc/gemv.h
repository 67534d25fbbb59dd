// gemv.h -- host interface of the skinny kernel (decode / small batches) and
// of the shared host helpers.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/qmm.h"

namespace qmm {

struct GemvParams {
    // a 2-D tensor map over the packed weights as 64-bit words [N][row_bytes / 8],
    // box pitch / 8 words x rb rows, so that one copy lands a stage (tma != 0)
    alignas(64) CUtensorMap tmw;
    int tma;
    const uint16_t *x;        // fp16 [M][K]                      (qmm_gemv)
    const int8_t *xq;         // int8 [M][K]                      (qmm_w4a8)
    const uint16_t *sa;       // fp16 [M] per-token scales        (qmm_w4a8)
    int32_t *acc_out;         // int32 [M][N][K/G] or nullptr     (qmm_w4a8)
    const uint8_t *packed;    // [N][K*b/8]
    const uint16_t *scales;   // fp16 [N][K/G]
    const uint8_t *zeros;     // uint8 [N][K/G] or nullptr
    void *y;                  // [M][N]
    int *status;              // device status word
    long long row_bytes;      // K*b/8
    int M, N, K, group, ng, zero_const, y_bf16;
    int use_bulk;             // rows 16-byte aligned: 1-D bulk copies, else plain copies
    // filled by skinny_plan
    int nchunks;              // ceil(K/128)
    int stages_per_block;     // K segments (pipeline stages) per row block
    int seg_chunks;           // 128-code chunks per K segment
    int seg_bytes;            // bytes of one row's segment (seg_chunks * 16 * b)
    int pitch;                // shared-memory row pitch of a stage
    int phase_chunks;         // chunks whose activations are staged at once
    int nphases;
    int rows_base, rows_rem;  // CTA c owns rows_base + (c < rows_rem) rows
    int rb, rbp;              // rows per block, rounded up to 16
    int ksplit_log2;          // 8 warps = 2^ksplit_log2 K splits x (8 >> ksplit_log2) tile groups
    int ring, stage_bytes;    // pipeline slots and the bytes of one
    int off_bar, off_x, off_xs, off_cs, off_sz, off_red, off_ring, sz_pitch;
    int sz_compact;           // scales staged as fp16 + uint8 zeros (M > 8), else float2 (s, z*s)
    int red_alias;            // the reduction buffer reuses the activation buffer
};

// Sets p.tma and p.tmw after skinny_plan when a stage can land with one tensor
// copy: bulk-copyable rows, a pitch that is a whole number of 16-byte units of
// at most 2048 bytes, segments on 16 bytes and a stage of rb rows.
void skinny_set_tma(GemvParams &p);

// Chooses grid, row blocking, K phases and the shared-memory layout.  A layout
// of at most `smem_pair` bytes (two CTAs per SM, so that consecutive calls
// overlap) is preferred; `smem_max` is the per-CTA limit.  QMM_ERR_UNSUPPORTED
// if no layout fits.
qmm_status skinny_plan(GemvParams &p, int bits, int num_sms, int smem_max, int smem_pair, int *grid,
                       int *smem);

// Per-width launchers (one translation unit each).
cudaError_t gemv_launch_w1(const GemvParams &, int, int, cudaStream_t);
cudaError_t gemv_launch_w2(const GemvParams &, int, int, cudaStream_t);
cudaError_t gemv_launch_w3(const GemvParams &, int, int, cudaStream_t);
cudaError_t gemv_launch_w4(const GemvParams &, int, int, cudaStream_t);
cudaError_t gemv_launch_w5(const GemvParams &, int, int, cudaStream_t);
cudaError_t gemv_launch_w6(const GemvParams &, int, int, cudaStream_t);
cudaError_t gemv_launch_w7(const GemvParams &, int, int, cudaStream_t);
cudaError_t gemv_launch_w8(const GemvParams &, int, int, cudaStream_t);
cudaError_t w4a8_launch(const GemvParams &, int, int, cudaStream_t);
cudaError_t w8a8_launch(const GemvParams &, int, int, cudaStream_t);

// fpgemv.cu: decode matmul with float weight codes (1 sign, e exponent, m mantissa bits).
cudaError_t launch_gemv_fp(const uint16_t *x, const uint8_t *packed, int ebits, int mbits, int group,
                           const uint16_t *scales, uint16_t *y, int M, int N, int K, cudaStream_t stream);
// quant.cu: per-token int8 quantization of fp16 activations (one CTA per token).
cudaError_t launch_quantize_act(const uint16_t *x, int8_t *xq, uint16_t *sa, int M, int K,
                                cudaStream_t stream);
cudaError_t launch_pack(const uint8_t *codes, uint8_t *packed, int N, int K, int bits,
                        int32_t *bad_count, cudaStream_t stream, int num_sms);
cudaError_t launch_unpack(const uint8_t *packed, uint8_t *codes, int N, int K, int bits,
                          cudaStream_t stream, int num_sms);
cudaError_t launch_flip_sign(uint8_t *packed, int N, int K, int bits, cudaStream_t stream, int num_sms);
cudaError_t launch_repack(const uint8_t *packed, uint8_t *out, int N, int K, int bits, int layout,
                          cudaStream_t stream, int num_sms);

// Tensor maps (api.cu).  A 2-D map over a byte matrix [rows][row_bytes] with a
// box_cols x box_rows box; and over a 16-bit matrix [rows][cols] with the
// 128-byte swizzle.
bool encode_byte_tmap(CUtensorMap *map, const void *base, long long row_bytes, long long rows,
                      int box_cols, int box_rows, bool swizzle128);
bool encode_u16_tmap(CUtensorMap *map, const void *base, long long cols, long long rows,
                     int box_cols, int box_rows);
// And over a matrix of 64-bit words [rows][cols], unswizzled, zero-filled
// outside (row pitch cols * 8 bytes).
bool encode_u64_tmap(CUtensorMap *map, const void *base, long long cols, long long rows,
                     int box_cols, int box_rows);

}  // namespace qmm
