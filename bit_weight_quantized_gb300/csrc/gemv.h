// gemv.h -- host interface of the skinny (M <= 16) kernel.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/qmm.h"

namespace qmm {

struct GemvParams {
    const uint16_t *x;        // fp16 [M][K]
    const uint8_t *packed;    // [N][K*b/8]
    const uint16_t *scales;   // fp16 [N][K/G]
    const uint8_t *zeros;     // uint8 [N][K/G] or nullptr
    void *y;                  // [M][N]
    int *status;              // device status word
    long long row_bytes;      // K*b/8
    int M, N, K, group, ng, zero_const, y_bf16, use_tma;
    // filled by gemv_plan
    int nchunks;              // ceil(K/128)
    int stages_per_block;     // TMA stages per row block
    int rows_base, rows_rem;  // CTA c owns rows_base + (c < rows_rem) rows
    int rb, rbp;              // rows per block, rounded up to 16
    int ring, stage_bytes, tile_bytes;
    int off_bar, off_x, off_xs, off_sz, off_red, sz_pitch;
};

// Chooses grid, row blocking and the shared-memory layout.  QMM_ERR_UNSUPPORTED
// if the activations do not fit in shared memory next to a 4-stage ring.
qmm_status gemv_plan(GemvParams &p, int bits, int num_sms, int smem_max, int *grid, int *smem);

// Launches the kernel for `bits` (tensor map used only when p.use_tma).
cudaError_t gemv_launch(const CUtensorMap &tmap, const GemvParams &p, int bits, int grid,
                        int smem, cudaStream_t stream);

// Chunks of 128 codes per TMA stage for width b (the stage box is
// 16*b*cs bytes wide).
int gemv_stage_chunks(int bits);

cudaError_t launch_pack(const uint8_t *codes, uint8_t *packed, int N, int K, int bits,
                        int32_t *bad_count, cudaStream_t stream, int num_sms);
cudaError_t launch_unpack(const uint8_t *packed, uint8_t *codes, int N, int K, int bits,
                          cudaStream_t stream, int num_sms);

}  // namespace qmm
