// decode.h -- the staged decode kernel (decode.cu): 1 <= M <= 16, groups of 64
// or 128, K a multiple of 8 groups, weights staged in shared memory by bulk copies.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qmm {

// Launch plan of one call: grid, row split, K segments and the shared-memory
// layout (byte offsets from the 128-byte aligned dynamic shared memory base).
struct DecodePlan {
    int grid;                 // CTAs: min(N, SMs)
    int rows_base, rows_rem;  // CTA c owns rows_base + (c < rows_rem) output columns (tile16: 16-row tiles)
    int max_rows;             // rows of the largest CTA
    int warps;                // warps per CTA (8)
    int kseg;                 // codes per K segment: one group per warp
    int nseg;                 // K / kseg
    int seg_bytes;            // kseg * b / 8: one row's bytes of one segment
    int span;                 // segments per ring slot: nseg (whole rows) or 1
    int pitch;                // bytes between rows in a ring slot (padded; 0 for tile16)
    int slot_bytes;           // min(32, max_rows) * pitch
    int slots;                // ring depth: segments in flight
    int x_pitch;              // bytes per token of one warp's activation stage
    int off_x, off_xsum, off_sc, off_zo, off_red, off_bar;
    int smem;                 // dynamic shared memory per CTA
};

struct DecodeParams {
    // canonical layout (tma != 0): a 2-D tensor map over the packed weights as
    // 64-bit words [N][row_bytes / 8], box pitch / 8 words x min(32, max_rows)
    // rows, so that one copy lands a ring chunk's rows at the slot pitch
    alignas(64) CUtensorMap tmw;
    int tma;
    const uint16_t *x;        // fp16 or bf16 [M][K], 16-byte aligned
    const uint8_t *packed;    // [N][K*b/8], 16-byte aligned
    const uint16_t *scales;   // fp16 [N][K/G]
    const uint8_t *zeros;     // uint8 [N][K/G] or nullptr (then zero_const)
    void *y;                  // fp16 or bf16 [M][N]
    int *status;              // device status word
    long long row_bytes;      // K * b / 8
    int M, N, K, group_log2, y_bf16;
    int x_bf16;               // activations are bf16 (converted to fp16 as they are staged)
    int zero_const;           // the zero of every group when zeros == nullptr
    int vec_sz;               // scales 16-byte and zeros 8-byte aligned: vector staging
    int ebits, mbits;         // float codes: exponent and mantissa bits (0 for integer codes)
    float fscale;             // float codes: 2^(15 - bias), folded into the scale
    // exact-integer mode (qmm_w4a8 / qmm_w8a8): x holds int8 [M][K], zero_const
    // is 2^(b-1), y = sa[m] * sum_g s * acc, and the int32 accumulators go to
    // acc_out [M][N][K/G] when it is not null
    const uint16_t *sa;       // fp16 [M] per-token activation scales
    int32_t *acc_out;
    DecodePlan pl;
};

// Whether the canonical ring of `plan` can land each chunk with one tensor-map
// box: a padded pitch that is a whole number of 16-byte units of at most 2048
// bytes (256 64-bit words, the box limit) and chunks that start on 16 bytes.
// The box covers min(32, max_rows) rows, exactly a slot.
inline bool decode_tma_fits(const DecodePlan &plan, long long row_bytes)
{
    return plan.pitch > 0 && plan.pitch % 16 == 0 && plan.pitch <= 2048 && row_bytes % 16 == 0 &&
           (static_cast<long long>(plan.span) * plan.seg_bytes) % 16 == 0;
}

// Rows of the canonical ring's tensor-map box (a slot's rows).
__host__ __device__ inline int decode_tma_rows(const DecodePlan &plan) { return plan.max_rows < 32 ? plan.max_rows : 32; }

// Plans a call; false if the kernel does not take the shape (the skinny kernel
// does).  smem_pair is the per-CTA shared memory with which two CTAs share an
// SM, smem_optin the most one CTA may use.  Host code only.
bool decode_plan(int M, int N, int K, int group, int bits, bool stored_zeros, bool tile16, int num_sms,
                 int smem_pair, int smem_optin, DecodePlan *plan);

// Launches the kernel for b = bits (1..8) with programmatic dependent launch;
// tile16: the weights are in the fragment-ordered layout (qmm_repack).
cudaError_t launch_decode(const DecodeParams &p, int bits, bool tile16, cudaStream_t stream);
cudaError_t launch_decode_tile16(const DecodeParams &p, int bits, cudaStream_t stream);
// Float codes (qmm_gemv_float): bits 2..8, at most 4 exponent bits.
cudaError_t launch_decode_float(const DecodeParams &p, int bits, cudaStream_t stream);
// Exact-integer mode (decode_int.cu): int8 activations, signed 4- or 8-bit weights.
cudaError_t launch_decode_int(const DecodeParams &p, int bits, cudaStream_t stream);
// Sets p.tma and p.tmw when the canonical ring can land its chunks by
// tensor-map boxes (decode_tma_fits); host code, in decode_int.cu.
void decode_set_tma(DecodeParams &p);

}  // namespace qmm
