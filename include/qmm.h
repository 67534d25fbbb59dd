/*
 * qmm.h -- C ABI of libqmm: FP16/BF16 activations x b-bit quantized weights
 * (b = 1..8), the integer-native W4A8 / W8A8 variants with their per-token
 * activation quantizer, and signed and float weight codes, on one GB300
 * (sm_103a).
 *
 * The operation (Tilus review, lead and pith_extraction.core_discovery: a
 * matmul of FP16 activations by weights of any width from 1 to 8 bits that
 * are loaded as packed bytes and reinterpreted; BitLLM sec. 2.2 Eq. (5) and
 * sec. 4.3-4.4 for the per-group affine dequantization and the int8 x int4
 * integer pipeline):
 *
 *     y[m][n] = sum_k x[m][k] * W[n][k],
 *     W[n][k] = (q[n][k] - z[n][k/G]) * s[n][k/G]          (BitLLM Eq. 5)
 *
 * Weight storage ("packed bitstream"): column n (output feature n) is its
 * own byte string of K*b/8 bytes at packed + n*K*b/8.  Code k occupies
 * stream bits [k*b, k*b+b); stream bit i is bit (i mod 8) of byte i/8
 * (LSB first); bit j of the code is stream bit k*b+j.  So 8 codes always
 * fill exactly b bytes, and a group of 32 codes is exactly b 32-bit words.
 *
 * Conventions for every call:
 *  - Pointers marked (device) are device memory owned by the caller; the
 *    library allocates nothing and keeps no per-call state.  Pointers marked
 *    (host) are host memory.
 *  - fp16 / bf16 tensors are passed as void* holding 16-bit IEEE binary16 /
 *    bfloat16 bit patterns.  Matrices are dense and row-major with the
 *    shapes given; there are no stride arguments.
 *  - Every call is asynchronous on `stream` (0 = the legacy default
 *    stream).  Argument errors are detected on the host before anything is
 *    launched and return a status without touching the device.  Launch
 *    failures return QMM_ERR_CUDA.  Device-side watchdog expiries (a
 *    pipeline wait that did not complete within about a second) do not trap:
 *    the kernel records QMM_ERR_TIMEOUT in a device status word, leaves its
 *    outputs unspecified and returns; qmm_device_status() reports and clears
 *    it.  Nothing in the library aborts, throws across the ABI or traps.
 *  - Outputs are written with round-to-nearest-even from fp32.
 *  - Overlap of consecutive calls.  qmm_gemv, qmm_gemm, qmm_w4a8, qmm_w8a8,
 *    qmm_gemv_float and qmm_quantize_act launch with programmatic dependent
 *    launch and let the next kernel on the stream start as soon as they start
 *    themselves.  The matmul calls read their weight arguments (packed / w4 /
 *    w8, scales / ws, zeros) BEFORE they wait for the preceding kernel;
 *    activations (x / xq, sa) are read only after that wait, which returns
 *    once every earlier kernel on the stream has completed.  Because each of
 *    these calls lets its successor start early, a whole run of consecutive
 *    such calls on one stream can be in flight at once.  So no call of such a
 *    run may write the weight arguments of a later call of the same run (for
 *    example as its y).  Any other work on the stream ends the run: qmm_pack,
 *    qmm_unpack, qmm_flip_sign, copies and ordinary CUDA / PyTorch kernels do
 *    not opt in to early launch, so the calls after them start only once they
 *    (and everything before them) have completed, and writing weights with
 *    them is fine.
 */
#ifndef QMM_H_
#define QMM_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define QMM_API __attribute__((visibility("default")))
#else
#define QMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QMM_OK = 0,
    QMM_ERR_NULL = 1,         /* a required pointer is NULL                      */
    QMM_ERR_BITS = 2,         /* bits outside the supported range               */
    QMM_ERR_SHAPE = 3,        /* negative size, K % group, unsupported M range  */
    QMM_ERR_ALIGN = 4,        /* a pointer or row pitch breaks an alignment rule */
    QMM_ERR_UNSUPPORTED = 5,  /* valid but not implemented (dtype, group, size) */
    QMM_ERR_CUDA = 6,         /* a CUDA runtime call or kernel launch failed     */
    QMM_ERR_TIMEOUT = 8,      /* device watchdog expired (see qmm_device_status) */
    QMM_ERR_DEVICE = 9        /* no usable sm_103a device                       */
} qmm_status;

typedef enum { QMM_F16 = 0, QMM_BF16 = 1 } qmm_dtype;

/* Pack b-bit codes into the column bitstream (packing is the storage format
 * above; BitLLM sec. 4.3 Fig. 8(a) is the b = 4 case).
 *   codes     (device) uint8 [N][K]; only the low `bits` bits of each code are
 *             stored.
 *   packed    (device) uint8 [N][K*bits/8], fully overwritten.
 *   bad_count (device, may be NULL) int32; the number of codes >= 2^bits is
 *             ADDED to it (the caller zeroes it first if a fresh count is
 *             wanted).
 * Requires 1 <= bits <= 8, N >= 0, K >= 0, K*bits % 8 == 0. */
QMM_API qmm_status qmm_pack(const uint8_t *codes, uint8_t *packed, int N, int K, int bits,
                    int32_t *bad_count, cudaStream_t stream);

/* Inverse of qmm_pack (a test aid): packed (device) [N][K*bits/8] ->
 * codes (device) uint8 [N][K]. */
QMM_API qmm_status qmm_unpack(const uint8_t *packed, uint8_t *codes, int N, int K, int bits,
                      cudaStream_t stream);

/* Decode / skinny matmul, 1 <= M <= 16 (BitLLM sec. 5.1 decodes at batch 1;
 * the skinny range covers small batches).  Streams the bitstream through
 * shared memory with bulk copies (TMA), extracts codes in registers and
 * accumulates in fp32 on tensor cores.
 *   x        (device) [M][K] activations, dtype x_dtype: QMM_F16, or QMM_BF16
 *            where the decode kernel takes the shape (see below; bf16 values
 *            are converted to fp16 as they are staged, exactly for magnitudes
 *            in [2^-14, 65504], to the fp16 subnormal grid below; magnitudes
 *            above 65504 are outside the contract).  16-byte aligned.
 *   packed   (device) [N][K*bits/8] bitstream, 16-byte aligned.
 *   bits     1..8.   group: G in {32, 64, 128}, K % G == 0.
 *   scales   (device) fp16 [N][K/G].
 *   zeros    (device) uint8 [N][K/G], or NULL to use zero_const for every
 *            group (0 <= zero_const <= 255).
 *   y        (device) [M][N], dtype y_dtype (QMM_F16 or QMM_BF16).
 * The tensor cores see the integer codes q exactly (as fp16 2^E + q) and the
 * fp16 activations, and accumulate each group in fp32; the group's offset,
 * scale and zero are applied in fp32 afterwards as s*(sum (2^E+q)*x - sum 2^E*x
 * - z*sum x), which equals sum s*(q - z)*x.  Results are deterministic run to
 * run.
 * Two kernels serve the call (qmm_gemv_route() tells which).  The decode kernel
 * takes G in {64, 128}, K % (8*G) == 0 and a 16-byte aligned `packed` when its
 * planner finds a shared-memory layout: each CTA copies its weight rows into
 * shared memory before waiting on the preceding kernel (one 2-D tensor copy
 * per ring slot, or one bulk copy per row where a slot's row pitch exceeds
 * 2048 bytes), then stages the activations.  The skinny kernel takes every
 * other shape (fp16 activations only: QMM_BF16 there returns
 * QMM_ERR_UNSUPPORTED); M x K fp16 must fit in
 * its shared memory next to the weight pipeline (larger return
 * QMM_ERR_UNSUPPORTED).  The two sum in different orders, so their outputs may
 * differ in the last bits.  qmm_set_gemv_kernel() forces the skinny kernel.
 * K % 32 == 0 is implied by the group rule. */
QMM_API qmm_status qmm_gemv(const void *x, qmm_dtype x_dtype, const uint8_t *packed, int bits,
                    int group, const void *scales, const uint8_t *zeros, int zero_const,
                    void *y, qmm_dtype y_dtype, int M, int N, int K, cudaStream_t stream);

/* Kernel choice of qmm_gemv for the calls that follow, process-wide:
 *   QMM_GEMV_AUTO   (0, the default) the decode kernel where it applies,
 *                   else the skinny kernel;
 *   QMM_GEMV_SKINNY (1) the skinny kernel for every shape (and qmm_w4a8 /
 *                   qmm_w8a8 off the decode kernel: the skinny or tcgen05 one).
 * Returns QMM_ERR_SHAPE for any other value.  The setting is read when a call
 * is issued; it does not change calls already issued. */
typedef enum { QMM_GEMV_AUTO = 0, QMM_GEMV_SKINNY = 1 } qmm_gemv_kernel;
QMM_API qmm_status qmm_set_gemv_kernel(int kernel);

/* Which kernel a qmm_gemv call of this shape would run on the current device
 * under the current qmm_set_gemv_kernel() setting, with a 16-byte aligned
 * `packed`: QMM_GEMV_AUTO (0) for the staged decode kernel, QMM_GEMV_SKINNY (1)
 * for the skinny kernel, or minus a status code (-QMM_ERR_SHAPE for a shape
 * qmm_gemv rejects, -QMM_ERR_DEVICE without a usable device).  stored_zeros is
 * nonzero when the call passes per-group zeros.  Launches nothing. */
QMM_API int qmm_gemv_route(int M, int N, int K, int bits, int group, int stored_zeros);

/* Tiled matmul for M >= 17 (the dense-contraction regime, Tilus review
 * supporting_citations [41]: tensor-core instruction layouts).  Same
 * arguments and storage as qmm_gemv, with these differences:
 *   - x and y may be QMM_BF16 or QMM_F16 (x_dtype == y_dtype);
 *   - x, y and packed must be 16-byte aligned and K * bits / 8 (the packed
 *     row pitch) a multiple of 16 bytes (else QMM_ERR_ALIGN);
 *   - any width 1..8 (the Tilus review's one matmul for every width).
 * Packed weights arrive by TMA in stages (128-byte swizzled boxes per row at
 * widths 1, 2, 4 and 8; two 64-code K steps per stage at the other widths),
 * are dequantized to bf16/fp16 (q - z) * s tiles in shared memory (one
 * rounding of the exact product; q - z itself is exact for every zero
 * 0..255) and multiplied with tcgen05 MMAs accumulating in fp32 in tensor
 * memory.  With fp16 the dequantized weight must be finite in fp16:
 * |q - z| * s < 65504. */
QMM_API qmm_status qmm_gemm(const void *x, qmm_dtype x_dtype, const uint8_t *packed, int bits,
                    int group, const void *scales, const uint8_t *zeros, int zero_const,
                    void *y, qmm_dtype y_dtype, int M, int N, int K, cudaStream_t stream);

/* Integer-native W4A8 (BitLLM sec. 4.3-4.4: int8 x int4 dot products into
 * int32, dequantization deferred to an epilogue):
 *   acc[m][n][g] = sum_{k in group g} xq[m][k] * w[n][k]          (int32, exact)
 *   y[m][n]      = sa[m] * sum_g ws[n][g] * acc[m][n][g]          (fp32 -> fp16)
 *   xq      (device) int8 [M][K] activations.
 *   sa      (device) fp16 [M] per-token activation scales.
 *   w4      (device) uint8 [N][K/2]: signed int4 weights in [-8, 7], 4-bit two's
 *           complement, the b = 4 bitstream (even k in the low nibble).
 *   ws      (device) fp16 [N][K/G] per-group weight scales, G in {32, 64, 128}.
 *   y       (device) fp16 [M][N].
 *   acc_out (device, may be NULL) int32 [M][N][K/G]: the integer accumulators.
 * Requires 1 <= M <= 64 (decode and small batches), K % G == 0.
 * Three kernels serve it, all on exact fp16 operands (every product and group
 * sum is an integer below 2^24, so fp32 accumulation is exact).  Up to M = 8,
 * with G in {64, 128}, K % (8*G) == 0 and xq, w4 16-byte aligned, the decode
 * kernel of qmm_gemv in its exact-integer mode (weights staged in shared
 * memory before the dependency wait).  Above that, and from M = 6 where the
 * decode kernel does not apply, a tcgen05 kernel when K is a multiple of 512
 * and K/G/4 <= 32: each group accumulates in its own tensor-memory
 * accumulator, a cluster of four CTAs splits K.  Every other shape takes the
 * skinny kernel (mma.sync).  qmm_set_gemv_kernel(QMM_GEMV_SKINNY) keeps this
 * call (and qmm_w8a8) off the decode kernel. */
QMM_API qmm_status qmm_w4a8(const int8_t *xq, const void *sa, const uint8_t *w4, const void *ws,
                    int group, void *y, int32_t *acc_out, int M, int N, int K,
                    cudaStream_t stream);

/* Float weight codes (the float3-float8 types of the Tilus review's arbitrary
 * low-precision types; the pages fix no exponent / mantissa split and no
 * special values).  Reading: a code of b = 1 + ebits + mbits bits holds a sign
 * bit, ebits exponent bits and mbits mantissa bits (top to bottom), bias
 * 2^(ebits-1) - 1, and every encoding is finite:
 *   E > 0: (-1)^s 2^(E - bias) (1 + M / 2^mbits),  E = 0: (-1)^s 2^(1 - bias) M / 2^mbits,
 * W[n][k] = value(code k of column n) * scales[n][k/G], y = x . W^T.
 *   x       (device) fp16 [M][K], 16-byte aligned; 1 <= M <= 16.
 *   packed  (device) uint8 [N][K*b/8]: the b-bit stream of qmm_pack, 4-byte aligned.
 *   scales  (device) fp16 [N][K/G]; G in {32, 64, 128}, K % G == 0.
 *   y       (device) fp16 [M][N], fully overwritten (fp32 accumulation, RNE).
 * Products of a weight and an activation are exact in fp32; the sums round.
 * Two kernels serve it.  Codes with ebits <= 4, G in {64, 128},
 * K % (8*G) == 0 and a 16-byte aligned `packed` run on the decode kernel's
 * tensor-core path: a code's exponent and mantissa fields placed at the top of
 * the fp16 fields and its sign at bit 15 read exactly as its value times
 * 2^(bias - 15), a power of two folded into the group scale.  Everything else
 * (ebits = 5, whose top exponent would read as inf in fp16; G = 32; other
 * shapes) runs on an FFMA kernel.
 * Errors: QMM_ERR_BITS (ebits < 1 or b outside 2..8), QMM_ERR_SHAPE,
 * QMM_ERR_NULL, QMM_ERR_ALIGN, QMM_ERR_DEVICE, QMM_ERR_CUDA. */
QMM_API qmm_status qmm_gemv_float(const void *x, const uint8_t *packed, int ebits, int mbits,
                                  int group, const void *scales, void *y, int M, int N, int K,
                                  cudaStream_t stream);

/* Pre-permuted weight layouts, written offline from the packed bitstream
 * (BitLLM sec. 4.3: weights are re-laid out ahead of time so that the kernel's
 * loads need no reordering; Fig. 6 / Fig. 8(b) for the int4 order).
 *   QMM_LAYOUT_TILE16 (any width): the fragment-ordered layout qmm_gemv_tile16
 *     reads.  Rows in tiles of 16 (the last tile padded with zero codes), K in
 *     blocks of 64 codes; unit (T, kb) is 128*bits bytes at byte
 *     (T*(K/64) + kb)*128*bits, and holds run r = (h*8 + g)*4 + t -- codes
 *     16t .. 16t+15 of the block for row 16T + 8h + g, LSB first -- at bytes
 *     [2*bits*r, 2*bits*r + 2*bits).  Each run is the 16-code slice one
 *     tensor-core thread reads, so a warp's reads are contiguous and a CTA's
 *     share of the weights is a few large bulk copies.  Needs K % 64 == 0.
 *     Size: ceil(N/16) * 16 * K * bits / 8 bytes.
 *   QMM_LAYOUT_INTERLEAVE4 (bits == 4): BitLLM's lane-interleaved order: in
 *     every 32-bit word the nibble slots hold codes 0 4 1 5 2 6 3 7 of the
 *     word's eight, so W & 0x0F0F0F0F gives codes 0..3 and
 *     (W >> 4) & 0x0F0F0F0F codes 4..7 as bytes.  Needs K % 8 == 0.
 *     Size: N * K / 2 bytes.  (A format conversion; no kernel here reads it:
 *     the fp16 operand extraction costs one shift and four LOP3s per word from
 *     the canonical stream already.) */
typedef enum { QMM_LAYOUT_TILE16 = 1, QMM_LAYOUT_INTERLEAVE4 = 2 } qmm_layout;

/* Bytes of the `layout` form of an N x K `bits`-bit weight matrix, or 0 if the
 * layout does not take these sizes. */
QMM_API size_t qmm_repack_bytes(int N, int K, int bits, int layout);

/* packed (device) [N][K*bits/8] canonical bitstream -> out (device,
 * qmm_repack_bytes(N, K, bits, layout) bytes, fully overwritten) in `layout`.
 * Byte-exact; an offline step like qmm_pack.  Errors: QMM_ERR_BITS,
 * QMM_ERR_SHAPE (sizes the layout does not take), QMM_ERR_NULL,
 * QMM_ERR_DEVICE, QMM_ERR_CUDA. */
QMM_API qmm_status qmm_repack(const uint8_t *packed, uint8_t *out, int N, int K, int bits, int layout,
                              cudaStream_t stream);

/* qmm_gemv on weights in the QMM_LAYOUT_TILE16 layout (`tiled`, 16-byte
 * aligned; everything else as for qmm_gemv).  Served by the decode kernel
 * only: shapes it does not take (M > 16, G = 32, K not a multiple of 8
 * groups, activations too large for shared memory) return
 * QMM_ERR_UNSUPPORTED.  Results equal qmm_gemv's on the canonical stream up
 * to the order of the fp32 sums. */
QMM_API qmm_status qmm_gemv_tile16(const void *x, qmm_dtype x_dtype, const uint8_t *tiled, int bits,
                                   int group, const void *scales, const uint8_t *zeros, int zero_const,
                                   void *y, qmm_dtype y_dtype, int M, int N, int K, cudaStream_t stream);

/* Signed b-bit weights.  Flips, in place, the top bit of every b-bit code of
 * a packed stream [N][K*bits/8] (two's complement <-> offset binary).  A
 * stream of signed codes c (w = c * s, the signed integer types among the
 * Tilus review's arbitrary low-precision types) becomes one of unsigned codes
 * u = c xor 2^(b-1) with c = u - 2^(b-1), so qmm_gemv / qmm_gemm with
 * zero_const = 2^(b-1) compute the signed matmul exactly.  An offline step
 * like qmm_pack; applying it twice restores the stream.
 *   packed (device) uint8 [N][K*bits/8], modified in place.
 * Errors: QMM_ERR_BITS, QMM_ERR_SHAPE (K*bits % 8), QMM_ERR_NULL,
 * QMM_ERR_DEVICE, QMM_ERR_CUDA. */
QMM_API qmm_status qmm_flip_sign(uint8_t *packed, int N, int K, int bits, cudaStream_t stream);

/* Integer-native W8A8: the qmm_w4a8 contract with signed 8-bit weights, the
 * other integer precision BitLLM evaluates (Experiment Setup: 8-bit weights and
 * activations, group-wise scaling, group 32).
 *   w8   (device) int8 [N][K] (two's complement; the 8-bit bitstream), 16-byte
 *        aligned.  Everything else as for qmm_w4a8:
 *   acc[m][n][g] = sum_{k in g} xq[m][k] * w8[n][k]   (exact int32)
 *   y[m][n]      = sa[m] * sum_g ws[n][g] * acc[m][n][g]   (fp32 -> fp16 RNE)
 * 1 <= M <= 64, G in {32, 64, 128}.  Errors as for qmm_w4a8.  The kernels
 * and their conditions are qmm_w4a8's (|acc| <= 128 * 128 * G stays exact),
 * except that the tcgen05 kernel starts at M = 2 where the decode kernel does
 * not apply. */
QMM_API qmm_status qmm_w8a8(const int8_t *xq, const void *sa, const int8_t *w8, const void *ws,
                            int group, void *y, int32_t *acc_out, int M, int N, int K,
                            cudaStream_t stream);

/* Per-token int8 quantization of fp16 activations, the step before qmm_w4a8
 * (BitLLM sec. 2.2, Eq. (1): q = clip(round(x / s) + z, q_min, q_max), with
 * the int8 range of Fig. 2(a)).  Reading of the pages (which do not fix how s
 * is chosen): symmetric per token, z = 0,
 *   sa[m]    = fp16( max_k |x[m][k]| / 127 )  -- IEEE single-precision
 *              division, then rounded to the nearest fp16 (ties to even);
 *   xq[m][k] = clip( round( x[m][k] / sa[m] ), -128, 127 )  -- IEEE
 *              single-precision division, rounded to the nearest integer
 *              (ties to even); xq = 0 for a token with sa[m] == 0.
 * The result is exact and reproducible: every integer is decided by the same
 * IEEE operations.  x must be finite.
 *   x    (device) fp16 [M][K], 16-byte aligned.
 *   xq   (device) int8 [M][K], 16-byte aligned, fully overwritten.
 *   sa   (device) fp16 [M], 2-byte aligned, fully overwritten (all 0 if K == 0).
 *   K % 8 == 0.  One CTA per token; like the matmul calls it launches with
 *   programmatic dependent launch and reads x only after waiting for the
 *   preceding kernel on the stream.
 * Errors: QMM_ERR_SHAPE (M or K negative, K % 8), QMM_ERR_NULL, QMM_ERR_ALIGN,
 * QMM_ERR_DEVICE, QMM_ERR_CUDA; nothing is launched on an argument error. */
QMM_API qmm_status qmm_quantize_act(const void *x, int8_t *xq, void *sa, int M, int K,
                                    cudaStream_t stream);

/* Synchronizes `stream`, then returns and clears the first device-side error
 * recorded by any qmm kernel on the current device (QMM_OK if none).  A
 * pending asynchronous CUDA error is reported as QMM_ERR_CUDA. */
QMM_API qmm_status qmm_device_status(cudaStream_t stream);

/* Watchdog self-test (no counterpart in the pages; it exists to test failure
 * detection without a GPU fault).  Launches one warp on `stream` that waits on
 * a shared-memory mbarrier no thread ever arrives at, through the same bounded
 * wait every qmm kernel uses: after about a second the wait gives up, records
 * QMM_ERR_TIMEOUT in the device status word and the kernel returns normally.
 * Returns QMM_OK if the launch succeeded; the following qmm_device_status()
 * then reports QMM_ERR_TIMEOUT.  Touches no caller memory. */
QMM_API qmm_status qmm_watchdog_selftest(cudaStream_t stream);

/* Static, NUL-terminated description of a status code. */
QMM_API const char *qmm_status_string(qmm_status status);

/* ABI version of this header (increases on incompatible change). */
QMM_API int qmm_abi_version(void);

#define QMM_ABI_VERSION 1

#ifdef __cplusplus
}
#endif
#endif /* QMM_H_ */
