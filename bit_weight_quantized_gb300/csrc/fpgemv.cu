// fpgemv.cu -- decode matmul with float weight codes (the float3-float8 types
// of the Tilus review's arbitrary low-precision types), 1 <= M <= 16, fp16
// activations and outputs.
//
// A b-bit code holds 1 sign bit, e exponent bits and m mantissa bits (top to
// bottom, b = 1 + e + m), bias 2^(e-1) - 1, every encoding finite:
//   E > 0: (-1)^s 2^(E - bias) (1 + M / 2^m),   E = 0: (-1)^s 2^(1 - bias) M / 2^m,
// and w = value * s[n][k/G].  Placing the code's exponent and mantissa bits in
// the exponent and top mantissa fields of an fp32 word gives exactly
// value * 2^(bias - 127) for normal and subnormal codes alike; one multiply by
// 2^(127 - bias) (exact, a power of two) restores the value, so every product
// with an fp16 activation is exact in fp32 and only the sums round.
//
// One warp per output column; lane l takes the 32-code runs l, l + 32, ... of
// the column's stream (a run is b whole 32-bit words, so the warp's loads are
// contiguous), multiplies the run by the tokens' activations, applies the
// run's group scale and finally the warp reduces in a fixed order.  Before
// waiting for the preceding kernel each lane prefetches its runs into L2 (the
// weights are not that kernel's output).  Compute-light per byte: FFMA per
// code and token, no tensor cores (M <= 16 rows of x).
#include <cuda_fp16.h>

#include "common.cuh"
#include "gemv.h"

namespace qmm {

namespace {

constexpr int kFpThreads = 256;
constexpr int kFpMaxM = 16;

template <int B>
__global__ void __launch_bounds__(kFpThreads)
gemv_fp_kernel(const uint16_t *__restrict__ x, const uint32_t *__restrict__ packed,
               const uint16_t *__restrict__ scales, uint16_t *__restrict__ y, int M, int N, int K,
               int group_log2, int mbits, float unbias)
{
    if (threadIdx.x == 0)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int n = blockIdx.x * (kFpThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int nruns = K / 32;
    const int ng = K >> group_log2;
    const uint32_t *row = packed + static_cast<long long>(min(n, N - 1)) * nruns * B;
    // the weights are not written by the preceding kernel: pull this lane's runs
    // into L2 while it may still be running
    for (int run = lane; run < nruns; run += 32)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row + run * B));
    // x may be the output of the preceding kernel on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (n >= N)
        return;
    const uint32_t mag_mask = (1u << (B - 1)) - 1u;
    const int mshift = 23 - mbits;

    float tot[kFpMaxM];
#pragma unroll
    for (int m = 0; m < kFpMaxM; ++m)
        tot[m] = 0.f;

#pragma unroll 1
    for (int run = lane; run < nruns; run += 32) {
        uint32_t w[B + 1];
#pragma unroll
        for (int i = 0; i < B; ++i)
            w[i] = row[run * B + i];
        w[B] = 0u;
        float wv[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int bit = i * B;   // compile-time: the word and the shift of code i
            const uint32_t code = (__funnelshift_r(w[bit >> 5], w[(bit >> 5) + 1], bit & 31)) & ((1u << B) - 1u);
            const uint32_t f = ((code >> (B - 1)) << 31) | ((code & mag_mask) << mshift);
            wv[i] = __uint_as_float(f) * unbias;
        }
        const float s = __half2float(__ushort_as_half(scales[static_cast<long long>(n) * ng + ((run * 32) >> group_log2)]));
#pragma unroll
        for (int m = 0; m < kFpMaxM; ++m) {
            if (m < M) {
                const uint4 *xr = reinterpret_cast<const uint4 *>(x + static_cast<long long>(m) * K + run * 32);
                float part = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 v = xr[c];
                    const uint32_t h[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        part = fmaf(wv[8 * c + 2 * j], __half2float(__ushort_as_half(static_cast<unsigned short>(h[j] & 0xFFFFu))), part);
                        part = fmaf(wv[8 * c + 2 * j + 1], __half2float(__ushort_as_half(static_cast<unsigned short>(h[j] >> 16))), part);
                    }
                }
                tot[m] = fmaf(s, part, tot[m]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < kFpMaxM; ++m) {
        if (m < M) {
            float v = tot[m];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0)
                y[static_cast<long long>(m) * N + n] = __half_as_ushort(__float2half_rn(v));
        }
    }
}

template <int B>
cudaError_t launch_fp(const uint16_t *x, const uint8_t *packed, const uint16_t *scales, uint16_t *y,
                      int M, int N, int K, int group_log2, int mbits, float unbias, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((N + kFpThreads / 32 - 1) / (kFpThreads / 32));
    cfg.blockDim = dim3(kFpThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemv_fp_kernel<B>, x, reinterpret_cast<const uint32_t *>(packed), scales,
                              y, M, N, K, group_log2, mbits, unbias);
}

}  // namespace

cudaError_t launch_gemv_fp(const uint16_t *x, const uint8_t *packed, int ebits, int mbits, int group,
                           const uint16_t *scales, uint16_t *y, int M, int N, int K, cudaStream_t stream)
{
    const int bits = 1 + ebits + mbits;
    const int group_log2 = group == 32 ? 5 : group == 64 ? 6 : 7;
    const int bias = (1 << (ebits - 1)) - 1;
    const float unbias = ldexpf(1.f, 127 - bias);   // exact: a power of two within fp32's range
    switch (bits) {
    case 2: return launch_fp<2>(x, packed, scales, y, M, N, K, group_log2, mbits, unbias, stream);
    case 3: return launch_fp<3>(x, packed, scales, y, M, N, K, group_log2, mbits, unbias, stream);
    case 4: return launch_fp<4>(x, packed, scales, y, M, N, K, group_log2, mbits, unbias, stream);
    case 5: return launch_fp<5>(x, packed, scales, y, M, N, K, group_log2, mbits, unbias, stream);
    case 6: return launch_fp<6>(x, packed, scales, y, M, N, K, group_log2, mbits, unbias, stream);
    case 7: return launch_fp<7>(x, packed, scales, y, M, N, K, group_log2, mbits, unbias, stream);
    case 8: return launch_fp<8>(x, packed, scales, y, M, N, K, group_log2, mbits, unbias, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
