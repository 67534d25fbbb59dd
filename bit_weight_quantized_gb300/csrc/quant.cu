// quant.cu -- per-token int8 quantization of fp16 activations, the step before
// the integer-native W4A8 matmul (BitLLM sec. 2.2, Eq. (1):
// q = clip(round(x / s) + z, q_min, q_max), with the int8 range of Fig. 2(a)).
//
// Symmetric per token (z = 0):
//   sa[m]    = fp16( max_k |x[m][k]| / 127 )          single-precision IEEE division,
//                                                     then round to nearest even
//   xq[m][k] = clip( rint( x[m][k] / sa[m] ), -128, 127 )   single-precision IEEE
//                                                     division, ties to even; 0 if sa[m] == 0
//
// The quotients that decide the integers are IEEE single-precision divisions
// (__fdiv_rn), so the result is reproducible bit for bit on any IEEE machine.
// One CTA per token: a max-|x| reduction over the row (a few 16-byte loads per
// thread, so the load latency is paid about once), then one pass that
// quantizes.  The second read of the row hits L1/L2.  One warp per token, with
// 16 dependent load rounds per lane at K = 4096, was three times slower.
// HBM-bound: 2 K bytes in, K + 2 bytes out per token.
#include <cuda_fp16.h>

#include "gemv.h"

namespace qmm {

namespace {

constexpr int kQuantThreads = 256;

__device__ __forceinline__ float half_bits_to_float(uint32_t h)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

__device__ __forceinline__ uint32_t quant8(uint32_t h, float s)
{
    int q = 0;
    if (s > 0.f)
        q = max(-128, min(127, __float2int_rn(__fdiv_rn(half_bits_to_float(h), s))));
    return static_cast<uint32_t>(q) & 0xFFu;
}

__global__ void __launch_bounds__(kQuantThreads)
quantize_act_kernel(const uint16_t *__restrict__ x, int8_t *__restrict__ xq, uint16_t *__restrict__ sa, int K)
{
    __shared__ float warp_max[kQuantThreads / 32];
    if (threadIdx.x == 0)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // x may be the output of the preceding kernel on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const long long row = static_cast<long long>(blockIdx.x) * K;
    const uint4 *xv = reinterpret_cast<const uint4 *>(x + row);
    const int nv = K / 8;

    float amax = 0.f;
    for (int v = threadIdx.x; v < nv; v += kQuantThreads) {
        const uint4 q = xv[v];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            amax = fmaxf(amax, fabsf(half_bits_to_float(w[i] & 0xFFFFu)));
            amax = fmaxf(amax, fabsf(half_bits_to_float(w[i] >> 16)));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if ((threadIdx.x & 31) == 0)
        warp_max[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < kQuantThreads / 32; ++i)
        amax = fmaxf(amax, warp_max[i]);

    const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.f));
    const float s = __half2float(s16);
    if (threadIdx.x == 0)
        sa[blockIdx.x] = __half_as_ushort(s16);

    // the second read of the row hits L1 / L2
    uint2 *qv = reinterpret_cast<uint2 *>(xq + row);
    for (int v = threadIdx.x; v < nv; v += kQuantThreads) {
        const uint4 q = xv[v];
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        uint32_t b[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            b[i] = quant8(w[i] & 0xFFFFu, s) | (quant8(w[i] >> 16, s) << 8);
        qv[v] = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
    }
}

}  // namespace

cudaError_t launch_quantize_act(const uint16_t *x, int8_t *xq, uint16_t *sa, int M, int K,
                                cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(M);
    cfg.blockDim = dim3(kQuantThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_act_kernel, x, xq, sa, K);
}

}  // namespace qmm
