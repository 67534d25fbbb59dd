// decode.cu -- the decode matmul without activation staging, for 1 <= M <= 8,
// groups of 64 or 128 and at most 32 output columns per CTA (the decode shapes).
//
//   y[m][n] = sum_g s[n][g] * ( sum_{k in g} (2^E + q[n][k]) x[m][k]  -  (2^E + z) X[m][g] ),
//   X[m][g] = sum_{k in g} x[m][k]
//
// which is sum_k x[m][k] s (q - z) (BitLLM Eq. (5)): every code enters the
// tensor core as the fp16 number 2^E + q, made by bit operations (BitLLM sec.
// 4.3), and the 2^E X term is removed per group in fp32.  For b = 4 and 8 a
// byte permute puts the code at the bottom of the mantissa under the exponent
// of 1024 (E = 10); for the other widths a shift puts it at the top, E = b, so
// that the offset is no larger than the codes and cancels least.
//
// Work split.  CTA c owns at most 32 consecutive columns (two 16-row MMA
// tiles); warp w owns K/8 codes of all of them, in blocks of 64.  In a block,
// quad thread t owns codes [16t, 16t + 16) of each of its rows: b/2 words,
// rounded up, read straight from global memory (one 8-byte load at b = 4, one
// 16-byte load at b = 8).  The MMA's k order is permuted to match: the 16
// codes of MMA step s of thread t are its codes 4s .. 4s + 3, so the B fragment
// is x[16t + 4s .. 16t + 4s + 3] of the block, one 32-byte load per thread and
// block.  No activation staging, no shared memory before the final reduction,
// one CTA barrier.  Loads run one block ahead in registers; before waiting for
// the preceding kernel the weights are prefetched into L2 (the weights are not
// that kernel's output).
#include "common.cuh"
#include "decode.h"

namespace qmm {

namespace {

constexpr int kDecThreads = 256;
constexpr int kDecRows = 32;   // columns per CTA, at most
constexpr int kDecMaxM = 8;

// Words a thread reads per row and block: its 16 codes start at bit 0 or 16
// of the first word (16 b t bits into the block), so (b + 1) / 2 words cover them.
template <int B>
__host__ __device__ constexpr int dec_words() { return (B + 1) / 2; }

// The exponent E of the fp16 operand 2^E + q.
template <int B>
__host__ __device__ constexpr int dec_exp() { return (B == 4 || B == 8) ? 10 : B; }

// fp16 pair (2^E + q_c, 2^E + q_{c+1}) of codes c, c + 1 (c even) of the
// thread's 16 codes, from its window (code 0 at bit 0 of win[0]).
template <int B>
__device__ __forceinline__ uint32_t dec_pair(const uint32_t (&win)[dec_words<B>() + 1], int c)
{
    if constexpr (B == 8) {   // one byte per code, under the exponent byte 0x64
        return prmt(win[c >> 2], 0x64646464u, (c & 2) ? 0x4342u : 0x4140u);
    } else if constexpr (B == 4) {   // codes c, c + 1 are the two nibbles of one byte
        const uint32_t w = win[c >> 3];
        const uint32_t byte = (c & 7) >> 1;
        return lop3_and_or(prmt(w, w >> 4, byte | ((4 + byte) << 8)), 0x000F000Fu, 0x64006400u);
    } else {
        // u: code c at bits [10 - B, 10), code c + 1 above it
        const int sh = c * B - (10 - B);
        const uint32_t u = sh < 0 ? win[0] << (-sh)
                                  : __funnelshift_r(win[sh >> 5], win[(sh >> 5) + 1], sh & 31);
        constexpr uint32_t mask = ((1u << B) - 1u) << (10 - B);
        constexpr uint32_t magic = static_cast<uint32_t>(B + 15) << 10;   // fp16 bits of 2^B
        const uint32_t lo = lop3_and_or(u, mask, magic | (magic << 16));
        return lop3_and_or(u << (16 - B), mask << 16, lo);
    }
}

// The thread's words of one row and block.  At b = 4 they are two words at an
// even word index, at b = 8 four at a multiple of four (K is a multiple of 512
// and the packed base 16-byte aligned), so one vector load reads them.
template <int B>
__device__ __forceinline__ void load_words(uint32_t (&w)[dec_words<B>()], const uint32_t *src)
{
    if constexpr (B == 8) {
        const uint4 v = *reinterpret_cast<const uint4 *>(src);
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    } else if constexpr (B == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(src);
        w[0] = v.x;
        w[1] = v.y;
    } else {
#pragma unroll
        for (int k = 0; k < dec_words<B>(); ++k)
            w[k] = src[k];
    }
}

template <int B>
__global__ void __launch_bounds__(kDecThreads, 2)
decode_kernel(const DecodeParams p)
{
    constexpr int NW = dec_words<B>();
    constexpr float kPow = static_cast<float>(1 << dec_exp<B>());
    __shared__ float red[kDecThreads / 32][kDecRows][kDecMaxM];
    if (threadIdx.x == 0)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int cta = blockIdx.x;
    const int r0 = cta * p.rows_base + min(cta, p.rows_rem);
    const int nrows = p.rows_base + (cta < p.rows_rem ? 1 : 0);
    const int K = p.K;
    const long long row_words = static_cast<long long>(K) * B / 32;
    const int ng = K >> p.group_log2;
    const int kw = K / 8;                  // codes of this warp
    const int k0w = warp * kw;
    const int nblk = kw / 64;
    const int group_end = (1 << (p.group_log2 - 6)) - 1;   // blocks per group - 1 (a power of two)
    const int o = (B & 1) ? 16 * (t & 1) : 0;   // bit offset of the thread's first code in its first word
    // this thread's rows (tile i, half h: row 16 i + 8 h + g; padding rows read row nrows - 1)
    const uint32_t *rowp[2][2];
    int rowi[2][2];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int lr = min(16 * i + 8 * h + g, nrows - 1);
            rowi[i][h] = r0 + lr;
            // first word of the thread's codes in block 0 of this warp
            rowp[i][h] = reinterpret_cast<const uint32_t *>(p.packed) + (r0 + lr) * row_words +
                         (static_cast<long long>(k0w) * B + 16 * B * t) / 32;
        }
    if (t == 0) {
        // one prefetch per 128-byte line of this warp's part of each row
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                for (int wd = 0; wd < kw * B / 32; wd += 32)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(rowp[i][h] + wd));
    }
    // x may be the output of the preceding kernel on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int m = min(g, p.M - 1);         // the token of this lane's B column
    const uint16_t *xr = p.x + static_cast<long long>(m) * K + k0w + 16 * t;
    float tot[2][4] = {};
    float acc[2][4] = {};
    float xsum = 0.f;

    uint32_t nw[2][2][NW];
    uint4 nxa, nxb;
    nxa = *reinterpret_cast<const uint4 *>(xr);
    nxb = *reinterpret_cast<const uint4 *>(xr + 8);
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h)
            load_words<B>(nw[i][h], rowp[i][h]);

#pragma unroll 1
    for (int j = 0; j < nblk; ++j) {
        uint32_t win[2][2][NW + 1];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                // shift the window so that the thread's code 0 sits at bit 0 (even widths: it does)
#pragma unroll
                for (int k = 0; k < NW; ++k)
                    win[i][h][k] = (B & 1) ? __funnelshift_r(nw[i][h][k], k + 1 < NW ? nw[i][h][k + 1] : 0u, o)
                                           : nw[i][h][k];
                win[i][h][NW] = 0u;
            }
        const uint4 xa = nxa, xb = nxb;
        if (j + 1 < nblk) {
            nxa = *reinterpret_cast<const uint4 *>(xr + 64 * (j + 1));
            nxb = *reinterpret_cast<const uint4 *>(xr + 64 * (j + 1) + 8);
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    load_words<B>(nw[i][h], rowp[i][h] + (j + 1) * 2 * B);
        }
        const uint32_t xw[8] = {xa.x, xa.y, xa.z, xa.w, xb.x, xb.y, xb.z, xb.w};
#pragma unroll
        for (int e = 0; e < 8; ++e)
            xsum += f16_bits_to_f32(static_cast<uint16_t>(xw[e])) + f16_bits_to_f32(static_cast<uint16_t>(xw[e] >> 16));
#pragma unroll
        for (int s = 0; s < 4; ++s) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
                mma_f16_16816(acc[i], dec_pair<B>(win[i][0], 4 * s), dec_pair<B>(win[i][1], 4 * s),
                              dec_pair<B>(win[i][0], 4 * s + 2), dec_pair<B>(win[i][1], 4 * s + 2),
                              xw[2 * s], xw[2 * s + 1]);
        }
        if (((j + 1) & group_end) == 0) {   // the end of a group
            // X_g of the quad's token: the sum of its four threads' 16-code slices of x
            float X = xsum;
            X += __shfl_xor_sync(0xffffffffu, X, 1);
            X += __shfl_xor_sync(0xffffffffu, X, 2);
            // the accumulator columns are tokens 2t and 2t + 1 (lanes 4 (2t), 4 (2t + 1))
            const float X0 = __shfl_sync(0xffffffffu, X, 8 * t);
            const float X1 = __shfl_sync(0xffffffffu, X, 8 * t + 4);
            const int gidx = (k0w + 64 * j) >> p.group_log2;
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const long long so = static_cast<long long>(rowi[i][h]) * ng + gidx;
                    const float sc = f16_bits_to_f32(p.scales[so]);
                    const float off = kPow + static_cast<float>(p.zeros ? p.zeros[so] : p.zero_const);
                    tot[i][2 * h] = fmaf(sc, fmaf(-off, X0, acc[i][2 * h]), tot[i][2 * h]);
                    tot[i][2 * h + 1] = fmaf(sc, fmaf(-off, X1, acc[i][2 * h + 1]), tot[i][2 * h + 1]);
                    acc[i][2 * h] = acc[i][2 * h + 1] = 0.f;
                }
            xsum = 0.f;
        }
    }

    // cross-warp reduction in a fixed order, then the store
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int tok = 2 * t + c;
                if (tok < p.M)
                    red[warp][16 * i + 8 * h + g][tok] = tot[i][2 * h + c];
            }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nrows * p.M; idx += kDecThreads) {
        const int row = idx / p.M, tok = idx - row * p.M;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kDecThreads / 32; ++w)
            v += red[w][row][tok];
        const long long out = static_cast<long long>(tok) * p.N + r0 + row;
        reinterpret_cast<uint16_t *>(p.y)[out] = p.y_bf16 ? f32_to_bf16_bits(v) : f32_to_f16_bits(v);
    }
}

template <int B>
cudaError_t launch_decode_b(const DecodeParams &p, int grid, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel<B>, p);
}

}  // namespace

bool decode_supports(int M, int N, int K, int group, int num_sms)
{
    if (M < 1 || M > kDecMaxM || (group != 64 && group != 128) || K < 8 * group || K % (8 * group))
        return false;
    const int grid = N < num_sms ? N : num_sms;
    return (N + grid - 1) / grid <= kDecRows;
}

cudaError_t launch_decode(DecodeParams p, int bits, int num_sms, cudaStream_t stream)
{
    const int grid = p.N < num_sms ? p.N : num_sms;
    p.rows_base = p.N / grid;
    p.rows_rem = p.N % grid;
    switch (bits) {
    case 1: return launch_decode_b<1>(p, grid, stream);
    case 2: return launch_decode_b<2>(p, grid, stream);
    case 3: return launch_decode_b<3>(p, grid, stream);
    case 4: return launch_decode_b<4>(p, grid, stream);
    case 5: return launch_decode_b<5>(p, grid, stream);
    case 6: return launch_decode_b<6>(p, grid, stream);
    case 7: return launch_decode_b<7>(p, grid, stream);
    case 8: return launch_decode_b<8>(p, grid, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace qmm
