// extract.cuh -- turning a run of b-bit codes into fp16 MMA operands with the
// generated extraction plans (unpack_plans.h): one LOP3 per pair of codes from
// a 32-bit window of the run (a word, a funnel shift or a byte permute), with
// exponent bits per half chosen so that each half reads exactly 2^E + q
// (BitLLM sec. 4.3: codes become numbers through bit operations, not
// conversions).  Shared by the skinny and the decode kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "unpack_plans.h"

namespace qmm {

template <int B, int R, int NW>
__device__ __forceinline__ uint32_t plan_window(const uint32_t (&w)[NW], int v)
{
    using P = UnpackPlan<B, R>;
    if (P::kind(v) == 1)
        return prmt(w[P::w0(v)], w[P::w1(v)], P::sel(v));
    const int o = P::off(v);
    if (o < 0)
        return w[0] << (-o);
    const int i = o >> 5, s = o & 31;
    if (s == 0)
        return w[i];
    if (i + 1 < NW)
        return __funnelshift_r(w[i], w[i + 1], s);
    return w[i] >> s;
}

__host__ __device__ constexpr uint32_t pow2_half_bits(int e)
{
    return static_cast<uint32_t>(e + 15) << 10;  // fp16 bits of 2^e
}

__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t mask, uint32_t bits)
{
    // (a & mask) ^ bits
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(mask), "r"(bits));
    return d;
}

// a[i] = fp16 pair of plan pair i.  With SUB the pair is (q_lo, q_hi), exact
// small integers; without it (2^E_lo + q_lo, 2^E_hi + q_hi), also exact, and
// the caller removes sum_k 2^E_k x_k from the dot product instead (one
// instruction per pair fewer on the integer/half pipe).  With FLIP8 each field's
// top bit is flipped first (signed int4 -> c xor 8, signed int8 -> c xor 128).
template <int B, int R, bool FLIP8, bool SUB>
__device__ __forceinline__ void extract_run(const uint32_t (&w)[(R * B + 31) / 32],
                                            uint32_t (&a)[R / 2])
{
    constexpr int NW = (R * B + 31) / 32;
    if constexpr (B == 8) {
#pragma unroll
        for (int i = 0; i < R / 2; ++i) {
            const uint32_t wb = FLIP8 ? (w[i >> 1] ^ 0x80808080u) : w[i >> 1];   // int8 -> c xor 128
            const uint32_t v = prmt(wb, 0x64646464u, (i & 1) ? 0x4342u : 0x4140u);
            a[i] = SUB ? hsub2(v, 0x64006400u) : v;
        }
    } else {
        using P = UnpackPlan<B, R>;
        uint32_t win[P::kWindows];
#pragma unroll
        for (int v = 0; v < P::kWindows; ++v)
            win[v] = plan_window<B, R, NW>(w, v);
#pragma unroll
        for (int i = 0; i < R / 2; ++i) {
            uint32_t v;
            if constexpr (FLIP8)   // xor the top bit of each of the two fields
                v = lop3_and_xor(win[P::win(i)], P::mask(i),
                                 P::magic(i) | (P::mask(i) & ~(P::mask(i) >> 1)));
            else
                v = lop3_and_or(win[P::win(i)], P::mask(i), P::magic(i));
            a[i] = SUB ? hsub2(v, pow2_half_bits(P::elo(i)) | (pow2_half_bits(P::ehi(i)) << 16)) : v;
        }
    }
}

// The exponent E of code c (0 <= c < R) of a run: without SUB its fp16 value
// is 2^E + q.
template <int B, int R>
__host__ __device__ constexpr int exp_of_code(int c)
{
    if constexpr (B == 8) {
        return 10;   // 0x64 exponent byte: 1024 + code
    } else {
        using P = UnpackPlan<B, R>;
        for (int i = 0; i < R / 2; ++i) {
            if (P::lo(i) == c)
                return P::elo(i);
            if (P::hi(i) == c)
                return P::ehi(i);
        }
        return -100;   // not reached: every code is in a pair
    }
}

// Code of the run that feeds slot s = 4*j + e of the activation fragments.
template <int B, int R>
__device__ __forceinline__ constexpr int code_of_slot(int s)
{
    if constexpr (B == 8) {
        return s;  // pairs are (2i, 2i+1): slot order is code order
    } else {
        using P = UnpackPlan<B, R>;
        const int i = 2 * (s >> 2) + ((s >> 1) & 1);
        return (s & 1) ? P::hi(i) : P::lo(i);
    }
}

}  // namespace qmm
