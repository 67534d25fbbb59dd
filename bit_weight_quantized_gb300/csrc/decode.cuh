// decode.cuh -- the decode / small-batch matmul for 1 <= M <= 16, groups of 64
// or 128 and K a multiple of 8 groups (BitLLM Eq. (5) on the per-column
// bitstream of the Tilus review's arbitrary-width weight types):
//
//   y[m][n] = sum_g s[n][g] * ( sum_{k in g} (2^E_k + q[n][k]) x[m][k]  -  C[m][g]  -  z[n][g] X[m][g] ),
//   X[m][g] = sum_{k in g} x[m][k],   C[m][g] = sum_{k in g} 2^E_k x[m][k]
//
// Codes reach the tensor core as exact fp16 numbers 2^E_k + q: the generated
// extraction plans (extract.cuh) turn each pair of codes into the fp16 pair
// (2^E_lo + q_lo, 2^E_hi + q_hi) with one LOP3 from a 32-bit window (BitLLM sec.
// 4.3: codes become numbers through bit operations, not conversions); E_k
// depends only on the position of code k in its run.  Every product is exact
// in fp32; mma.sync accumulates a group in fp32, and the group's offset C, zero
// and scale are applied in fp32 afterwards.  C and X are summed in fp32 when
// the activations are staged, so no per-code subtraction is needed.  Two
// variants share the kernel: float weight codes (FL: the code's fields placed
// in an fp16 number, no offset), and the exact-integer mode of qmm_w4a8 /
// qmm_w8a8 (IX: int8 activations, signed codes read as offset binary, the
// offset 2^E taken off each operand so that every group sum is an exact
// integer in fp32, y = sa[m] * sum_g s (acc - 2^(b-1) X)).
//
// Staging.  The weights are the one large operand and are never the output of
// the preceding kernel, so every CTA copies its share of them into shared
// memory with 1-D bulk copies (TMA) as soon as it starts, BEFORE it waits for
// the preceding kernel on the stream (programmatic dependent launch).  In a
// stream of calls this streams call i+1's weights from HBM while call i
// computes.  After the wait each warp loads the activations of its K slices
// (one round trip), stores them in shared memory in the order its MMA
// fragments read them, and forms X and C per group.
//
// Work split.  CTA c owns consecutive output columns (rows of the packed
// matrix), taken in row blocks of at most 32 (two 16-row MMA tiles).  A row
// block's K range is cut into segments of 8 groups; one segment of one row
// block fills one slot of a ring in shared memory (one tensor-map copy of the
// slot's rows, or one bulk copy per row where the pitch is too wide for a box;
// rows at a padded pitch that keeps the fragment reads free of bank conflicts).
// Warp w owns group w of every segment, in 64-code blocks.  In a block, quad
// thread t owns the run of codes [16t, 16t + 16) of each of its four rows; the
// plan pairs the run's codes, and the MMA's k order follows the pairing (the
// activations are stored permuted the same way), which relabels k inside one
// MMA and leaves the sum unchanged.  The warps' partial sums meet in shared
// memory and are added in a fixed order.
#pragma once

#include "common.cuh"
#include "decode.h"
#include "extract.cuh"

namespace qmm {

namespace {

constexpr int kRowBlock = 32;   // rows per row block: two 16-row MMA tiles
constexpr int kMaxSlots = 16;

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;

// Words holding a thread's 16-code run of one row and block: the run starts at
// bit 0 or 16 of its first word (16 b t bits into the block).
template <int B>
__host__ __device__ constexpr int run_words() { return (B + 1) / 2; }

// Residue (mod 128 bytes) of a ring slot's row pitch that spreads the eight
// rows of one fragment load over distinct banks: the quad's four threads read
// 8b consecutive bytes of a row, and eight rows meet in one load.
__host__ __device__ constexpr int pitch_residue(int b) { return b == 8 ? 64 : b == 4 ? 32 : 16; }

// The thread's run of one row and block from shared memory, shifted so that
// code 0 sits at bit 0 (odd widths, odd t: the run starts at bit 16).  At b = 4
// the words are 8-byte aligned, at b = 8 16-byte aligned (block offsets are
// multiples of 8b bytes and the slot pitch a multiple of 16), so one vector load
// reads them.
template <int B>
__device__ __forceinline__ void load_run(uint32_t (&w)[run_words<B>()], const uint8_t *src, int o)
{
    constexpr int NW = run_words<B>();
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
        uint32_t r[NW];
#pragma unroll
        for (int k = 0; k < NW; ++k)
            r[k] = reinterpret_cast<const uint32_t *>(src)[k];
#pragma unroll
        for (int k = 0; k < NW; ++k)
            w[k] = (B & 1) ? __funnelshift_r(r[k], k + 1 < NW ? r[k + 1] : 0u, o) : r[k];
    }
}

// Byte-permute selector taking fp16 half c1 of word A (lo) and half c2 of word
// B (hi), c1, c2 in {0, 1}.
__host__ __device__ constexpr uint32_t half_sel(int c1, int c2)
{
    return static_cast<uint32_t>(2 * c1) | static_cast<uint32_t>(2 * c1 + 1) << 4 |
           static_cast<uint32_t>(4 + 2 * c2) << 8 | static_cast<uint32_t>(5 + 2 * c2) << 12;
}

// 16-byte asynchronous copy global -> shared through L2 only.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Issues ring chunk i of this CTA (row block i / nchunk, segments
// [span (i % nchunk), span (i % nchunk + 1))) into its slot, all completing on
// full[slot].  Canonical layout: one bulk copy of span segments per row, rows
// at the slot pitch; or, with the tensor map (p.tma), one box of a slot's rows,
// each row's chunk and the pad up to the pitch (the pad holds the next
// segment's first bytes, or zeros past the row's end, and is never read; rows
// past the CTA's last belong to the next CTA or are zeros, and are not used).
// Fragment-ordered layout (TILE): one bulk copy per 16-row tile of the row
// block, the tile's blocks back to back.  Called by all lanes of warp 0.
template <bool TILE>
__device__ __forceinline__ void issue_chunk(const DecodeParams &p, uint8_t *slots, uint64_t *full, int i,
                                            int r0, int nrows, uint64_t pol, int lane)
{
    const DecodePlan &pl = p.pl;
    const int nchunk = pl.nseg / pl.span;
    const int rb = i / nchunk, c = i - rb * nchunk;
    const int slot = i % pl.slots;
    const int rr = rb * kRowBlock;
    const int cnt = min(kRowBlock, nrows - rr);
    const int bytes = pl.span * pl.seg_bytes;               // one row's share of the chunk
    uint8_t *dst = slots + static_cast<size_t>(slot) * pl.slot_bytes;
    if constexpr (TILE) {
        const int ntiles = (cnt + 15) / 16;
        const int tbytes = 16 * bytes;                      // one tile's share
        if (lane == 0)
            mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(ntiles * tbytes));
        __syncwarp();
        const uint8_t *src = p.packed + static_cast<long long>(r0 + rr) * p.row_bytes + static_cast<long long>(c) * tbytes;
        if (lane < ntiles)
            bulk_load_hint(dst + lane * tbytes, src + lane * 16 * p.row_bytes, static_cast<uint32_t>(tbytes),
                           &full[slot], pol);
    } else if (p.tma && (smem_u32(dst) & 127u) == 0) {   // a tensor copy lands on 128 bytes
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(decode_tma_rows(pl) * pl.pitch));
            tma_load_2d_hint(dst, &p.tmw, &full[slot], c * (bytes >> 3), r0 + rr, pol);
        }
        __syncwarp();
    } else {
        if (lane == 0)
            mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(cnt * bytes));
        __syncwarp();
        const uint8_t *src = p.packed + static_cast<long long>(r0 + rr) * p.row_bytes + static_cast<long long>(c) * bytes;
        for (int r = lane; r < cnt; r += 32)
            bulk_load_hint(dst + r * pl.pitch, src + r * p.row_bytes, static_cast<uint32_t>(bytes), &full[slot], pol);
    }
}

// One warp's 64-code block: the thread's runs of its four rows turned into
// exact code pairs, its activation fragments (already in pair order), and the
// MMAs into the group accumulators.  With two token tiles (NT = 2, one CTA per
// SM) MMAs j = 0, 2 and j = 1, 3 go to separate accumulator sets (summed at
// the fold), which halves the dependent chains; with one (two CTAs per SM, 128
// registers) a single set measured faster.
// Code k of a run whose code 0 sits at bit 0 of w[0], at bit 0 of the result
// (higher bits hold the following codes).
template <int B>
__device__ __forceinline__ uint32_t run_code_at0(const uint32_t (&w)[run_words<B>()], int k)
{
    constexpr int NW = run_words<B>();
    const int bit = B * k, i = bit >> 5, sh = bit & 31;
    if (sh == 0)
        return w[i];
    return i + 1 < NW ? __funnelshift_r(w[i], w[i + 1], sh) : w[i] >> sh;
}

// Float codes (sign, e exponent bits, m mantissa bits; e <= 4) of the 16-code
// run in w, as fp16 pairs in code order (pair q = codes 2q, 2q + 1): the
// exponent and mantissa fields go to the top of the fp16 exponent and mantissa
// fields and the sign to bit 15, which reads exactly the code's value times
// 2^(bias - 15) (normal and subnormal codes alike).  fl = {mask of the e + m low
// bits in both halves, shift of that field, shift of the sign}.
template <int B>
__device__ __forceinline__ void extract_float_run(const uint32_t (&w)[run_words<B>()], uint3 fl, uint32_t (&a)[8])
{
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        uint32_t t;
        if constexpr (B == 4) {   // nibbles 2j, 2j + 1 of word q / 4 to the low nibble of each half
            const uint32_t wq = w[q >> 2];
            const uint32_t j = static_cast<uint32_t>(q & 3);
            t = prmt(wq, wq >> 4, j | ((4u + j) << 8));
        } else if constexpr (B == 8) {   // bytes 2q, 2q + 1 to the low byte of each half
            const uint32_t b0 = static_cast<uint32_t>(2 * (q & 1));
            t = prmt(w[q >> 1], 0u, b0 | (4u << 4) | ((b0 + 1u) << 8) | (4u << 12));
        } else {   // other widths: each code of the pair shifted to bit 0, low halves joined
            t = prmt(run_code_at0<B>(w, 2 * q), run_code_at0<B>(w, 2 * q + 1), 0x5410u);
        }
        uint32_t r;
        asm("lop3.b32 %0, %1, %2, %3, 0xF8;"   // a | (b & c)
            : "=r"(r)
            : "r"((t & fl.x) << fl.y), "r"(t << fl.z), "r"(0x80008000u));
        a[q] = r;
    }
}

// The fp16 bits of the pair (2^E_lo, 2^E_hi) that the integer plans add to the
// codes of pair q of a run (slot order), for the exact-integer mode.
template <int B>
__host__ __device__ constexpr uint32_t offset_pair(int q)
{
    return static_cast<uint32_t>(exp_of_code<B, 16>(code_of_slot<B, 16>(2 * q)) + 15) << 10 |
           static_cast<uint32_t>(exp_of_code<B, 16>(code_of_slot<B, 16>(2 * q + 1)) + 15) << 26;
}

template <int B, int NT, bool FL, bool IX = false>
__device__ __forceinline__ void block_mma(const uint8_t *const (&run0)[2][2], int boff, const uint8_t *xb,
                                          int x_pitch, int m0, int m1, int o, uint3 fl, float (&acc)[2][2][NT][4])
{
    constexpr int NW = run_words<B>();
    uint32_t a[2][2][8];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t w[NW];
            load_run<B>(w, run0[i][h] + boff, o);
            if constexpr (IX) {   // signed codes: two's complement -> offset binary (c xor 2^(b-1))
#pragma unroll
                for (int k = 0; k < NW; ++k)
                    w[k] ^= B == 4 ? 0x88888888u : 0x80808080u;
            }
            if constexpr (FL)
                extract_float_run<B>(w, fl, a[i][h]);
            else
                extract_run<B, 16, false, false>(w, a[i][h]);
            if constexpr (IX) {   // 2^E + u - 2^E: the code u itself, so that every sum stays exact
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    a[i][h][q] = hsub2(a[i][h][q], offset_pair<B>(q));
            }
        }
    uint32_t xw[NT][8];
#pragma unroll
    for (int tt = 0; tt < NT; ++tt) {
        const uint8_t *xt = xb + (tt ? m1 : m0) * x_pitch;
        const uint4 lo = *reinterpret_cast<const uint4 *>(xt);
        const uint4 hi = *reinterpret_cast<const uint4 *>(xt + 16);
        xw[tt][0] = lo.x; xw[tt][1] = lo.y; xw[tt][2] = lo.z; xw[tt][3] = lo.w;
        xw[tt][4] = hi.x; xw[tt][5] = hi.y; xw[tt][6] = hi.z; xw[tt][7] = hi.w;
    }
    // MMA j takes pairs 2j (k = 2t, 2t + 1) and 2j + 1 (k = 2t + 8, 2t + 9)
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int tt = 0; tt < NT; ++tt)
                mma_f16_16816(acc[NT == 2 ? (j & 1) : 0][i][tt], a[i][0][2 * j], a[i][1][2 * j], a[i][0][2 * j + 1],
                              a[i][1][2 * j + 1], xw[tt][2 * j], xw[tt][2 * j + 1]);
}

// Stores one 16-code run of activations (in[8] = its 16 fp16 values in code
// order) in fragment (slot) order: slot s of the run holds x of the run's code
// code_of_slot(s).  Returns the run's sums X = sum x and C = sum 2^E x (E of
// each code's position in the plan; 0 for float codes and the exact-integer
// mode), in fp32.  IX: raw[0] holds 16 int8 activations instead.
template <int B, bool FL, bool IX = false>
__device__ __forceinline__ float2 stage_run(uint8_t *dst, const uint4 (&raw)[2], bool x_bf16)
{
    uint32_t in[8] = {raw[0].x, raw[0].y, raw[0].z, raw[0].w, raw[1].x, raw[1].y, raw[1].z, raw[1].w};
    if constexpr (IX) {
        // 16 int8 activations (raw[0]) as exact fp16 pairs: byte v + 128 under
        // the fp16 exponent byte 0x64 reads 1152 + v; minus 1152 leaves v
        const uint32_t wv[4] = {raw[0].x ^ 0x80808080u, raw[0].y ^ 0x80808080u, raw[0].z ^ 0x80808080u,
                                raw[0].w ^ 0x80808080u};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t b0 = static_cast<uint32_t>(2 * (q & 1));
            in[q] = hsub2(prmt(wv[q >> 1], 0x64646464u, b0 | (4u << 4) | ((b0 + 1u) << 8) | (4u << 12)),
                          0x64806480u);
        }
    } else if (x_bf16) {
        // bf16 activations become fp16: exact for magnitudes in [2^-14, 65504]
        // (8 significant bits fit in 11), rounded to the fp16 subnormal grid below
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            uint32_t h;
            asm("cvt.rn.f16x2.f32 %0, %1, %2;"
                : "=r"(h)
                : "f"(__uint_as_float(in[q] & 0xFFFF0000u)), "f"(__uint_as_float(in[q] << 16)));
            in[q] = h;
        }
    }
    uint32_t out[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        // float codes pair in code order (slot s = code s)
        const int c1 = FL ? 2 * q : code_of_slot<B, 16>(2 * q), c2 = FL ? 2 * q + 1 : code_of_slot<B, 16>(2 * q + 1);
        out[q] = prmt(in[c1 >> 1], in[c2 >> 1], half_sel(c1 & 1, c2 & 1));
    }
    *reinterpret_cast<uint4 *>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
    *reinterpret_cast<uint4 *>(dst + 16) = make_uint4(out[4], out[5], out[6], out[7]);
    float X = 0.f, C = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
        const float v = f16_bits_to_f32(static_cast<uint16_t>(in[c >> 1] >> (16 * (c & 1))));
        X += v;
        if constexpr (!FL && !IX)   // float codes carry no offset, exact-integer operands neither
            C = fmaf(static_cast<float>(1 << exp_of_code<B, 16>(c)), v, C);
    }
    return make_float2(X, C);
}

// The activation staging of more than one round (several tokens or long K),
// kept out of line so that the one-round path of the decode shapes stays compact.
template <int B, int NB, bool FL, bool IX = false>
__device__ __noinline__ void stage_rounds(const DecodeParams &p, uint8_t *xw, float2 *xs, int warp, int lane,
                                          int rounds)
{
    constexpr int kBatch = 4;
    constexpr int jstep = 8 / NB;                       // segments per round
    const DecodePlan &pl = p.pl;
    const int tq = lane & 3, bb = (lane >> 2) & (NB - 1), jl = lane >> (NB == 2 ? 3 : 2);
        int mr = 0, jr = 0;                             // token and first segment of the next round
        for (int r0 = 0; r0 < rounds; r0 += kBatch) {
            uint4 raw[kBatch][2];
            int mq[kBatch], jq[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                mq[q] = mr;
                jq[q] = r0 + q < rounds ? jr + jl : pl.nseg;   // nseg marks an idle lane
                if (jq[q] < pl.nseg && IX) {   // 16 int8 activations
                    const int8_t *src = reinterpret_cast<const int8_t *>(p.x) + static_cast<long long>(mq[q]) * p.K +
                                        jq[q] * pl.kseg + 64 * (warp * NB + bb) + 16 * tq;
                    raw[q][0] = *reinterpret_cast<const uint4 *>(src);
                    raw[q][1] = make_uint4(0u, 0u, 0u, 0u);
                } else if (jq[q] < pl.nseg) {
                    const uint16_t *src = p.x + static_cast<long long>(mq[q]) * p.K + jq[q] * pl.kseg +
                                          64 * (warp * NB + bb) + 16 * tq;
                    raw[q][0] = *reinterpret_cast<const uint4 *>(src);
                    raw[q][1] = *reinterpret_cast<const uint4 *>(src + 8);
                } else {
                    raw[q][0] = raw[q][1] = make_uint4(0u, 0u, 0u, 0u);
                }
                jr += jstep;
                if (jr >= pl.nseg) {
                    jr = 0;
                    ++mr;
                }
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                if (r0 + q >= rounds)
                    break;
                float2 v = make_float2(0.f, 0.f);
                if (jq[q] < pl.nseg)
                    v = stage_run<B, FL, IX>(xw + mq[q] * pl.x_pitch + ((jq[q] * NB + bb) * 64 + 16 * tq) * 2, raw[q],
                                     p.x_bf16 != 0);
#pragma unroll
                for (int off = 1; off < 4 * NB; off <<= 1) {
                    v.x += __shfl_xor_sync(0xffffffffu, v.x, off);
                    v.y += __shfl_xor_sync(0xffffffffu, v.y, off);
                }
                if (jq[q] < pl.nseg && (lane & (4 * NB - 1)) == 0)
                    xs[mq[q] * pl.nseg + jq[q]] = v;   // (X, C) of the token, this warp's group of segment jq
            }
        }
}

// NB = G / 64 blocks per group; warp w owns group w of every 8-group segment.
// TILE: the weights are in the fragment-ordered (tile16) layout.
template <int B, int NT, int NB, bool TILE, bool FL, bool IX = false>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 2 : 1)
decode_kernel(const __grid_constant__ DecodeParams p)
{
    const DecodePlan &pl = p.pl;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *slots = smem;
    uint16_t *sc = reinterpret_cast<uint16_t *>(smem + pl.off_sc);
    uint16_t *zo = reinterpret_cast<uint16_t *>(smem + pl.off_zo);
    float *xsum = reinterpret_cast<float *>(smem + pl.off_xsum);
    float *red = reinterpret_cast<float *>(smem + pl.off_red);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + pl.off_bar);
    uint64_t *empty = full + pl.slots;
    volatile int *fail = reinterpret_cast<volatile int *>(empty + pl.slots);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int cta = blockIdx.x;
    // canonical layout: CTA c owns rows_base + (c < rows_rem) rows; tile16: as many 16-row tiles
    const int u0 = cta * pl.rows_base + min(cta, pl.rows_rem);
    const int nu = pl.rows_base + (cta < pl.rows_rem ? 1 : 0);
    const int r0 = TILE ? 16 * u0 : u0;
    const int nrows = TILE ? min(16 * nu, p.N - r0) : nu;
    const int nrb = (nrows + kRowBlock - 1) / kRowBlock;
    const int nchunk = pl.nseg / pl.span;
    const int total = nrb * nchunk;   // ring chunks of this CTA
    const int ng = p.K >> p.group_log2;

    // warp 0: barriers, then the first ring of weight chunks, before the wait
    uint64_t pol = 0;
    int issued = 0;
    if (warp == 0) {
        if (lane == 0) {
            asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
            for (int s = 0; s < pl.slots; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kWarps);
            }
            *fail = 0;
            fence_barrier_init();
        }
        __syncwarp();
        pol = l2_evict_first_policy();
        issued = min(pl.slots, total);
        for (int i = 0; i < issued; ++i)
            issue_chunk<TILE>(p, slots, full, i, r0, nrows, pol, lane);
    }
    // the CTA's scales and zeros (fp16) into shared memory, transposed to
    // [group][row] so that the eight rows of a fragment meet consecutive halves
    if (NT == 2 && p.vec_sz) {
        // eight groups of a row per step: one 16-byte load of scales and one
        // 8-byte load of zeros; (row, c) advance by a fixed stride without
        // divisions (the one-token-tile variant keeps the smaller scalar loop:
        // there the staging overlaps the preceding call, and the code size shows)
        const int vpr = ng >> 3;                        // 8-group vectors per row
        const int total = nrows * vpr;
        const int dq = kThreads / vpr, dr = kThreads - dq * vpr;
        int row = threadIdx.x / vpr, c = threadIdx.x - row * vpr;
        const uint4 *gs = reinterpret_cast<const uint4 *>(p.scales + static_cast<long long>(r0) * ng);
        const uint2 *gz = reinterpret_cast<const uint2 *>(p.zeros + static_cast<long long>(r0) * ng);
        for (int v = threadIdx.x; v < total; v += kThreads) {
            const uint4 sv = gs[v];
            const uint32_t sw[4] = {sv.x, sv.y, sv.z, sv.w};
            uint16_t *sd = sc + 8 * c * nrows + row;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                sd[e * nrows] = static_cast<uint16_t>(sw[e >> 1] >> (16 * (e & 1)));
            if (p.zeros) {
                const uint2 zv = gz[v];
                uint16_t *zd = zo + 8 * c * nrows + row;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    zd[e * nrows] = f32_to_f16_bits(static_cast<float>(((e < 4 ? zv.x : zv.y) >> (8 * (e & 3))) & 0xFFu));
            }
            row += dq;
            c += dr;
            if (c >= vpr) {
                c -= vpr;
                ++row;
            }
        }
    } else {
        const uint16_t *gs = p.scales + static_cast<long long>(r0) * ng;
        for (int e = threadIdx.x; e < nrows * ng; e += kThreads) {
            const int row = e / ng, gi = e - row * ng;
            sc[gi * nrows + row] = gs[e];
        }
        if (p.zeros) {
            const uint8_t *gz = p.zeros + static_cast<long long>(r0) * ng;
            for (int e = threadIdx.x; e < nrows * ng; e += kThreads) {
                const int row = e / ng, gi = e - row * ng;
                zo[gi * nrows + row] = f32_to_f16_bits(static_cast<float>(gz[e]));
            }
        }
    }
    __syncthreads();
    // x may be the output of the preceding kernel on the stream
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // this warp's group of every segment, for every token, in fragment order:
    // run (m, j, block bb, thread tq) holds x[m][j kseg + 64 (warp NB + bb) + 16 tq + (0 .. 16)];
    // the 4 NB runs of one (m, j) are summed into X[m][j]
    uint8_t *xw = smem + pl.off_x + warp * (p.M * pl.x_pitch);
    float2 *xs = reinterpret_cast<float2 *>(xsum) + warp * p.M * pl.nseg;
    {
        // A round is 32 runs, one per lane: lane l takes run tq = l & 3 of block
        // bb = (l >> 2) % NB of segment jb + (l >> 2) / NB of one token; the
        // 4 NB lanes of one (token, segment) meet in the shuffle sum.  Rounds go
        // token by token, segment block by segment block, and kBatch rounds'
        // loads are issued before any is used.
        constexpr int jstep = 8 / NB;                   // segments per round
        const int tq = lane & 3, bb = (lane >> 2) & (NB - 1), jl = lane >> (NB == 2 ? 3 : 2);
        const int rounds = p.M * ((pl.nseg + jstep - 1) / jstep);
        if (rounds == 1) {   // one round (a single token and at most jstep segments)
            float2 v = make_float2(0.f, 0.f);
            if (jl < pl.nseg) {
                uint4 raw[2];
                if constexpr (IX) {   // 16 int8 activations
                    raw[0] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const int8_t *>(p.x) + jl * pl.kseg +
                                                              64 * (warp * NB + bb) + 16 * tq);
                    raw[1] = make_uint4(0u, 0u, 0u, 0u);
                } else {
                    const uint16_t *src = p.x + jl * pl.kseg + 64 * (warp * NB + bb) + 16 * tq;
                    raw[0] = *reinterpret_cast<const uint4 *>(src);
                    raw[1] = *reinterpret_cast<const uint4 *>(src + 8);
                }
                v = stage_run<B, FL, IX>(xw + ((jl * NB + bb) * 64 + 16 * tq) * 2, raw, p.x_bf16 != 0);
            }
#pragma unroll
            for (int off = 1; off < 4 * NB; off <<= 1) {
                v.x += __shfl_xor_sync(0xffffffffu, v.x, off);
                v.y += __shfl_xor_sync(0xffffffffu, v.y, off);
            }
            if (jl < pl.nseg && (lane & (4 * NB - 1)) == 0)
                xs[jl] = v;
        }
        if (rounds > 1)
            stage_rounds<B, NB, FL, IX>(p, xw, xs, warp, lane, rounds);
        __syncwarp();
    }

    const int m0 = min(g, p.M - 1);                     // token of the lane's B column, tile 0
    const int m1 = min(g + 8, p.M - 1);                 // tile 1 (NT = 2)
    const int first_b = (16 * B * t) / 32 * 4;          // byte of the thread's first word in a block
    const int o = (B & 1) ? 16 * (t & 1) : 0;           // bit offset of its run in that word
    const float zc = p.zeros ? 0.f : static_cast<float>(p.zero_const);
    const uint3 fl = make_uint3(((1u << (p.ebits + p.mbits)) - 1u) * 0x00010001u, static_cast<uint32_t>(10 - p.mbits),
                                static_cast<uint32_t>(15 - p.ebits - p.mbits));
    bool ok = true;
    int slot = 0;
    uint32_t par = 0;

    for (int rb = 0; rb < nrb; ++rb) {
        const int rr = rb * kRowBlock;
        const int cnt = min(kRowBlock, nrows - rr);
        int lr[2][2];   // slot row of (tile i, half h); padding rows repeat the last row
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h)
                lr[i][h] = min(16 * i + 8 * h + g, cnt - 1);
        float tot[2][NT][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    tot[i][tt][e] = 0.f;

#pragma unroll 1
        for (int c = 0; c < nchunk; ++c) {
            const int ichunk = rb * nchunk + c;
            if (ok && *fail)
                ok = false;
            if (ok && !mbar_wait(&full[slot], par, p.status)) {
                ok = false;
                *fail = 1;
            }
            if (ok) {
                const uint8_t *sb = slots + static_cast<size_t>(slot) * pl.slot_bytes;
                // where the thread's run of (tile i, half h) starts in block 0 of the chunk
                const uint8_t *run0[2][2];
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        run0[i][h] = TILE ? sb + i * 16 * pl.span * pl.seg_bytes + ((8 * h + g) * 4 + t) * 2 * B -
                                                ((B & 1) && (t & 1) ? 2 : 0)
                                          : sb + lr[i][h] * pl.pitch + first_b;
#pragma unroll 1
                for (int jj = 0; jj < pl.span; ++jj) {
                    const int j = c * pl.span + jj;
                    float acc[2][2][NT][4];
#pragma unroll
                    for (int u = 0; u < 2; ++u)
#pragma unroll
                        for (int i = 0; i < 2; ++i)
#pragma unroll
                            for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    acc[u][i][tt][e] = 0.f;
#pragma unroll
                    for (int bb = 0; bb < NB; ++bb) {
                        // block kblock of the chunk: 8 b bytes apart per row (canonical), or one
                        // 16-row unit of 128 b bytes apart (tile16)
                        const int kblock = jj * (pl.kseg / 64) + warp * NB + bb;
                        block_mma<B, NT, FL, IX>(run0, kblock * (TILE ? 128 * B : 8 * B),
                                             xw + ((j * NB + bb) * 64 + 16 * t) * 2, pl.x_pitch, m0, m1, o, fl,
                                             acc);
                    }
                    // the group's offset, zero and scale: tot += s (acc - C - z X)
                    const int gidx = j * kWarps + warp;
                    float X[NT][2], D[NT][2];
#pragma unroll
                    for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                        for (int cc = 0; cc < 2; ++cc) {
                            const int tok = 8 * tt + 2 * t + cc;
                            const float2 xc = tok < p.M ? xs[tok * pl.nseg + j] : make_float2(0.f, 0.f);
                            X[tt][cc] = xc.x;
                            D[tt][cc] = fmaf(zc, xc.x, xc.y);   // C + z X for a constant zero
                        }
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const int e = gidx * nrows + rr + lr[i][h];
                            const float s = FL ? f16_bits_to_f32(sc[e]) * p.fscale : f16_bits_to_f32(sc[e]);
                            const float z = p.zeros ? f16_bits_to_f32(zo[e]) : 0.f;
#pragma unroll
                            for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                                for (int cc = 0; cc < 2; ++cc)
                                    tot[i][tt][2 * h + cc] = fmaf(
                                        s, fmaf(-z, X[tt][cc], (NT == 2 ? acc[0][i][tt][2 * h + cc] + acc[1][i][tt][2 * h + cc]
                                                                        : acc[0][i][tt][2 * h + cc]) - D[tt][cc]),
                                    tot[i][tt][2 * h + cc]);
                            if constexpr (IX) {
                                // the exact integer accumulator sum (u - z) x of the group, when asked
                                const int row = 16 * i + 8 * h + g;
                                if (p.acc_out && row < cnt) {
#pragma unroll
                                    for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                                        for (int cc = 0; cc < 2; ++cc) {
                                            const int tok = 8 * tt + 2 * t + cc;
                                            const float a = (NT == 2 ? acc[0][i][tt][2 * h + cc] + acc[1][i][tt][2 * h + cc]
                                                                     : acc[0][i][tt][2 * h + cc]) - D[tt][cc];
                                            if (tok < p.M)
                                                p.acc_out[(static_cast<long long>(tok) * p.N + r0 + rr + row) * ng + gidx] =
                                                    static_cast<int32_t>(a);
                                        }
                                }
                            }
                        }
                }
            }
            // release the slot; warp 0 refills it with chunk ichunk + slots
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[slot]);
            if (warp == 0 && ichunk + pl.slots < total) {
                if (ok && !mbar_wait(&empty[slot], par, p.status)) {
                    ok = false;
                    *fail = 1;
                }
                if (ok) {
                    fence_proxy_async_smem();
                    issue_chunk<TILE>(p, slots, full, ichunk + pl.slots, r0, nrows, pol, lane);
                    issued = ichunk + pl.slots + 1;
                }
            }
            if (++slot == pl.slots) {
                slot = 0;
                par ^= 1u;
            }
        }

        // the row block's partial sums meet in shared memory, added in warp order
        float *rw = red + warp * kRowBlock * p.M;
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int row = 16 * i + 8 * h + g, tok = 8 * tt + 2 * t + c;
                        if (row < cnt && tok < p.M)
                            rw[row * p.M + tok] = tot[i][tt][2 * h + c];
                    }
        __syncthreads();
        for (int idx = threadIdx.x; idx < cnt * p.M; idx += kThreads) {
            const int tok = idx / cnt, row = idx - tok * cnt;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w)
                v += red[(w * kRowBlock + row) * p.M + tok];
            const long long out = static_cast<long long>(tok) * p.N + r0 + rr + row;
            if constexpr (IX)   // the per-token activation scale
                v *= f16_bits_to_f32(p.sa[tok]);
            reinterpret_cast<uint16_t *>(p.y)[out] = p.y_bf16 ? f32_to_bf16_bits(v) : f32_to_f16_bits(v);
        }
        if (rb + 1 < nrb)
            __syncthreads();
    }

    // after a timed-out wait, no bulk copy may still be landing when the CTA exits
    __syncthreads();
    if (warp == 0 && lane == 0 && *fail) {
        for (int i = max(0, issued - pl.slots); i < issued; ++i)
            if (!mbar_wait(&full[i % pl.slots], static_cast<uint32_t>(i / pl.slots) & 1u, p.status))
                break;
    }
}

template <int B, int NT, int NB, bool TILE, bool FL, bool IX = false>
cudaError_t launch_decode_b(const DecodeParams &p, cudaStream_t stream)
{
    auto kern = decode_kernel<B, NT, NB, TILE, FL, IX>;
    static SmemLimit limit;
    if (const cudaError_t e = ensure_smem_limit(limit, kern, p.pl.smem, true); e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.pl.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int NT, int NB, bool TILE>
cudaError_t launch_decode_cfg(const DecodeParams &p, int bits, cudaStream_t stream)
{
    switch (bits) {
    case 1: return launch_decode_b<1, NT, NB, TILE, false>(p, stream);
    case 2: return launch_decode_b<2, NT, NB, TILE, false>(p, stream);
    case 3: return launch_decode_b<3, NT, NB, TILE, false>(p, stream);
    case 4: return launch_decode_b<4, NT, NB, TILE, false>(p, stream);
    case 5: return launch_decode_b<5, NT, NB, TILE, false>(p, stream);
    case 6: return launch_decode_b<6, NT, NB, TILE, false>(p, stream);
    case 7: return launch_decode_b<7, NT, NB, TILE, false>(p, stream);
    case 8: return launch_decode_b<8, NT, NB, TILE, false>(p, stream);
    default: return cudaErrorInvalidValue;
    }
}

// All configurations of one layout.
template <bool TILE>
cudaError_t launch_decode_layout(const DecodeParams &p, int bits, cudaStream_t stream)
{
    const bool g128 = p.group_log2 == 7;
    if (p.M > 8)
        return g128 ? launch_decode_cfg<2, 2, TILE>(p, bits, stream) : launch_decode_cfg<2, 1, TILE>(p, bits, stream);
    return g128 ? launch_decode_cfg<1, 2, TILE>(p, bits, stream) : launch_decode_cfg<1, 1, TILE>(p, bits, stream);
}

// Exact-integer mode (int8 activations, signed b-bit weights), every configuration.
template <int B>
cudaError_t launch_decode_int_width(const DecodeParams &p, cudaStream_t stream)
{
    const bool g128 = p.group_log2 == 7;
    if (p.M > 8)
        return g128 ? launch_decode_b<B, 2, 2, false, false, true>(p, stream)
                    : launch_decode_b<B, 2, 1, false, false, true>(p, stream);
    return g128 ? launch_decode_b<B, 1, 2, false, false, true>(p, stream)
                : launch_decode_b<B, 1, 1, false, false, true>(p, stream);
}

// Float codes of width B (canonical layout), every configuration.
template <int B>
cudaError_t launch_decode_float_width(const DecodeParams &p, cudaStream_t stream)
{
    const bool g128 = p.group_log2 == 7;
    if (p.M > 8)
        return g128 ? launch_decode_b<B, 2, 2, false, true>(p, stream) : launch_decode_b<B, 2, 1, false, true>(p, stream);
    return g128 ? launch_decode_b<B, 1, 2, false, true>(p, stream) : launch_decode_b<B, 1, 1, false, true>(p, stream);
}

}  // namespace

}  // namespace qmm
