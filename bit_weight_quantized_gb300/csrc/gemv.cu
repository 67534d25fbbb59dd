// gemv.cu -- decode / skinny quantized matmul (1 <= M <= 16) for sm_103a.
//
// y[m][n] = sum_g s[n][g] * ( sum_{k in g} q[n][k] x[m][k]  -  z[n][g] * X[m][g] ),
// X[m][g] = sum_{k in g} x[m][k]   -- Eq. (5) of BitLLM, w = s (q - z), with the
// zero-point term factored out of the group sum so that the tensor cores only
// ever see exact integer codes.
//
// Work split.  CTA c owns a contiguous range of output columns (rows of the
// packed weight matrix) and the whole K range; rows are processed in blocks
// of at most 128 (eight 16-row MMA tiles).  Warp 0 is the producer: it streams
// the block's packed bitstream through a ring of shared-memory stages with
// TMA tile loads (one load per stage: rows x Cs 128-code chunks).  Warps 1..8
// consume: warp w takes every 8th chunk, so the K reduction is split over the
// eight warps and finished through shared memory in a fixed order (the result
// is deterministic).
//
// Inside a chunk, each 16-row tile is one mma.sync.m16n8k16 (f16 in, f32
// accumulate) per 16 codes.  The four threads of an MMA quad each own a run of
// R = G/4 consecutive codes of the same group, so every MMA accumulates within
// one group and the group scale can be applied in fp32.  Codes become fp16 in
// registers with no shared-memory round trip: a LOP3 keeps one code in each
// half of a 32-bit window and sets the half's exponent so that the half reads
// 2^E + q exactly; an exact HSUB2 removes 2^E.  The code-to-slot pairing is a
// per-width plan (unpack_plans.h); activations are staged once per CTA in the
// same slot order, so the sum over k is unchanged.
#include <cuda.h>

#include "common.cuh"
#include "gemv.h"
#include "unpack_plans.h"

namespace qmm {

// ---- per-width compile-time facts -------------------------------------------------
template <int B> struct Width {
    // 128-code chunks per TMA stage.  Odd, so that the dense smem row pitch
    // 16*B*CS makes the quad-strided run reads bank-conflict free; 16*B*CS <= 256
    // (TMA box limit).  B = 8 uses one chunk of 128 B with the 128-byte swizzle.
    static constexpr int CS = B == 1 ? 15 : B == 2 ? 7 : B == 3 ? 5 : (B == 4 || B == 5) ? 3 : 1;
    static constexpr int CHUNK_BYTES = 16 * B;
    static constexpr int ROW_BYTES = CHUNK_BYTES * CS;   // bytes of one row in a stage
    static constexpr bool SWIZZLE = (B == 8);
};

__host__ __device__ constexpr int width_cs(int b)
{
    return b == 1 ? 15 : b == 2 ? 7 : b == 3 ? 5 : (b == 4 || b == 5) ? 3 : 1;
}

// ---- reading a run of a row out of a stage ---------------------------------------------
// Byte offset of (row, byte) inside a stage, applying the 128-byte swizzle
// (16-byte chunk index XOR row mod 8) when the stage was loaded with it.
template <int B>
__device__ __forceinline__ uint32_t stage_off(int row, int byte)
{
    const uint32_t logical = static_cast<uint32_t>(row * Width<B>::ROW_BYTES + byte);
    if constexpr (Width<B>::SWIZZLE)
        return logical ^ (((logical >> 7) & 7u) << 4);
    else
        return logical;
}

// Loads the run of R codes that starts at code `code0` of the stage row into
// NW words, shifted so that the run starts at bit 0 of w[0].
template <int B, int R>
__device__ __forceinline__ void load_run(const uint8_t *stage, int row, int code0,
                                         uint32_t (&w)[(R * B + 31) / 32])
{
    constexpr int NW = (R * B + 31) / 32;
    const int bit0 = code0 * B;
    if constexpr ((R * B) % 32 == 0 && (B % 4 == 0) && B != 8) {
        // 16-byte aligned run of NW words (B = 4: R*B/8 bytes at a multiple of 16)
        static_assert(NW % 4 == 0 || NW < 4, "");
        if constexpr (NW >= 4) {
#pragma unroll
            for (int i = 0; i < NW; i += 4) {
                const uint4 v = *reinterpret_cast<const uint4 *>(stage + stage_off<B>(row, bit0 / 8 + 4 * i));
                w[i] = v.x; w[i + 1] = v.y; w[i + 2] = v.z; w[i + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < NW; ++i)
                w[i] = *reinterpret_cast<const uint32_t *>(stage + stage_off<B>(row, bit0 / 8 + 4 * i));
        }
    } else if constexpr (B == 8) {
        // byte-aligned codes; runs are R bytes at a multiple of R, 16-byte swizzle chunks
        if constexpr (R >= 16) {
#pragma unroll
            for (int i = 0; i < NW; i += 4) {
                const uint4 v = *reinterpret_cast<const uint4 *>(stage + stage_off<B>(row, code0 + 4 * i));
                w[i] = v.x; w[i + 1] = v.y; w[i + 2] = v.z; w[i + 3] = v.w;
            }
        } else {
            const uint2 v = *reinterpret_cast<const uint2 *>(stage + stage_off<B>(row, code0));
            w[0] = v.x; w[1] = v.y;
        }
    } else if constexpr ((R * B) % 32 == 0) {
        // word aligned; B = 2 and 6 are also 8-byte aligned
        const int wi = bit0 / 32;
        if constexpr (B % 2 == 0 && NW % 2 == 0) {
#pragma unroll
            for (int i = 0; i < NW; i += 2) {
                const uint2 v = *reinterpret_cast<const uint2 *>(stage + stage_off<B>(row, 4 * (wi + i)));
                w[i] = v.x; w[i + 1] = v.y;
            }
        } else {
#pragma unroll
            for (int i = 0; i < NW; ++i)
                w[i] = *reinterpret_cast<const uint32_t *>(stage + stage_off<B>(row, 4 * (wi + i)));
        }
    } else {
        // run starts inside a word: read NW+1 words and funnel-shift
        const int wi = bit0 / 32;
        const int sh = bit0 & 31;
        uint32_t src[NW + 1];
#pragma unroll
        for (int i = 0; i <= NW; ++i)
            src[i] = *reinterpret_cast<const uint32_t *>(stage + stage_off<B>(row, 4 * (wi + i)));
#pragma unroll
        for (int i = 0; i < NW; ++i)
            w[i] = __funnelshift_r(src[i], src[i + 1], sh);
    }
}

// ---- codes -> fp16 pairs (q exact) ---------------------------------------------------------
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

// a[i] = fp16 pair (q_lo, q_hi) of plan pair i (exact small integers)
template <int B, int R>
__device__ __forceinline__ void extract_run(const uint32_t (&w)[(R * B + 31) / 32],
                                            uint32_t (&a)[R / 2])
{
    constexpr int NW = (R * B + 31) / 32;
    if constexpr (B == 8) {
        // pair i = codes (2i, 2i+1): bytes into the low mantissa of 1024.0
#pragma unroll
        for (int i = 0; i < R / 2; ++i) {
            const uint32_t v = prmt(w[i >> 1], 0x64646464u, (i & 1) ? 0x4342u : 0x4140u);
            a[i] = hsub2(v, 0x64006400u);
        }
    } else {
        using P = UnpackPlan<B, R>;
        uint32_t win[P::kWindows];
#pragma unroll
        for (int v = 0; v < P::kWindows; ++v)
            win[v] = plan_window<B, R, NW>(w, v);
#pragma unroll
        for (int i = 0; i < R / 2; ++i) {
            const uint32_t v = lop3_and_or(win[P::win(i)], P::mask(i), P::magic(i));
            a[i] = hsub2(v, pow2_half_bits(P::elo(i)) | (pow2_half_bits(P::ehi(i)) << 16));
        }
    }
}

// activation slot order of code c within a run (inverse of the pairing)
template <int B, int R>
__device__ __forceinline__ constexpr int code_of_slot(int s)
{
    // s = 4*j + e -> pair 2j + (e >> 1), lo if e even else hi
    if constexpr (B == 8) {
        return s;  // pairs are (2i, 2i+1), so slot order is code order
    } else {
        using P = UnpackPlan<B, R>;
        const int i = 2 * (s >> 2) + ((s >> 1) & 1);
        return (s & 1) ? P::hi(i) : P::lo(i);
    }
}

// ---- the kernel ----------------------------------------------------------------------------
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kMaxTiles = 8;   // 16-row MMA tiles per row block

template <int B, int NT, int R>
__global__ void __launch_bounds__(kThreads, 1)
gemv_kernel(const __grid_constant__ CUtensorMap tmap, const GemvParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *ring = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    uint64_t *empty = full + p.ring;
    uint16_t *xp = reinterpret_cast<uint16_t *>(smem + p.off_x);      // [chunk][8][M][4][4]
    float *xs = reinterpret_cast<float *>(smem + p.off_xs);           // [group][MP]
    float2 *sz = reinterpret_cast<float2 *>(smem + p.off_sz);         // [row][sz_pitch] (s, z*s)
    float *red = reinterpret_cast<float *>(smem + p.off_red);         // [warp][RBP][MP]

    constexpr int MP = 8 * NT;           // padded token count of the D fragments
    constexpr int NGC = 128 / (4 * R);   // groups per 128-code chunk
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int cta = blockIdx.x;
    const int r0 = cta * p.rows_base + min(cta, p.rows_rem);
    const int nrows = p.rows_base + (cta < p.rows_rem ? 1 : 0);
    const int nblocks = (nrows + p.rb - 1) / p.rb;
    const int total_stages = nblocks * p.stages_per_block;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.ring; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ================= producer =================
        bool ok = true;
        int issued = 0;
        for (int it = 0; it < total_stages && ok; ++it) {
            const int slot = it % p.ring;
            const int round = it / p.ring;
            if (round > 0)
                ok = mbar_wait(&empty[slot], (round - 1) & 1, p.status);
            if (!ok)
                break;
            const int blk = it / p.stages_per_block;
            const int s = it - blk * p.stages_per_block;
            const int row0 = r0 + blk * p.rb;
            uint8_t *dst = ring + static_cast<size_t>(slot) * p.stage_bytes;
            if (p.use_tma) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(&full[slot], p.tile_bytes);
                    tma_load_2d(dst, &tmap, &full[slot], s * Width<B>::ROW_BYTES, row0);
                }
            } else {
                // plain 4-byte copies (row pitch of the packed matrix not 16-byte aligned)
                const int words_per_row = Width<B>::ROW_BYTES / 4;
                for (int e = lane; e < p.rb * words_per_row; e += 32) {
                    const int r = e / words_per_row;
                    const int wo = e - r * words_per_row;
                    const long long byte = static_cast<long long>(s) * Width<B>::ROW_BYTES + 4 * wo;
                    uint32_t v = 0;
                    if (row0 + r < p.N && byte < p.row_bytes)
                        v = *reinterpret_cast<const uint32_t *>(p.packed + static_cast<long long>(row0 + r) * p.row_bytes + byte);
                    *reinterpret_cast<uint32_t *>(dst + stage_off<B>(r, 4 * wo)) = v;
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&full[slot]);
            }
            ++issued;
        }
        // drain: make sure no copy into this CTA's shared memory is still in flight
        if (lane == 0) {
            const int first = issued > p.ring ? issued - p.ring : 0;
            for (int it = first; it < issued; ++it)
                if (!mbar_wait(&full[it % p.ring], (it / p.ring) & 1, p.status))
                    break;
        }
        return;
    }

    // ================= consumers =================
    const int cw = warp - 1;              // consumer warp 0..7
    const int ct = threadIdx.x - 32;      // consumer thread 0..255
    const int g = lane >> 2, t = lane & 3;
    const int M = p.M;

    // ---- stage activations in slot order and the per-group sums X[m][grp] ----
    {
        const int G = 4 * R;
        const int ngp = p.nchunks * NGC;  // groups incl. the padding of the last chunk
        for (int idx = ct; idx < M * ngp; idx += 32 * kConsumerWarps) {
            const int m = idx / ngp;
            const int grp = idx - m * ngp;
            const int cg = grp / NGC;
            const int gi = grp - cg * NGC;
            float sum = 0.f;
#pragma unroll 1
            for (int tt = 0; tt < 4; ++tt) {
                const int k0 = grp * G + tt * R;
                uint16_t v[R];
#pragma unroll
                for (int c = 0; c < R; c += 8) {
                    uint4 q = make_uint4(0, 0, 0, 0);
                    if (k0 + c < p.K)
                        q = *reinterpret_cast<const uint4 *>(p.x + static_cast<long long>(m) * p.K + k0 + c);
                    v[c + 0] = q.x & 0xFFFF; v[c + 1] = q.x >> 16;
                    v[c + 2] = q.y & 0xFFFF; v[c + 3] = q.y >> 16;
                    v[c + 4] = q.z & 0xFFFF; v[c + 5] = q.z >> 16;
                    v[c + 6] = q.w & 0xFFFF; v[c + 7] = q.w >> 16;
                }
#pragma unroll
                for (int c = 0; c < R; ++c)
                    sum += f16_bits_to_f32(v[c]);
#pragma unroll
                for (int j = 0; j < R / 4; ++j) {
                    uint2 o;
                    o.x = v[code_of_slot<B, R>(4 * j + 0)] | (static_cast<uint32_t>(v[code_of_slot<B, R>(4 * j + 1)]) << 16);
                    o.y = v[code_of_slot<B, R>(4 * j + 2)] | (static_cast<uint32_t>(v[code_of_slot<B, R>(4 * j + 3)]) << 16);
                    const int jj = gi * (R / 4) + j;
                    *reinterpret_cast<uint2 *>(xp + ((static_cast<long long>(cg) * 8 + jj) * M + m) * 16 + tt * 4) = o;
                }
            }
            xs[grp * MP + m] = sum;
        }
        // zero the padded tokens of X
        for (int idx = ct; idx < (MP - M) * ngp; idx += 32 * kConsumerWarps) {
            const int mm = M + idx / ngp;
            const int grp = idx % ngp;
            xs[grp * MP + mm] = 0.f;
        }
    }

    const int ng = p.ng;
    bool ok = true;
    int it = 0;
    for (int blk = 0; blk < nblocks; ++blk) {
        const int row0 = r0 + blk * p.rb;
        const int rows_valid = min(p.rb, r0 + nrows - row0);
        const int T = (rows_valid + 15) / 16;

        // ---- scales and zero*scale for the block's rows ----
        named_sync(1, 32 * kConsumerWarps);   // previous block's epilogue is done with sz/red
        for (int idx = ct; idx < rows_valid * ng; idx += 32 * kConsumerWarps) {
            const int r = idx / ng;
            const int grp = idx - r * ng;
            const long long off = static_cast<long long>(row0 + r) * ng + grp;
            const float s = f16_bits_to_f32(p.scales[off]);
            const float z = p.zeros ? static_cast<float>(p.zeros[off]) : static_cast<float>(p.zero_const);
            sz[r * p.sz_pitch + grp] = make_float2(s, z * s);
        }
        named_sync(1, 32 * kConsumerWarps);

        float tot[kMaxTiles][NT][4];
#pragma unroll
        for (int mt = 0; mt < kMaxTiles; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    tot[mt][nt][e] = 0.f;

        for (int s = 0; s < p.stages_per_block; ++s, ++it) {
            const int slot = it % p.ring;
            if (ok)
                ok = mbar_wait(&full[slot], (it / p.ring) & 1, p.status);
            if (ok) {
                const uint8_t *stage = ring + static_cast<size_t>(slot) * p.stage_bytes;
#pragma unroll 1
                for (int ci = 0; ci < Width<B>::CS; ++ci) {
                    const int cg = s * Width<B>::CS + ci;
                    if (cg >= p.nchunks)
                        break;
                    if ((cg & (kConsumerWarps - 1)) != cw)
                        continue;
#pragma unroll 1
                    for (int gi = 0; gi < NGC; ++gi) {
                        const int grp = cg * NGC + gi;
                        if (grp >= ng)
                            break;
                        // activation fragments for the R/4 MMAs of this group
                        uint32_t bf[R / 4][NT][2];
#pragma unroll
                        for (int j = 0; j < R / 4; ++j)
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const int m = g + 8 * nt;
                                uint2 v = make_uint2(0, 0);
                                if (m < M)
                                    v = *reinterpret_cast<const uint2 *>(
                                        xp + ((static_cast<long long>(cg) * 8 + gi * (R / 4) + j) * M + m) * 16 + t * 4);
                                bf[j][nt][0] = v.x;
                                bf[j][nt][1] = v.y;
                            }
                        float2 xv[NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            xv[nt] = *reinterpret_cast<const float2 *>(xs + grp * MP + 8 * nt + 2 * t);
                        const int code0 = ci * 128 + gi * 4 * R + t * R;   // within the stage row
#pragma unroll
                        for (int mt = 0; mt < kMaxTiles; ++mt) {
                            if (mt < T) {
                                const int lr0 = mt * 16 + g;
                                uint32_t w0[(R * B + 31) / 32], w1[(R * B + 31) / 32];
                                load_run<B, R>(stage, lr0, code0, w0);
                                load_run<B, R>(stage, lr0 + 8, code0, w1);
                                uint32_t a0[R / 2], a1[R / 2];
                                extract_run<B, R>(w0, a0);
                                extract_run<B, R>(w1, a1);
                                float d[NT][4];
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        d[nt][e] = 0.f;
#pragma unroll
                                for (int j = 0; j < R / 4; ++j)
#pragma unroll
                                    for (int nt = 0; nt < NT; ++nt)
                                        mma_f16_16816(d[nt], a0[2 * j], a1[2 * j], a0[2 * j + 1],
                                                      a1[2 * j + 1], bf[j][nt][0], bf[j][nt][1]);
                                const float2 sz0 = sz[lr0 * p.sz_pitch + grp];
                                const float2 sz1 = sz[(lr0 + 8) * p.sz_pitch + grp];
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    tot[mt][nt][0] = fmaf(sz0.x, d[nt][0], tot[mt][nt][0]);
                                    tot[mt][nt][0] = fmaf(-sz0.y, xv[nt].x, tot[mt][nt][0]);
                                    tot[mt][nt][1] = fmaf(sz0.x, d[nt][1], tot[mt][nt][1]);
                                    tot[mt][nt][1] = fmaf(-sz0.y, xv[nt].y, tot[mt][nt][1]);
                                    tot[mt][nt][2] = fmaf(sz1.x, d[nt][2], tot[mt][nt][2]);
                                    tot[mt][nt][2] = fmaf(-sz1.y, xv[nt].x, tot[mt][nt][2]);
                                    tot[mt][nt][3] = fmaf(sz1.x, d[nt][3], tot[mt][nt][3]);
                                    tot[mt][nt][3] = fmaf(-sz1.y, xv[nt].y, tot[mt][nt][3]);
                                }
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[slot]);
        }

        // ---- cross-warp reduction in a fixed order, then the store ----
#pragma unroll
        for (int mt = 0; mt < kMaxTiles; ++mt) {
            if (mt < T) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int row = mt * 16 + g;
                    const int tok = 8 * nt + 2 * t;
                    *reinterpret_cast<float2 *>(red + (cw * p.rbp + row) * MP + tok) =
                        make_float2(tot[mt][nt][0], tot[mt][nt][1]);
                    *reinterpret_cast<float2 *>(red + (cw * p.rbp + row + 8) * MP + tok) =
                        make_float2(tot[mt][nt][2], tot[mt][nt][3]);
                }
            }
        }
        named_sync(1, 32 * kConsumerWarps);
        for (int idx = ct; idx < M * rows_valid; idx += 32 * kConsumerWarps) {
            const int tok = idx / rows_valid;
            const int row = idx - tok * rows_valid;
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w)
                v += red[(w * p.rbp + row) * MP + tok];
            const long long o = static_cast<long long>(tok) * p.N + row0 + row;
            if (p.y_bf16)
                reinterpret_cast<uint16_t *>(p.y)[o] = f32_to_bf16_bits(v);
            else
                reinterpret_cast<uint16_t *>(p.y)[o] = f32_to_f16_bits(v);
        }
    }
}

// ---- host side -----------------------------------------------------------------------------
template <int B, int NT, int R>
static cudaError_t launch_one(const CUtensorMap &tmap, const GemvParams &p, int grid, int smem,
                              cudaStream_t stream)
{
    auto kern = gemv_kernel<B, NT, R>;
    static thread_local int configured_dev = -1;
    static thread_local int configured_smem = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev || configured_smem < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess)
            return e;
        configured_dev = dev;
        configured_smem = smem;
    }
    kern<<<grid, kThreads, smem, stream>>>(tmap, p);
    return cudaGetLastError();
}

template <int B, int NT>
static cudaError_t launch_r(const CUtensorMap &tmap, const GemvParams &p, int grid, int smem,
                            cudaStream_t stream)
{
    switch (p.group) {
    case 32: return launch_one<B, NT, 8>(tmap, p, grid, smem, stream);
    case 64: return launch_one<B, NT, 16>(tmap, p, grid, smem, stream);
    default: return launch_one<B, NT, 32>(tmap, p, grid, smem, stream);
    }
}

template <int B>
static cudaError_t launch_nt(const CUtensorMap &tmap, const GemvParams &p, int grid, int smem,
                             cudaStream_t stream)
{
    if (p.M <= 8)
        return launch_r<B, 1>(tmap, p, grid, smem, stream);
    return launch_r<B, 2>(tmap, p, grid, smem, stream);
}

static int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Shared-memory layout for a given row-block size; returns total bytes (0 if
// it does not fit with at least `min_ring` stages).
static int plan_smem(GemvParams &p, int bits, int rb, int smem_max, int min_ring)
{
    const int MP = p.M <= 8 ? 8 : 16;
    const int ngp = p.nchunks * (128 / p.group);
    p.rb = rb;
    p.rbp = align_up(rb, 16);
    const int row_bytes = 16 * bits * width_cs(bits);
    p.tile_bytes = rb * row_bytes;
    // room for the 16-row tile padding the consumers read (never stored) and
    // for the one word a shifted run may read past its row
    p.stage_bytes = align_up(p.rbp * row_bytes + 16, 1024);
    p.sz_pitch = p.ng + ((p.ng & 1) ? 0 : 1);
    int off = 0;
    const int x_bytes = align_up(p.M * p.nchunks * 128 * 2, 16);
    const int xs_bytes = align_up(ngp * MP * 4, 16);
    const int sz_bytes = align_up(p.rbp * p.sz_pitch * 8, 16);
    const int red_bytes = align_up(kConsumerWarps * p.rbp * MP * 4, 16);
    const int fixed = x_bytes + xs_bytes + sz_bytes + red_bytes;
    const int budget = smem_max - 1024 /*alignment slack*/ - fixed;
    int ring = budget / (p.stage_bytes + 16);
    const int total_stages_max = p.stages_per_block * 8;
    if (ring > total_stages_max)
        ring = total_stages_max;
    if (ring > 32)
        ring = 32;
    if (ring < min_ring)
        return 0;
    p.ring = ring;
    off = ring * p.stage_bytes;
    p.off_bar = off;
    off += align_up(2 * ring * 8, 16);
    p.off_x = off;
    off += x_bytes;
    p.off_xs = off;
    off += xs_bytes;
    p.off_sz = off;
    off += sz_bytes;
    p.off_red = off;
    off += red_bytes;
    return off + 1024;
}

qmm_status gemv_plan(GemvParams &p, int bits, int num_sms, int smem_max, int *grid_out,
                     int *smem_out)
{
    p.nchunks = (p.K + 127) / 128;
    p.stages_per_block = (p.nchunks + width_cs(bits) - 1) / width_cs(bits);
    int grid = (p.N + 15) / 16;
    if (grid > num_sms)
        grid = num_sms;
    if (grid < 1)
        grid = 1;
    p.rows_base = p.N / grid;
    p.rows_rem = p.N % grid;
    const int rows_max = p.rows_base + (p.rows_rem ? 1 : 0);
    for (int nblk = (rows_max + 127) / 128; nblk <= rows_max; ++nblk) {
        const int rb = (rows_max + nblk - 1) / nblk;
        const int smem = plan_smem(p, bits, rb, smem_max, 4);
        if (smem) {
            *grid_out = grid;
            *smem_out = smem;
            return QMM_OK;
        }
        if (rb <= 16)
            break;
    }
    return QMM_ERR_UNSUPPORTED;  // activations of M x K do not fit in shared memory
}

cudaError_t gemv_launch(const CUtensorMap &tmap, const GemvParams &p, int bits, int grid,
                        int smem, cudaStream_t stream)
{
    switch (bits) {
    case 1: return launch_nt<1>(tmap, p, grid, smem, stream);
    case 2: return launch_nt<2>(tmap, p, grid, smem, stream);
    case 3: return launch_nt<3>(tmap, p, grid, smem, stream);
    case 4: return launch_nt<4>(tmap, p, grid, smem, stream);
    case 5: return launch_nt<5>(tmap, p, grid, smem, stream);
    case 6: return launch_nt<6>(tmap, p, grid, smem, stream);
    case 7: return launch_nt<7>(tmap, p, grid, smem, stream);
    default: return launch_nt<8>(tmap, p, grid, smem, stream);
    }
}

}  // namespace qmm

namespace qmm {
int gemv_stage_chunks(int bits) { return width_cs(bits); }
}  // namespace qmm
