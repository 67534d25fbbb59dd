// skinny.cuh -- the decode / skinny quantized matmul kernel (sm_103a).
//
// Computes, for a weight matrix stored as per-column LSB-first b-bit streams,
//
//   y[m][n] = sum_g s[n][g] * ( sum_{k in g} q[n][k] x[m][k]  -  z[n][g] X[m][g] ),
//   X[m][g] = sum_{k in g} x[m][k],
//
// which is sum_k x[m][k] * s (q - z) -- BitLLM Eq. (5) with the zero-point term
// factored out of each group so that the tensor cores only see exact integer
// codes.  The same kernel runs the integer-native W4A8 variant (BitLLM
// sec. 4.3-4.4): signed int4 weights w = (c xor 8) - 8, int8 activations, an
// exact per-group integer accumulator acc = sum u x - 8 X (u = c xor 8), and a
// deferred epilogue y = sa[m] * sum_g ws[n][g] * acc.  Products of 4-bit and
// 8-bit integers and their group sums (|sum| <= 128*15*127 < 2^24) are exact in
// fp16 x fp16 -> fp32 tensor-core arithmetic, and GB300's fp16 tensor path is
// several times faster than its int8 paths, so the integer pipeline runs there.
//
// Work split.  CTA c owns a contiguous range of output columns (rows of the
// packed matrix) and the whole K range; rows are processed in blocks of at most
// 128.  A block's bitstream moves through a ring of shared-memory stages: a
// stage is one K segment of every row of the block, one 1-D bulk copy (TMA) per
// row, landing at a padded pitch that keeps the MMA quads' reads bank-conflict
// free.  There is no producer warp: the first ring of stages is issued at entry
// and the last warp to finish a stage issues the stage that reuses its slot.
// The eight warps split K (warp w takes the chunks = w mod ksplit) and the
// block's 16-row tiles (at most two per warp); partial sums meet in shared
// memory and are added in a fixed order (deterministic).
//
// Decode sequences.  A decode-size CTA uses at most half of an SM (shared
// memory, 256 threads x 128 registers), and the kernel signals its dependents
// at entry, so with programmatic dependent launch the next call's CTAs start
// beside this call's and stream their weights while this call finishes.  The
// packed weights, scales and zeros are read before the dependency wait (the
// ABI requires that the preceding kernel on the stream does not write them);
// only the activations wait for the preceding kernel.
//
// Inside a chunk each 16-row tile takes one mma.sync.m16n8k16 per 16 codes and
// 8 tokens.  The four threads of an MMA quad own runs of R = G/4 consecutive
// codes of one group, so every MMA stays inside a group and the group's scale
// is applied in fp32.  Codes become fp16 in registers with no shared-memory
// round trip: a LOP3 keeps one code in each half of a 32-bit window and sets the
// half's exponent so that it reads 2^E + q exactly.  The fp16 path keeps 2^E in
// the MMA operand and subtracts C[m][g] = sum_k 2^E_k x[m][k], formed exactly
// by the activation staging, from each group's dot product in fp32; the W4A8
// path removes 2^E with an exact HSUB2 so that its sums stay integers below
// 2^24.  Activations are staged once per CTA (or once per K phase when M x K
// does not fit) in "slot" order -- the order in which codes come out of the
// registers -- with 16-byte chunks XOR-swizzled against bank conflicts.
#pragma once

#include <cuda.h>

#include <type_traits>

#include "common.cuh"
#include "gemv.h"
#include "extract.cuh"
#include "unpack_plans.h"

namespace qmm {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kTilesPerWarp = 2;   // 16-row tiles a warp computes per block, at most

// The run of R codes starting at code `code0` of the stage row at `rowp`, as
// NW words shifted so that the run starts at bit 0 of w[0].
template <int B, int R>
__device__ __forceinline__ void load_run(const uint8_t *rowp, int code0, uint32_t (&w)[(R * B + 31) / 32])
{
    constexpr int NW = (R * B + 31) / 32;
    const int bit0 = code0 * B;
    if constexpr (B == 8) {
        if constexpr (R >= 16) {
#pragma unroll
            for (int i = 0; i < NW; i += 4) {
                const uint4 v = *reinterpret_cast<const uint4 *>(rowp + code0 + 4 * i);
                w[i] = v.x; w[i + 1] = v.y; w[i + 2] = v.z; w[i + 3] = v.w;
            }
        } else {
            const uint2 v = *reinterpret_cast<const uint2 *>(rowp + code0);
            w[0] = v.x; w[1] = v.y;
        }
    } else if constexpr ((R * B) % 32 == 0 && B == 4 && NW == 4) {
        const uint4 v = *reinterpret_cast<const uint4 *>(rowp + bit0 / 8);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr ((R * B) % 32 == 0) {
        const int wi = bit0 / 32;
        if constexpr (B % 2 == 0 && NW % 2 == 0) {
#pragma unroll
            for (int i = 0; i < NW; i += 2) {
                const uint2 v = *reinterpret_cast<const uint2 *>(rowp + 4 * (wi + i));
                w[i] = v.x; w[i + 1] = v.y;
            }
        } else {
#pragma unroll
            for (int i = 0; i < NW; ++i)
                w[i] = *reinterpret_cast<const uint32_t *>(rowp + 4 * (wi + i));
        }
    } else {
        // the run starts inside a word: read NW+1 words and funnel-shift
        const int wi = bit0 / 32;
        const int sh = bit0 & 31;
        uint32_t src[NW + 1];
#pragma unroll
        for (int i = 0; i <= NW; ++i)
            src[i] = *reinterpret_cast<const uint32_t *>(rowp + 4 * (wi + i));
#pragma unroll
        for (int i = 0; i < NW; ++i)
            w[i] = __funnelshift_r(src[i], src[i + 1], sh);
    }
}

// Four int8 values (one word) -> two fp16x2 words, exactly: with u = x + 128
// (the sign bit flipped), the byte permute forms fp16 1024 + u under the
// exponent byte 0x64, and subtracting 1152 leaves x.
__device__ __forceinline__ void s8x4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi)
{
    const uint32_t u = w ^ 0x80808080u;
    lo = hsub2(prmt(u, 0x64646464u, 0x4140u), 0x64806480u);
    hi = hsub2(prmt(u, 0x64646464u, 0x4342u), 0x64806480u);
}

// Loads run `idx` (R codes of one token) of the chunks [ch0, ch0 + nch) as fp16
// bit patterns (zeros past K).  MODE 0 reads fp16 x; MODE 1 reads int8 xq,
// converts it exactly and also returns the run's integer sum in `isum`.
template <int R, int MODE>
__device__ __forceinline__ void load_act_run(const GemvParams &p, int ch0, int runs_per_tok,
                                             int idx, uint16_t (&v)[R], int &isum)
{
    constexpr int G = 4 * R;
    constexpr int RPC = 128 / R;                 // runs per chunk
    const int m = idx / runs_per_tok;
    const int rr = idx - m * runs_per_tok;
    const int k0 = ch0 * 128 + (rr / RPC) * 128 + ((rr % RPC) / 4) * G + (rr % 4) * R;
    if constexpr (MODE == 0) {
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
    } else {
        isum = 0;
#pragma unroll
        for (int c = 0; c < R; c += 8) {
            uint2 q = make_uint2(0, 0);
            if (k0 + c < p.K)
                q = *reinterpret_cast<const uint2 *>(p.xq + static_cast<long long>(m) * p.K + k0 + c);
            isum = __dp4a(static_cast<int>(q.x), 0x01010101, isum);
            isum = __dp4a(static_cast<int>(q.y), 0x01010101, isum);
            uint32_t h[4];
            s8x4_to_f16x2(q.x, h[0], h[1]);
            s8x4_to_f16x2(q.y, h[2], h[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[c + 2 * e] = static_cast<uint16_t>(h[e] & 0xFFFFu);
                v[c + 2 * e + 1] = static_cast<uint16_t>(h[e] >> 16);
            }
        }
    }
}

// Chunk swizzle of the staged activations.  A run of R fp16 slots is R / 8
// 16-byte chunks; the run of (token, quad thread) index i stores its chunk c at
// chunk c ^ act_swizzle<R>(i).  Without it the 32 lanes of a fragment load (runs
// i = 0..31, the same chunk) would hit only 128 / (2 R) distinct 16-byte bank
// groups; with it every wavefront of 16-byte loads is conflict-free.
template <int R>
__device__ __forceinline__ int act_swizzle(int i)
{
    constexpr int NCH = R / 8;                   // chunks per run
    return NCH > 1 ? (i / (8 / NCH)) & (NCH - 1) : 0;
}

// Stages the activations of chunks [ch0, ch0 + nch) in slot order, and the
// per-group sums X[group][token]: each run summed pairwise in a fixed order,
// the four runs of a group added in order across the quad's lanes, so the
// result does not depend on the launch.
// MP - M padded tokens get X = 0.
template <int B, int R, int MODE, int MP>
__device__ __forceinline__ void stage_activations(const GemvParams &p, uint16_t *xp, float *xs,
                                                  float *cs, int ch0, int nch)
{
    constexpr int RPC = 128 / R;                 // runs per chunk
    constexpr int NGC = 128 / (4 * R);           // groups per chunk
    constexpr int U = R >= 32 ? 1 : 2;           // runs in flight per thread
    const int M = p.M;
    const int lane = threadIdx.x & 31;
    const int runs_per_tok = nch * RPC;
    const int nruns = M * runs_per_tok;
    if (MP > M) {
        const int ngp = nch * NGC;
        for (int idx = threadIdx.x; idx < ngp * (MP - M); idx += kThreads) {
            const int lg = idx / (MP - M);
            xs[lg * MP + M + (idx - lg * (MP - M))] = 0.f;
            if (MODE == 0)
                cs[lg * MP + M + (idx - lg * (MP - M))] = 0.f;
        }
    }
    // With at most half as many runs as threads, the runs go to every other lane
    // of all eight warps (two warps per scheduler instead of one).
    const int sp = 2 * nruns <= kThreads ? 2 : 1;
    const int rpw = 32 / sp;                         // runs per warp and pass
    const int rstep = kWarps * rpw;
    const int mylane = (lane % sp == 0) ? lane / sp : rpw;   // rpw: no run
    // warp-uniform trip count: the quad shuffles need every lane
    for (int wbase = (threadIdx.x >> 5) * rpw; wbase < nruns; wbase += U * rstep) {
        uint16_t v[U][R];
        int isum[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            isum[u] = 0;
            if (mylane < rpw && wbase + mylane + u * rstep < nruns)
                load_act_run<R, MODE>(p, ch0, runs_per_tok, wbase + mylane + u * rstep, v[u], isum[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int idx = wbase + mylane + u * rstep;
            const bool valid = mylane < rpw && idx < nruns;   // whole quads: nruns % 4 == 0
            float sum = 0.f, csum = 0.f;
            int m = 0, lc = 0, gi = 0, tt = 0;
            if (valid) {
                m = idx / runs_per_tok;
                const int rr = idx - m * runs_per_tok;
                lc = rr / RPC;
                gi = (rr % RPC) / 4;
                tt = rr % 4;
                if constexpr (MODE == 1) {
                    sum = static_cast<float>(isum[u]);   // exact: |sum| <= 128 R
                } else {
                    // pairwise, in a fixed order
                    float ps[R];
#pragma unroll
                    for (int c = 0; c < R; ++c)
                        ps[c] = f16_bits_to_f32(v[u][c]);
#pragma unroll
                    for (int w = 1; w < R; w *= 2)
#pragma unroll
                        for (int c = 0; c < R; c += 2 * w)
                            ps[c] += ps[c + w];
                    sum = ps[0];
                    // sum_k 2^E_k x_k: x summed per exponent, then scaled (exact)
                    // and added in increasing exponent order
                    float se[11];
#pragma unroll
                    for (int e = 0; e < 11; ++e)
                        se[e] = 0.f;
#pragma unroll
                    for (int c = 0; c < R; ++c)
                        se[exp_of_code<B, R>(c)] += f16_bits_to_f32(v[u][c]);
#pragma unroll
                    for (int e = 0; e < 11; ++e)
                        csum += se[e] * static_cast<float>(1 << e);   // exact: a power of two
                }
                // the run's R slots: [chunk][group][token][quad thread][R], chunks swizzled
                uint16_t *dst = xp + ((static_cast<long long>(lc * NGC + gi) * M + m) * 4 + tt) * R;
                const int swz = act_swizzle<R>(m * 4 + tt);
#pragma unroll
                for (int j = 0; j < R / 4; j += 2) {
                    uint4 o;
                    o.x = v[u][code_of_slot<B, R>(4 * j + 0)] | (static_cast<uint32_t>(v[u][code_of_slot<B, R>(4 * j + 1)]) << 16);
                    o.y = v[u][code_of_slot<B, R>(4 * j + 2)] | (static_cast<uint32_t>(v[u][code_of_slot<B, R>(4 * j + 3)]) << 16);
                    o.z = v[u][code_of_slot<B, R>(4 * j + 4)] | (static_cast<uint32_t>(v[u][code_of_slot<B, R>(4 * j + 5)]) << 16);
                    o.w = v[u][code_of_slot<B, R>(4 * j + 6)] | (static_cast<uint32_t>(v[u][code_of_slot<B, R>(4 * j + 7)]) << 16);
                    *reinterpret_cast<uint4 *>(dst + 8 * ((j >> 1) ^ swz)) = o;
                }
            }
            const float s1 = __shfl_down_sync(0xffffffffu, sum, 1 * sp);
            const float s2 = __shfl_down_sync(0xffffffffu, sum, 2 * sp);
            const float s3 = __shfl_down_sync(0xffffffffu, sum, 3 * sp);
            if (valid && tt == 0)
                xs[(lc * NGC + gi) * MP + m] = ((sum + s1) + s2) + s3;
            if constexpr (MODE == 0) {
                const float c1 = __shfl_down_sync(0xffffffffu, csum, 1 * sp);
                const float c2 = __shfl_down_sync(0xffffffffu, csum, 2 * sp);
                const float c3 = __shfl_down_sync(0xffffffffu, csum, 3 * sp);
                if (valid && tt == 0)
                    cs[(lc * NGC + gi) * MP + m] = ((csum + c1) + c2) + c3;
            }
        }
    }
}

// Scales of a block's rows: as float2 (s, z*s), or as stored (fp16 scale, uint8
// zero) when p.sz_compact.  Warp w takes rows w, w + 8, ..., four rows' loads in
// flight per lane.
static __device__ __noinline__ void stage_scales(const GemvParams &p, uint8_t *szb, int row0, int rows_valid)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ng = p.ng;
    for (int r = warp; r < rows_valid; r += 4 * kWarps) {
        for (int g = lane; g < ng; g += 32) {
            uint16_t sv[4];
            uint8_t zv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int rr = r + u * kWarps;
                sv[u] = 0;
                zv[u] = static_cast<uint8_t>(p.zero_const);
                if (rr < rows_valid) {
                    const long long off = static_cast<long long>(row0 + rr) * ng + g;
                    sv[u] = p.scales[off];
                    if (p.zeros)
                        zv[u] = p.zeros[off];
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int rr = r + u * kWarps;
                if (rr < rows_valid) {
                    const int o = rr * p.sz_pitch + g;
                    if (p.sz_compact) {
                        reinterpret_cast<uint16_t *>(szb)[o] = sv[u];
                        if (p.zeros)
                            szb[p.rbp * p.sz_pitch * 2 + o] = zv[u];
                    } else {
                        const float sf = f16_bits_to_f32(sv[u]);
                        reinterpret_cast<float2 *>(szb)[o] = make_float2(sf, static_cast<float>(zv[u]) * sf);
                    }
                }
            }
        }
    }
}

// Issues pipeline stage `it` (K segment s of row block blk) into ring slot
// `slot`, completing on full[slot]: one tensor copy of rb rows x pitch bytes
// (p.tma; bytes past a row's end arrive as zeros, rows past the CTA's are the
// next CTA's or zeros and are not used), else one bulk copy per row.  Called
// by a whole warp.  Without 16-byte aligned rows the warp copies with 4-byte
// loads.
static __device__ __noinline__ void issue_stage(const GemvParams &p, int it, int slot, uint8_t *ring,
                                            uint64_t *full, int r0, int nrows, uint64_t policy)
{
    const int lane = threadIdx.x & 31;
    const int blk = it / p.stages_per_block;
    const int s = it - blk * p.stages_per_block;
    const int row0 = r0 + blk * p.rb;
    const int rows_here = min(p.rb, r0 + nrows - row0);
    const long long seg_off = static_cast<long long>(s) * p.seg_bytes;
    const int seg_len = static_cast<int>(min(static_cast<long long>(p.seg_bytes), p.row_bytes - seg_off));
    uint8_t *dst = ring + static_cast<size_t>(slot) * p.stage_bytes;
    const uint8_t *src = p.packed + static_cast<long long>(row0) * p.row_bytes + seg_off;
    if (p.tma && (smem_u32(dst) & 127u) == 0) {   // a tensor copy lands on 128 bytes
        if (lane == 0) {
            mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(p.rb * p.pitch));
            tma_load_2d_hint(dst, &p.tmw, &full[slot], static_cast<int>(seg_off >> 3), row0, policy);
        }
        __syncwarp();
    } else if (p.use_bulk) {
        if (lane == 0)
            mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(rows_here * seg_len));
        __syncwarp();
#pragma unroll 1
        for (int r = lane; r < rows_here; r += 32)
            bulk_load_hint(dst + r * p.pitch, src + static_cast<long long>(r) * p.row_bytes, seg_len,
                           &full[slot], policy);
    } else {
        // rows one after another, the warp's lanes along the row
        const int words = seg_len / 4;
#pragma unroll 1
        for (int r = 0; r < rows_here; ++r) {
            const uint32_t *srow = reinterpret_cast<const uint32_t *>(src + static_cast<long long>(r) * p.row_bytes);
            uint32_t *drow = reinterpret_cast<uint32_t *>(dst + r * p.pitch);
#pragma unroll 1
            for (int wo = lane; wo < words; wo += 32)
                drow[wo] = srow[wo];
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&full[slot]);
    }
}

template <int B, int NT, int R, int MODE>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 2 : 1)
skinny_kernel(const __grid_constant__ GemvParams p)
{
    constexpr int MP = 8 * NT;                 // padded token count of the D fragments
    constexpr int NGC = 128 / (4 * R);         // groups per 128-code chunk
    constexpr bool FLIP8 = (MODE == 1);
    constexpr int TPW = kTilesPerWarp;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                                ~static_cast<uintptr_t>(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    int *done_count = reinterpret_cast<int *>(full + p.ring);       // warps done per slot (monotonic)
    uint16_t *xp = reinterpret_cast<uint16_t *>(smem + p.off_x);   // [chunk][group][M][4][R]
    float *xs = reinterpret_cast<float *>(smem + p.off_xs);        // [group][MP] sum x
    float *cs = reinterpret_cast<float *>(smem + p.off_cs);        // [group][MP] sum 2^E x
    uint8_t *szb = smem + p.off_sz;   // scales: float2 (s, z*s) or fp16 + uint8 zeros, [row][sz_pitch]
    const float2 *sz2 = reinterpret_cast<const float2 *>(szb);
    const uint16_t *s16 = reinterpret_cast<const uint16_t *>(szb);
    const uint8_t *z8 = szb + p.rbp * p.sz_pitch * 2;
    float *red = reinterpret_cast<float *>(smem + p.off_red);      // [ksplit][rbp][MP]
    uint8_t *ring = smem + p.off_ring;

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
            done_count[i] = 0;
        }
        fence_barrier_init();
    }
    __syncthreads();
    // the next kernel on the stream may start now; it reads nothing that this
    // one writes before its own griddepcontrol.wait
    if (threadIdx.x == 0)
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- before the dependency wait: weights and scales (not written by the
    // preceding kernel) ----
    const uint64_t policy = l2_evict_first_policy();   // the bitstream is read once
    if (warp == 0) {
        const int first = min(p.ring, total_stages);
        for (int it = 0; it < first; ++it)
            issue_stage(p, it, it, ring, full, r0, nrows, policy);
    }
    stage_scales(p, szb, r0, min(p.rb, nrows));

    // ---- the activations may come from the preceding kernel ----
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int ksplit = 1 << p.ksplit_log2;
    const int kid = warp & (ksplit - 1);          // K split: chunks = kid (mod ksplit)
    const int tg = warp >> p.ksplit_log2;         // tile group: tiles tg, tg + ntg
    const int ntg = kWarps >> p.ksplit_log2;
    const int g = lane >> 2, t = lane & 3;
    const int M = p.M;
    const int ng = p.ng;
    // activation fragments of token g + 8 nt and quad thread t: R slots at
    // xp[(chunk * NGC + group) * M * 4 R + xlane[nt]], 16-byte chunks swizzled by
    // xswz[nt]; tokens past M read token M - 1 (their accumulator columns are never
    // stored)
    const int gstride = M * 4 * R;
    int xlane[NT], xswz[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int i = min(g + 8 * nt, M - 1) * 4 + t;
        xlane[nt] = i * R;
        xswz[nt] = act_swizzle<R>(i);
    }

    bool ok = true;
    int it = 0;                 // pipeline stage, and its slot and phase parity
    int slot = 0;
    uint32_t parity = 0;
    for (int blk = 0; blk < nblocks; ++blk) {
        const int row0 = r0 + blk * p.rb;
        const int rows_valid = min(p.rb, r0 + nrows - row0);
        const int T = (rows_valid + 15) / 16;

        if (blk > 0) {
            __syncthreads();   // the previous block's epilogue is done with sz / red
            stage_scales(p, szb, row0, rows_valid);
            __syncthreads();
        }

        float tot[TPW][NT][4];
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    tot[i][nt][e] = 0.f;

        // this warp's tiles (tg, tg + ntg) and their row offsets in a stage and in sz
        const int ntl = (tg < T ? 1 : 0) + (tg + ntg < T ? 1 : 0);
        // rows past the block's end read row rb - 1 (in the slot); their results are dropped
        int roff[TPW][2], szo[TPW][2];
#pragma unroll
        for (int i = 0; i < TPW; ++i)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int lr = min((tg + i * ntg) * 16 + g + 8 * h, p.rb - 1);
                roff[i][h] = lr * p.pitch;
                szo[i][h] = lr * p.sz_pitch;
            }

        // activations: staged at the first stage of block 0, or per phase of every
        // block when they are staged in K phases
        int cur_phase = (p.nphases == 1 && blk > 0) ? 0 : -1;
        int phase = 0, phase_end = p.phase_chunks;
        for (int s = 0; s < p.stages_per_block; ++s, ++it) {
            while (s * p.seg_chunks >= phase_end) {
                ++phase;
                phase_end += p.phase_chunks;
            }
            if (phase != cur_phase) {
                __syncthreads();   // everyone is done with the previous phase
                const int ch0 = phase * p.phase_chunks;
                stage_activations<B, R, MODE, MP>(p, xp, xs, cs, ch0, min(p.phase_chunks, p.nchunks - ch0));
                __syncthreads();
                cur_phase = phase;
            }
            if (ok)
                ok = mbar_wait(&full[slot], parity, p.status);
            if (ok) {
                const uint8_t *stage = ring + static_cast<size_t>(slot) * p.stage_bytes;
                // this warp's chunks of the stage: cg = kid (mod ksplit)
                const int cg_first = s * p.seg_chunks + ((kid - s * p.seg_chunks) & (ksplit - 1));
                const int cg_end = min((s + 1) * p.seg_chunks, p.nchunks);
                // NTL = this warp's tiles in the block (1 or 2), a compile-time count
                auto run_chunks = [&](auto ntl_c) {
                    constexpr int NTL = decltype(ntl_c)::value;
#pragma unroll 1
                    for (int cg = cg_first; cg < cg_end; cg += ksplit) {
                        const int ci = cg - s * p.seg_chunks;
                        const int lc = cg - phase * p.phase_chunks;   // chunk within the phase
#pragma unroll 1
                        for (int gi = 0; gi < NGC; ++gi) {
                            const int grp = cg * NGC + gi;
                            if (grp >= ng)
                                break;
                            const int lg = lc * NGC + gi;
                            const uint16_t *xg = xp + (lc * NGC + gi) * gstride;
                            // activation fragments of the R/4 MMAs, shared by the tiles
                            [[maybe_unused]] uint32_t bf[NT <= 2 ? R / 4 : 1][NT <= 2 ? NT : 1][2];
                            if constexpr (NT <= 2) {
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                                    for (int j = 0; j < R / 4; j += 2) {
                                        const uint4 v = *reinterpret_cast<const uint4 *>(xg + xlane[nt] + 8 * ((j >> 1) ^ xswz[nt]));
                                        bf[j][nt][0] = v.x;
                                        bf[j][nt][1] = v.y;
                                        bf[j + 1][nt][0] = v.z;
                                        bf[j + 1][nt][1] = v.w;
                                    }
                            }
                            float2 xv[NT];
                            [[maybe_unused]] float2 cv[NT];   // MODE 0 only
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                xv[nt] = *reinterpret_cast<const float2 *>(xs + lg * MP + 8 * nt + 2 * t);
                                if constexpr (MODE == 0)
                                    cv[nt] = *reinterpret_cast<const float2 *>(cs + lg * MP + 8 * nt + 2 * t);
                            }
                            const int code0 = ci * 128 + gi * 4 * R + t * R;   // within the stage row
                            // raw words and scales of every tile first, so their loads overlap
                            uint32_t w[NTL][2][(R * B + 31) / 32];
                            float sc[NTL][2], zs[NTL][2];
#pragma unroll
                            for (int i = 0; i < NTL; ++i)
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    load_run<B, R>(stage + roff[i][h], code0, w[i][h]);
                                    const int so = szo[i][h] + grp;
                                    if constexpr (NT >= 2) {   // staged as stored (p.sz_compact)
                                        sc[i][h] = f16_bits_to_f32(s16[so]);
                                        zs[i][h] = (p.zeros ? static_cast<float>(z8[so]) : static_cast<float>(p.zero_const)) * sc[i][h];
                                    } else {
                                        const float2 v = sz2[so];
                                        sc[i][h] = v.x;
                                        zs[i][h] = v.y;
                                    }
                                }
                            uint32_t a0[NTL][R / 2], a1[NTL][R / 2];
#pragma unroll
                            for (int i = 0; i < NTL; ++i) {
                                extract_run<B, R, FLIP8, MODE == 1>(w[i][0], a0[i]);
                                extract_run<B, R, FLIP8, MODE == 1>(w[i][1], a1[i]);
                            }
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                // per tile two independent accumulator chains (even / odd j),
                                // the tiles' MMAs interleaved
                                float d[NTL][2][4];
#pragma unroll
                                for (int i = 0; i < NTL; ++i)
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        d[i][0][e] = d[i][1][e] = 0.f;
                                uint4 bv = make_uint4(0u, 0u, 0u, 0u);   // NT > 2: chunk of j, j + 1
#pragma unroll
                                for (int j = 0; j < R / 4; ++j) {
                                    uint32_t b0, b1;
                                    if constexpr (NT <= 2) {
                                        b0 = bf[j][nt][0];
                                        b1 = bf[j][nt][1];
                                    } else {
                                        if ((j & 1) == 0)
                                            bv = *reinterpret_cast<const uint4 *>(xg + xlane[nt] + 8 * ((j >> 1) ^ xswz[nt]));
                                        b0 = (j & 1) ? bv.z : bv.x;
                                        b1 = (j & 1) ? bv.w : bv.y;
                                    }
#pragma unroll
                                    for (int i = 0; i < NTL; ++i)
                                        mma_f16_16816(d[i][j & 1], a0[i][2 * j], a1[i][2 * j], a0[i][2 * j + 1],
                                                      a1[i][2 * j + 1], b0, b1);
                                }
#pragma unroll
                                for (int i = 0; i < NTL; ++i) {
                                    float dd[4];
#pragma unroll
                                    for (int e = 0; e < 4; ++e)
                                        dd[e] = d[i][0][e] + d[i][1][e];
                                    if constexpr (MODE == 0) {
                                        // the products carried 2^E x as well
                                        dd[0] -= cv[nt].x;
                                        dd[1] -= cv[nt].y;
                                        dd[2] -= cv[nt].x;
                                        dd[3] -= cv[nt].y;
                                        tot[i][nt][0] = fmaf(-zs[i][0], xv[nt].x, fmaf(sc[i][0], dd[0], tot[i][nt][0]));
                                        tot[i][nt][1] = fmaf(-zs[i][0], xv[nt].y, fmaf(sc[i][0], dd[1], tot[i][nt][1]));
                                        tot[i][nt][2] = fmaf(-zs[i][1], xv[nt].x, fmaf(sc[i][1], dd[2], tot[i][nt][2]));
                                        tot[i][nt][3] = fmaf(-zs[i][1], xv[nt].y, fmaf(sc[i][1], dd[3], tot[i][nt][3]));
                                    } else {
                                        // exact integers: d and 2^(B-1) X are below 2^24
                                        constexpr float kOff = static_cast<float>(1 << (B - 1));
                                        const float acc0 = dd[0] - kOff * xv[nt].x, acc1 = dd[1] - kOff * xv[nt].y;
                                        const float acc2 = dd[2] - kOff * xv[nt].x, acc3 = dd[3] - kOff * xv[nt].y;
                                        tot[i][nt][0] = fmaf(sc[i][0], acc0, tot[i][nt][0]);
                                        tot[i][nt][1] = fmaf(sc[i][0], acc1, tot[i][nt][1]);
                                        tot[i][nt][2] = fmaf(sc[i][1], acc2, tot[i][nt][2]);
                                        tot[i][nt][3] = fmaf(sc[i][1], acc3, tot[i][nt][3]);
                                        if (p.acc_out) {
                                            const int lr0 = (tg + i * ntg) * 16 + g;
                                            const int tok = 8 * nt + 2 * t;
                                            const int n0 = row0 + lr0;
                                            const bool v0 = lr0 < rows_valid, v1 = lr0 + 8 < rows_valid;
                                            const long long base0 = static_cast<long long>(n0) * ng + grp;
                                            const long long base1 = static_cast<long long>(n0 + 8) * ng + grp;
                                            const long long tstride = static_cast<long long>(p.N) * ng;
                                            if (v0 && tok < M) p.acc_out[tok * tstride + base0] = static_cast<int>(acc0);
                                            if (v0 && tok + 1 < M) p.acc_out[(tok + 1) * tstride + base0] = static_cast<int>(acc1);
                                            if (v1 && tok < M) p.acc_out[tok * tstride + base1] = static_cast<int>(acc2);
                                            if (v1 && tok + 1 < M) p.acc_out[(tok + 1) * tstride + base1] = static_cast<int>(acc3);
                                        }
                                    }
                                }
                            }
                        }
                    }
                };
                if (ntl == 2)
                    run_chunks(std::integral_constant<int, 2>{});
                else if (ntl == 1)
                    run_chunks(std::integral_constant<int, 1>{});
            }
            // The last warp done with this slot refills it with stage it + ring.
            if (it + p.ring < total_stages) {
                __syncwarp();
                int last = 0;
                if (lane == 0) {
                    __threadfence_block();
                    last = (atomicAdd(&done_count[slot], 1) % kWarps) == kWarps - 1;
                    __threadfence_block();
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    // the other warps' reads of the slot come before the copy's writes
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue_stage(p, it + p.ring, slot, ring, full, r0, nrows, policy);
                }
            }
            if (++slot == p.ring) {
                slot = 0;
                parity ^= 1u;
            }
        }

        // ---- cross-warp reduction in a fixed order, then the store ----
        if (p.red_alias)
            __syncthreads();   // every warp is done reading the activations it overwrites
#pragma unroll
        for (int i = 0; i < TPW; ++i) {
            const int mt = tg + i * ntg;
            if (mt < T) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int row = mt * 16 + g;
                    const int tok = 8 * nt + 2 * t;
                    *reinterpret_cast<float2 *>(red + (kid * p.rbp + row) * MP + tok) =
                        make_float2(tot[i][nt][0], tot[i][nt][1]);
                    *reinterpret_cast<float2 *>(red + (kid * p.rbp + row + 8) * MP + tok) =
                        make_float2(tot[i][nt][2], tot[i][nt][3]);
                }
            }
        }
        __syncthreads();
#pragma unroll 1
        for (int idx = threadIdx.x; idx < rows_valid * MP; idx += kThreads) {
            const int tok = idx & (MP - 1);
            const int row = idx / MP;   // MP is a power of two
            if (tok >= M)
                continue;
            float v = 0.f;
#pragma unroll 1
            for (int w = 0; w < ksplit; ++w)
                v += red[(w * p.rbp + row) * MP + tok];
            if constexpr (MODE == 1)
                v *= f16_bits_to_f32(p.sa[tok]);
            const long long o = static_cast<long long>(tok) * p.N + row0 + row;
            if (p.y_bf16)
                reinterpret_cast<uint16_t *>(p.y)[o] = f32_to_bf16_bits(v);
            else
                reinterpret_cast<uint16_t *>(p.y)[o] = f32_to_f16_bits(v);
        }
    }

    // After a timed-out wait some copies may not have been waited for: none may
    // still be landing in shared memory when the CTA exits.
    __syncthreads();
    if (!ok && threadIdx.x == 0) {
        const int first = total_stages > p.ring ? total_stages - p.ring : 0;
        for (int j = first; j < total_stages; ++j)
            if (!mbar_wait(&full[j % p.ring], (j / p.ring) & 1, p.status))
                break;
    }
}

// ---- host-side launch of one instantiation ----------------------------------------------
template <int B, int NT, int R, int MODE>
cudaError_t launch_skinny(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    auto kern = skinny_kernel<B, NT, R, MODE>;
    static SmemLimit limit;
    if (const cudaError_t e = ensure_smem_limit(limit, kern, smem, true); e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess)
        return e;
    return cudaGetLastError();
}

template <int B, int MODE>
cudaError_t launch_skinny_width(const GemvParams &p, int grid, int smem, cudaStream_t stream)
{
    const int nt = p.M <= 8 ? 1 : p.M <= 16 ? 2 : p.M <= 32 ? 4 : 8;   // as skinny_plan
#define QMM_R(NTV)                                                                          \
    switch (p.group) {                                                                      \
    case 32: return launch_skinny<B, NTV, 8, MODE>(p, grid, smem, stream);            \
    case 64: return launch_skinny<B, NTV, 16, MODE>(p, grid, smem, stream);           \
    default: return launch_skinny<B, NTV, 32, MODE>(p, grid, smem, stream);           \
    }
    if (nt <= 1) { QMM_R(1) }
    if (nt <= 2) { QMM_R(2) }
    if constexpr (MODE == 1) {
        if (nt <= 4) { QMM_R(4) }
        QMM_R(8)
    }
#undef QMM_R
    return cudaErrorInvalidValue;
}

}  // namespace qmm
