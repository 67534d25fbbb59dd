// gemm.cuh -- tiled quantized matmul for M >= 17 on the 5th-generation tensor
// cores (tcgen05, sm_103a).
//
//   y[m][n] = sum_k x[m][k] * W[n][k],   W[n][k] = (q[n][k] - z) * s[n][k/G]
//
// This is the dense-contraction regime: every dequantized weight is reused by
// up to 256 tokens, so the kernel dequantizes each weight tile once into shared
// memory and feeds tcgen05 MMAs that accumulate in tensor memory (TMEM).
//
// Tiles.  A CTA owns kBN = 192 weight columns (the MMA's N; 150 tiles cover
// N = 28672 in one wave on 152 SMs) and walks the tokens in passes of MT
// 128-token M tiles, one TMEM accumulator each (MT = 2 for M > 128, MT = 1 with
// a deeper pipeline for M <= 128).  Per 64-wide K step: the x tiles (A operand,
// K-major, 128-byte swizzle) and, every four K steps, a 192 x 256-code
// packed-weight tile arrive by TMA; twelve dequant warps (two threads per
// weight column) turn 64 codes into bf16/fp16 (q - z) * s and write them in the
// same canonical K-major swizzled layout (B operand); one thread issues
// 4 x MT MMAs of K = 16; four epilogue warps move the accumulators TMEM ->
// registers -> global memory.  The roles meet on mbarriers; every wait is
// bounded and reports QMM_ERR_TIMEOUT.
#pragma once

#include <cstring>

#include "common.cuh"
#include "gemm.h"

namespace qmm {

namespace {

constexpr int kBN = 192;           // weight columns per tile (MMA N)
constexpr int kBM = 128;           // tokens per M tile (MMA M)
constexpr int kBK = 64;            // K per step: one 128-byte swizzle atom of 16-bit values
// Packed-weight stages.  Widths 1, 2, 4, 8: a 128-byte box per row (16 / b K
// steps), 128-byte swizzled so that the dequant threads' reads of 32 rows are
// free of bank conflicts.  Widths 3, 5, 6, 7: two K steps, 16 b bytes per row,
// unswizzled (a 128-byte box is not a whole number of K steps).
__host__ __device__ constexpr bool w_swizzled(int b) { return b == 1 || b == 2 || b == 4 || b == 8; }
__host__ __device__ constexpr int w_ksteps(int b) { return w_swizzled(b) ? 16 / b : 2; }   // K steps per stage
__host__ __device__ constexpr int w_box(int b) { return w_ksteps(b) * 8 * b; }             // bytes per row
constexpr int kWStages = 2;
constexpr int kAccCols = 256;      // TMEM column stride between the accumulators
constexpr int kTmemCols = 512;

constexpr int kEpiWarps = 4;       // warps 0..3: epilogue, TMEM lane quarter = warp id
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kDeqWarp0 = 6;       // warps 6..: dequant, kDeqPerCol threads per tile column
constexpr int kDeqPerCol = 2;      // each takes 64 / kDeqPerCol codes of every 64
constexpr int kDeqWords = 8 / kDeqPerCol;
constexpr int kDeqWarps = kDeqPerCol * kBN / 32;
constexpr int kThreads = 32 * (kDeqWarp0 + kDeqWarps);

constexpr int kXTileBytes = kBM * kBK * 2;     // 16 KB
constexpr int kWTileBytes = kBN * 128;          // 24 KB: the largest stage (w_box <= 128)
constexpr int kBTileBytes = kBN * kBK * 2;      // 24 KB

// Shared-memory layout of one configuration: MT accumulators (128-token M
// tiles) per pass and S stages of x tiles and of B tiles (x and B stages share
// their empty barriers, so they advance together).  Two configurations exist:
// <2, 3> for M > 128, and <1, 4> for M <= 128, which spends the room of the
// unused second x tile on a fourth stage.
template <int MT, int S>
struct Layout {
    static constexpr int kOffX = 0;
    static constexpr int kOffW = kOffX + S * MT * kXTileBytes;
    static constexpr int kOffB = kOffW + kWStages * kWTileBytes;
    static constexpr int kOffBar = kOffB + S * kBTileBytes;
    // b_full [S], x_empty (= b_empty) [S], w_full / w_empty [kWStages], d_full, d_empty, drain
    static constexpr int kNumBars = 2 * S + 2 * kWStages + 3;
    static constexpr int kOffTmemAddr = kOffBar + kNumBars * 8;
    static constexpr int kBytes = kOffTmemAddr + 16 + 1024;   // + alignment slack
};
static_assert(Layout<2, 3>::kBytes <= 227 * 1024 && Layout<1, 4>::kBytes <= 227 * 1024,
              "shared memory per CTA");



// ---- tcgen05 / TMEM helpers -------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16, one CTA
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on `bar` once all previously issued tcgen05 MMAs of this thread are done
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile with the 128-byte swizzle:
// rows of 128 bytes, 8-row atoms of 1024 bytes (the stride between atoms).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);        // start address
    d |= static_cast<uint64_t>(1) << 16;                       // leading byte offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;               // stride byte offset: 8-row atom
    d |= static_cast<uint64_t>(1) << 46;                       // descriptor version (tcgen05)
    d |= static_cast<uint64_t>(2) << 61;                       // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16, fp32 accumulator, A and B K-major.
__host__ __device__ constexpr uint32_t f16_idesc(bool bf16, int m, int n)
{
    return (1u << 4)                                           // D = f32
           | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) // A, B = bf16 or f16
           | (static_cast<uint32_t>(n >> 3) << 17)             // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);            // M / 16
}

__device__ __forceinline__ uint32_t sub2(uint32_t a, uint32_t b, bool bf16)
{
    uint32_t d;
    if (bf16)
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else
        asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b, bool bf16)
{
    uint32_t d;
    if (bf16)
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t fma2_bf16(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// fp32 -> two 16-bit values packed (lo = a)
__device__ __forceinline__ uint32_t pack2(float a, float b, bool bf16)
{
    uint32_t d;
    if (bf16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(b), "f"(a));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(b), "f"(a));
    return d;
}

// scale and (2^E + z) of one group as packed 16-bit pairs.  For bf16 the fp16
// scale is split s = s_hi + s_lo with both parts exact in bf16 (s_hi = the
// scale rounded to 8 significant bits, s_lo = the remaining <= 4 bits), so that
// (q - z) * s_lo is exact and one bf16 FMA rounds the exact product once.
// bf16 holds every integer up to 256 but not the odd ones above, so 128 + z is
// exact only for z <= 128.  For larger zeros the subtraction goes in two exact
// steps: 128 + min(z, 128) first (leaving q - min(z, 128), at most 128 in
// magnitude), then the rest z - 128 (the result |q - z| <= 255 is exact).
struct GroupConst {
    uint32_t s2;      // fp16: s;  bf16: s_hi
    uint32_t slo2;    // bf16: s_lo
    uint32_t off2;
    uint32_t zrest2;  // bf16 with zsplit: max(z - 128, 0), else 0
};

// Scales and zeros of eight consecutive groups 8w .. 8w + 7 of one column, held
// in registers.  Where the rows allow it one 16-byte load (and one 8-byte load
// of the zeros) fetches the window: a warp's 32 columns are 32 different rows,
// so scattered 2-byte loads would cost the L1 data pipe one wavefront per
// column per group, the same pipe the B-tile stores use.
struct ScaleWindow {
    uint4 s;   // fp16 scale of group 8w + i in half (i & 1) of word i / 2
    uint2 z;   // zero of group 8w + i in byte (i & 3) of word i / 4
};

__device__ __forceinline__ void load_window(const GemmParams &p, int n, int w, ScaleWindow &r)
{
    const int g0 = 8 * w;
    const uint32_t zc = static_cast<uint32_t>(p.zero_const) * 0x01010101u;
    r.s = make_uint4(0u, 0u, 0u, 0u);
    r.z = make_uint2(zc, zc);
    if (n >= p.N || g0 >= p.ng)
        return;
    const long long base = static_cast<long long>(n) * p.ng + g0;
    if (p.vec_scales) {   // 16-byte aligned rows, ng % 8 == 0: the window lies inside the row
        r.s = *reinterpret_cast<const uint4 *>(p.scales + base);
        if (p.zeros)
            r.z = *reinterpret_cast<const uint2 *>(p.zeros + base);
        return;
    }
    uint32_t sw[4] = {0u, 0u, 0u, 0u};
    uint32_t zw[2] = {zc, zc};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (g0 + i >= p.ng)
            break;
        sw[i >> 1] |= static_cast<uint32_t>(p.scales[base + i]) << (16 * (i & 1));
        if (p.zeros) {
            const int sh = 8 * (i & 3);
            zw[i >> 2] = (zw[i >> 2] & ~(0xFFu << sh)) | (static_cast<uint32_t>(p.zeros[base + i]) << sh);
        }
    }
    r.s = make_uint4(sw[0], sw[1], sw[2], sw[3]);
    r.z = make_uint2(zw[0], zw[1]);
}

__device__ __forceinline__ uint16_t window_scale(const ScaleWindow &w, int i)
{
    const uint32_t a = (i & 4) ? ((i & 2) ? w.s.w : w.s.z) : ((i & 2) ? w.s.y : w.s.x);
    return static_cast<uint16_t>((i & 1) ? (a >> 16) : (a & 0xFFFFu));
}

__device__ __forceinline__ uint8_t window_zero(const ScaleWindow &w, int i)
{
    const uint32_t a = (i & 4) ? w.z.y : w.z.x;
    return static_cast<uint8_t>(a >> (8 * (i & 3)));
}

__device__ __forceinline__ GroupConst group_const(uint16_t s_bits, uint8_t z, bool bf16)
{
    GroupConst c;
    const float s = f16_bits_to_f32(s_bits);
    c.s2 = pack2(s, s, bf16);
    c.slo2 = 0;
    c.zrest2 = 0;
    if (bf16) {
        const float s_hi = __uint_as_float((c.s2 & 0xFFFFu) << 16);
        const float s_lo = s - s_hi;                              // exact in fp32 and in bf16
        c.slo2 = pack2(s_lo, s_lo, true);
        const float rest = static_cast<float>(z > 128 ? z - 128 : 0);
        c.zrest2 = pack2(rest, rest, true);
        z = z > 128 ? 128 : z;
    }
    const float off = (bf16 ? 128.f : 1024.f) + static_cast<float>(z);   // exact in 16 bits
    c.off2 = pack2(off, off, bf16);
    return c;
}

// 8 packed 4-bit codes (one word, k = 8i..8i+7) -> four 16-bit pairs (k, k+1),
// each (q - z) * s.  A byte permute puts code 2j in the low half and code 2j+1
// (pre-shifted by 4) in the high half; a LOP3 sets the exponent so each half
// reads 2^E + q; the subtraction is exact and the scaling rounds once.
__device__ __forceinline__ void dequant_word4(uint32_t w, const GroupConst &c, bool bf16, bool zsplit,
                                              uint32_t (&o)[4])
{
    const uint32_t hi = w >> 4;
    const uint32_t magic = bf16 ? 0x43004300u : 0x64006400u;   // 128.0 / 1024.0
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t sel = static_cast<uint32_t>(j) | (static_cast<uint32_t>(4 + j) << 8);
        const uint32_t t = prmt(w, hi, sel);
        const uint32_t v = lop3_and_or(t, 0x000F000Fu, magic);
        uint32_t qz = sub2(v, c.off2, bf16);                       // q - min(z, 128), exact
        if (zsplit)
            qz = sub2(qz, c.zrest2, true);                         // q - z, exact
        if (bf16)
            o[j] = fma2_bf16(qz, c.s2, mul2(qz, c.slo2, true));     // one rounding of (q - z) * s
        else
            o[j] = mul2(qz, c.s2, false);                           // one rounding in fp16
    }
}

// Widths other than 4: the fp16 / bf16 pair (2^b + q_c, 2^b + q_{c+1}) of codes
// c, c + 1 (c even) of a 32-code run (b words, code 0 at bit 0 of w[0]).  A
// funnel shift puts code c at the top of the low half's mantissa (MB mantissa
// bits: 10 for fp16, 7 for bf16) and code c + 1 just above it; two LOP3s
// (one after a shift) set each half's exponent to that of 2^b, so each half
// reads exactly 2^b + q.
template <int B, int MB>
__device__ __forceinline__ uint32_t run_pair(const uint32_t (&w)[B], int c)
{
    const int sh = c * B - (MB - B);
    uint32_t u;
    if (sh < 0) {
        u = w[0] << (-sh);
    } else {
        const int i = sh >> 5, s = sh & 31;
        const uint32_t hi = i + 1 < B ? w[i + 1] : 0u;
        u = s == 0 ? w[i] : __funnelshift_r(w[i], hi, s);
    }
    constexpr uint32_t mask = ((1u << B) - 1u) << (MB - B);
    constexpr uint32_t magic = MB == 10 ? static_cast<uint32_t>(B + 15) << 10 : static_cast<uint32_t>(B + 127) << 7;
    const uint32_t lo = lop3_and_or(u, mask, magic | (magic << 16));
    return lop3_and_or(u << (16 - B), mask << 16, lo);
}

// 32 codes of one run (b words) -> 16 pairs (2j, 2j + 1) of (q - z) * s, with
// q - z exact and one rounding by the scale.
template <int B>
__device__ __forceinline__ void dequant_run(const uint32_t (&w)[B], uint16_t s_bits, uint8_t z, bool bf16,
                                            bool zsplit, uint32_t (&o)[16])
{
    if constexpr (B == 4) {
        const GroupConst gc = group_const(s_bits, z, bf16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t q[4];
            dequant_word4(w[i], gc, bf16, zsplit, q);
            o[4 * i] = q[0];
            o[4 * i + 1] = q[1];
            o[4 * i + 2] = q[2];
            o[4 * i + 3] = q[3];
        }
    } else if constexpr (B == 8) {
        const float s = f16_bits_to_f32(s_bits);
        const float off = 1024.f + static_cast<float>(z);   // exact in fp16
        const uint32_t off2 = pack2(off, off, false);
        const uint32_t s2 = pack2(s, s, false);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            // one byte per code under the fp16 exponent byte 0x64: 1024 + q; minus 1024 + z: q - z, exact
            const uint32_t qz = sub2(prmt(w[j >> 1], 0x64646464u, (j & 1) ? 0x4342u : 0x4140u), off2, false);
            if (bf16) {   // (q - z) s is exact in fp32; one rounding to bf16
                o[j] = pack2(f16_bits_to_f32(static_cast<uint16_t>(qz)) * s,
                             f16_bits_to_f32(static_cast<uint16_t>(qz >> 16)) * s, true);
            } else {
                o[j] = mul2(qz, s2, false);
            }
        }
    } else {
        const float s = f16_bits_to_f32(s_bits);
        if (bf16) {
            // 2^b + q and 2^b are bf16 numbers (b <= 7); q - z is exact in bf16 (|q - z| <= 255)
            const uint32_t s2 = pack2(s, s, true);
            const float s_hi = __uint_as_float((s2 & 0xFFFFu) << 16);
            const float s_lo = s - s_hi;                              // exact in bf16
            const uint32_t slo2 = pack2(s_lo, s_lo, true);
            const float p2 = static_cast<float>(1 << B);
            const uint32_t p22 = pack2(p2, p2, true);
            const uint32_t z2 = pack2(static_cast<float>(z), static_cast<float>(z), true);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint32_t qz = sub2(sub2(run_pair<B, 7>(w, 2 * j), p22, true), z2, true);
                o[j] = fma2_bf16(qz, s2, mul2(qz, slo2, true));
            }
        } else {
            const float off = static_cast<float>((1 << B) + z);   // exact in fp16 (< 2048)
            const uint32_t off2 = pack2(off, off, false);
            const uint32_t s2 = pack2(s, s, false);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                o[j] = mul2(sub2(run_pair<B, 10>(w, 2 * j), off2, false), s2, false);
        }
    }
}

template <int B, int MT, int S>
__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
            const GemmParams p)
{
    constexpr int kKPerW = w_ksteps(B);   // K steps per packed-weight stage
    constexpr int kWBytes = kBN * w_box(B);
    constexpr int kMTiles = MT;   // accumulators per pass
    constexpr int kXStages = S;
    constexpr int kBStages = S;
    using L = Layout<MT, S>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    uint8_t *sx = smem + L::kOffX;
    uint8_t *sw = smem + L::kOffW;
    uint8_t *sb = smem + L::kOffB;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    // K step k uses x slot k % 3 and B slot k % 3.  One barrier per slot says both
    // are full (the x tiles' bytes and the dequant warps' arrivals), one that both
    // are free again (one MMA commit per K step).
    uint64_t *b_full = bars;
    uint64_t *x_empty = b_full + kBStages;
    uint64_t *b_empty = x_empty;
    uint64_t *w_full = x_empty + kXStages;
    uint64_t *w_empty = w_full + kWStages;
    uint64_t *d_full = w_empty + kWStages;
    uint64_t *d_empty = d_full + 1;
    uint64_t *drain = d_empty + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffTmemAddr);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool bf16 = p.bf16 != 0;
    const bool zsplit = p.zsplit != 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kXStages; ++i)
            mbar_init(&x_empty[i], 1);
        for (int i = 0; i < kWStages; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], kDeqWarps);
        }
        for (int i = 0; i < kBStages; ++i) {
            // the dequant warps' arrivals plus the producer's (with the x tiles' bytes)
            mbar_init(&b_full[i], kDeqWarps + 1);
        }
        mbar_init(d_full, 1);
        mbar_init(d_empty, kEpiWarps);
        mbar_init(drain, 1);
        fence_barrier_init();
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    if (warp == kMmaWarp)
        tmem_alloc(tmem_slot, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int nks = p.ksteps;
    bool ok = true;

    if (warp == kProdWarp) {
        // ================= TMA producer =================
        if (lane == 0) {
            prefetch_tmap(&tmx);
            prefetch_tmap(&tmw);
            int xi = 0, wi = 0;
            for (int tile = blockIdx.x; tile < p.tiles_n && ok; tile += gridDim.x) {
                const int n0 = tile * kBN;
                for (int pass = 0; pass < p.passes && ok; ++pass) {
                    const int mt0 = pass * kMTiles;
                    const int cnt = min(kMTiles, p.mtiles - mt0);
                    for (int ks = 0; ks < nks && ok; ++ks) {
                        if (ks % kKPerW == 0) {
                            const int slot = wi % kWStages, round = wi / kWStages;
                            if (round > 0 && !(ok = mbar_wait(&w_empty[slot], (round - 1) & 1, p.status)))
                                break;
                            mbar_arrive_expect_tx(&w_full[slot], kWBytes);
                            tma_load_2d(sw + slot * kWTileBytes, &tmw, &w_full[slot], ks * 8 * B, n0);
                            ++wi;
                        }
                        const int slot = xi % kXStages, round = xi / kXStages;
                        if (round > 0 && !(ok = mbar_wait(&x_empty[slot], (round - 1) & 1, p.status)))
                            break;
                        mbar_arrive_expect_tx(&b_full[slot], cnt * kXTileBytes);
                        for (int j = 0; j < cnt; ++j)
                            tma_load_2d(sx + (slot * kMTiles + j) * kXTileBytes, &tmx, &b_full[slot], ks * kBK,
                                        (mt0 + j) * kBM);
                        ++xi;
                    }
                }
            }
            // drain: the last copies into shared memory have landed
            for (int i = max(0, xi - kXStages); i < xi; ++i)
                if (!mbar_wait(&b_full[i % kXStages], (i / kXStages) & 1, p.status))
                    break;
            for (int i = max(0, wi - kWStages); i < wi; ++i)
                if (!mbar_wait(&w_full[i % kWStages], (i / kWStages) & 1, p.status))
                    break;
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ================= MMA issuer =================
        if (lane == 0) {
            const uint32_t idesc = f16_idesc(bf16, kBM, kBN);
            // operand descriptors of slot 0, built once; the start-address field
            // (bits 0..13, in 16-byte units; shared memory stays below 2^18 bytes) is
            // advanced by the slot's offset and, per 16-wide K step, by 32 bytes (+2)
            const uint64_t a_desc0 = sw128_desc(smem_u32(sx));
            const uint64_t b_desc0 = sw128_desc(smem_u32(sb));
            int slot = 0, np = 0;       // x and B stage slot (they advance together)
            uint32_t parity = 0;
            for (int tile = blockIdx.x; tile < p.tiles_n && ok; tile += gridDim.x) {
                for (int pass = 0; pass < p.passes && ok; ++pass) {
                    const int cnt = min(kMTiles, p.mtiles - pass * kMTiles);
                    if (np > 0 && !(ok = mbar_wait(d_empty, (np - 1) & 1, p.status)))
                        break;
                    tc_fence_after();
                    for (int ks = 0; ks < nks && ok; ++ks) {
                        // x tiles landed and the B tile written: one barrier
                        if (!(ok = mbar_wait(&b_full[slot], parity, p.status)))
                            break;
                        tc_fence_after();
                        const uint32_t acc0 = ks > 0 ? 1u : 0u;
#pragma unroll
                        for (int j = 0; j < kMTiles; ++j) {
                            if (j < cnt) {
#pragma unroll
                                for (int kk = 0; kk < kBK / 16; ++kk)
                                    tc_mma(tmem_base + j * kAccCols,
                                           a_desc0 + (((slot * kMTiles + j) * kXTileBytes) >> 4) + 2 * kk,
                                           b_desc0 + ((slot * kBTileBytes) >> 4) + 2 * kk, idesc, kk > 0 ? 1u : acc0);
                            }
                        }
                        tc_commit(&x_empty[slot]);   // frees x slot and B slot
                        if (++slot == kXStages) {
                            slot = 0;
                            parity ^= 1u;
                        }
                    }
                    if (ok)
                        tc_commit(d_full);
                    ++np;
                }
            }
            // drain: every MMA this thread issued has completed
            tc_commit(drain);
            mbar_wait(drain, 0, p.status);
        }
        __syncwarp();
    } else if (warp >= kDeqWarp0) {
        // ================= dequant: two threads per tile column =================
        // Thread (r, h) turns codes 32h .. 32h + 31 of every 64 of column r into
        // 16-bit values.  Work goes by packed-weight stage (kKPerW K steps,
        // unrolled).  Scales come from a register window of eight groups, the
        // next window loaded one window ahead.
        const int dt = threadIdx.x - 32 * kDeqWarp0;
        const int r = dt % kBN;                         // column
        const int qd = dt / kBN;                        // part of each 64 codes
        const int h = qd * kDeqWords / 4;               // its half (the scale group of 32 codes)
        const int nws = (nks + kKPerW - 1) / kKPerW;
        int wi = 0, bi = 0;
        for (int tile = blockIdx.x; tile < p.tiles_n && ok; tile += gridDim.x) {
            const int n = tile * kBN + r;
            for (int pass = 0; pass < p.passes && ok; ++pass) {
                // group g = (64 ks + 32 h) / G grows by at most 2 per K step (G >= 32),
                // so the window index g / 8 grows by at most one
                ScaleWindow cur, nxt;
                int wcur = 0;
                load_window(p, n, 0, cur);
                load_window(p, n, 1, nxt);
                for (int wsi = 0; wsi < nws && ok; ++wsi) {
                    const int ws = wi % kWStages;
                    if (!(ok = mbar_wait(&w_full[ws], (wi / kWStages) & 1, p.status)))
                        break;
                    const uint8_t *wrow = sw + ws * kWTileBytes + r * w_box(B);
#pragma unroll
                    for (int j = 0; j < kKPerW; ++j) {
                        const int ks = wsi * kKPerW + j;
                        if (ks < nks && ok) {
                            const int bs = bi % kBStages, bround = bi / kBStages;
                            if (bround > 0 && !(ok = mbar_wait(&b_empty[bs], (bround - 1) & 1, p.status)))
                                break;
                            // this part's run of 32 codes: b words at byte (2 j + qd) 4 b of the
                            // row; in a swizzled stage the row is 128 B with its 16-byte chunks
                            // permuted by r & 7
                            uint32_t wv[B];
                            const int ob = (2 * j + qd) * 4 * B;
                            if constexpr (B == 4) {   // one 16-byte chunk
                                const uint4 v = *reinterpret_cast<const uint4 *>(wrow + (((ob >> 4) ^ (r & 7)) << 4));
                                wv[0] = v.x; wv[1] = v.y; wv[2] = v.z; wv[3] = v.w;
                            } else if constexpr (B == 8) {   // two 16-byte chunks
                                const uint4 v0 = *reinterpret_cast<const uint4 *>(wrow + (((ob >> 4) ^ (r & 7)) << 4));
                                const uint4 v1 = *reinterpret_cast<const uint4 *>(wrow + ((((ob >> 4) + 1) ^ (r & 7)) << 4));
                                wv[0] = v0.x; wv[1] = v0.y; wv[2] = v0.z; wv[3] = v0.w;
                                wv[4] = v1.x; wv[5] = v1.y; wv[6] = v1.z; wv[7] = v1.w;
                            } else if constexpr (w_swizzled(B)) {   // 1 or 2 words inside one chunk
#pragma unroll
                                for (int i = 0; i < B; ++i)
                                    wv[i] = *reinterpret_cast<const uint32_t *>(
                                        wrow + ((((ob + 4 * i) >> 4) ^ (r & 7)) << 4) + ((ob + 4 * i) & 15));
                            } else {
#pragma unroll
                                for (int i = 0; i < B; ++i)
                                    wv[i] = *reinterpret_cast<const uint32_t *>(wrow + ob + 4 * i);
                            }
                            const int g = (64 * ks + 32 * h) >> p.group_log2;
                            if ((g >> 3) != wcur) {
                                cur = nxt;
                                ++wcur;
                                load_window(p, n, wcur + 1, nxt);
                            }
                            uint32_t o[16];
                            dequant_run<B>(wv, window_scale(cur, g & 7), window_zero(cur, g & 7), bf16, zsplit, o);
                            uint8_t *brow = sb + bs * kBTileBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                *reinterpret_cast<uint4 *>(brow + (((4 * qd + i) ^ (r & 7)) << 4)) =
                                    make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(&b_full[bs]);
                            ++bi;
                        }
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&w_empty[ws]);
                    ++wi;
                }
            }
        }
    } else {
        // ================= epilogue: warp q reads TMEM lanes 32q..32q+31 =================
        const int q = warp;
        int np = 0;
        for (int tile = blockIdx.x; tile < p.tiles_n && ok; tile += gridDim.x) {
            const int n0 = tile * kBN;
            for (int pass = 0; pass < p.passes && ok; ++pass) {
                const int mt0 = pass * kMTiles;
                const int cnt = min(kMTiles, p.mtiles - mt0);
                if (!(ok = mbar_wait(d_full, np & 1, p.status)))
                    break;
                tc_fence_after();
                for (int j = 0; j < cnt; ++j) {
                    const int m = (mt0 + j) * kBM + q * 32 + lane;
                    for (int c0 = 0; c0 < kBN; c0 += 32) {
                        uint32_t v[32];
                        tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + j * kAccCols + c0, v);
                        if (m < p.M) {
                            uint16_t *yrow = p.y + static_cast<long long>(m) * p.N + n0 + c0;
                            if (n0 + c0 + 32 <= p.N && (p.N % 8) == 0) {
#pragma unroll
                                for (int e = 0; e < 32; e += 8) {
                                    uint4 o;
                                    o.x = pack2(__uint_as_float(v[e]), __uint_as_float(v[e + 1]), bf16);
                                    o.y = pack2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]), bf16);
                                    o.z = pack2(__uint_as_float(v[e + 4]), __uint_as_float(v[e + 5]), bf16);
                                    o.w = pack2(__uint_as_float(v[e + 6]), __uint_as_float(v[e + 7]), bf16);
                                    *reinterpret_cast<uint4 *>(yrow + e) = o;
                                }
                            } else {
                                for (int e = 0; e < 32; ++e)
                                    if (n0 + c0 + e < p.N)
                                        yrow[e] = bf16 ? f32_to_bf16_bits(__uint_as_float(v[e]))
                                                       : f32_to_f16_bits(__uint_as_float(v[e]));
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(d_empty);
                ++np;
            }
        }
    }

    // teardown: every role is done (or gave up); release tensor memory
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp)
        tmem_dealloc(tmem_base, kTmemCols);
}

template <int B, int MT, int S>
qmm_status launch_gemm(const CUtensorMap &tmx, const CUtensorMap &tmw, GemmParams p, int grid,
                       int smem_optin, cudaStream_t stream)
{
    constexpr int smem = Layout<MT, S>::kBytes;
    if (smem_optin < smem)
        return QMM_ERR_UNSUPPORTED;
    p.passes = (p.mtiles + MT - 1) / MT;
    static SmemLimit limit;
    if (ensure_smem_limit(limit, gemm_kernel<B, MT, S>, smem, true) != cudaSuccess)
        return QMM_ERR_CUDA;
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
    if (cudaLaunchKernelEx(&cfg, gemm_kernel<B, MT, S>, tmx, tmw, p) != cudaSuccess)
        return QMM_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

// One width's two configurations (M <= 128: <1, 4>; M > 128: <2, 3>).
template <int B>
qmm_status launch_gemm_width(const CUtensorMap &tmx, const CUtensorMap &tmw, const GemmParams &p, int grid,
                             int smem_optin, cudaStream_t stream)
{
    if (p.mtiles == 1)
        return launch_gemm<B, 1, 4>(tmx, tmw, p, grid, smem_optin, stream);
    return launch_gemm<B, 2, 3>(tmx, tmw, p, grid, smem_optin, stream);
}

}  // namespace

}  // namespace qmm

// Instantiates the launcher of width W (one translation unit per width).
#define QMM_GEMM_WIDTH(W)                                                                              \
    namespace qmm {                                                                                    \
    qmm_status gemm_launch_w##W(const CUtensorMap &tmx, const CUtensorMap &tmw, const GemmParams &p,   \
                                int grid, int smem_optin, cudaStream_t stream)                         \
    {                                                                                                  \
        return launch_gemm_width<W>(tmx, tmw, p, grid, smem_optin, stream);                            \
    }                                                                                                  \
    }
