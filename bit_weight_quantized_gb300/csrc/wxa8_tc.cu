// wxa8_tc.cu -- integer-native W4A8 / W8A8 (BitLLM sec. 4.3-4.4: int8 x intb
// products accumulated exactly per group, dequantization deferred to an
// epilogue) on the 5th-generation tensor cores, for batches of up to 64 tokens.
//
//   acc[m][n][g] = sum_{k in g} xq[m][k] * w[n][k]        (exact)
//   y[m][n]      = sa[m] * sum_g ws[n][g] * acc[m][n][g]
//
// Every operand is an integer of at most 8 bits, exact in fp16, so tcgen05.mma
// kind::f16 computes the products exactly and its fp32 accumulation stays exact
// while a group's sum is below 2^24 (|acc| <= 128 * 128 * 128 = 2^21).  Each
// group accumulates into its own TMEM accumulator; fold warps read it back, write
// the int32 accumulators when asked and add ws * acc into per-row totals.
//
// Shape.  The weights are the MMA's A operand (M = 128 weight rows per CTA), the
// tokens its B operand (N = the batch rounded up to 16).  A cluster of kKSplit
// CTAs shares one row tile and splits K; at the end each CTA sends each quarter
// of its partial totals to the CTA of the cluster that owns that quarter, by a
// bulk copy between shared memories that completes on the receiver's mbarrier,
// and each CTA sums and stores its quarter.  N = 4096 gives 32 row tiles, 128
// CTAs.
//
// Pipeline per 128-code super step: a producer thread loads the packed weights
// (before the dependency wait: they are never the preceding kernel's output)
// and the int8 activations by TMA; eight converter warps turn both into fp16
// (K-major, 128-byte swizzled operand tiles); one thread issues the MMAs; four
// fold warps drain the per-group accumulators.  Every wait is bounded.
#include <cstring>

#include "gemm.cuh"
#include "w4a8.h"

namespace qmm {

namespace {

constexpr int kKSplit = 4;            // CTAs per cluster, splitting K
constexpr int kTRows = 128;           // weight rows per CTA (MMA M)
constexpr int kSuper = 128;           // codes per super step (two 64-code K steps)
constexpr int kRawStages = 3;
constexpr int kOpStages = 2;
constexpr int kAccSlots = 8;          // TMEM accumulators (one per group in flight)
constexpr int kTThreads = 512;        // warps 0-3 fold (TMEM lane quarter = warp), 4 TMA, 5 MMA, 6-15 convert
constexpr int kFoldWarp0 = 0;
constexpr int kTProdWarp = 4;
constexpr int kTMmaWarp = 5;
constexpr int kConvWarp0 = 6;
constexpr int kConvWarps = 10;       // 256 threads for the weights, 64 for the activations
constexpr int kMaxLocalGroups = 32;   // groups of one CTA's K range (scales staged in shared memory)

struct TcParams {
    const uint16_t *sa;     // fp16 [M]
    const uint16_t *ws;     // fp16 [N][K/G]
    uint16_t *y;            // fp16 [M][N]
    int32_t *acc_out;       // int32 [M][N][K/G] or nullptr
    int *status;
    int M, N, K, ng, group, group_log2;
    int vec_ws;             // ws 16-byte aligned, K/G and each CTA's group count multiples of 8
};

// Shared-memory layout for `bits`-bit weights and NP token columns.
template <int BITS, int NP>
struct TcLayout {
    static constexpr int kWRow = kSuper * BITS / 8;                   // packed bytes per row per super step
    static constexpr int kWBytes = kTRows * kWRow;
    static constexpr int kXBytes = NP * 128;                           // int8 tokens x 128 codes
    static constexpr int kRawBytes = kWBytes + ((kXBytes + 1023) / 1024) * 1024;
    static constexpr int kATile = kTRows * 128;                        // fp16 128 rows x 64 codes
    static constexpr int kBTile = ((NP * 128 + 1023) / 1024) * 1024;   // fp16 NP tokens x 64 codes
    static constexpr int kOpBytes = 2 * kATile + 2 * kBTile;
    static constexpr int kOffRaw = 0;
    static constexpr int kOffOp = kOffRaw + kRawStages * kRawBytes;
    static constexpr int kOffWs = kOffOp + kOpStages * kOpBytes;
    static constexpr int kWsBytes = kMaxLocalGroups * kTRows * 2;
    static constexpr int kOffSa = kOffWs + kWsBytes;                  // fp32 [NP] token scales
    static constexpr int kPartBytes = NP * 32 * 4;                     // one quarter's partial totals [NP][32]
    static constexpr int kOffRecv = kOffSa + NP * 4;                   // [kKSplit sources] partials
    static constexpr int kOffBar = kOffRecv + kKSplit * kPartBytes;
    static constexpr int kNumBars = 3 * kRawStages + 2 * kOpStages + 2 * kAccSlots + 2;
    static constexpr int kOffTmem = kOffBar + kNumBars * 8;
    static constexpr int kBytes = kOffTmem + 16;
    static_assert(4 * kPartBytes <= kOpStages * kOpBytes, "the outgoing partials alias the operand stages");
};

__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));   // (a & b) ^ c
    return d;
}

__device__ __forceinline__ uint32_t sub_f16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// 16 consecutive 32-bit TMEM columns of this thread's lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Bulk copy of `bytes` from this CTA's shared memory to the same offset as
// `dst_local` in CTA `rank` of the cluster, completing on that CTA's copy of
// the barrier at `bar_local`.
__device__ __forceinline__ void bulk_to_cluster(const void *dst_local, const void *src, uint32_t bytes,
                                                const uint64_t *bar_local, uint32_t rank)
{
    uint32_t dst, bar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(smem_u32(dst_local)), "r"(rank));
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(bar) : "r"(smem_u32(bar_local)), "r"(rank));
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "r"(smem_u32(src)), "r"(bytes), "r"(bar)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Eight signed int8 values (two words) -> four exact fp16 pairs: the sign bit
// flipped (u = v + 128), each byte put under the exponent byte 0x64 (1024 + u),
// minus 1152.
__device__ __forceinline__ void int8x8_to_f16(uint32_t w0, uint32_t w1, uint32_t (&o)[4])
{
    const uint32_t u0 = w0 ^ 0x80808080u, u1 = w1 ^ 0x80808080u;
    const uint32_t off = 0x64806480u;   // fp16 1152 in both halves
    o[0] = sub_f16x2(prmt(u0, 0x64646464u, 0x5140u), off);
    o[1] = sub_f16x2(prmt(u0, 0x64646464u, 0x5342u), off);
    o[2] = sub_f16x2(prmt(u1, 0x64646464u, 0x5140u), off);
    o[3] = sub_f16x2(prmt(u1, 0x64646464u, 0x5342u), off);
}

// Eight signed int4 codes (one word of the 4-bit stream, code 2j in the low
// nibble of byte j) -> four exact fp16 pairs (code 2j, code 2j + 1): a byte
// permute puts the pair's nibbles in the low nibble of each half, one LOP3
// flips their sign bit under the exponent of 1024 (1024 + (c xor 8)), minus 1032.
__device__ __forceinline__ void int4x8_to_f16(uint32_t w, uint32_t (&o)[4])
{
    const uint32_t hi = w >> 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t sel = static_cast<uint32_t>(j) | (static_cast<uint32_t>(4 + j) << 8);
        o[j] = sub_f16x2(lop3_and_xor(prmt(w, hi, sel), 0x000F000Fu, 0x64086408u), 0x64086408u);
    }
}

// Stores 64 fp16 values (32 words, k order) as row r of a K-major 128-byte
// swizzled tile: 16-byte chunk c of the row at chunk position c ^ (r & 7).
__device__ __forceinline__ void store_row64(uint8_t *tile, int r, const uint32_t (&v)[32])
{
    uint8_t *row = tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(row + ((c ^ (r & 7)) << 4)) =
            make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}

// The eight MMAs of super step i (two 64-code K steps of four k16 MMAs) for
// groups of 2^GLOG2 codes: each group into its own TMEM accumulator slot, the
// slot's accumulator committed to acc_full when the group ends.  The group
// bookkeeping is compile-time; only the super step's first group index is not.
template <int GLOG2, int NP, int ATILE, int BTILE>
__device__ __forceinline__ bool mma_superstep(int i, uint32_t tmem_base, uint64_t desc0, uint32_t a0, uint32_t b0,
                                              uint32_t idesc, uint64_t *acc_full, uint64_t *acc_empty, int *status)
{
    constexpr int G = 1 << GLOG2;
    constexpr int gps = kSuper / G;
#pragma unroll
    for (int hh = 0; hh < 2; ++hh)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int kg = hh * 64 + kk * 16;               // code offset in the super step (compile time)
            const bool first = (kg & (G - 1)) == 0;
            const bool last = ((kg + 16) & (G - 1)) == 0;
            const int gl = i * gps + (kg >> GLOG2);          // local group
            const int slot = gl & (kAccSlots - 1);
            if (first && gl >= kAccSlots) {
                if (!mbar_wait(&acc_empty[slot], ((gl / kAccSlots) - 1) & 1, status))
                    return false;
                tc_fence_after();
            }
            tc_mma(tmem_base + slot * NP, desc0 + a0 + ((hh * ATILE) >> 4) + 2 * kk,
                   desc0 + b0 + ((hh * BTILE) >> 4) + 2 * kk, idesc, first ? 0u : 1u);
            if (last)
                tc_commit(&acc_full[slot]);
        }
    return true;
}

template <int BITS, int NP>
__global__ void __cluster_dims__(kKSplit, 1, 1) __launch_bounds__(kTThreads, 1)
wxa8_tc_kernel(const __grid_constant__ CUtensorMap tmw, const __grid_constant__ CUtensorMap tmx, const TcParams p)
{
    using L = TcLayout<BITS, NP>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled stages, by pointer arithmetic so the
    // compiler keeps the shared state space
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBar);
    uint64_t *w_full = bars;
    uint64_t *x_full = w_full + kRawStages;
    uint64_t *raw_empty = x_full + kRawStages;
    uint64_t *op_full = raw_empty + kRawStages;
    uint64_t *op_empty = op_full + kOpStages;
    uint64_t *acc_full = op_empty + kOpStages;
    uint64_t *acc_empty = acc_full + kAccSlots;
    uint64_t *drain = acc_empty + kAccSlots;
    uint64_t *red_full = drain + 1;   // the four partials of this CTA's quarter have landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::kOffTmem);
    uint16_t *ws_s = reinterpret_cast<uint16_t *>(smem + L::kOffWs);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int tile = blockIdx.x / kKSplit;
    const int n0 = tile * kTRows;
    const int klocal = p.K / kKSplit;
    const int k0 = static_cast<int>(rank) * klocal;
    const int nsuper = klocal / kSuper;
    const int ngl = klocal / p.group;                 // groups of this CTA
    const int gbase = k0 / p.group;

    if (threadIdx.x == 0) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        for (int i = 0; i < kRawStages; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&x_full[i], 1);
            mbar_init(&raw_empty[i], kConvWarps);
        }
        for (int i = 0; i < kOpStages; ++i) {
            mbar_init(&op_full[i], kConvWarps);
            mbar_init(&op_empty[i], 1);
        }
        for (int i = 0; i < kAccSlots; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], 4);
        }
        mbar_init(drain, 1);
        mbar_init(red_full, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(red_full, kKSplit * L::kPartBytes);
    }
    __syncthreads();
    if (warp == kTProdWarp && lane == 0) {
        // weights first, while the rest of the set-up runs: not the preceding kernel's output
        prefetch_tmap(&tmw);
        prefetch_tmap(&tmx);
        const int pre = nsuper < kRawStages ? nsuper : kRawStages;
        for (int i = 0; i < pre; ++i) {
            mbar_arrive_expect_tx(&w_full[i], L::kWBytes);
            tma_load_2d(smem + L::kOffRaw + i * L::kRawBytes, &tmw, &w_full[i], (k0 + i * kSuper) * BITS / 8, n0);
        }
    }
    if (warp == kTMmaWarp)
        tmem_alloc(tmem_slot, 512);
    // this CTA's weight scales, [local group][row]: eight groups of a row per
    // 16-byte load where the rows allow it
    if (p.vec_ws) {
        const int vpr = ngl >> 3;
        for (int e = threadIdx.x; e < vpr * kTRows; e += kTThreads) {
            const int r = e / vpr, c = e - r * vpr;
            const int n = n0 + r;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (n < p.N)
                v = *reinterpret_cast<const uint4 *>(p.ws + static_cast<long long>(n) * p.ng + gbase + 8 * c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 8; ++j)
                ws_s[(8 * c + j) * kTRows + r] = static_cast<uint16_t>(w[j >> 1] >> (16 * (j & 1)));
        }
    } else {
        for (int e = threadIdx.x; e < ngl * kTRows; e += kTThreads) {
            const int g = e / kTRows, r = e - g * kTRows;
            const int n = n0 + r;
            ws_s[e] = n < p.N ? p.ws[static_cast<long long>(n) * p.ng + gbase + g] : static_cast<uint16_t>(0);
        }
    }
    // every CTA of the cluster has its barriers set up before any partial can arrive
    tc_fence_before();
    cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    bool ok = true;

    if (warp == kTProdWarp) {
        // ================= TMA producer =================
        int issued_w = nsuper < kRawStages ? nsuper : kRawStages, issued_x = 0;
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (lane == 0) {
            for (int i = 0; i < nsuper && ok; ++i) {
                const int s = i % kRawStages;
                uint8_t *sw = smem + L::kOffRaw + s * L::kRawBytes;
                if (i >= kRawStages) {
                    if (!(ok = mbar_wait(&raw_empty[s], ((i / kRawStages) - 1) & 1, p.status)))
                        break;
                    mbar_arrive_expect_tx(&w_full[s], L::kWBytes);
                    tma_load_2d(sw, &tmw, &w_full[s], (k0 + i * kSuper) * BITS / 8, n0);
                    issued_w = i + 1;
                }
                mbar_arrive_expect_tx(&x_full[s], L::kXBytes);
                tma_load_2d(sw + L::kWBytes, &tmx, &x_full[s], k0 + i * kSuper, 0);
                issued_x = i + 1;
            }
            // drain: no copy may still be landing when the CTA moves on
            for (int i = issued_w > kRawStages ? issued_w - kRawStages : 0; i < issued_w; ++i)
                if (!mbar_wait(&w_full[i % kRawStages], (i / kRawStages) & 1, p.status))
                    break;
            for (int i = issued_x > kRawStages ? issued_x - kRawStages : 0; i < issued_x; ++i)
                if (!mbar_wait(&x_full[i % kRawStages], (i / kRawStages) & 1, p.status))
                    break;
        }
        __syncwarp();
    } else {
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    float *sa_s = reinterpret_cast<float *>(smem + L::kOffSa);
    if (threadIdx.x < NP)   // the token scales (may be the preceding kernel's output)
        sa_s[threadIdx.x] = threadIdx.x < p.M ? f16_bits_to_f32(p.sa[threadIdx.x]) : 0.f;

    if (warp == kTMmaWarp) {
        // ================= MMA issuer =================
        if (lane == 0) {
            const uint32_t idesc = f16_idesc(false, kTRows, NP);
            const uint64_t op_desc0 = sw128_desc(smem_u32(smem + L::kOffOp));
            for (int i = 0; i < nsuper && ok; ++i) {
                const int t = i % kOpStages;
                if (!(ok = mbar_wait(&op_full[t], (i / kOpStages) & 1, p.status)))
                    break;
                tc_fence_after();
                const uint32_t a0 = (t * L::kOpBytes) >> 4, b0 = (t * L::kOpBytes + 2 * L::kATile) >> 4;
                switch (p.group_log2) {
                case 5: ok = mma_superstep<5, NP, L::kATile, L::kBTile>(i, tmem_base, op_desc0, a0, b0, idesc, acc_full, acc_empty, p.status); break;
                case 6: ok = mma_superstep<6, NP, L::kATile, L::kBTile>(i, tmem_base, op_desc0, a0, b0, idesc, acc_full, acc_empty, p.status); break;
                default: ok = mma_superstep<7, NP, L::kATile, L::kBTile>(i, tmem_base, op_desc0, a0, b0, idesc, acc_full, acc_empty, p.status); break;
                }
                if (!ok)
                    break;
                tc_commit(&op_empty[t]);
            }
            tc_commit(drain);
            mbar_wait(drain, 0, p.status);
        }
        __syncwarp();
    } else if (warp >= kConvWarp0) {
        // ================= converters: packed / int8 -> fp16 operand tiles =================
        const int ct = threadIdx.x - 32 * kConvWarp0;    // 0 .. 319
        const int h = (ct >> 7) & 1, r = ct & 127;        // weights: K step h of the super step, row r
        const int m = ct - 256;                           // activations: token m, both K steps
        for (int i = 0; i < nsuper && ok; ++i) {
            const int s = i % kRawStages, t = i % kOpStages;
            const uint32_t par = (i / kRawStages) & 1;
            ok = mbar_wait(&w_full[s], par, p.status) && mbar_wait(&x_full[s], par, p.status) &&
                 (i < kOpStages || mbar_wait(&op_empty[t], ((i / kOpStages) - 1) & 1, p.status));
            if (!(ok = __all_sync(0xffffffffu, ok)))   // the warp leaves together (its syncs stay whole)
                break;
            const uint8_t *raw = smem + L::kOffRaw + s * L::kRawBytes;
            uint8_t *op = smem + L::kOffOp + t * L::kOpBytes;
            uint32_t v[32];
            if (ct < 256) {
                if constexpr (BITS == 4) {
                    // row r: 64 B per super step; this thread's 32 B = codes 64h .. 64h + 63
                    const uint8_t *src = raw + r * L::kWRow + 32 * h;
                    const uint4 q0 = *reinterpret_cast<const uint4 *>(src);
                    const uint4 q1 = *reinterpret_cast<const uint4 *>(src + 16);
                    const uint32_t wv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                    for (int i8 = 0; i8 < 8; ++i8) {
                        uint32_t o[4];
                        int4x8_to_f16(wv[i8], o);
                        v[4 * i8] = o[0];
                        v[4 * i8 + 1] = o[1];
                        v[4 * i8 + 2] = o[2];
                        v[4 * i8 + 3] = o[3];
                    }
                } else {
                    // row r: 128 B per super step, 128-byte swizzled by TMA; chunks 4h .. 4h + 3
                    const uint8_t *row = raw + r * L::kWRow;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 q = *reinterpret_cast<const uint4 *>(row + (((4 * h + c) ^ (r & 7)) << 4));
                        uint32_t o[4];
                        int8x8_to_f16(q.x, q.y, o);
                        v[8 * c] = o[0];
                        v[8 * c + 1] = o[1];
                        v[8 * c + 2] = o[2];
                        v[8 * c + 3] = o[3];
                        int8x8_to_f16(q.z, q.w, o);
                        v[8 * c + 4] = o[0];
                        v[8 * c + 5] = o[1];
                        v[8 * c + 6] = o[2];
                        v[8 * c + 7] = o[3];
                    }
                }
                store_row64(op + h * L::kATile, r, v);
            } else if (m < NP) {
                // token m: 64 int8 per K step hx of the 128-byte swizzled row
                const uint8_t *row = raw + L::kWBytes + m * 128;
#pragma unroll 1
                for (int hx = 0; hx < 2; ++hx) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint4 q = *reinterpret_cast<const uint4 *>(row + (((4 * hx + c) ^ (m & 7)) << 4));
                    uint32_t o[4];
                    int8x8_to_f16(q.x, q.y, o);
                    v[8 * c] = o[0];
                    v[8 * c + 1] = o[1];
                    v[8 * c + 2] = o[2];
                    v[8 * c + 3] = o[3];
                    int8x8_to_f16(q.z, q.w, o);
                    v[8 * c + 4] = o[0];
                    v[8 * c + 5] = o[1];
                    v[8 * c + 6] = o[2];
                    v[8 * c + 7] = o[3];
                }
                store_row64(op + 2 * L::kATile + hx * L::kBTile, m, v);
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&raw_empty[s]);
                mbar_arrive(&op_full[t]);
            }
        }
    } else if (warp < kFoldWarp0 + 4) {
        // ================= fold: per-group accumulators -> scaled totals =================
        const int qd = warp - kFoldWarp0;                // TMEM lane quarter
        const int r = 32 * qd + lane;                    // weight row of this thread
        const int n = n0 + r;
        float tot[NP];
#pragma unroll
        for (int m = 0; m < NP; ++m)
            tot[m] = 0.f;
        for (int gl = 0; gl < ngl && ok; ++gl) {
            const int slot = gl % kAccSlots;
            ok = mbar_wait(&acc_full[slot], (gl / kAccSlots) & 1, p.status);
            if (!(ok = __all_sync(0xffffffffu, ok)))
                break;
            tc_fence_after();
            const float s = f16_bits_to_f32(ws_s[gl * kTRows + r]);
            int32_t *ao = p.acc_out && n < p.N ? p.acc_out + static_cast<long long>(n) * p.ng + gbase + gl : nullptr;
#pragma unroll
            for (int c0 = 0; c0 < NP; c0 += 32) {
                // 32 columns per TMEM load (one wait), 16 for the last of NP = 16 or 48
                const uint32_t ta = tmem_base + (static_cast<uint32_t>(32 * qd) << 16) + slot * NP + c0;
                if (c0 + 32 <= NP) {
                    uint32_t a[32];
                    tmem_ld32(ta, a);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        tot[c0 + e] = fmaf(s, __uint_as_float(a[e]), tot[c0 + e]);
                    if (ao)
                        for (int e = 0; e < 32 && c0 + e < p.M; ++e)
                            ao[static_cast<long long>(c0 + e) * p.N * p.ng] = __float2int_rn(__uint_as_float(a[e]));
                } else {
                    uint32_t a[16];
                    tmem_ld16(ta, a);
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        tot[c0 + e] = fmaf(s, __uint_as_float(a[e]), tot[c0 + e]);
                    if (ao)
                        for (int e = 0; e < 16 && c0 + e < p.M; ++e)
                            ao[static_cast<long long>(c0 + e) * p.N * p.ng] = __float2int_rn(__uint_as_float(a[e]));
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&acc_empty[slot]);
        }
        // this CTA's MMAs and conversions are over, so the operand stages can
        // hold the outgoing partials: fold warp q writes its 32 rows [token][row]
        // and one bulk copy sends them to CTA q of the cluster
        float *out = reinterpret_cast<float *>(smem + L::kOffOp) + qd * NP * 32;
#pragma unroll
        for (int m = 0; m < NP; ++m)
            out[m * 32 + lane] = tot[m];
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            bulk_to_cluster(smem + L::kOffRecv + rank * L::kPartBytes, out, L::kPartBytes, red_full,
                            static_cast<uint32_t>(qd));
            bulk_wait_read();   // the copy has read its source before the CTA moves on
        }
        __syncwarp();
    }
    // this CTA's quarter of the rows: sum the four partials, scale by the token's scale
    const bool got = mbar_wait(red_full, 0, p.status);
    const float *recv = reinterpret_cast<const float *>(smem + L::kOffRecv);
    for (int idx = threadIdx.x; got && idx < 32 * NP; idx += kTThreads) {
        const int i = idx & 31, m = idx >> 5;
        const int n = n0 + static_cast<int>(rank) * 32 + i;
        if (m < p.M && n < p.N) {
            float v = 0.f;
#pragma unroll
            for (int src = 0; src < kKSplit; ++src)
                v += recv[(src * NP + m) * 32 + i];
            p.y[static_cast<long long>(m) * p.N + n] = f32_to_f16_bits(v * sa_s[m]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kTMmaWarp)
        tmem_dealloc(tmem_base, 512);
}

template <int BITS, int NP>
cudaError_t launch_tc(const CUtensorMap &tmw, const CUtensorMap &tmx, const TcParams &p, int grid, int smem_optin,
                      cudaStream_t stream)
{
    using L = TcLayout<BITS, NP>;
    const int smem = L::kBytes + 1024;
    if (smem > smem_optin)
        return cudaErrorInvalidConfiguration;
    auto kern = wxa8_tc_kernel<BITS, NP>;
    static SmemLimit limit;
    if (const cudaError_t e = ensure_smem_limit(limit, kern, smem); e != cudaSuccess)
        return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmw, tmx, p);
}

template <int BITS>
cudaError_t launch_tc_np(int np, const CUtensorMap &tmw, const CUtensorMap &tmx, const TcParams &p, int grid,
                         int smem_optin, cudaStream_t stream)
{
    switch (np) {
    case 16: return launch_tc<BITS, 16>(tmw, tmx, p, grid, smem_optin, stream);
    case 32: return launch_tc<BITS, 32>(tmw, tmx, p, grid, smem_optin, stream);
    case 48: return launch_tc<BITS, 48>(tmw, tmx, p, grid, smem_optin, stream);
    default: return launch_tc<BITS, 64>(tmw, tmx, p, grid, smem_optin, stream);
    }
}

}  // namespace

bool wxa8_tc_takes(int bits, int M, int N, int K, int group, const void *xq, const void *w)
{
    if ((bits != 4 && bits != 8) || M < 1 || M > 64 || N < 1 || K % (kKSplit * kSuper) != 0)
        return false;
    if ((K / kKSplit) / group > kMaxLocalGroups)
        return false;
    return reinterpret_cast<uintptr_t>(xq) % 16 == 0 && reinterpret_cast<uintptr_t>(w) % 16 == 0;
}

qmm_status wxa8_tc_dispatch(int bits, const int8_t *xq, const void *sa, const uint8_t *w, const void *ws,
                            int group, void *y, int32_t *acc_out, int M, int N, int K, int *status,
                            int smem_optin, cudaStream_t stream)
{
    const int np = (M + 15) / 16 * 16;
    CUtensorMap tmw, tmx;
    std::memset(&tmw, 0, sizeof(tmw));
    std::memset(&tmx, 0, sizeof(tmx));
    const long long row_bytes = static_cast<long long>(K) * bits / 8;
    if (!encode_byte_tmap(&tmw, w, row_bytes, N, kSuper * bits / 8, kTRows, bits == 8))
        return QMM_ERR_CUDA;
    if (!encode_byte_tmap(&tmx, xq, K, M, kSuper, np, true))
        return QMM_ERR_CUDA;
    TcParams p;
    std::memset(&p, 0, sizeof(p));
    p.sa = static_cast<const uint16_t *>(sa);
    p.ws = static_cast<const uint16_t *>(ws);
    p.y = static_cast<uint16_t *>(y);
    p.acc_out = acc_out;
    p.status = status;
    p.M = M;
    p.N = N;
    p.K = K;
    p.ng = K / group;
    p.group = group;
    p.group_log2 = group == 32 ? 5 : group == 64 ? 6 : 7;
    p.vec_ws = reinterpret_cast<uintptr_t>(ws) % 16 == 0 && p.ng % 8 == 0 && (p.ng / kKSplit) % 8 == 0;
    const int grid = kKSplit * ((N + kTRows - 1) / kTRows);
    const cudaError_t e = bits == 8 ? launch_tc_np<8>(np, tmw, tmx, p, grid, smem_optin, stream)
                                    : launch_tc_np<4>(np, tmw, tmx, p, grid, smem_optin, stream);
    return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA;
}

}  // namespace qmm
