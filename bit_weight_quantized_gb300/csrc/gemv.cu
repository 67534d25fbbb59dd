// gemv.cu -- host planning for the skinny kernel (shared by qmm_gemv and
// qmm_w4a8): grid, row blocks, K segments and phases, shared-memory layout.
#include "gemv.h"
#include "skinny.cuh"

#include <mutex>
#include <unordered_map>

namespace qmm {

static int align_up(int v, int a) { return (v + a - 1) / a * a; }

// shortest per-row segment (bytes) tried before falling back to anything that fits
constexpr int kMinSegBytes = 256;
// most pipeline slots per CTA
constexpr int kMaxRing = 16;

// n-tiles of 8 tokens the kernel is instantiated with (1, 2, 4 or 8)
static int token_tiles(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8; }

// Lays out shared memory for row blocks of `rb` rows, K phases of `cp` chunks and
// at most `max_ring` slots; returns the dynamic shared-memory size, or 0 if
// fewer than `min_ring` slots fit in `budget` bytes.
static int plan_layout(GemvParams &p, int rb, int nblk, int cp, int budget, int max_ring, int min_ring)
{
    const int MP = 8 * token_tiles(p.M);
    const int ngc = 128 / p.group;
    p.rb = rb;
    p.rbp = align_up(rb, 16);
    p.phase_chunks = cp;
    p.nphases = (p.nchunks + cp - 1) / cp;
    // a slot holds rb rows (tile rows past rb read row rb - 1); a run that starts
    // inside a word reads one word past its end: 16 bytes of slack after the ring
    p.stage_bytes = align_up(rb * p.pitch, 128);
    const int overrun = 128;
    p.sz_pitch = p.ng + ((p.ng & 1) ? 0 : 1);   // odd: the eight rows of a tile hit different banks
    const int bar_bytes = align_up(kMaxRing * 12, 128);
    const int x_bytes = align_up(p.M * cp * 128 * 2, 128);
    const int xs_bytes = align_up(cp * ngc * MP * 4, 128);
    // scales as float2 (s, z*s) for one token tile, as stored (fp16 + uint8 zeros)
    // for more, where activations and row blocks are large
    p.sz_compact = token_tiles(p.M) >= 2;
    const int sz_bytes = align_up(p.rbp * p.sz_pitch * (p.sz_compact ? (p.zeros ? 3 : 2) : 8), 128);
    const int red_bytes = align_up((1 << p.ksplit_log2) * p.rbp * MP * 4, 128);
    // group sums of x and of 2^E x
    int fixed = 128 /* base alignment */ + bar_bytes + x_bytes + 2 * xs_bytes + sz_bytes + red_bytes + overrun;
    // The reduction buffer may reuse the activation buffer when the activations
    // are not needed after a block's loop (one block, or restaged per phase); it
    // costs a barrier, so it is taken only when it buys ring slots.
    p.red_alias = 0;
    if ((p.nphases > 1 || nblk == 1) && red_bytes <= x_bytes && (budget - fixed) / p.stage_bytes < max_ring &&
        (budget - fixed + red_bytes) / p.stage_bytes > (budget - fixed) / p.stage_bytes) {
        p.red_alias = 1;
        fixed -= red_bytes;
    }
    if (budget - fixed < p.stage_bytes * min_ring)
        return 0;
    int ring = (budget - fixed) / p.stage_bytes;
    if (ring > max_ring)
        ring = max_ring;
    p.ring = ring;
    int off = 0;
    p.off_bar = off;
    off += bar_bytes;
    p.off_x = off;
    off += x_bytes;
    p.off_xs = off;
    off += xs_bytes;
    p.off_cs = off;
    off += xs_bytes;
    p.off_sz = off;
    off += sz_bytes;
    p.off_red = p.red_alias ? p.off_x : off;
    if (!p.red_alias)
        off += red_bytes;
    p.off_ring = off;
    off += ring * p.stage_bytes + overrun;
    return off + 128;
}

// Sets the K segment of `seg` chunks (pitch: 16*b mod 128, or 16 for b = 8, so
// that the four threads of a quad and the eight rows of a tile read distinct
// banks).
static void set_segment(GemvParams &p, int bits, int seg)
{
    p.seg_chunks = seg;
    p.seg_bytes = seg * 16 * bits;
    const int want = bits == 8 ? 16 : (16 * bits) % 128;
    const int pad = ((want - p.seg_bytes % 128) % 128 + 128) % 128;
    p.pitch = p.seg_bytes + pad;
    p.stages_per_block = (p.nchunks + seg - 1) / seg;
}

static qmm_status skinny_plan_search(GemvParams &p, int bits, int num_sms, int smem_max, int smem_pair,
                                     int *grid_out, int *smem_out)
{
    p.nchunks = (p.K + 127) / 128;
    int grid = (p.N + 15) / 16;
    if (grid > num_sms)
        grid = num_sms;
    if (grid < 1)
        grid = 1;
    p.rows_base = p.N / grid;
    p.rows_rem = p.N % grid;
    const int rows_max = p.rows_base + (p.rows_rem ? 1 : 0);
    // a block holds at most 8 tiles of 16 rows (two per warp of a K split of 2)
    const int rbmax = 16 * kWarps * kTilesPerWarp / 2;
    const int nblk0 = (rows_max + rbmax - 1) / rbmax;
    // K segment: about a kilobyte of each row per stage, at least 8 chunks; longer
    // ones (up to 2 KB) are tried first, since fewer, larger bulk copies stream
    // faster when the ring still holds as much
    int seg0 = (1024 + 16 * bits - 1) / (16 * bits);
    if (seg0 < 8)
        seg0 = 8;
    if (seg0 > p.nchunks)
        seg0 = p.nchunks;
    int seg_hi = (2048 + 16 * bits - 1) / (16 * bits);
    if (seg_hi < seg0)
        seg_hi = seg0;
    if (seg_hi > p.nchunks)
        seg_hi = p.nchunks;
    const int budgets[2] = {smem_pair, smem_max};
    // Candidates are ranked by: how often the activations are staged (once with
    // one phase or one block, else once per block), row blocks (a block switch
    // drains the pipeline), phases, then bytes in flight (a shorter segment only
    // for at least 15% more), then segment length.  Segments under
    // kMinSegBytes, or not a multiple of the K split, are tried only when
    // nothing else fits.  A layout that lets
    // two CTAs share an SM is taken first, if it needs one phase, the fewest
    // blocks and no short segments.
    struct Cand {
        int nph, nblk, seg, kl;
        long long inflight;
    };
    auto better = [](const Cand &a, const Cand &b) {   // a ranks before b
        const int ra = (a.nph == 1 || a.nblk == 1) ? 1 : a.nblk;
        const int rb_ = (b.nph == 1 || b.nblk == 1) ? 1 : b.nblk;
        if (ra != rb_)
            return ra < rb_;
        if (a.nblk != b.nblk)
            return a.nblk < b.nblk;
        if (a.nph != b.nph)
            return a.nph < b.nph;
        if (a.inflight * 100 > b.inflight * 115)
            return true;
        if (b.inflight * 100 > a.inflight * 115)
            return false;
        return a.seg > b.seg;
    };
    for (int bi = 0; bi < 2; ++bi) {
        const int budget = budgets[bi];
        if (budget <= 0 || budget > smem_max)
            continue;
        const int nph_max = bi == 0 ? 1 : p.nchunks;
        const int nblk_max = bi == 0 ? nblk0 : nblk0 + 8;
        for (int pass = 0; pass < (bi == 0 ? 1 : 2); ++pass) {
            bool found = false;
            Cand best = {0, 0, 0, 0, 0};
            for (int nph = 1; nph <= nph_max; ++nph) {
                for (int nblk = nblk0; nblk <= nblk_max; ++nblk) {
                    const int rb = (rows_max + nblk - 1) / nblk;
                    if (rb < 1)
                        break;
                    // the largest K split whose tile groups cover the tiles, two per warp
                    const int tiles = (rb + 15) / 16;
                    int kl = 3;
                    while (kl > 0 && tiles > kTilesPerWarp * (kWarps >> kl))
                        --kl;
                    p.ksplit_log2 = kl;
                    for (int seg = seg_hi; seg >= 1; --seg) {
                        if (pass == 0 && seg < seg0 && seg * 16 * bits < kMinSegBytes)
                            break;
                        // every warp of the K split gets the same number of a stage's
                        // chunks (a stage ends when its slowest warp does)
                        if (pass == 0 && seg < p.nchunks && seg % (1 << kl) != 0)
                            continue;
                        set_segment(p, bits, seg);
                        // phase = a whole number of segments covering nchunks in nph phases
                        const int cp = ((p.stages_per_block + nph - 1) / nph) * seg;
                        if ((p.nchunks + cp - 1) / cp != nph)
                            continue;
                        const int total = nblk * p.stages_per_block;
                        const int max_ring = total < kMaxRing ? total : kMaxRing;
                        if (!plan_layout(p, rb, nblk, cp, budget, max_ring, max_ring < 2 ? max_ring : 2))
                            continue;
                        // bytes in flight from the start: the ring, or the whole slice if less
                        long long inflight = static_cast<long long>(p.ring) * p.seg_bytes;
                        if (inflight > p.row_bytes * nblk)
                            inflight = p.row_bytes * nblk;
                        inflight *= rb;
                        const Cand c = {nph, nblk, seg, kl, inflight};
                        if (!found || better(c, best)) {
                            best = c;
                            found = true;
                        }
                    }
                }
            }
            if (found) {
                const int rb = (rows_max + best.nblk - 1) / best.nblk;
                p.ksplit_log2 = best.kl;
                set_segment(p, bits, best.seg);
                const int cp = ((p.stages_per_block + best.nph - 1) / best.nph) * best.seg;
                const int total = best.nblk * p.stages_per_block;
                const int max_ring = total < kMaxRing ? total : kMaxRing;
                *smem_out = plan_layout(p, rb, best.nblk, cp, budget, max_ring, max_ring < 2 ? max_ring : 2);
                *grid_out = grid;
                return QMM_OK;
            }
        }
    }
    return QMM_ERR_UNSUPPORTED;
}

// The search above costs microseconds; decode calls repeat the same shapes, so
// plans are kept per (shape, width, group, zero mode, device limits).
namespace {

struct PlanKey {
    int M, N, K, bits, group, zeros, num_sms, smem_max, smem_pair;
    bool operator==(const PlanKey &o) const
    {
        return M == o.M && N == o.N && K == o.K && bits == o.bits && group == o.group &&
               zeros == o.zeros && num_sms == o.num_sms && smem_max == o.smem_max &&
               smem_pair == o.smem_pair;
    }
};

struct PlanKeyHash {
    size_t operator()(const PlanKey &k) const
    {
        uint64_t h = 1469598103934665603ull;
        const int v[9] = {k.M, k.N, k.K, k.bits, k.group, k.zeros, k.num_sms, k.smem_max, k.smem_pair};
        for (int x : v) {
            h ^= static_cast<uint32_t>(x);
            h *= 1099511628211ull;
        }
        return static_cast<size_t>(h);
    }
};

struct PlanEntry {
    qmm_status status;
    GemvParams plan;   // only the fields the search fills are used
    int grid, smem;
};

std::mutex g_plan_mutex;
std::unordered_map<PlanKey, PlanEntry, PlanKeyHash> g_plans;
constexpr size_t kMaxPlans = 1024;

void copy_plan_fields(GemvParams &d, const GemvParams &s)
{
    d.nchunks = s.nchunks;
    d.stages_per_block = s.stages_per_block;
    d.seg_chunks = s.seg_chunks;
    d.seg_bytes = s.seg_bytes;
    d.pitch = s.pitch;
    d.phase_chunks = s.phase_chunks;
    d.nphases = s.nphases;
    d.rows_base = s.rows_base;
    d.rows_rem = s.rows_rem;
    d.rb = s.rb;
    d.rbp = s.rbp;
    d.ksplit_log2 = s.ksplit_log2;
    d.ring = s.ring;
    d.stage_bytes = s.stage_bytes;
    d.off_bar = s.off_bar;
    d.off_x = s.off_x;
    d.off_xs = s.off_xs;
    d.off_cs = s.off_cs;
    d.off_sz = s.off_sz;
    d.off_red = s.off_red;
    d.off_ring = s.off_ring;
    d.sz_pitch = s.sz_pitch;
    d.sz_compact = s.sz_compact;
    d.red_alias = s.red_alias;
}

}  // namespace

qmm_status skinny_plan(GemvParams &p, int bits, int num_sms, int smem_max, int smem_pair,
                       int *grid_out, int *smem_out)
{
    const PlanKey key = {p.M, p.N, p.K, bits, p.group, p.zeros ? 1 : 0, num_sms, smem_max, smem_pair};
    {
        std::lock_guard<std::mutex> lock(g_plan_mutex);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) {
            copy_plan_fields(p, it->second.plan);
            *grid_out = it->second.grid;
            *smem_out = it->second.smem;
            return it->second.status;
        }
    }
    int grid = 0, smem = 0;
    const qmm_status st = skinny_plan_search(p, bits, num_sms, smem_max, smem_pair, &grid, &smem);
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    if (g_plans.size() >= kMaxPlans)
        g_plans.clear();
    g_plans[key] = PlanEntry{st, p, grid, smem};
    *grid_out = grid;
    *smem_out = smem;
    return st;
}

}  // namespace qmm

