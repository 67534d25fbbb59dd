// gemv.cu -- host planning for the skinny kernel (shared by qmm_gemv and
// qmm_w4a8): grid, row blocks, K phases and the shared-memory layout.
#include "gemv.h"
#include "skinny.cuh"

namespace qmm {

static int align_up(int v, int a) { return (v + a - 1) / a * a; }

// pipeline stages in flight per CTA
constexpr int kLookahead = 3;

// n-tiles of 8 tokens the kernel is instantiated with (1, 2, 4 or 8)
static int token_tiles(int M) { return M <= 8 ? 1 : M <= 16 ? 2 : M <= 32 ? 4 : 8; }

// Lays out shared memory for row blocks of `rb` rows and K phases of `cp`
// chunks; returns the dynamic shared-memory size, or 0 if it does not fit with
// at least `min_ring` pipeline stages.
static int plan_smem(GemvParams &p, int bits, int rb, int cp, int smem_max, int min_ring)
{
    const int nt = token_tiles(p.M);
    const int MP = 8 * nt;
    const int ngc = 128 / p.group;
    p.rb = rb;
    p.rbp = align_up(rb, 16);
    p.phase_chunks = cp;
    p.nphases = (p.nchunks + cp - 1) / cp;
    p.stage_bytes = align_up(p.rbp * p.pitch + 16, 128);
    p.sz_pitch = p.ng + ((p.ng & 1) ? 0 : 1);
    const int x_bytes = align_up(p.M * cp * 128 * 2, 16);
    const int xs_bytes = align_up(cp * ngc * MP * 4, 16);
    const int sz_bytes = align_up(p.rbp * p.sz_pitch * 8, 16);
    // the reduction buffer also holds the per-run activation sums while staging
    const int runsum_bytes = p.M * cp * (128 / (p.group / 4)) * 4;
    int red_bytes = align_up(kConsumerWarps * p.rbp * MP * 4, 16);
    if (red_bytes < align_up(runsum_bytes, 16))
        red_bytes = align_up(runsum_bytes, 16);
    const int fixed = x_bytes + xs_bytes + sz_bytes + red_bytes;
    const int budget = smem_max - 1024 /* alignment slack */ - fixed;
    if (budget <= 0)
        return 0;
    // A few stages of look-ahead keep enough bytes in flight for HBM while
    // letting the stages land roughly in order (issuing a whole block at once
    // makes every stage complete near the end, so compute cannot overlap).
    int ring = budget / (p.stage_bytes + 16);
    if (ring > kLookahead)
        ring = kLookahead;
    if (ring < min_ring)
        return 0;
    p.ring = ring;
    int off = ring * p.stage_bytes;
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

qmm_status skinny_plan(GemvParams &p, int bits, int num_sms, int smem_max, int *grid_out,
                       int *smem_out)
{
    p.nchunks = (p.K + 127) / 128;
    const int maxt = 2;   // as the kernel's MAXT
    const int rbmax = 16 * maxt;
    int grid = (p.N + 15) / 16;
    if (grid > num_sms)
        grid = num_sms;
    if (grid < 1)
        grid = 1;
    p.rows_base = p.N / grid;
    p.rows_rem = p.N % grid;
    const int rows_max = p.rows_base + (p.rows_rem ? 1 : 0);
    // K segment: about a kilobyte of each row per stage, at least 8 chunks;
    // smaller when the activations of a segment do not fit (large M)
    int seg0 = (1024 + 16 * bits - 1) / (16 * bits);
    if (seg0 < 8)
        seg0 = 8;
    if (seg0 > p.nchunks)
        seg0 = p.nchunks;
    for (int seg = seg0; seg >= 1; seg = seg > 1 ? seg / 2 : 0) {
        p.seg_chunks = seg;
        p.seg_bytes = seg * 16 * bits;
        // pitch = 16*b (mod 128), or 16 for b = 8: with it the four threads of a
        // quad and the eight rows of an MMA tile read distinct banks
        const int want = bits == 8 ? 16 : (16 * bits) % 128;
        const int pad = ((want - p.seg_bytes % 128) % 128 + 128) % 128;
        p.pitch = p.seg_bytes + pad;
        p.stages_per_block = (p.nchunks + seg - 1) / seg;
        const int cp_full = p.stages_per_block * seg;
        for (int nblk = (rows_max + rbmax - 1) / rbmax; nblk <= rows_max; ++nblk) {
            const int rb = (rows_max + nblk - 1) / nblk;
            // prefer one activation phase; otherwise the largest phase that fits
            for (int cp = cp_full; cp >= seg; cp = (cp / 2 / seg) * seg) {
                const int smem = plan_smem(p, bits, rb, cp, smem_max, 2);
                if (smem) {
                    *grid_out = grid;
                    *smem_out = smem;
                    return QMM_OK;
                }
                if (cp == seg)
                    break;
            }
            if (rb <= 16)
                break;
        }
        if (seg == 1)
            break;
    }
    return QMM_ERR_UNSUPPORTED;
}

}  // namespace qmm
