// gemv.cu -- host planning for the skinny kernel (shared by qmm_gemv and
// qmm_w4a8): grid, row blocks, K phases and the shared-memory layout.
#include "gemv.h"
#include "skinny.cuh"

namespace qmm {

int skinny_stage_chunks(int bits) { return width_cs(bits); }

static int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Lays out shared memory for row blocks of `rb` rows and K phases of `cp`
// chunks; returns the dynamic shared-memory size, or 0 if it does not fit with
// at least `min_ring` pipeline stages.
static int plan_smem(GemvParams &p, int bits, int rb, int cp, int smem_max, int min_ring)
{
    const int nt = (p.M + 7) / 8;
    const int MP = 8 * nt;
    const int ngc = 128 / p.group;
    p.rb = rb;
    p.rbp = align_up(rb, 16);
    p.phase_chunks = cp;
    p.nphases = (p.nchunks + cp - 1) / cp;
    const int row_bytes = 16 * bits * width_cs(bits);
    p.tile_bytes = rb * row_bytes;
    // room for the 16-row tile padding the consumers read (never stored) and
    // for the one word a shifted run may read past its row
    p.stage_bytes = align_up(p.rbp * row_bytes + 16, 1024);
    p.sz_pitch = p.ng + ((p.ng & 1) ? 0 : 1);
    const int x_bytes = align_up(p.M * cp * 128 * 2, 16);
    const int xs_bytes = align_up(cp * ngc * MP * 4, 16);
    const int sz_bytes = align_up(p.rbp * p.sz_pitch * 8, 16);
    const int red_bytes = align_up(kConsumerWarps * p.rbp * MP * 4, 16);
    const int fixed = x_bytes + xs_bytes + sz_bytes + red_bytes;
    const int budget = smem_max - 1024 /* alignment slack */ - fixed;
    if (budget <= 0)
        return 0;
    int ring = budget / (p.stage_bytes + 16);
    const int total_stages_max = p.stages_per_block * 8;
    if (ring > total_stages_max)
        ring = total_stages_max;
    if (ring > 32)
        ring = 32;
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
    const int cs = width_cs(bits);
    p.nchunks = (p.K + 127) / 128;
    p.stages_per_block = (p.nchunks + cs - 1) / cs;
    const int nt = (p.M + 7) / 8;
    const int maxt = nt <= 2 ? 8 : 16 / nt;
    const int rbmax = 16 * maxt;
    int grid = (p.N + 15) / 16;
    if (grid > num_sms)
        grid = num_sms;
    if (grid < 1)
        grid = 1;
    p.rows_base = p.N / grid;
    p.rows_rem = p.N % grid;
    const int rows_max = p.rows_base + (p.rows_rem ? 1 : 0);
    const int cp_full = p.stages_per_block * cs;
    for (int nblk = (rows_max + rbmax - 1) / rbmax; nblk <= rows_max; ++nblk) {
        const int rb = (rows_max + nblk - 1) / nblk;
        // prefer one activation phase; otherwise the largest phase that fits
        for (int cp = cp_full; cp >= cs; cp = (cp / 2 / cs) * cs) {
            const int smem = plan_smem(p, bits, rb, cp, smem_max, 6);
            if (smem) {
                *grid_out = grid;
                *smem_out = smem;
                return QMM_OK;
            }
            if (cp == cs)
                break;
        }
        if (rb <= 16)
            break;
    }
    return QMM_ERR_UNSUPPORTED;
}

}  // namespace qmm
