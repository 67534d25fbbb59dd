// decode.cu -- host side of the staged decode kernel (decode.cuh): the
// launch plan and the launcher for the canonical weight layout (the
// fragment-ordered layout's launcher is in decode_tile.cu).
#include "decode.cuh"

namespace qmm {

namespace {

constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

}  // namespace

bool decode_plan(int M, int N, int K, int group, int bits, bool stored_zeros, bool tile16, int num_sms,
                 int smem_pair, int smem_optin, DecodePlan *plan)
{
    if (M < 1 || M > 16 || N < 1 || bits < 1 || bits > 8 || (group != 64 && group != 128) ||
        K < 8 * group || K % (8 * group) || num_sms < 1)
        return false;
    DecodePlan pl = {};
    pl.warps = kWarps;
    pl.kseg = kWarps * group;           // warp w owns group w of a segment
    pl.nseg = K / pl.kseg;
    // the units CTAs share out: rows (canonical layout) or 16-row tiles (tile16)
    const int units = tile16 ? (N + 15) / 16 : N;
    pl.grid = units < num_sms ? units : num_sms;
    pl.rows_base = units / pl.grid;
    pl.rows_rem = units % pl.grid;
    pl.max_rows = pl.rows_base + (pl.rows_rem > 0 ? 1 : 0);
    if (tile16)
        pl.max_rows = 16 * pl.max_rows < N ? 16 * pl.max_rows : N;
    const int nrb = (pl.max_rows + kRowBlock - 1) / kRowBlock;
    const int slot_rows = pl.max_rows < kRowBlock ? pl.max_rows : kRowBlock;
    const int ng = K / group;
    pl.x_pitch = K / kWarps * 2 + 16;                   // + 16: tokens of one load on other banks
    const int x_bytes = align_up(kWarps * M * pl.x_pitch, 16);
    const int xsum_bytes = align_up(kWarps * M * pl.nseg * 8, 16);
    const int sc_bytes = align_up(pl.max_rows * ng * 2, 16);
    const int zo_bytes = stored_zeros ? sc_bytes : 0;
    const int red_bytes = kWarps * kRowBlock * M * 4;
    pl.seg_bytes = pl.kseg * bits / 8;
    const int fixed = x_bytes + xsum_bytes + sc_bytes + zo_bytes + red_bytes + 2 * kMaxSlots * 8 + 16;
    // two CTAs per SM (the next call's weights stream in while this one computes)
    // when at least two slots, or every chunk, fit beside the rest; else one.
    // A slot holds a whole row block's K (one bulk copy per row) when every row
    // block fits at once, else one segment (a ring of segments).
    for (int pair = 1; pair >= 0; --pair) {
        const int budget = pair ? smem_pair : smem_optin;
        int slots = 0;
        for (int whole = 1; whole >= 0; --whole) {
            pl.span = whole ? pl.nseg : 1;
            const int bytes = pl.span * pl.seg_bytes;
            // tile16: a slot holds two dense 16-row tiles (fragment reads are contiguous)
            pl.pitch = tile16 ? 0 : bytes + ((pitch_residue(bits) - bytes % 128) + 128) % 128;
            pl.slot_bytes = tile16 ? 32 * bytes : slot_rows * pl.pitch;
            // slots a tensor-map box fills (decode_tma_fits) start on 128 bytes
            if (!tile16 && pl.pitch <= 2048)
                pl.slot_bytes = align_up(pl.slot_bytes, 128);
            const int total = nrb * (pl.nseg / pl.span);
            slots = budget > fixed ? (budget - fixed) / pl.slot_bytes : 0;
            slots = slots < total ? slots : total;
            slots = slots < kMaxSlots ? slots : kMaxSlots;
            if (whole ? slots == total : (slots >= 2 || (slots >= 1 && slots == total)))
                break;
            slots = 0;
        }
        if (slots < 1)
            continue;
        pl.slots = slots;
        pl.off_x = align_up(slots * pl.slot_bytes, 16);
        pl.off_xsum = pl.off_x + x_bytes;
        pl.off_sc = pl.off_xsum + xsum_bytes;
        pl.off_zo = pl.off_sc + sc_bytes;
        pl.off_red = pl.off_zo + zo_bytes;
        pl.off_bar = align_up(pl.off_red + red_bytes, 8);
        pl.smem = pl.off_bar + 2 * slots * 8 + 16;
        if (pl.smem > budget)
            continue;
        *plan = pl;
        return true;
    }
    return false;
}

cudaError_t launch_decode(const DecodeParams &p, int bits, bool tile16, cudaStream_t stream)
{
    return tile16 ? launch_decode_tile16(p, bits, stream) : launch_decode_layout<false>(p, bits, stream);
}

}  // namespace qmm
