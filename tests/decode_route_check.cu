// Prints decode_plan() (the staged decode kernel's shape rule and shared-memory
// plan) for shapes read from stdin, one per line:
//   "M N K group bits stored_zeros num_sms smem_pair smem_optin [tile16]"
// (the tenth field, tile16, is 0 or 1).  Output per line: the first nine inputs, then 0 (the skinny kernel takes the shape)
// or 1 followed by the plan's fields in DecodePlan order.  Host code only: it
// runs without a GPU.  tests/test_planner.py checks the answers.
#include <cstdio>

#include "../bit_weight_quantized_gb300/csrc/decode.cu"
#include "../bit_weight_quantized_gb300/csrc/decode_tile.cu"

int main()
{
    int M, N, K, group, bits, zeros, num_sms, pair, optin, tile;
    while (std::scanf("%d %d %d %d %d %d %d %d %d %d", &M, &N, &K, &group, &bits, &zeros, &num_sms, &pair,
                      &optin, &tile) == 10) {
        qmm::DecodePlan p;
        const bool ok = qmm::decode_plan(M, N, K, group, bits, zeros != 0, tile != 0, num_sms, pair, optin, &p);
        std::printf("%d %d %d %d %d %d %d %d %d %d", M, N, K, group, bits, zeros, num_sms, pair, optin, ok ? 1 : 0);
        if (ok)
            std::printf(" %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d %d", p.grid, p.rows_base,
                        p.rows_rem, p.max_rows, p.warps, p.kseg, p.nseg, p.seg_bytes, p.span, p.pitch,
                        p.slot_bytes, p.slots, p.x_pitch, p.off_x, p.off_xsum, p.off_sc, p.off_zo, p.off_red,
                        p.off_bar, p.smem);
        std::printf("\n");
    }
    return 0;
}
