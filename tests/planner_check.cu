// Prints the skinny-kernel planner's choices as one JSON object per line, for
// shapes read from stdin ("M N K bits group zeros" per line).  Host code only:
// it plans for GB300's limits (152 SMs, 227 KB per CTA, 113 KB for two CTAs per
// SM) and runs without a GPU.  tests/test_planner.py checks the invariants.
#include <cstdio>
#include <cstring>

#include "../bit_weight_quantized_gb300/csrc/gemv.cu"

int main()
{
    using namespace qmm;
    const int num_sms = 152, smem_max = 232448, smem_pair = 115712;
    int M, N, K, bits, group, zeros;
    while (std::scanf("%d %d %d %d %d %d", &M, &N, &K, &bits, &group, &zeros) == 6) {
        GemvParams p;
        std::memset(&p, 0, sizeof(p));
        p.M = M;
        p.N = N;
        p.K = K;
        p.group = group;
        p.ng = K / group;
        p.row_bytes = static_cast<long long>(K) * bits / 8;
        p.zeros = zeros ? reinterpret_cast<const uint8_t *>(16) : nullptr;   // only tested for null
        p.zero_const = zeros ? 0 : 8;
        int grid = 0, smem = 0;
        const qmm_status st = skinny_plan(p, bits, num_sms, smem_max, smem_pair, &grid, &smem);
        std::printf("{\"M\":%d,\"N\":%d,\"K\":%d,\"bits\":%d,\"group\":%d,\"zeros\":%d,\"st\":%d,"
                    "\"grid\":%d,\"smem\":%d,\"num_sms\":%d,\"smem_max\":%d,\"smem_pair\":%d,"
                    "\"nchunks\":%d,\"stages_per_block\":%d,\"seg_chunks\":%d,\"seg_bytes\":%d,"
                    "\"pitch\":%d,\"phase_chunks\":%d,\"nphases\":%d,\"rows_base\":%d,\"rows_rem\":%d,"
                    "\"rb\":%d,\"rbp\":%d,\"ksplit_log2\":%d,\"ring\":%d,\"stage_bytes\":%d,"
                    "\"off_bar\":%d,\"off_x\":%d,\"off_xs\":%d,\"off_cs\":%d,\"off_sz\":%d,"
                    "\"off_red\":%d,\"off_ring\":%d,\"sz_pitch\":%d,\"sz_compact\":%d,\"red_alias\":%d}\n",
                    M, N, K, bits, group, zeros, static_cast<int>(st), grid, smem, num_sms, smem_max,
                    smem_pair, p.nchunks, p.stages_per_block, p.seg_chunks, p.seg_bytes, p.pitch,
                    p.phase_chunks, p.nphases, p.rows_base, p.rows_rem, p.rb, p.rbp, p.ksplit_log2,
                    p.ring, p.stage_bytes, p.off_bar, p.off_x, p.off_xs, p.off_cs, p.off_sz,
                    p.off_red, p.off_ring, p.sz_pitch, p.sz_compact, p.red_alias);
    }
    return 0;
}
