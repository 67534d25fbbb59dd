// Prints decode_supports() (the decode kernel's shape rule) for shapes read from
// stdin ("M N K group num_sms" per line), one "M N K group num_sms answer" line
// each.  Host code only: it runs without a GPU.  tests/test_planner.py checks
// the answers against the documented rule.
#include <cstdio>

#include "../bit_weight_quantized_gb300/csrc/decode.cu"

int main()
{
    int M, N, K, group, num_sms;
    while (std::scanf("%d %d %d %d %d", &M, &N, &K, &group, &num_sms) == 5)
        std::printf("%d %d %d %d %d %d\n", M, N, K, group, num_sms,
                    qmm::decode_supports(M, N, K, group, num_sms) ? 1 : 0);
    return 0;
}
