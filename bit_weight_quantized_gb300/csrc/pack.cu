// pack.cu -- b-bit codes <-> per-column LSB-first bitstream (offline step).
//
// Column n's stream is K*b/8 bytes; code k occupies stream bits [k*b, k*b+b)
// and stream bit i is bit (i mod 8) of byte i/8.  Packing is not on the timed
// decode path, so these kernels favour simplicity: one thread per output
// byte (pack, sign flip) or per code (unpack).
#include "common.cuh"

namespace qmm {

__global__ void pack_kernel(const uint8_t *__restrict__ codes, uint8_t *__restrict__ packed,
                            long long N, long long K, int bits, int32_t *bad_count)
{
    const long long row_bytes = K * bits / 8;
    const long long total = N * row_bytes;
    const int mask = (1 << bits) - 1;
    int bad = 0;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long n = idx / row_bytes;
        const long long j = idx - n * row_bytes;        // byte within the row
        const long long bit0 = 8 * j;                   // first stream bit of this byte
        const long long k0 = bit0 / bits;
        const long long k1 = (bit0 + 7) / bits;         // last code touching the byte
        const uint8_t *row = codes + n * K;
        uint32_t out = 0;
        for (long long k = k0; k <= k1 && k < K; ++k) {
            const int q = row[k];
            const long long sh = k * bits - bit0;       // in [-7, 7]
            const uint32_t v = static_cast<uint32_t>(q & mask);
            out |= sh >= 0 ? (v << sh) : (v >> (-sh));
            if (k * bits >= bit0 && (q & ~mask))        // count each code once, at its first byte
                ++bad;
        }
        packed[idx] = static_cast<uint8_t>(out & 0xFF);
    }
    if (bad_count) {
        // one atomic per warp
        for (int o = 16; o > 0; o >>= 1)
            bad += __shfl_xor_sync(0xffffffffu, bad, o);
        if ((threadIdx.x & 31) == 0 && bad)
            atomicAdd(bad_count, bad);
    }
}

__global__ void unpack_kernel(const uint8_t *__restrict__ packed, uint8_t *__restrict__ codes,
                              long long N, long long K, int bits)
{
    const long long row_bytes = K * bits / 8;
    const long long total = N * K;
    const int mask = (1 << bits) - 1;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long n = idx / K;
        const long long k = idx - n * K;
        const uint8_t *row = packed + n * row_bytes;
        const long long b0 = k * bits;
        const long long byte = b0 >> 3;
        uint32_t v = row[byte];
        if (byte + 1 < row_bytes)
            v |= static_cast<uint32_t>(row[byte + 1]) << 8;
        codes[idx] = static_cast<uint8_t>((v >> (b0 & 7)) & mask);
    }
}

// Flips the top bit of every b-bit code in place: byte j of a row is XORed
// with the bits p in [8j, 8j + 8) that are a code's top bit, (p + 1) % b == 0
// (codes restart at each row, which starts byte-aligned).
__global__ void flip_sign_kernel(uint8_t *__restrict__ packed, long long N, long long K, int bits)
{
    const long long row_bytes = K * bits / 8;
    const long long total = N * row_bytes;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long bit0 = 8 * (idx % row_bytes);
        uint32_t m = 0;
        for (int t = 0; t < 8; ++t)
            if ((bit0 + t + 1) % bits == 0)
                m |= 1u << t;
        packed[idx] ^= static_cast<uint8_t>(m);
    }
}

// Fragment-ordered (tile16) layout: rows in tiles of 16 (the last padded with
// zero bytes), K in blocks of 64; unit (T, kb) = 128 b bytes at (T K/64 + kb)
// 128 b, holding run r = (h 8 + g) 4 + t (codes 16t .. 16t + 15 of row
// 16T + 8h + g) at bytes [2 b r, 2 b r + 2 b).  A run of 16 codes is 2b whole
// bytes of the canonical row starting at byte 8 b kb + 2 b t, so the layout is a
// byte gather.  One thread per output byte.
__global__ void tile16_kernel(const uint8_t *__restrict__ packed, uint8_t *__restrict__ out, long long N,
                              long long K, int bits)
{
    const long long row_bytes = K * bits / 8;
    const long long kbs = K / 64;
    const long long unit_bytes = 128LL * bits;
    const long long total = (N + 15) / 16 * 16 * row_bytes;
    const int run_bytes = 2 * bits;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long unit = idx / unit_bytes;
        const int w = static_cast<int>(idx - unit * unit_bytes);
        const long long T = unit / kbs, kb = unit - T * kbs;
        const int run = w / run_bytes, rb = w - run * run_bytes;
        const int h = run >> 5, g = (run >> 2) & 7, t = run & 3;
        const long long n = 16 * T + 8 * h + g;
        out[idx] = n < N ? packed[n * row_bytes + 8LL * bits * kb + 2LL * bits * t + rb] : 0;
    }
}

// Lane-interleaved int4 layout (BitLLM Fig. 6): in every 32-bit word the nibble
// slots hold codes 0 4 1 5 2 6 3 7 of the word's eight, so byte y of word w is
// code 8w + y (low nibble) and code 8w + y + 4 (high nibble).  One thread per
// output byte.
__global__ void interleave4_kernel(const uint8_t *__restrict__ packed, uint8_t *__restrict__ out, long long N,
                                   long long K)
{
    const long long row_bytes = K / 2;
    const long long total = N * row_bytes;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const long long n = idx / row_bytes;
        const long long j = idx - n * row_bytes;
        const uint8_t *row = packed + n * row_bytes;
        const long long k0 = 8 * (j >> 2) + (j & 3), k1 = k0 + 4;
        const uint32_t c0 = (row[k0 >> 1] >> (4 * (k0 & 1))) & 15u;
        const uint32_t c1 = (row[k1 >> 1] >> (4 * (k1 & 1))) & 15u;
        out[idx] = static_cast<uint8_t>(c0 | (c1 << 4));
    }
}

cudaError_t launch_repack(const uint8_t *packed, uint8_t *out, int N, int K, int bits, int layout,
                          cudaStream_t stream, int num_sms)
{
    const long long total = layout == QMM_LAYOUT_TILE16 ? (long long)(N + 15) / 16 * 16 * K * bits / 8
                                                         : (long long)N * K / 2;
    long long blocks = (total + 255) / 256;
    if (blocks > (long long)num_sms * 16)
        blocks = (long long)num_sms * 16;
    if (layout == QMM_LAYOUT_TILE16)
        tile16_kernel<<<(int)blocks, 256, 0, stream>>>(packed, out, N, K, bits);
    else
        interleave4_kernel<<<(int)blocks, 256, 0, stream>>>(packed, out, N, K);
    return cudaGetLastError();
}

cudaError_t launch_flip_sign(uint8_t *packed, int N, int K, int bits, cudaStream_t stream, int num_sms)
{
    const long long total = (long long)N * K * bits / 8;
    long long blocks = (total + 255) / 256;
    if (blocks > (long long)num_sms * 16)
        blocks = (long long)num_sms * 16;
    flip_sign_kernel<<<(int)blocks, 256, 0, stream>>>(packed, N, K, bits);
    return cudaGetLastError();
}

cudaError_t launch_pack(const uint8_t *codes, uint8_t *packed, int N, int K, int bits,
                        int32_t *bad_count, cudaStream_t stream, int num_sms)
{
    const long long total = (long long)N * K * bits / 8;
    long long blocks = (total + 255) / 256;
    if (blocks > (long long)num_sms * 16)
        blocks = (long long)num_sms * 16;
    pack_kernel<<<(int)blocks, 256, 0, stream>>>(codes, packed, N, K, bits, bad_count);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t *packed, uint8_t *codes, int N, int K, int bits,
                          cudaStream_t stream, int num_sms)
{
    const long long total = (long long)N * K;
    long long blocks = (total + 255) / 256;
    if (blocks > (long long)num_sms * 16)
        blocks = (long long)num_sms * 16;
    unpack_kernel<<<(int)blocks, 256, 0, stream>>>(packed, codes, N, K, bits);
    return cudaGetLastError();
}

}  // namespace qmm
