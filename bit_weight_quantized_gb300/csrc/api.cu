// api.cu -- the C ABI of libqmm (include/qmm.h): argument checks, device
// facts, TMA descriptors and dispatch to the kernels.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "decode.h"
#include "gemv.h"
#include "w4a8.h"
#include "gemm.h"

namespace qmm {

// The library's device status word (one per device that loads the library).
__device__ int g_status_word = 0;

// One warp waits on an mbarrier that nothing arrives at; the bounded wait gives
// up, records QMM_ERR_TIMEOUT and the kernel returns.
__global__ void watchdog_selftest_kernel(int *status)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    mbar_wait(&bar, 0, status);
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceFacts {
    bool ready = false;
    qmm_status usable = QMM_ERR_DEVICE;
    int num_sms = 0;
    int smem_optin = 0;
    int smem_pair = 0;   // per-CTA shared memory with which two CTAs share an SM
    int *status = nullptr;
};

DeviceFacts g_facts[kMaxDevices];
std::mutex g_mutex;
std::atomic<int> g_gemv_kernel{QMM_GEMV_AUTO};

// Facts about the current device, computed once per device.
const DeviceFacts *device_facts()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceFacts &f = g_facts[dev];
    if (!f.ready) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&f.num_sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&f.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        int smem_sm = 0, reserved = 0;
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
        f.smem_pair = (smem_sm / 2 - reserved) / 128 * 128;
        void *addr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&addr, g_status_word);
        if (e != cudaSuccess || major != 10 || minor != 3 || f.num_sms <= 0) {
            cudaGetLastError();
            f.usable = QMM_ERR_DEVICE;
        } else {
            f.status = static_cast<int *>(addr);
            f.usable = QMM_OK;
        }
        f.ready = true;
    }
    return &f;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qmm_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QMM_OK : QMM_ERR_CUDA; }

}  // namespace

// 2-D tensor map over a byte matrix [rows][row_bytes] with a box of
// box_cols bytes x box_rows rows.  Returns false if the driver refuses it.
bool encode_byte_tmap(CUtensorMap *map, const void *base, long long row_bytes, long long rows,
                      int box_cols, int box_rows, bool swizzle128)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D tensor map over a 16-bit matrix [rows][cols] (elements) with the
// 128-byte swizzle, box box_cols x box_rows elements.
bool encode_u16_tmap(CUtensorMap *map, const void *base, long long cols, long long rows,
                     int box_cols, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_u64_tmap(CUtensorMap *map, const void *base, long long cols, long long rows,
                     int box_cols, int box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 8)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

void skinny_set_tma(GemvParams &p)
{
    p.tma = 0;
    if (p.use_bulk && p.pitch % 16 == 0 && p.pitch > 0 && p.pitch <= 2048 && p.row_bytes % 16 == 0 &&
        p.seg_bytes % 16 == 0 && p.rb >= 1 && p.rb <= 256 &&
        static_cast<long long>(p.stage_bytes) >= static_cast<long long>(p.rb) * p.pitch &&
        encode_u64_tmap(&p.tmw, p.packed, p.row_bytes / 8, p.N, p.pitch / 8, p.rb))
        p.tma = 1;
}

// Shared checks of qmm_gemv / qmm_gemm (everything that needs no device).
static qmm_status check_qmm_args(const void *x, const uint8_t *packed, int bits, int group,
                                 const void *scales, int zero_const, const uint8_t *zeros,
                                 void *y, int M, int N, int K)
{
    if (M < 0 || N < 0 || K < 0)
        return QMM_ERR_SHAPE;
    if (bits < 1 || bits > 8)
        return QMM_ERR_BITS;
    if (group != 32 && group != 64 && group != 128)
        return QMM_ERR_SHAPE;
    if (K % group)
        return QMM_ERR_SHAPE;
    if (!zeros && (zero_const < 0 || zero_const > 255))
        return QMM_ERR_SHAPE;
    if (M == 0 || N == 0)
        return QMM_OK;
    if (!y)
        return QMM_ERR_NULL;
    if (K == 0)
        return QMM_OK;
    if (!x || !packed || !scales)
        return QMM_ERR_NULL;
    if (!aligned(x, 16) || !aligned(packed, 4) || !aligned(scales, 2) || !aligned(y, 2))
        return QMM_ERR_ALIGN;
    return QMM_OK;
}

}  // namespace qmm

using namespace qmm;

extern "C" {

int qmm_abi_version(void) { return QMM_ABI_VERSION; }

const char *qmm_status_string(qmm_status s)
{
    switch (s) {
    case QMM_OK: return "ok";
    case QMM_ERR_NULL: return "a required pointer is NULL";
    case QMM_ERR_BITS: return "bits outside the supported range";
    case QMM_ERR_SHAPE: return "invalid shape or group size";
    case QMM_ERR_ALIGN: return "pointer or pitch breaks an alignment rule";
    case QMM_ERR_UNSUPPORTED: return "valid request that is not implemented";
    case QMM_ERR_CUDA: return "CUDA runtime or launch failure";
    case QMM_ERR_TIMEOUT: return "device watchdog expired";
    case QMM_ERR_DEVICE: return "no usable sm_103a device";
    }
    return "unknown status";
}

qmm_status qmm_pack(const uint8_t *codes, uint8_t *packed, int N, int K, int bits,
                    int32_t *bad_count, cudaStream_t stream)
{
    if (bits < 1 || bits > 8)
        return QMM_ERR_BITS;
    if (N < 0 || K < 0 || (static_cast<long long>(K) * bits) % 8)
        return QMM_ERR_SHAPE;
    if (N == 0 || K == 0)
        return QMM_OK;
    if (!codes || !packed)
        return QMM_ERR_NULL;
    if (bad_count && !aligned(bad_count, 4))
        return QMM_ERR_ALIGN;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    return from_cuda(launch_pack(codes, packed, N, K, bits, bad_count, stream, f->num_sms));
}

qmm_status qmm_unpack(const uint8_t *packed, uint8_t *codes, int N, int K, int bits,
                      cudaStream_t stream)
{
    if (bits < 1 || bits > 8)
        return QMM_ERR_BITS;
    if (N < 0 || K < 0 || (static_cast<long long>(K) * bits) % 8)
        return QMM_ERR_SHAPE;
    if (N == 0 || K == 0)
        return QMM_OK;
    if (!codes || !packed)
        return QMM_ERR_NULL;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    return from_cuda(launch_unpack(packed, codes, N, K, bits, stream, f->num_sms));
}

qmm_status qmm_gemv_float(const void *x, const uint8_t *packed, int ebits, int mbits, int group,
                          const void *scales, void *y, int M, int N, int K, cudaStream_t stream)
{
    if (ebits < 1 || mbits < 0 || 1 + ebits + mbits < 2 || 1 + ebits + mbits > 8)
        return QMM_ERR_BITS;
    if (M < 0 || N < 0 || K < 0 || M > 16)
        return QMM_ERR_SHAPE;
    if (group != 32 && group != 64 && group != 128)
        return QMM_ERR_SHAPE;
    if (K % group)
        return QMM_ERR_SHAPE;
    if (M == 0 || N == 0)
        return QMM_OK;
    if (!y)
        return QMM_ERR_NULL;
    if (K > 0 && (!x || !packed || !scales))
        return QMM_ERR_NULL;
    if (!aligned(x, 16) || !aligned(packed, 4) || !aligned(scales, 2) || !aligned(y, 2))
        return QMM_ERR_ALIGN;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    if (K == 0)
        return from_cuda(cudaMemsetAsync(y, 0, static_cast<size_t>(M) * N * 2, stream));
    // codes with at most 4 exponent bits are exact fp16 numbers (times a power
    // of two; a 5-bit exponent field of 31 would read as inf): the decode
    // kernel runs them on the tensor cores
    const int bits = 1 + ebits + mbits;
    DecodePlan plan;
    if (ebits <= 4 && aligned(packed, 16) &&
        decode_plan(M, N, K, group, bits, false, false, f->num_sms, f->smem_pair, f->smem_optin, &plan)) {
        DecodeParams d;
        std::memset(&d, 0, sizeof(d));
        d.x = static_cast<const uint16_t *>(x);
        d.packed = packed;
        d.scales = static_cast<const uint16_t *>(scales);
        d.zeros = nullptr;
        d.y = y;
        d.status = f->status;
        d.row_bytes = static_cast<long long>(K) * bits / 8;
        d.M = M;
        d.N = N;
        d.K = K;
        d.group_log2 = group == 64 ? 6 : 7;
        d.zero_const = 0;
        d.ebits = ebits;
        d.mbits = mbits;
        d.fscale = static_cast<float>(1 << (15 - ((1 << (ebits - 1)) - 1)));
        d.pl = plan;
        decode_set_tma(d);
        return from_cuda(launch_decode_float(d, bits, stream));
    }
    return from_cuda(launch_gemv_fp(static_cast<const uint16_t *>(x), packed, ebits, mbits, group,
                                    static_cast<const uint16_t *>(scales), static_cast<uint16_t *>(y), M, N,
                                    K, stream));
}

qmm_status qmm_flip_sign(uint8_t *packed, int N, int K, int bits, cudaStream_t stream)
{
    if (bits < 1 || bits > 8)
        return QMM_ERR_BITS;
    if (N < 0 || K < 0 || (static_cast<long long>(K) * bits) % 8)
        return QMM_ERR_SHAPE;
    if (N == 0 || K == 0)
        return QMM_OK;
    if (!packed)
        return QMM_ERR_NULL;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    return from_cuda(launch_flip_sign(packed, N, K, bits, stream, f->num_sms));
}

qmm_status qmm_gemv(const void *x, qmm_dtype x_dtype, const uint8_t *packed, int bits,
                    int group, const void *scales, const uint8_t *zeros, int zero_const,
                    void *y, qmm_dtype y_dtype, int M, int N, int K, cudaStream_t stream)
{
    qmm_status st = check_qmm_args(x, packed, bits, group, scales, zero_const, zeros, y, M, N, K);
    if (st != QMM_OK)
        return st;
    if (M > 16)
        return QMM_ERR_SHAPE;
    if ((x_dtype != QMM_F16 && x_dtype != QMM_BF16) || (y_dtype != QMM_F16 && y_dtype != QMM_BF16))
        return QMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0)
        return QMM_OK;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    if (K == 0)
        return from_cuda(cudaMemsetAsync(y, 0, static_cast<size_t>(M) * N * 2, stream));
    DecodePlan plan;
    if (g_gemv_kernel.load(std::memory_order_relaxed) == QMM_GEMV_AUTO && aligned(packed, 16) &&
        decode_plan(M, N, K, group, bits, zeros != nullptr, false, f->num_sms, f->smem_pair, f->smem_optin,
                    &plan)) {
        DecodeParams d;
        std::memset(&d, 0, sizeof(d));
        d.x = static_cast<const uint16_t *>(x);
        d.packed = packed;
        d.scales = static_cast<const uint16_t *>(scales);
        d.zeros = zeros;
        d.y = y;
        d.status = f->status;
        d.row_bytes = static_cast<long long>(K) * bits / 8;
        d.M = M;
        d.N = N;
        d.K = K;
        d.group_log2 = group == 64 ? 6 : 7;
        d.y_bf16 = y_dtype == QMM_BF16;
        d.x_bf16 = x_dtype == QMM_BF16;
        d.zero_const = zeros ? 0 : zero_const;
        d.vec_sz = aligned(scales, 16) && (!zeros || aligned(zeros, 8));
        d.pl = plan;
        decode_set_tma(d);
        return from_cuda(launch_decode(d, bits, false, stream));
    }

    if (x_dtype != QMM_F16)   // the skinny kernel stages fp16 activations only
        return QMM_ERR_UNSUPPORTED;
    GemvParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = static_cast<const uint16_t *>(x);
    p.packed = packed;
    p.scales = static_cast<const uint16_t *>(scales);
    p.zeros = zeros;
    p.y = y;
    p.status = f->status;
    p.row_bytes = static_cast<long long>(K) * bits / 8;
    p.M = M;
    p.N = N;
    p.K = K;
    p.group = group;
    p.ng = K / group;
    p.zero_const = zeros ? 0 : zero_const;
    p.y_bf16 = y_dtype == QMM_BF16;
    int grid = 0, smem = 0;
    st = skinny_plan(p, bits, f->num_sms, f->smem_optin, f->smem_pair, &grid, &smem);
    if (st != QMM_OK)
        return st;
    p.use_bulk = aligned(packed, 16) && p.row_bytes % 16 == 0;
    skinny_set_tma(p);
    cudaError_t e;
    switch (bits) {
    case 1: e = gemv_launch_w1(p, grid, smem, stream); break;
    case 2: e = gemv_launch_w2(p, grid, smem, stream); break;
    case 3: e = gemv_launch_w3(p, grid, smem, stream); break;
    case 4: e = gemv_launch_w4(p, grid, smem, stream); break;
    case 5: e = gemv_launch_w5(p, grid, smem, stream); break;
    case 6: e = gemv_launch_w6(p, grid, smem, stream); break;
    case 7: e = gemv_launch_w7(p, grid, smem, stream); break;
    default: e = gemv_launch_w8(p, grid, smem, stream); break;
    }
    return from_cuda(e);
}

int qmm_gemv_route(int M, int N, int K, int bits, int group, int stored_zeros)
{
    if (M < 1 || M > 16 || N < 1 || K < 1 || bits < 1 || bits > 8 ||
        (group != 32 && group != 64 && group != 128) || K % group)
        return -static_cast<int>(QMM_ERR_SHAPE);
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return -static_cast<int>(QMM_ERR_DEVICE);
    if (g_gemv_kernel.load(std::memory_order_relaxed) != QMM_GEMV_AUTO)
        return QMM_GEMV_SKINNY;
    DecodePlan plan;
    return decode_plan(M, N, K, group, bits, stored_zeros != 0, false, f->num_sms, f->smem_pair, f->smem_optin,
                       &plan)
               ? QMM_GEMV_AUTO
               : QMM_GEMV_SKINNY;
}

size_t qmm_repack_bytes(int N, int K, int bits, int layout)
{
    if (N < 0 || K < 0 || bits < 1 || bits > 8)
        return 0;
    if (layout == QMM_LAYOUT_TILE16)
        return K % 64 ? 0 : static_cast<size_t>((N + 15) / 16) * 16 * K * bits / 8;
    if (layout == QMM_LAYOUT_INTERLEAVE4)
        return bits != 4 || K % 8 ? 0 : static_cast<size_t>(N) * K / 2;
    return 0;
}

qmm_status qmm_repack(const uint8_t *packed, uint8_t *out, int N, int K, int bits, int layout, cudaStream_t stream)
{
    if (bits < 1 || bits > 8)
        return QMM_ERR_BITS;
    if (N < 0 || K < 0 || (layout != QMM_LAYOUT_TILE16 && layout != QMM_LAYOUT_INTERLEAVE4))
        return QMM_ERR_SHAPE;
    if ((layout == QMM_LAYOUT_TILE16 && K % 64) || (layout == QMM_LAYOUT_INTERLEAVE4 && (bits != 4 || K % 8)))
        return QMM_ERR_SHAPE;
    if (N == 0 || K == 0)
        return QMM_OK;
    if (!packed || !out)
        return QMM_ERR_NULL;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    return from_cuda(launch_repack(packed, out, N, K, bits, layout, stream, f->num_sms));
}

qmm_status qmm_gemv_tile16(const void *x, qmm_dtype x_dtype, const uint8_t *tiled, int bits, int group,
                           const void *scales, const uint8_t *zeros, int zero_const, void *y, qmm_dtype y_dtype,
                           int M, int N, int K, cudaStream_t stream)
{
    qmm_status st = check_qmm_args(x, tiled, bits, group, scales, zero_const, zeros, y, M, N, K);
    if (st != QMM_OK)
        return st;
    if (M > 16)
        return QMM_ERR_SHAPE;
    if ((x_dtype != QMM_F16 && x_dtype != QMM_BF16) || (y_dtype != QMM_F16 && y_dtype != QMM_BF16))
        return QMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0)
        return QMM_OK;
    if (K > 0 && !aligned(tiled, 16))
        return QMM_ERR_ALIGN;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    if (K == 0)
        return from_cuda(cudaMemsetAsync(y, 0, static_cast<size_t>(M) * N * 2, stream));
    DecodePlan plan;
    if (!decode_plan(M, N, K, group, bits, zeros != nullptr, true, f->num_sms, f->smem_pair, f->smem_optin, &plan))
        return QMM_ERR_UNSUPPORTED;
    DecodeParams d;
    std::memset(&d, 0, sizeof(d));
    d.x = static_cast<const uint16_t *>(x);
    d.packed = tiled;
    d.scales = static_cast<const uint16_t *>(scales);
    d.zeros = zeros;
    d.y = y;
    d.status = f->status;
    d.row_bytes = static_cast<long long>(K) * bits / 8;
    d.M = M;
    d.N = N;
    d.K = K;
    d.group_log2 = group == 64 ? 6 : 7;
    d.y_bf16 = y_dtype == QMM_BF16;
    d.x_bf16 = x_dtype == QMM_BF16;
    d.zero_const = zeros ? 0 : zero_const;
    d.vec_sz = aligned(scales, 16) && (!zeros || aligned(zeros, 8));
    d.pl = plan;
    return from_cuda(launch_decode(d, bits, true, stream));
}

qmm_status qmm_set_gemv_kernel(int kernel)
{
    if (kernel != QMM_GEMV_AUTO && kernel != QMM_GEMV_SKINNY)
        return QMM_ERR_SHAPE;
    g_gemv_kernel.store(kernel, std::memory_order_relaxed);
    return QMM_OK;
}

qmm_status qmm_gemm(const void *x, qmm_dtype x_dtype, const uint8_t *packed, int bits,
                    int group, const void *scales, const uint8_t *zeros, int zero_const,
                    void *y, qmm_dtype y_dtype, int M, int N, int K, cudaStream_t stream)
{
    qmm_status st = check_qmm_args(x, packed, bits, group, scales, zero_const, zeros, y, M, N, K);
    if (st != QMM_OK)
        return st;
    if (M != 0 && M < 17)
        return QMM_ERR_SHAPE;
    if (x_dtype != y_dtype || (x_dtype != QMM_F16 && x_dtype != QMM_BF16))
        return QMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0)
        return QMM_OK;
    if (K > 0 && (!aligned(x, 16) || !aligned(packed, 16) || !aligned(y, 16) ||
                  (static_cast<long long>(K) * bits / 8) % 16))
        return QMM_ERR_ALIGN;
    if (K > 0 && !gemm_supports_bits(bits))
        return QMM_ERR_UNSUPPORTED;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    if (K == 0)
        return from_cuda(cudaMemsetAsync(y, 0, static_cast<size_t>(M) * N * 2, stream));
    return gemm_dispatch(x, x_dtype == QMM_BF16, packed, bits, group, scales, zeros, zero_const,
                         y, M, N, K, f->status, f->num_sms, f->smem_optin, stream);
}

qmm_status qmm_w4a8(const int8_t *xq, const void *sa, const uint8_t *w4, const void *ws,
                    int group, void *y, int32_t *acc_out, int M, int N, int K,
                    cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0)
        return QMM_ERR_SHAPE;
    if (group != 32 && group != 64 && group != 128)
        return QMM_ERR_SHAPE;
    if (K % group || M > 64)
        return QMM_ERR_SHAPE;
    if (M == 0 || N == 0)
        return QMM_OK;
    if (!y)
        return QMM_ERR_NULL;
    if (K > 0 && (!xq || !sa || !w4 || !ws))
        return QMM_ERR_NULL;
    if (!aligned(xq, 16) || !aligned(w4, 16) || !aligned(ws, 2) || !aligned(sa, 2) ||
        !aligned(y, 2) || (acc_out && !aligned(acc_out, 4)))
        return QMM_ERR_ALIGN;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    if (K == 0) {
        cudaError_t e = cudaMemsetAsync(y, 0, static_cast<size_t>(M) * N * 2, stream);
        return from_cuda(e);
    }
    return wxa8_dispatch(4, xq, sa, w4, ws, group, y, acc_out, M, N, K, f->status, f->num_sms,
                         f->smem_optin, f->smem_pair,
                         g_gemv_kernel.load(std::memory_order_relaxed) == QMM_GEMV_AUTO, stream);
}

qmm_status qmm_w8a8(const int8_t *xq, const void *sa, const int8_t *w8, const void *ws,
                    int group, void *y, int32_t *acc_out, int M, int N, int K,
                    cudaStream_t stream)
{
    if (M < 0 || N < 0 || K < 0)
        return QMM_ERR_SHAPE;
    if (group != 32 && group != 64 && group != 128)
        return QMM_ERR_SHAPE;
    if (K % group || M > 64)
        return QMM_ERR_SHAPE;
    if (M == 0 || N == 0)
        return QMM_OK;
    if (!y)
        return QMM_ERR_NULL;
    if (K > 0 && (!xq || !sa || !w8 || !ws))
        return QMM_ERR_NULL;
    if (!aligned(xq, 16) || !aligned(w8, 16) || !aligned(ws, 2) || !aligned(sa, 2) ||
        !aligned(y, 2) || (acc_out && !aligned(acc_out, 4)))
        return QMM_ERR_ALIGN;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    if (K == 0)
        return from_cuda(cudaMemsetAsync(y, 0, static_cast<size_t>(M) * N * 2, stream));
    return wxa8_dispatch(8, xq, sa, reinterpret_cast<const uint8_t *>(w8), ws, group, y, acc_out, M, N,
                         K, f->status, f->num_sms, f->smem_optin, f->smem_pair,
                         g_gemv_kernel.load(std::memory_order_relaxed) == QMM_GEMV_AUTO, stream);
}

qmm_status qmm_quantize_act(const void *x, int8_t *xq, void *sa, int M, int K, cudaStream_t stream)
{
    if (M < 0 || K < 0 || K % 8)
        return QMM_ERR_SHAPE;
    if (M == 0)
        return QMM_OK;
    if (!sa || (K > 0 && (!x || !xq)))
        return QMM_ERR_NULL;
    if (!aligned(sa, 2) || (K > 0 && (!aligned(x, 16) || !aligned(xq, 16))))
        return QMM_ERR_ALIGN;
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    if (K == 0)   // max over an empty row is 0: every scale is 0
        return from_cuda(cudaMemsetAsync(sa, 0, static_cast<size_t>(M) * 2, stream));
    return from_cuda(launch_quantize_act(static_cast<const uint16_t *>(x), xq, static_cast<uint16_t *>(sa),
                                         M, K, stream));
}

qmm_status qmm_watchdog_selftest(cudaStream_t stream)
{
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>(f->status);
    return from_cuda(cudaGetLastError());
}

qmm_status qmm_device_status(cudaStream_t stream)
{
    const DeviceFacts *f = device_facts();
    if (!f || f->usable != QMM_OK)
        return QMM_ERR_DEVICE;
    if (cudaStreamSynchronize(stream) != cudaSuccess) {
        cudaGetLastError();
        return QMM_ERR_CUDA;
    }
    int v = 0;
    if (cudaMemcpy(&v, f->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return QMM_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        cudaMemcpy(f->status, &zero, sizeof(int), cudaMemcpyHostToDevice);
    }
    return static_cast<qmm_status>(v);
}

}  // extern "C"
