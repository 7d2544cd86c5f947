// bi_runtime.cu -- per-device state, the sticky device error word, tensor-map
// encoding and the small ABI utilities (status strings, version).
#include <limits.h>
#include <string.h>

#include <mutex>

#include "bi_device.cuh"
#include "bi_internal.h"

namespace bi {

static_assert(kErrTimeout == (unsigned int)BI_ERR_TIMEOUT, "the device code of a wait that ran out");

// Sticky error word: a kernel that gives up a bounded wait records
// (status | where << 8) here; bi_get_last_device_error() reads and clears it.
__device__ unsigned int g_device_error;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
Device g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

bi_status current_device(Device **out)
{
    int ord = -1;
    if (cudaGetDevice(&ord) != cudaSuccess || ord < 0 || ord >= kMaxDevices) return BI_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    Device &d = g_dev[ord];
    if (d.ordinal < 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ord) != cudaSuccess)
            return BI_ERR_CUDA;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return BI_ERR_CUDA;
        d.sm_count = sms;
        d.err = static_cast<unsigned int *>(p);
        d.ordinal = ord;
    }
    *out = &d;
    return BI_OK;
}

bi_status encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, uint32_t rank,
                       const void *gaddr, const uint64_t *dims, const uint64_t *strides_bytes,
                       const uint32_t *box, CUtensorMapSwizzle swizzle)
{
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return BI_ERR_CUDA;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = g_encode(map, dt, rank, const_cast<void *>(gaddr),
                          reinterpret_cast<const cuuint64_t *>(dims),
                          reinterpret_cast<const cuuint64_t *>(strides_bytes),
                          reinterpret_cast<const cuuint32_t *>(box), estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? BI_OK : BI_ERR_CUDA;
}

namespace {
// One thread waits on an mbarrier that nothing ever arrives at; the bounded
// wait gives up after limit_ns and records BI_ERR_TIMEOUT (where = 0xFE).
__global__ void selftest_wait_kernel(unsigned int *err, unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait_limit(&bar, 0, err, 0xFEu, limit_ns);
}
// FP32 FMA rate probe: every thread runs 8 independent fused multiply-add
// chains in registers (enough independent work to fill the FMA pipe), and
// one thread per block writes a value that depends on all of them so that
// nothing is optimised away.  PACKED runs each chain as a pair of lanes of
// the two-wide f32 FMA (fma.rn.f32x2: two independent f32 fused
// multiply-adds, each rounded once, in one instruction).
constexpr int kFmaChains = 8;

template <bool PACKED>
__global__ void __launch_bounds__(256) fma_rate_kernel(int iters, float a, float b, float *sink)
{
    float t = 0.0f;
    if constexpr (!PACKED) {
        float x[kFmaChains];
#pragma unroll
        for (int c = 0; c < kFmaChains; ++c) x[c] = (float)(threadIdx.x + c);
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int u = 0; u < 16; ++u) {
#pragma unroll
                for (int c = 0; c < kFmaChains; ++c) x[c] = __fmaf_rn(x[c], a, b);
            }
        }
#pragma unroll
        for (int c = 0; c < kFmaChains; ++c) t += x[c];
    } else {
        uint64_t x[kFmaChains];
        const uint64_t a2 = (uint64_t)__float_as_uint(a) | ((uint64_t)__float_as_uint(a) << 32);
        const uint64_t b2 = (uint64_t)__float_as_uint(b) | ((uint64_t)__float_as_uint(b) << 32);
#pragma unroll
        for (int c = 0; c < kFmaChains; ++c)
            x[c] = (uint64_t)__float_as_uint((float)(threadIdx.x + c)) |
                   ((uint64_t)__float_as_uint((float)(threadIdx.x + 2 * c)) << 32);
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int u = 0; u < 16; ++u) {
#pragma unroll
                for (int c = 0; c < kFmaChains; ++c)
                    asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[c]) : "l"(a2), "l"(b2));
            }
        }
#pragma unroll
        for (int c = 0; c < kFmaChains; ++c)
            t += __uint_as_float((uint32_t)x[c]) + __uint_as_float((uint32_t)(x[c] >> 32));
    }
    if (t == 12345.678f) sink[blockIdx.x] = t;     // practically never true; keeps the chains live
}
}  // namespace

}  // namespace bi

extern "C" {

bi_status bi_selftest_fma_rate(int32_t iters, int32_t packed, float *sink, bi_stream s, double *flops_launched)
{
    if (iters < 1 || iters > (1 << 20) || (packed != 0 && packed != 1) || !sink || !flops_launched)
        return BI_ERR_INVALID_ARG;
    bi::Device *d = nullptr;
    bi_status st = bi::current_device(&d);
    if (st != BI_OK) return st;
    const int blocks = 8 * d->sm_count;      // 8 blocks of 256 threads per SM: 64 warps
    *flops_launched = 2.0 * blocks * 256.0 * (double)iters * 16.0 * bi::kFmaChains * (packed ? 2 : 1);
    if (packed)
        bi::fma_rate_kernel<true><<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(s)>>>(iters, 0.999f, 0.001f, sink);
    else
        bi::fma_rate_kernel<false><<<blocks, 256, 0, reinterpret_cast<cudaStream_t>(s)>>>(iters, 0.999f, 0.001f, sink);
    return bi::from_cuda(cudaGetLastError());
}

bi_status bi_selftest_wait_timeout(uint32_t limit_us, bi_stream s)
{
    if (limit_us == 0 || limit_us > 2000000u) return BI_ERR_INVALID_ARG;
    bi::Device *d = nullptr;
    bi_status st = bi::current_device(&d);
    if (st != BI_OK) return st;
    bi::selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(s)>>>(d->err,
                                                                          1000ull * limit_us);
    return bi::from_cuda(cudaGetLastError());
}

const char *bi_status_string(bi_status st)
{
    switch (st) {
    case BI_OK: return "BI_OK";
    case BI_ERR_INVALID_ARG: return "BI_ERR_INVALID_ARG: a pointer is NULL or a size is negative or inconsistent";
    case BI_ERR_UNSUPPORTED_SHAPE: return "BI_ERR_UNSUPPORTED_SHAPE: a size is outside the library's limits";
    case BI_ERR_MISALIGNED: return "BI_ERR_MISALIGNED: a pointer or stride is not 16-byte aligned";
    case BI_ERR_CUDA: return "BI_ERR_CUDA: the CUDA runtime reported an error";
    case BI_ERR_TIMEOUT: return "BI_ERR_TIMEOUT: a device-side bounded wait ran out";
    }
    return "unknown bi_status";
}

bi_status bi_get_last_device_error(void)
{
    unsigned int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return BI_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, bi::g_device_error, sizeof v) != cudaSuccess) return BI_ERR_CUDA;
    unsigned int zero = 0;
    if (cudaMemcpyToSymbol(bi::g_device_error, &zero, sizeof zero) != cudaSuccess) return BI_ERR_CUDA;
    return static_cast<bi_status>(v & 0xFFu);
}

int32_t bi_abi_version(void) { return BI_ABI_VERSION; }

bi_status bi_get_config(bi_config *out, size_t out_size)
{
    if (!out || out_size < 2 * sizeof(int32_t)) return BI_ERR_INVALID_ARG;
    bi_config c;
    memset(&c, 0, sizeof c);
    c.struct_size = (int32_t)sizeof(bi_config);
    c.abi_version = BI_ABI_VERSION;
    c.router_slab = bi::kRouterSlab;
    c.router_block = bi::kRouterBlock;
    c.router_partitions = bi::kRouterParts;
    c.router_partition_order = 1;
    c.router_tree = BI_TREE_PAIRWISE;
    c.router_accum = BI_F32;
    c.gemm_tile_m = bi::kGemmTileM;
    c.gemm_tile_n = bi::kGemmTileN;
    c.gemm_block_k = bi::kGemmBlockK;
    c.gemm_mma_k = bi::kGemmMmaK;
    c.gemm_accum = BI_F32;
    c.gemm_split_k = 0;
    c.topk_tie_rule = 1;
    c.softmax_sum_order = 1;
    memcpy(out, &c, out_size < sizeof c ? out_size : sizeof c);
    return BI_OK;
}

bi_status bi_prefix_split(const int32_t *lengths, int32_t n_requests, int32_t block, int32_t *cached_out,
                          int32_t *suffix_offsets_out)
{
    if (!lengths || !cached_out || !suffix_offsets_out || n_requests < 0 || block < 1) return BI_ERR_INVALID_ARG;
    int64_t total = 0;
    for (int32_t r = 0; r < n_requests; ++r) {
        if (lengths[r] < 0) return BI_ERR_INVALID_ARG;
        total += lengths[r];
    }
    if (total > INT32_MAX) return BI_ERR_INVALID_ARG;
    int32_t off = 0;
    suffix_offsets_out[0] = 0;
    for (int32_t r = 0; r < n_requests; ++r) {
        const int32_t n = lengths[r];
        int32_t suffix = n % block;            // rows past the last full block
        if (suffix == 0) suffix = n < block ? n : block;   // none: recompute the last full block
        cached_out[r] = n - suffix;
        off += suffix;
        suffix_offsets_out[r + 1] = off;
    }
    return BI_OK;
}

}  // extern "C"
