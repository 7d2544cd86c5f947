// bi_internal.h -- host-side state shared by the translation units of libbi.
// Not part of the public ABI (include/bi.h is).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "bi.h"

namespace bi {

// The numeric contract: the kernels are built from these constants, and
// bi_get_config reports them.  Changing one changes the bits of the results.
constexpr int kRouterSlab = 128;      // h is cut into slabs of 128
constexpr int kRouterBlock = 8;       // each slab into 16 blocks of 8
constexpr int kRouterParts = 16;      // partition q owns block q of every slab
constexpr int kGemmTileM = 128, kGemmTileN = 256;
constexpr int kGemmBlockK = 64;       // K in blocks of 64, increasing
constexpr int kGemmMmaK = 16;         // each block as four 16-deep tensor-core steps
static_assert(kRouterSlab == kRouterBlock * kRouterParts, "a slab is one block per partition");

// Per-device state, created on the first call made with that device current.
struct Device {
    int ordinal = -1;
    int sm_count = 0;
    unsigned int *err = nullptr;   // device address of the sticky error word
    void *scratch = nullptr;       // router partial sums (see router.cu)
    size_t scratch_bytes = 0;
    uint64_t attr_done = 0;        // kernels whose smem attribute is set (bit per kernel id)
};

// The state of the current device (never NULL on BI_OK).
bi_status current_device(Device **out);

// Grow-only device scratch owned by the library (allocated at most a few
// times per device over the process lifetime, never per call).
bi_status device_scratch(Device *d, size_t bytes, void **out);

// cuTensorMapEncodeTiled, resolved once through the runtime.
bi_status encode_tiled(CUtensorMap *map, CUtensorMapDataType dt, uint32_t rank,
                       const void *gaddr, const uint64_t *dims, const uint64_t *strides_bytes,
                       const uint32_t *box, CUtensorMapSwizzle swizzle);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bi_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BI_OK : BI_ERR_CUDA; }

// Launch with programmatic dependent launch enabled: the kernel may start
// while the previous kernel in the stream drains; every kernel of this
// library waits (griddepcontrol.wait) before touching global memory.
template <typename... KArgs, typename... Args>
bi_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t s, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return from_cuda(e);
}

// Once per device and kernel: the dynamic shared memory limit, and the
// largest shared-memory carveout.  Every kernel of the library asks for the
// same carveout, so a small kernel resident on an SM never leaves it
// configured for less shared memory than the next large-tile block needs
// (an SM changes its carveout only when it is empty, so a mismatch would
// make the large block wait for the small one to finish).
template <typename K>
bi_status set_smem_once(Device *d, int kernel_id, K kernel, size_t bytes)
{
    uint64_t bit = 1ull << kernel_id;
    if (d->attr_done & bit) return BI_OK;
    if (bytes > 0 &&
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
        return BI_ERR_CUDA;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared) != cudaSuccess)
        return BI_ERR_CUDA;
    d->attr_done |= bit;
    return BI_OK;
}

// kernel ids for set_smem_once (one bit each)
enum : int {
    KID_ROUTER_PROJ = 0,   // 10 instantiations: 0..9
    KID_GEMM = 16,
    KID_SELECT = 20,       // 4 instantiations: 20..23 (two group sums or none)
    KID_GATE = 24,
    KID_HASH = 25,         // 4 instantiations: 25..28
    KID_ROUTER_GEMV = 30,  // 2 instantiations (8 tokens per block): 30..31
    KID_SELECT_GATE = 34,  // 4 instantiations: 34..37 (two group sums or none)
    KID_MOE = 40,          // 5 kernels: 40..44
    KID_NORM = 45,         // 2 instantiations: 45..46
    KID_ROUTER_PROJ_SHALLOW = 49,   // 2 instantiations: 49..50
    KID_SELECT_GENERAL = 51,        // 4 instantiations: 51..54
    KID_SELECT_GATE_GENERAL = 55,   // 4 instantiations: 55..58
    KID_ROUTER_GEMV1 = 59,          // 2 instantiations (one token per block): 59..60
};

}  // namespace bi
