// bi_internal.h -- host-side state shared by the translation units of libbi.
// Not part of the public ABI (include/bi.h is).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>

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
// The library keeps no device buffers of its own beyond the sticky error word
// (and the fixed array of bi_router_topk_noalloc): every call's working
// memory is the caller's.
struct Device {
    int ordinal = -1;
    int sm_count = 0;
    unsigned int *err = nullptr;   // device address of the sticky error word
    // kernels whose attributes are set (bit per kernel id); concurrent first
    // calls from several host threads may both set them, which is harmless
    std::atomic<uint64_t> attr_done[2] = {};
    // whether one block of the persistent router projection fits an SM
    // (f32, bf16 inputs; without, with the shared gate): -1 not yet asked,
    // 0 no, 1 yes
    std::atomic<int> persist_fits[4] = {-1, -1, -1, -1};
};

// The state of the current device (never NULL on BI_OK).
bi_status current_device(Device **out);

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

// Once per device and kernel: run `set` (which sets the kernel's function
// attributes and returns false on a CUDA error) unless it already succeeded.
template <typename F>
bi_status set_attr_once(Device *d, int kernel_id, F &&set)
{
    const uint64_t bit = 1ull << (kernel_id & 63);
    std::atomic<uint64_t> &word = d->attr_done[kernel_id >> 6];
    if (word.load(std::memory_order_acquire) & bit) return BI_OK;
    if (!set()) return BI_ERR_CUDA;
    word.fetch_or(bit, std::memory_order_acq_rel);
    return BI_OK;
}

// The dynamic shared memory limit and the largest shared-memory carveout.
// Every kernel of the library asks for the same carveout, so a small kernel
// resident on an SM never leaves it configured for less shared memory than
// the next large-tile block needs (an SM changes its carveout only when it
// is empty, so a mismatch would make the large block wait for the small one
// to finish).
template <typename K>
bi_status set_smem_once(Device *d, int kernel_id, K kernel, size_t bytes)
{
    return set_attr_once(d, kernel_id, [&]() -> bool {
        if (bytes > 0 &&
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
            return false;
        return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    (int)cudaSharedmemCarveoutMaxShared) == cudaSuccess;
    });
}

// kernel ids for set_attr_once (one bit each, 128 in all)
enum : int {
    KID_ROUTER_PROJ = 0,   // 10 instantiations: 0..9
    KID_GEMM = 16,
    KID_SELECT = 20,       // 4 instantiations: 20..23 (two group sums or none)
    KID_GATE = 24,
    KID_HASH = 25,         // 4 instantiations: 25..28
    KID_SELECT_GATE = 34,  // 4 instantiations: 34..37 (two group sums or none)
    KID_MOE = 40,          // 5 kernels: 40..44
    KID_NORM = 45,         // 2 instantiations: 45..46
    KID_ROUTER_PROJ_SHALLOW = 49,   // 2 instantiations: 49..50
    KID_SELECT_GENERAL = 51,        // 4 instantiations: 51..54
    KID_SELECT_GATE_GENERAL = 55,   // 4 instantiations: 55..58
    KID_ROUTER_CLUSTER = 64,        // 10 instantiations: 64..73
    KID_FLOOR = 74,
    KID_ROUTER_PERSIST = 75,        // 4 instantiations: 75..78
    KID_ATTN = 79,                  // 2 instantiations: 79..80
};

// Batches of at most this many rows (and E <= kClusterMaxE) take the
// one-launch cluster router (csrc/bi_router_cluster.cu); larger ones the
// tiled projection + selection.  112 = 7 clusters of 16 tokens, the clusters
// of 16 blocks a GB300 places at once.
constexpr int kClusterMaxM = 112, kClusterMaxE = 512;

// How the cluster router cuts one call (see bi_router_cluster.cu).
struct ClusterPlan {
    bool ok;          // false: the cluster router does not apply to this call
    int CS;           // blocks per cluster (each owns E / CS experts)
    int TM, NT;       // tokens per cluster; the compiled token tile (>= TM)
    int NC;           // clusters
    int warps;        // warps per block
    int Eb4;          // gate rows per block, rounded up to a multiple of 4
    int nst, stage_bytes, x_off, g_off, gather_off, tile_off, smem;   // shared-memory layout
};

ClusterPlan cluster_plan(Device *d, int M, int E, int H, int es, bool gate);

bi_status router_cluster_call(Device *d, const ClusterPlan &p, const void *x, const void *w_gate, bool f32in,
                              int logit_bf16, int M, int H, int E, int k, void *logits, int32_t *ids,
                              float *weights, float *margin, int32_t *ulps, const void *w_sg, float *gdot,
                              float *gsig, cudaStream_t s);

// The persistent projection for large batches (csrc/bi_router_persist.cu).
// Workspace layout of that plan: the call epoch (one word), the hand-off
// flags (16 words per CTA), the hand-off accumulators (128 KB per CTA), the
// shared gate's hand-off (2 KB per CTA), then the two halves' group sums
// [2][M][E] and the gate's [2][M], read by the selection kernel.
constexpr int kPersistMaxCtas = 160;        // CTAs at most (one per SM)
constexpr int kPersistMinItems = 128;       // below this many items the split plans are used
constexpr long long kPersistSumsMax = 64ll << 20;
constexpr int kPersistFlagsPerCta = 16;     // 8 compute warps, 2 gate warps, spare
constexpr size_t kPersistFlagsOffset = 256;
constexpr size_t kPersistHandoffOffset = 16384;
constexpr size_t kPersistGateHandoffOffset = kPersistHandoffOffset + (size_t)kPersistMaxCtas * 8 * 128 * 32 * 4;
constexpr size_t kPersistGroupSumsOffset = kPersistGateHandoffOffset + (size_t)kPersistMaxCtas * 8 * 2 * 32 * 4;
static_assert(kPersistFlagsOffset + (size_t)kPersistMaxCtas * kPersistFlagsPerCta * 4 <= kPersistHandoffOffset,
              "flag words");

struct PersistArgs {
    int M, E, H, n_et, ns, n_items;
    float *part;              // group sums [2][M][E]
    unsigned int *epoch;      // advanced by the selection kernel of each call
    unsigned int *flags;      // [G][kPersistFlagsPerCta]
    float *handoff;           // [G][8][128][32]
    const void *w_sg;         // the shared gate's row (NULL: no gate)
    float *gpart;             // the gate's group sums [2][M]
    float *ghandoff;          // [G][2 gate warps][8 partitions][32]
    unsigned int *err;
};

struct PersistPlan {
    bool ok;
    int G, n_et, n_items;
};

PersistPlan persist_plan(Device *d, int M, int E, bool f32in, bool gate);
size_t persist_workspace_bytes(long long M, long long E);
bi_status launch_persist(Device *d, const PersistPlan &p, bool f32in, const void *x, const void *w,
                         const void *w_sg, int M, int E, int H, void *workspace, cudaStream_t s);

}  // namespace bi
