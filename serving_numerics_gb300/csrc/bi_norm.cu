// bi_norm.cu -- bi_rmsnorm: batch-invariant RMSNorm ("The Illusion of
// Determinism in Disaggregated Inference", section "The physics of the
// cascade": one root-mean-square over the whole hidden state divides every
// element, so its reduction order decides every output of the row).
//
//   ss[m]   = sum_h x[m, h]^2     in the router's reduction contract: h cut
//             into slabs of 128 and blocks of 8, partition q (0..15) runs
//             one f32 fused multiply-add chain over block q of every slab
//             from +0, the 16 partials added by the pairwise tree
//   r[m]    = 1 / sqrt(ss[m] / H + eps)   (each operation rounded once)
//   y[m, h] = bf16_rne((x[m, h] * r[m]) * w[h])
//
// Half a warp per row, lane q = partition q (the shared gate's layout): the
// butterfly shuffles with offsets 1, 2, 4, 8 add the partials in the
// pairwise tree.  y is written in 16-byte stores.  Nothing depends on M or
// on the other rows.
//
// Two kernels compute exactly that, differing only in how x reaches the
// lanes:
//  - rmsnorm_staged_kernel (rows of at most 3072 f32 / 6144 bf16 values):
//    each row is read from device memory once.  A persistent block of four
//    warps owns groups of 8 consecutive rows (one contiguous span of x); TMA
//    stages each group into a ring of shared-memory stages, the sum of
//    squares and then the output read the staged row, and w is staged once
//    per block.  f32 rows are staged with the 32-byte swizzle, so that the
//    16 lanes of a half-warp reading the first (then the second) 16 bytes of
//    their 8-value blocks meet each bank at most twice.
//  - rmsnorm_kernel (longer rows): the row is read twice from device memory,
//    eight slabs of loads in flight per pass (the second pass finds it in
//    L2; holding whole rows in registers instead needs 169 registers per
//    thread and measured slower, two waves of rows instead of one).
#include <cuda_bf16.h>

#include "bi_device.cuh"
#include "bi_internal.h"

namespace bi {
namespace {

constexpr int kNormWarps = 8;
static_assert(kRouterParts == 16 && kRouterBlock == 8 && kRouterSlab == 128, "norm lane layout");

__device__ __forceinline__ void ld8(const float *p, float (&v)[8])
{
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void ld8(const __nv_bfloat16 *p, float (&v)[8])
{
    const uint4 r = *reinterpret_cast<const uint4 *>(p);
    v[0] = bf16lo(r.x); v[1] = bf16hi(r.x); v[2] = bf16lo(r.y); v[3] = bf16hi(r.y);
    v[4] = bf16lo(r.z); v[5] = bf16hi(r.z); v[6] = bf16lo(r.w); v[7] = bf16hi(r.w);
}

__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&v);
}

constexpr int kStreamSlabs = 8;

// Two passes over the row (the second re-reads it from L2), kStreamSlabs
// slabs of loads in flight per pass.
template <typename InT>
__global__ void __launch_bounds__(32 * kNormWarps)
rmsnorm_kernel(const InT *__restrict__ x, const InT *__restrict__ w, int M, int H, float eps,
               __nv_bfloat16 *__restrict__ y, float *__restrict__ rstd)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    pdl_wait();
    const int lane = threadIdx.x & 31, q = lane & 15;
    const int m = (blockIdx.x * kNormWarps + (threadIdx.x >> 5)) * 2 + (lane >> 4);
    const bool active = m < M;
    const InT *xr = x + (size_t)(active ? m : 0) * H;
    const int ns = (H + kRouterSlab - 1) / kRouterSlab;

    float acc = 0.0f;
    for (int s0 = 0; s0 < ns; s0 += kStreamSlabs) {
        float v[kStreamSlabs][8];
#pragma unroll
        for (int u = 0; u < kStreamSlabs; ++u) {
            const int h0 = kRouterSlab * (s0 + u) + kRouterBlock * q;
            if (h0 < H) ld8(xr + h0, v[u]);
        }
#pragma unroll
        for (int u = 0; u < kStreamSlabs; ++u) {
            const int h0 = kRouterSlab * (s0 + u) + kRouterBlock * q;
            if (h0 < H) {
#pragma unroll
                for (int i = 0; i < 8; ++i) acc = __fmaf_rn(v[u][i], v[u][i], acc);
            }
        }
    }
#pragma unroll
    for (int d = 1; d < 16; d *= 2) acc = acc + __shfl_xor_sync(0xFFFFFFFFu, acc, d);
    const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc, (float)H), eps)));
    if (!active) return;
    if (q == 0 && rstd) rstd[m] = r;

    __nv_bfloat16 *yr = y + (size_t)m * H;
    for (int s0 = 0; s0 < ns; s0 += kStreamSlabs / 2) {
        float xv[kStreamSlabs / 2][8], wv[kStreamSlabs / 2][8];
#pragma unroll
        for (int u = 0; u < kStreamSlabs / 2; ++u) {
            const int h0 = kRouterSlab * (s0 + u) + kRouterBlock * q;
            if (h0 < H) {
                ld8(xr + h0, xv[u]);
                ld8(w + h0, wv[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kStreamSlabs / 2; ++u) {
            const int h0 = kRouterSlab * (s0 + u) + kRouterBlock * q;
            if (h0 < H) {
                float o[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = __fmul_rn(__fmul_rn(xv[u][i], r), wv[u][i]);
                uint4 p;
                p.x = pack2(o[0], o[1]);
                p.y = pack2(o[2], o[3]);
                p.z = pack2(o[4], o[5]);
                p.w = pack2(o[6], o[7]);
                *reinterpret_cast<uint4 *>(yr + h0) = p;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// One read of each row: groups of kGroupRows consecutive rows staged by TMA.
constexpr int kStagedWarps = 4, kGroupRows = 2 * kStagedWarps, kStagedMaxStages = 4;
constexpr int kStagedSmemMax = 226 * 1024;
constexpr int kBoxBlocks = 128;       // 8-value blocks per TMA box along a row (1024 values)

// Partition q's 8 values of slab s of a staged row (h increasing).  A group
// is staged box by box: box b holds values [1024 b, 1024 (b + 1)) of the 8
// rows, row after row.  f32 boxes are 32-byte swizzled (halves of block q
// swapped when bit 2 of q is set); bf16 blocks are 16 bytes, unswizzled.
__device__ __forceinline__ void staged8(const uint8_t *grp, int row, int s, int q, float (&v)[8], float)
{
    const int blk = 16 * s + q, box = blk / kBoxBlocks, inb = blk % kBoxBlocks;
    const uint8_t *p = grp + ((size_t)box * kGroupRows + row) * (kBoxBlocks * 32) + inb * 32;
    const int sw = (q >> 2) & 1;
    const float4 a = *reinterpret_cast<const float4 *>(p + 16 * sw);
    const float4 b = *reinterpret_cast<const float4 *>(p + 16 * (sw ^ 1));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void staged8(const uint8_t *grp, int row, int s, int q, float (&v)[8], __nv_bfloat16)
{
    const int blk = 16 * s + q, box = blk / kBoxBlocks, inb = blk % kBoxBlocks;
    const uint4 r = *reinterpret_cast<const uint4 *>(grp + ((size_t)box * kGroupRows + row) * (kBoxBlocks * 16) +
                                                     inb * 16);
    v[0] = bf16lo(r.x); v[1] = bf16hi(r.x); v[2] = bf16lo(r.y); v[3] = bf16hi(r.y);
    v[4] = bf16lo(r.z); v[5] = bf16hi(r.z); v[6] = bf16lo(r.w); v[7] = bf16hi(r.w);
}

struct StagedArgs {
    int M, H, nst, stage_bytes, nbox, w_off;
    float eps;
    __nv_bfloat16 *y;
    float *rstd;
    unsigned int *err;
};

template <typename InT>
__global__ void __launch_bounds__(32 * kStagedWarps, 1)
rmsnorm_staged_kernel(const __grid_constant__ CUtensorMap tmx, const InT *__restrict__ w, StagedArgs a)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    constexpr int ES = (int)sizeof(InT);
    constexpr int BOX_BYTES_ROW = kBoxBlocks * 8 * ES;          // one row's share of a box
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStagedMaxStages];
    __shared__ __align__(8) uint64_t w_bar;
    __shared__ int released[kStagedMaxStages];
    uint8_t *smem = smem_align1024(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, q = lane & 15;
    const int hrow = 2 * warp + (lane >> 4);                     // this half-warp's row in a group
    const int H = a.H, ns = (H + kRouterSlab - 1) / kRouterSlab, NST = a.nst;
    const int groups = (a.M + kGroupRows - 1) / kGroupRows;
    const int G = gridDim.x;
    const int mine = groups > (int)blockIdx.x ? (groups - 1 - (int)blockIdx.x) / G + 1 : 0;
    const InT *ws = reinterpret_cast<const InT *>(smem + a.w_off);

    if (tid == 0) {
        prefetch_tmap(&tmx);
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full_bar[i], 1);
            released[i] = 0;
        }
        mbar_init(&w_bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    auto issue = [&](int j, int slot) {        // this block's j-th group into ring slot `slot`
        const int g = (int)blockIdx.x + j * G;
        uint8_t *st = smem + slot * a.stage_bytes;
        mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)(a.nbox * kGroupRows * BOX_BYTES_ROW));
        for (int bx = 0; bx < a.nbox; ++bx) {
            uint8_t *dst = st + (size_t)bx * kGroupRows * BOX_BYTES_ROW;
            tma_load_3d(dst, &tmx, &full_bar[slot], 0, bx * kBoxBlocks, g * kGroupRows);
        }
    };
    if (tid == 0) {
        // w is a weight, not the preceding kernel's output: staged before the wait
        mbar_arrive_expect_tx(&w_bar, (uint32_t)(H * ES));
        bulk_load(smem + a.w_off, w, (uint32_t)(H * ES), &w_bar);
    }
    pdl_wait();       // x may be the preceding kernel's output
    if (tid == 0)
        for (int j = 0; j < mine && j < NST; ++j) issue(j, j);
    mbar_wait(&w_bar, 0, a.err, 0x46);

    int slot = 0;
    uint32_t phase = 0;
    for (int j = 0; j < mine; ++j) {
        mbar_wait(&full_bar[slot], phase, a.err, 0x45);
        const uint8_t *grp = smem + slot * a.stage_bytes;
        const int m = ((int)blockIdx.x + j * G) * kGroupRows + hrow;
        float acc = 0.0f;
        for (int s = 0; s < ns; ++s) {
            if (kRouterSlab * s + kRouterBlock * q < H) {
                float v[8];
                staged8(grp, hrow, s, q, v, InT());
#pragma unroll
                for (int i = 0; i < 8; ++i) acc = __fmaf_rn(v[i], v[i], acc);
            }
        }
#pragma unroll
        for (int d = 1; d < 16; d *= 2) acc = acc + __shfl_xor_sync(0xFFFFFFFFu, acc, d);
        const float r = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc, (float)H), a.eps)));
        if (m < a.M) {
            if (q == 0 && a.rstd) a.rstd[m] = r;
            __nv_bfloat16 *yr = a.y + (size_t)m * H;
            for (int s = 0; s < ns; ++s) {
                const int h0 = kRouterSlab * s + kRouterBlock * q;
                if (h0 < H) {
                    float v[8], wv[8];
                    staged8(grp, hrow, s, q, v, InT());
                    ld8(ws + h0, wv);
                    float o[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = __fmul_rn(__fmul_rn(v[i], r), wv[i]);
                    uint4 p;
                    p.x = pack2(o[0], o[1]);
                    p.y = pack2(o[2], o[3]);
                    p.z = pack2(o[4], o[5]);
                    p.w = pack2(o[6], o[7]);
                    *reinterpret_cast<uint4 *>(yr + h0) = p;
                }
            }
        }
        // release the slot: the last warp done with it stages group j + NST
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&released[slot], 1) == kStagedWarps - 1) {
                released[slot] = 0;
                if (j + NST < mine) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(j + NST, slot);
                }
            }
        }
        if (++slot == NST) {
            slot = 0;
            phase ^= 1u;
        }
    }
}

}  // namespace
}  // namespace bi

using namespace bi;

extern "C" bi_status bi_rmsnorm(const void *x, const void *w, bi_dtype dtype, int32_t M, int32_t H, float eps,
                                void *y_out, float *rstd_out, bi_stream s)
{
    if (dtype != BI_F32 && dtype != BI_BF16) return BI_ERR_INVALID_ARG;
    if (M < 0 || H <= 0 || !(eps >= 0.0f) || eps > 3.0e38f) return BI_ERR_INVALID_ARG;
    if (H > BI_MAX_H || (H % 8) != 0 || M > (1 << 24)) return BI_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return BI_OK;
    if (!x || !w || !y_out) return BI_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y_out) || (reinterpret_cast<uintptr_t>(rstd_out) & 3u))
        return BI_ERR_MISALIGNED;
    Device *d = nullptr;
    bi_status st = current_device(&d);
    if (st != BI_OK) return st;
    cudaStream_t cs0 = reinterpret_cast<cudaStream_t>(s);
    {
        // one read of each row where a ring of at least two 8-row groups fits
        const int es = dtype == BI_F32 ? 4 : 2;
        const int nbox = (H / 8 + kBoxBlocks - 1) / kBoxBlocks;
        const int stage = ((nbox * kGroupRows * kBoxBlocks * 8 * es) + 1023) & ~1023;
        const int w_bytes = ((H * es) + 1023) & ~1023;
        int nst = (kStagedSmemMax - 1024 - w_bytes) / stage;
        const int groups = (M + kGroupRows - 1) / kGroupRows;
        if (nst > kStagedMaxStages) nst = kStagedMaxStages;
        if (nst >= 2) {
            StagedArgs a;
            a.M = M;
            a.H = H;
            a.nst = nst;
            a.stage_bytes = stage;
            a.nbox = nbox;
            a.w_off = nst * stage;
            a.eps = eps;
            a.y = static_cast<__nv_bfloat16 *>(y_out);
            a.rstd = rstd_out;
            a.err = d->err;
            const size_t smem = (size_t)a.w_off + w_bytes + 1024;
            const int grid = groups < d->sm_count ? groups : d->sm_count;
            alignas(64) CUtensorMap tmx;
            if (dtype == BI_F32) {
                const uint64_t dims[3] = {8, (uint64_t)H / 8, (uint64_t)M};
                const uint64_t str[2] = {32, (uint64_t)H * 4};
                const uint32_t box[3] = {8, (uint32_t)kBoxBlocks, (uint32_t)kGroupRows};
                if ((st = encode_tiled(&tmx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, x, dims, str, box,
                                       CU_TENSOR_MAP_SWIZZLE_32B)) != BI_OK)
                    return st;
                auto kern = rmsnorm_staged_kernel<float>;
                if ((st = set_smem_once(d, KID_NORM + 2, kern, kStagedSmemMax)) != BI_OK) return st;
                return launch_pdl(kern, dim3(grid), dim3(32 * kStagedWarps), smem, cs0, tmx,
                                  static_cast<const float *>(w), a);
            }
            const uint64_t dims[3] = {8, (uint64_t)H / 8, (uint64_t)M};
            const uint64_t str[2] = {16, (uint64_t)H * 2};
            const uint32_t box[3] = {8, (uint32_t)kBoxBlocks, (uint32_t)kGroupRows};
            if ((st = encode_tiled(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, x, dims, str, box,
                                   CU_TENSOR_MAP_SWIZZLE_NONE)) != BI_OK)
                return st;
            auto kern = rmsnorm_staged_kernel<__nv_bfloat16>;
            if ((st = set_smem_once(d, KID_NORM + 3, kern, kStagedSmemMax)) != BI_OK) return st;
            return launch_pdl(kern, dim3(grid), dim3(32 * kStagedWarps), smem, cs0, tmx,
                              static_cast<const __nv_bfloat16 *>(w), a);
        }
    }
    const int rows_per_block = 2 * kNormWarps;
    dim3 grid((M + rows_per_block - 1) / rows_per_block), block(32 * kNormWarps);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(y_out);
    if (dtype == BI_F32) {
        if ((st = set_smem_once(d, KID_NORM + 0, rmsnorm_kernel<float>, 0)) != BI_OK) return st;
        return launch_pdl(rmsnorm_kernel<float>, grid, block, 0, cs, static_cast<const float *>(x),
                          static_cast<const float *>(w), (int)M, (int)H, eps, y, rstd_out);
    }
    auto kern = rmsnorm_kernel<__nv_bfloat16>;
    if ((st = set_smem_once(d, KID_NORM + 1, kern, 0)) != BI_OK) return st;
    return launch_pdl(kern, grid, block, 0, cs, static_cast<const __nv_bfloat16 *>(x),
                      static_cast<const __nv_bfloat16 *>(w), (int)M, (int)H, eps, y, rstd_out);
}
