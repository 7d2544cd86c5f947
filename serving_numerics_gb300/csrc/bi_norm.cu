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
// pairwise tree.  The row is read twice, eight slabs of loads in flight per
// pass (the second pass finds it in L2; holding whole rows in registers
// instead needs 169 registers per thread and measured slower, two waves of
// rows instead of one).  y is written in 16-byte stores.  Nothing depends
// on M or on the other rows.
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
