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
// pairwise tree.  One block per SM takes an equal share of the rows and
// copies all of them (up to the shared memory it has) into shared memory at
// once, each row on its own barrier, so every row's read is in flight from
// the start and each half-warp starts on its row as soon as it lands; the
// sum of squares and the output both read the staged row, w is staged once
// per block.  y is written in 16-byte stores.  Nothing depends on M or on
// the other rows.  (Same-box timings at M = 4096, H = 2048: 12.3 us against
// 14.2 us for a two-pass kernel that read each row twice; loading each
// lane's two 16-byte halves in swapped order to spread a half-warp over all
// bank groups measured slower, 13.9 us.)
#include <cuda_bf16.h>

#include <algorithm>

#include "bi_device.cuh"
#include "bi_internal.h"

namespace bi {
namespace {

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

constexpr int kNormMaxRows = 32;                // rows a block stages at once (half a warp each)
constexpr int kNormSmemMax = 226 * 1024;         // dynamic; 227 KB a block with the static barriers

// Rows [m_begin, m_end) of block b: an equal share, staged in chunks of at
// most `chunk` rows (one chunk when they fit the shared memory at once).
// stage_w: w is staged too (rows so long that w and one row do not fit
// together read w from device memory instead).
template <typename InT>
__global__ void __launch_bounds__(16 * kNormMaxRows, 1)
rmsnorm_kernel(const InT *__restrict__ x, const InT *__restrict__ w, int M, int H, float eps,
               __nv_bfloat16 *__restrict__ y, float *__restrict__ rstd, int rows_per_block, int chunk,
               int stage_w, unsigned int *err)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t row_bar[kNormMaxRows];
    __shared__ __align__(8) uint64_t w_bar;
    uint8_t *smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
    const uint32_t row_bytes = (uint32_t)H * sizeof(InT);
    const uint32_t w_span = stage_w ? (row_bytes + 127u) & ~127u : 0u;
    const InT *ws = stage_w ? reinterpret_cast<const InT *>(smem) : w;
    uint8_t *rows = smem + w_span;

    const int tid = threadIdx.x, r_loc = tid >> 4, q = tid & 15;
    const int m_begin = blockIdx.x * rows_per_block;
    const int m_end = min(M, m_begin + rows_per_block);
    const int ns = (H + kRouterSlab - 1) / kRouterSlab;
    if (tid == 0) {
        for (int r = 0; r < kNormMaxRows; ++r) mbar_init(&row_bar[r], 1);
        mbar_init(&w_bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (stage_w && tid == 0) {     // w is a weight, not a preceding kernel's output
        mbar_arrive_expect_tx(&w_bar, row_bytes);
        bulk_load(smem, w, row_bytes, &w_bar);
    }
    pdl_wait();
    bool ok = true;        // every wait of this thread completed
    if (stage_w) ok &= mbar_wait(&w_bar, 0, err, 0x30);

    // every block has rows: the grid is cut so that m_begin < m_end
    uint32_t parity = 0;
    int nrows = 0;
    for (int c0 = m_begin;; c0 += chunk, parity ^= 1u) {
        nrows = min(chunk, m_end - c0);
        if (tid == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // the previous chunk's reads first
            for (int r = 0; r < nrows; ++r) {
                mbar_arrive_expect_tx(&row_bar[r], row_bytes);
                bulk_load(rows + (size_t)r * row_bytes, x + (size_t)(c0 + r) * H, row_bytes, &row_bar[r]);
            }
        }
        if (r_loc < nrows) {
            const int m = c0 + r_loc;
            ok &= mbar_wait(&row_bar[r_loc], parity, err, 0x31);
            const InT *xr = reinterpret_cast<const InT *>(rows + (size_t)r_loc * row_bytes);
            float acc = 0.0f;
            for (int s0 = 0; s0 < ns; ++s0) {
                const int h0 = kRouterSlab * s0 + kRouterBlock * q;
                if (h0 < H) {
                    float v[8];
                    ld8(xr + h0, v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc = __fmaf_rn(v[i], v[i], acc);
                }
            }
#pragma unroll
            for (int d = 1; d < 16; d *= 2) acc = acc + __shfl_xor_sync(0xFFFFu << (tid & 16), acc, d);
            const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc, (float)H), eps)));
            if (q == 0 && rstd) rstd[m] = rs;
            __nv_bfloat16 *yr = y + (size_t)m * H;
            for (int s0 = 0; s0 < ns; ++s0) {
                const int h0 = kRouterSlab * s0 + kRouterBlock * q;
                if (h0 < H) {
                    float xv[8], wv[8], o[8];
                    ld8(xr + h0, xv);
                    ld8(ws + h0, wv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = __fmul_rn(__fmul_rn(xv[i], rs), wv[i]);
                    uint4 p;
                    p.x = pack2(o[0], o[1]);
                    p.y = pack2(o[2], o[3]);
                    p.z = pack2(o[4], o[5]);
                    p.w = pack2(o[6], o[7]);
                    *reinterpret_cast<uint4 *>(yr + h0) = p;
                }
            }
        }
        // the last chunk; else every staged row is read before the next
        // chunk's copies, and after a wait that gave up none is issued
        if (c0 + chunk >= m_end || __syncthreads_or(!ok)) break;
    }
    // a wait gave up: the rows still landing finish before the block exits
    if (__syncthreads_or(!ok) && tid == 0) {
        for (int r = 0; r < nrows; ++r) mbar_drain(&row_bar[r], parity);
        if (stage_w) mbar_drain(&w_bar, 0);
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
    // one block per SM, an equal share of rows each; as many rows staged at
    // once as the shared memory holds next to w (at most kNormMaxRows)
    const size_t es = dtype == BI_F32 ? 4 : 2, row_bytes = (size_t)H * es;
    const int stage_w = (long long)((row_bytes + 127) & ~(size_t)127) + (long long)row_bytes + 128 <= kNormSmemMax;
    const size_t w_span = stage_w ? (row_bytes + 127) & ~(size_t)127 : 0;
    const int blocks = (int)std::min<long long>(d->sm_count, M);
    const int per_block = (int)((M + blocks - 1) / blocks);
    const long long fit = ((long long)kNormSmemMax - 128 - (long long)w_span) / (long long)row_bytes;
    if (fit < 1) return BI_ERR_UNSUPPORTED_SHAPE;      // never for H <= BI_MAX_H
    const int chunk = (int)std::min<long long>({fit, (long long)kNormMaxRows, (long long)per_block});
    const size_t smem = 128 + w_span + (size_t)chunk * row_bytes;
    const dim3 grid((M + per_block - 1) / per_block), block(16 * ((chunk + 1) & ~1));
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    __nv_bfloat16 *y = static_cast<__nv_bfloat16 *>(y_out);
    if (dtype == BI_F32) {
        if ((st = set_smem_once(d, KID_NORM + 0, rmsnorm_kernel<float>, kNormSmemMax)) != BI_OK) return st;
        return launch_pdl(rmsnorm_kernel<float>, grid, block, smem, cs, static_cast<const float *>(x),
                          static_cast<const float *>(w), (int)M, (int)H, eps, y, rstd_out, per_block, chunk, stage_w,
                          d->err);
    }
    auto kern = rmsnorm_kernel<__nv_bfloat16>;
    if ((st = set_smem_once(d, KID_NORM + 1, kern, kNormSmemMax)) != BI_OK) return st;
    return launch_pdl(kern, grid, block, smem, cs, static_cast<const __nv_bfloat16 *>(x),
                      static_cast<const __nv_bfloat16 *>(w), (int)M, (int)H, eps, y, rstd_out, per_block, chunk,
                      stage_w, d->err);
}
