// bi_gate.cu -- bi_shared_gate: the one-output shared-expert gate,
// dot = X[m,:] . w_sg and sigmoid(dot) ("batch changed the model's mind",
// "m-scan: the staircase" and "The fix: m-invariant twins").
//
// Same reduction contract as the router: partition q (0..15) owns the 8-wide
// block q of every 128-wide slab of h (h < H only) and runs one f32 FMA chain
// from +0; the 16 partials meet in the pairwise tree (0+1),(2+3),... .
// Half a warp serves one token: lane q of the half is partition q, so one
// slab is a 512-byte coalesced read per token, and the butterfly shuffles
// with offsets 1, 2, 4, 8 reproduce the pairwise tree exactly (fp addition
// is commutative, so both lanes of a pair hold the same sum).
#include "bi_device.cuh"
#include "bi_internal.h"

namespace bi {
namespace {

constexpr int kGateWarps = 8;
// the lane layout below is the contract's: 16 lanes = 16 partitions, 8-wide
// blocks, 128-wide slabs
static_assert(kRouterParts == 16 && kRouterBlock == 8 && kRouterSlab == 128, "gate lane layout");

__global__ void __launch_bounds__(32 * kGateWarps)
shared_gate_kernel(const float *__restrict__ x, const float *__restrict__ w, int M, int H,
                   float *__restrict__ dot, float *__restrict__ sig)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    pdl_wait();
    const int lane = threadIdx.x & 31, q = lane & 15;
    const int m = (blockIdx.x * kGateWarps + (threadIdx.x >> 5)) * 2 + (lane >> 4);
    const bool active = m < M;
    const float *xr = x + (size_t)(active ? m : 0) * H;
    float acc = 0.0f;
    const int ns = (H + 127) / 128;
    int s = 0;
    // four slabs per step so that eight 16-byte loads are in flight per lane
    for (; s + 4 <= ns; s += 4) {
        float4 xv[8], wv[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int h0 = 128 * (s + u) + 8 * q;
            if (h0 < H) {
                xv[2 * u] = *reinterpret_cast<const float4 *>(xr + h0);
                xv[2 * u + 1] = *reinterpret_cast<const float4 *>(xr + h0 + 4);
                wv[2 * u] = *reinterpret_cast<const float4 *>(w + h0);
                wv[2 * u + 1] = *reinterpret_cast<const float4 *>(w + h0 + 4);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int h0 = 128 * (s + u) + 8 * q;
            if (h0 < H) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    acc = __fmaf_rn(xv[2 * u + c].x, wv[2 * u + c].x, acc);
                    acc = __fmaf_rn(xv[2 * u + c].y, wv[2 * u + c].y, acc);
                    acc = __fmaf_rn(xv[2 * u + c].z, wv[2 * u + c].z, acc);
                    acc = __fmaf_rn(xv[2 * u + c].w, wv[2 * u + c].w, acc);
                }
            }
        }
    }
    for (; s < ns; ++s) {
        const int h0 = 128 * s + 8 * q;
        if (h0 < H) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float4 a = *reinterpret_cast<const float4 *>(xr + h0 + 4 * c);
                const float4 b = *reinterpret_cast<const float4 *>(w + h0 + 4 * c);
                acc = __fmaf_rn(a.x, b.x, acc);
                acc = __fmaf_rn(a.y, b.y, acc);
                acc = __fmaf_rn(a.z, b.z, acc);
                acc = __fmaf_rn(a.w, b.w, acc);
            }
        }
    }
#pragma unroll
    for (int d = 1; d < 16; d *= 2) acc = acc + __shfl_xor_sync(0xFFFFFFFFu, acc, d);
    if (active && q == 0) {
        dot[m] = acc;
        if (sig) sig[m] = 1.0f / (1.0f + expf(-acc));
    }
}

}  // namespace
}  // namespace bi

using namespace bi;

extern "C" bi_status bi_shared_gate(const float *x, const float *w_sg, int32_t M, int32_t H,
                                    float *dot_out, float *sigmoid_out, bi_stream s)
{
    if (M < 0 || H <= 0) return BI_ERR_INVALID_ARG;
    if (H > BI_MAX_H || (H % 8) != 0 || M > (1 << 24)) return BI_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return BI_OK;
    if (!x || !w_sg || !dot_out) return BI_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_sg) || (reinterpret_cast<uintptr_t>(dot_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(sigmoid_out) & 3u))
        return BI_ERR_MISALIGNED;
    Device *d = nullptr;
    bi_status st = current_device(&d);
    if (st != BI_OK) return st;
    if ((st = set_smem_once(d, KID_GATE, shared_gate_kernel, 0)) != BI_OK) return st;
    const int tokens_per_block = 2 * kGateWarps;
    dim3 grid((M + tokens_per_block - 1) / tokens_per_block);
    return launch_pdl(shared_gate_kernel, grid, dim3(32 * kGateWarps), 0,
                      reinterpret_cast<cudaStream_t>(s), x, w_sg, (int)M, (int)H, dot_out, sigmoid_out);
}
