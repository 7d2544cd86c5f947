// bi_moe.cu -- bi_moe_expert_gemm: the grouped expert projection that
// consumes the router's ids and weights ("diag(MODEL-MM-QWEN4-EXP): the MoE
// expert selections DIFFER, and a third of the boundaries are exact bf16
// ties", section "Why a value tap could never have said this": the
// assembled per-slot expert outputs, and the grouped expert GEMM as the
// place where run-to-run differences grow).
//
// Every token-slot (m, j) is one row through expert ids[m, j]:
//   Y[m, j, :] = bf16_rne( X[m, :] . W[ids[m, j]]^T ),  f32 accumulation,
// and the combined row out[m, :] = bf16_rne( sum_j weights[m, j] Y[m, j, :] ),
// an f32 fused multiply-add chain over j = 0 .. k-1 (rank order).
//
// Invariance by construction: the per-expert row counts change with the
// batch, but a row's arithmetic does not depend on them.  Rows are grouped by
// expert into 128-row tiles padded with unused rows, and every tile runs the
// dense projection's schedule (128 x 256 output tile, K in blocks of 64 in
// increasing order, each block as four 16-deep tcgen05 steps, accumulation
// in f32 in tensor memory, one rounding): a row's result is the same in
// whichever tile, at whichever position, next to whichever other rows it
// lands.  The order of rows inside an expert's group is set by atomic
// counters and may differ run to run; nothing numeric depends on it.
//
// Launch sequence (all on the caller's stream, no host synchronisation):
//   plan        one block: rows per expert, padded exclusive scan over the
//               experts -> tile table; resets the cursors and the row map
//   place       one warp per token-slot: claim a row of its expert's group,
//               record it in the row map, copy X[m] there
//   gemm        persistent tcgen05 kernel over the tile table (count of
//               tiles read on the device); the epilogue stores each row
//               straight to its token-slot of Y
//   combine     out[m] from the k rows of Y[m] (when asked for)
#include <cuda_bf16.h>

#include "bi_device.cuh"
#include "bi_internal.h"
#include "bi_tcgen05.cuh"

namespace bi {
namespace {

constexpr int kPlanThreads = 1024;   // the plan kernel's one block: one thread per expert

// Workspace: one caller-owned device buffer, cut into these arrays (each
// 256-byte aligned).  cap = M*k + E*(BM-1) rows, rounded up to BM: every
// expert's rows padded up to whole tiles always fit.
struct MoeWs {
    int32_t *counts, *cursor, *offsets, *ntiles, *tile_row0, *tile_expert, *row_src;
    __nv_bfloat16 *Ag, *Y;
    int64_t cap, max_tiles;
};

size_t moe_layout(int64_t M, int64_t k, int64_t E, int64_t N, int64_t K, uint8_t *base, MoeWs *ws)
{
    const int64_t cap = ((M * k + E * (BM - 1)) + BM - 1) / BM * BM;
    const int64_t max_tiles = cap / BM;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = base ? base + off : nullptr;
        off += (bytes + 255) & ~(size_t)255;
        return p;
    };
    uint8_t *counts = take(sizeof(int32_t) * 2 * E);      // (spare) then the placement cursors
    uint8_t *offsets = take(sizeof(int32_t) * (E + 1));
    uint8_t *ntiles = take(sizeof(int32_t));
    uint8_t *tr0 = take(sizeof(int32_t) * max_tiles);
    uint8_t *tex = take(sizeof(int32_t) * max_tiles);
    uint8_t *rsrc = take(sizeof(int32_t) * cap);
    uint8_t *ag = take(sizeof(__nv_bfloat16) * cap * K);
    uint8_t *y = take(sizeof(__nv_bfloat16) * M * k * N);
    if (ws) {
        ws->counts = reinterpret_cast<int32_t *>(counts);
        ws->cursor = ws->counts ? ws->counts + E : nullptr;
        ws->offsets = reinterpret_cast<int32_t *>(offsets);
        ws->ntiles = reinterpret_cast<int32_t *>(ntiles);
        ws->tile_row0 = reinterpret_cast<int32_t *>(tr0);
        ws->tile_expert = reinterpret_cast<int32_t *>(tex);
        ws->row_src = reinterpret_cast<int32_t *>(rsrc);
        ws->Ag = reinterpret_cast<__nv_bfloat16 *>(ag);
        ws->Y = reinterpret_cast<__nv_bfloat16 *>(y);
        ws->cap = cap;
        ws->max_tiles = max_tiles;
    }
    return off;
}

// One block does the whole plan: rows per expert (a histogram in shared
// memory), each expert's rows padded up to whole tiles, the exclusive scan
// over experts, the tile table (first gathered row and expert of every
// tile), the placement cursors reset to 0 and the padding rows of every
// expert's last tile marked -1 in the row map (the placement writes every
// other row the tiles cover).  An
// id outside [0, E) is recorded in the device error word
// (BI_ERR_INVALID_ARG) and its slot is left out everywhere.
__global__ void __launch_bounds__(kPlanThreads)
moe_plan_kernel(const int32_t *__restrict__ ids, int Mk, int E, int32_t *__restrict__ cursor,
                int32_t *__restrict__ offsets, int32_t *__restrict__ ntiles, int32_t *__restrict__ tile_row0,
                int32_t *__restrict__ tile_expert, int32_t *__restrict__ row_src, unsigned int *err)
{
    pdl_trigger();
    __shared__ int32_t hist[kPlanThreads], scan_t[kPlanThreads];
    const int e = threadIdx.x;
    hist[e] = 0;
    pdl_wait();
    __syncthreads();
    auto count = [&](int x) {
        if (x < 0 || x >= E)
            report_error(err, (unsigned int)BI_ERR_INVALID_ARG, 0x50u);
        else
            atomicAdd(&hist[x], 1);
    };
    // one block is latency-bound on the id loads: 16-byte loads, eight in
    // flight per thread (ids 16-byte aligned; otherwise one id at a time)
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(ids) & 15u) == 0) {
        const int4 *ids4 = reinterpret_cast<const int4 *>(ids);
        const int n4 = Mk / 4;
        for (int base = 0; base < n4; base += 8 * kPlanThreads) {
            int4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int q = base + u * kPlanThreads + e;
                if (q < n4) v[u] = ids4[q];
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (base + u * kPlanThreads + e < n4) {
                    count(v[u].x);
                    count(v[u].y);
                    count(v[u].z);
                    count(v[u].w);
                }
            }
        }
        done = n4 * 4;
    }
    for (int i = done + e; i < Mk; i += kPlanThreads) count(ids[i]);
    __syncthreads();
    const int c = e < E ? hist[e] : 0;
    const int t = (c + BM - 1) / BM;                  // this expert's tiles
    scan_t[e] = t;
    __syncthreads();
    for (int d = 1; d < kPlanThreads; d *= 2) {       // inclusive scan (Hillis-Steele)
        const int v = e >= d ? scan_t[e - d] : 0;
        __syncthreads();
        scan_t[e] += v;
        __syncthreads();
    }
    const int t0 = scan_t[e] - t;                     // exclusive
    if (e < E) {
        offsets[e] = t0 * BM;
        cursor[e] = 0;
        for (int i = 0; i < t; ++i) {
            tile_row0[t0 + i] = (t0 + i) * BM;
            tile_expert[t0 + i] = e;
        }
    }
    // padding rows of every expert's last tile, one warp per expert
    for (int x = e >> 5; x < E; x += kPlanThreads / 32) {
        const int cx = hist[x], end = scan_t[x] * BM;                 // expert x's rows end here
        const int first = end - (cx + BM - 1) / BM * BM + cx;         // its first unclaimed row
        for (int r = first + (e & 31); r < end; r += 32) row_src[r] = -1;
    }
    if (e == kPlanThreads - 1) {
        *ntiles = scan_t[e];
        offsets[E] = scan_t[e] * BM;
    }
}

// One warp per token-slot: claim a row in the expert's group, record where
// it came from, copy X[m] (K bf16) into it.
__global__ void __launch_bounds__(256)
moe_place_kernel(const __nv_bfloat16 *__restrict__ X, const int32_t *__restrict__ ids, int Mk, int k, int K,
                 const int32_t *__restrict__ offsets, int32_t *__restrict__ cursor, int32_t *__restrict__ row_src,
                 __nv_bfloat16 *__restrict__ Ag, int E)
{
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (i >= Mk) return;
    const int e = ids[i];
    if (e < 0 || e >= E) return;
    int p = 0;
    if (lane == 0) p = atomicAdd(&cursor[e], 1);
    p = __shfl_sync(0xFFFFFFFFu, p, 0);
    const int64_t pos = (int64_t)offsets[e] + p;
    if (lane == 0) row_src[pos] = i;
    const uint4 *src = reinterpret_cast<const uint4 *>(X + (int64_t)(i / k) * K);
    uint4 *dst = reinterpret_cast<uint4 *>(Ag + pos * K);
    const int n16 = K / 8;                            // 16-byte pieces of the row
    for (int c0 = 0; c0 < n16; c0 += 8 * 32) {         // eight loads in flight per lane
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < n16) v[u] = src[c];
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < n16) dst[c] = v[u];
        }
    }
}

// The grouped projection: persistent, one block per SM, the dense kernel's
// warp roles (warp 0 TMA, warp 1 tensor memory + MMA issue, warps 2..5
// epilogue) and schedule.  Work item t = (row tile t / n_tiles, column tile
// t % n_tiles); the number of row tiles is read from the device after the
// dependency wait.  A comes from the gathered rows (2-D map), B from the
// expert's slice of W (3-D map [E][N][K], box 64 x 256 x 1).
__global__ void __launch_bounds__(GEMM_THREADS, 1)
moe_gemm_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmw,
                const int32_t *__restrict__ ntiles_p, const int32_t *__restrict__ tile_row0,
                const int32_t *__restrict__ tile_expert, const int32_t *__restrict__ row_src,
                __nv_bfloat16 *__restrict__ Y, int N, int K, unsigned int *err)
{
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES], tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ uint32_t tmem_base_sh;
    uint8_t *smem = smem_align1024(smem_raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (N + BN - 1) / BN, kblocks = K / BK;

    if (threadIdx.x == 0) {
        prefetch_tmap(&tma);
        prefetch_tmap(&tmw);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], 4);
        }
        mbar_init(&drain_bar, 1);
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(&tmem_base_sh, TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_sh;

    pdl_wait();
    const int num_items = *ntiles_p * n_tiles;

    if (warp == 0) {
        if (lane == 0) {   // TMA producer
            // a stage is released only by the MMA thread, after it saw the
            // stage full (it stops at its first wait that gives up), so a
            // stage is never refilled before its last load landed; after a
            // wait has given up nothing more is issued
            uint32_t it = 0;                 // ring steps issued
            bool run = true;
            for (int item = blockIdx.x; run && item < num_items; item += gridDim.x) {
                const int mt = item / n_tiles, nt = item % n_tiles;
                const int row0 = tile_row0[mt], e = tile_expert[mt];
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!(run = mbar_wait(&empty_bar[s], ph ^ 1u, err, 0x51))) break;
                    uint8_t *st = smem + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full_bar[s], STAGE_BYTES);
                    tma_load_2d(st, &tma, &full_bar[s], kb * BK, row0);
                    tma_load_3d(st + A_BYTES, &tmw, &full_bar[s], kb * BK, nt * BN, e);
                }
            }
            // the block outlives its copies (free in a healthy pipeline: the
            // MMA thread waits for the same loads)
            drain_ring(full_bar, STAGES, (int)it);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // MMA issuer
            // stops at its first wait that gives up: it then issues and
            // releases nothing more
            uint32_t it = 0, tc = 0;
            bool run = true;
            for (int item = blockIdx.x; run && item < num_items; item += gridDim.x, ++tc) {
                const uint32_t b = tc & 1u, tph = (tc >> 1) & 1u;
                if (!(run = mbar_wait(&tempty_bar[b], tph ^ 1u, err, 0x52))) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * ACC_COLS;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    if (!(run = mbar_wait(&full_bar[s], ph, err, 0x53))) break;
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        umma_bf16(d_tmem, sw128_desc(a_addr + kk * UMMA_K * 2), sw128_desc(b_addr + kk * UMMA_K * 2),
                                  IDESC, (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(&empty_bar[s]);
                }
                if (!run) break;
                umma_commit(&tfull_bar[b]);
            }
            // every product issued is complete before the tensor memory is
            // freed (free in a healthy pipeline: the epilogue waits for the
            // last of them)
            umma_drain(&drain_bar);
        }
    } else {
        // epilogue: warp w reads tensor-memory lanes 32*(w%4) .. +31; row r
        // of the tile is gathered row tile_row0 + r, stored to its token-slot
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        uint32_t tc = 0;
        for (int item = blockIdx.x; item < num_items; item += gridDim.x, ++tc) {
            const int mt = item / n_tiles, nt = item % n_tiles;
            const int src = row_src[tile_row0[mt] + row];      // -1: a padding row
            const uint32_t b = tc & 1u, tph = (tc >> 1) & 1u;
            mbar_wait(&tfull_bar[b], tph, err, 0x54);
            tc_fence_after();
            __nv_bfloat16 *yrow = Y + (int64_t)(src >= 0 ? src : 0) * N;
#pragma unroll 1
            for (int chunk = 0; chunk < BN / 32; ++chunk) {
                uint32_t r[32];
                tmem_ld32(tmem_base + ((uint32_t)(quad * 32) << 16) + b * ACC_COLS + chunk * 32, r);
                const int n0 = nt * BN + chunk * 32;
                if (src >= 0) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (n0 + 8 * g < N) {
                            uint4 v;
                            v.x = pack_bf16x2(r[8 * g + 0], r[8 * g + 1]);
                            v.y = pack_bf16x2(r[8 * g + 2], r[8 * g + 3]);
                            v.z = pack_bf16x2(r[8 * g + 4], r[8 * g + 5]);
                            v.w = pack_bf16x2(r[8 * g + 6], r[8 * g + 7]);
                            *reinterpret_cast<uint4 *>(yrow + n0 + 8 * g) = v;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty_bar[b]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// out[m, n] = bf16_rne(sum_j weights[m, j] * Y[m, j, n]): one f32 fused
// multiply-add chain over j = 0 .. k-1 from +0; one thread per 8 columns.
__global__ void __launch_bounds__(256)
moe_combine_kernel(const __nv_bfloat16 *__restrict__ Y, const float *__restrict__ weights, int M, int k, int N,
                   __nv_bfloat16 *__restrict__ out)
{
    pdl_trigger();
    pdl_wait();
    const int groups = N / 8;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)M * groups) return;
    const int m = (int)(t / groups), g = (int)(t % groups);
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[c] = 0.0f;
    for (int j = 0; j < k; ++j) {
        const float w = weights[(int64_t)m * k + j];
        const uint4 r = *reinterpret_cast<const uint4 *>(Y + ((int64_t)m * k + j) * N + 8 * g);
        const float y[8] = {bf16lo(r.x), bf16hi(r.x), bf16lo(r.y), bf16hi(r.y),
                            bf16lo(r.z), bf16hi(r.z), bf16lo(r.w), bf16hi(r.w)};
#pragma unroll
        for (int c = 0; c < 8; ++c) acc[c] = __fmaf_rn(w, y[c], acc[c]);
    }
    uint4 o;
    o.x = pack_bf16x2(__float_as_uint(acc[0]), __float_as_uint(acc[1]));
    o.y = pack_bf16x2(__float_as_uint(acc[2]), __float_as_uint(acc[3]));
    o.z = pack_bf16x2(__float_as_uint(acc[4]), __float_as_uint(acc[5]));
    o.w = pack_bf16x2(__float_as_uint(acc[6]), __float_as_uint(acc[7]));
    *reinterpret_cast<uint4 *>(out + (int64_t)m * N + 8 * g) = o;
}

}  // namespace
}  // namespace bi

using namespace bi;

extern "C" size_t bi_moe_workspace_bytes(int32_t M, int32_t k, int32_t E, int32_t N, int32_t K)
{
    if (M < 0 || k <= 0 || E <= 0 || N <= 0 || K <= 0) return 0;
    return moe_layout(M, k, E, N, K, nullptr, nullptr);
}

extern "C" bi_status bi_moe_expert_gemm(const void *X, const int32_t *ids, const float *weights, const void *W,
                                        int32_t M, int32_t k, int32_t E, int32_t N, int32_t K, void *Y_out,
                                        void *out, void *workspace, size_t workspace_bytes, bi_stream s)
{
    if (M < 0 || k <= 0 || E <= 0 || N <= 0 || K <= 0) return BI_ERR_INVALID_ARG;
    if (E > BI_MAX_E || k > BI_MAX_K || (K % BK) != 0 || (N % 16) != 0 || K > 65536 || N > 65536 ||
        (int64_t)M * k > (1 << 24))
        return BI_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return BI_OK;
    if (!X || !ids || !W || !workspace || (!Y_out && !out) || (out && !weights)) return BI_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y_out) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) || (reinterpret_cast<uintptr_t>(ids) & 3u) ||
        (reinterpret_cast<uintptr_t>(weights) & 3u))
        return BI_ERR_MISALIGNED;
    MoeWs ws;
    const size_t need = moe_layout(M, k, E, N, K, static_cast<uint8_t *>(workspace), &ws);
    if (workspace_bytes < need) return BI_ERR_INVALID_ARG;
    __nv_bfloat16 *Y = Y_out ? static_cast<__nv_bfloat16 *>(Y_out) : ws.Y;

    Device *d = nullptr;
    bi_status st = current_device(&d);
    if (st != BI_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);

    alignas(64) CUtensorMap tma, tmw;
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)ws.cap};
        const uint64_t strides[1] = {(uint64_t)K * 2};
        const uint32_t box[2] = {(uint32_t)BK, (uint32_t)BM};
        if ((st = encode_tiled(&tma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ws.Ag, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B)) != BI_OK)
            return st;
    }
    {
        const uint64_t dims[3] = {(uint64_t)K, (uint64_t)N, (uint64_t)E};
        const uint64_t strides[2] = {(uint64_t)K * 2, (uint64_t)N * K * 2};
        const uint32_t box[3] = {(uint32_t)BK, (uint32_t)BN, 1u};
        if ((st = encode_tiled(&tmw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, W, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B)) != BI_OK)
            return st;
    }

    const int Mk = M * k;
    if ((st = set_smem_once(d, KID_MOE + 1, moe_plan_kernel, 0)) != BI_OK) return st;
    if ((st = launch_pdl(moe_plan_kernel, dim3(1), dim3(kPlanThreads), 0, cs, ids, Mk, (int)E, ws.cursor,
                         ws.offsets, ws.ntiles, ws.tile_row0, ws.tile_expert, ws.row_src, d->err)) != BI_OK)
        return st;
    if ((st = set_smem_once(d, KID_MOE + 2, moe_place_kernel, 0)) != BI_OK) return st;
    if ((st = launch_pdl(moe_place_kernel, dim3((Mk + 7) / 8), dim3(256), 0, cs,
                         static_cast<const __nv_bfloat16 *>(X), ids, Mk, (int)k, (int)K,
                         (const int32_t *)ws.offsets, ws.cursor, ws.row_src, ws.Ag, (int)E)) != BI_OK)
        return st;
    if ((st = set_smem_once(d, KID_MOE + 3, moe_gemm_kernel, GEMM_SMEM)) != BI_OK) return st;
    if ((st = launch_pdl(moe_gemm_kernel, dim3(d->sm_count), dim3(GEMM_THREADS), (size_t)GEMM_SMEM, cs, tma, tmw,
                         (const int32_t *)ws.ntiles, (const int32_t *)ws.tile_row0, (const int32_t *)ws.tile_expert,
                         (const int32_t *)ws.row_src, Y, (int)N, (int)K, d->err)) != BI_OK)
        return st;
    if (!out) return BI_OK;
    if ((st = set_smem_once(d, KID_MOE + 4, moe_combine_kernel, 0)) != BI_OK) return st;
    const int64_t threads = (int64_t)M * (N / 8);
    return launch_pdl(moe_combine_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, cs,
                      (const __nv_bfloat16 *)Y, weights, (int)M, (int)k, (int)N, static_cast<__nv_bfloat16 *>(out));
}
