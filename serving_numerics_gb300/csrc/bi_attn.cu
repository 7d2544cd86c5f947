// bi_attn.cu -- bi_attention_prefill: batch-invariant causal prefill
// attention over ragged requests on the tcgen05 tensor cores.
//
// Source page: "The Illusion of Determinism in Disaggregated Inference",
// section "The physics of the cascade": a one-ULP difference that reaches
// attention is stretched by the softmax's exponential and spread over every
// feature by the product with the value matrix, so attention is the next
// operation on the path after RMSNorm whose result must not depend on the
// batch; the page's references name attention among the kernels a
// batch-invariant engine rewrites.
//
// Invariance by construction.  Every query row walks the keys of its own
// request in blocks of 64 at fixed absolute key positions (block b holds
// keys 64b .. 64b+63 of the context), from block 0 up to the block holding
// the row's own position, and does the same arithmetic on each block:
//
//   s_j   = q . k_j               f32, on the tensor cores: d = 0..127 as
//                                 eight 16-deep steps in increasing order
//   bm    = max over visible j of s_j           (exact: order-free)
//   m'    = max(m, bm * c)        c = scale * log2(e), m the running maximum
//   p_j   = bf16_rne(exp2f(fmaf(s_j, c, -m')))  visible j, else 0
//   l'    = fmaf(l, a, pairwise sum of the 64 widened p_j), a = exp2f(m - m')
//   O_b   = sum_j p_j v_j         f32, on the tensor cores: four 16-deep
//                                 steps over the block's keys, in order
//   acc'  = fmaf(acc, a, O_b)     per output column
//
// and finally o = bf16_rne(acc / l), lse = (m + log2f(l)) * ln(2).  A
// block that holds no key the row can see changes nothing (a = 1, the p_j
// are 0, O_b is a sum of zero products), so a row's bits are the same
// whichever query tile it falls in, whatever tile boundaries the batch, a
// cached prefix or a chunked prefill put around it, and whatever else is in
// the launch.  Which tile a row lands in, how many tiles run and in which
// order never enter its arithmetic.
//
// Structure (one CTA per query tile of 128 rows and one head, 192 threads):
//   warp 0      TMA producer: the Q tile once (two 64-column boxes, 128-byte
//               swizzle), then K and V of each key block into a ring of 4
//               stages (32 KB each)
//   warp 1      allocates 512 tensor-memory columns (two S buffers of
//               128 x 64 f32, two O buffers of 128 x 128 f32); one lane
//               issues S = Q K^T for block b+1 before O_b = P_b V_b, so the
//               tensor cores compute the next scores while the softmax of
//               the current block runs
//   warps 2..5  one thread per query row: the softmax of block b (P_b as
//               bf16 into shared memory in the swizzled K-major layout the
//               next MMA reads), then the correction of block b-1 (O_{b-1}
//               from tensor memory folded into registers), then the output
// V is read by the PV product straight from its TMA box as an MN-major
// operand (keys along K, head dimension contiguous), so V needs no
// transpose.  Every wait on an mbarrier is bounded (about 2 s); on expiry
// the kernel records BI_ERR_TIMEOUT in the device error word and carries on.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "bi_device.cuh"
#include "bi_internal.h"
#include "bi_tcgen05.cuh"

namespace bi {
namespace {

constexpr int AT_D = 128;                          // head dimension
constexpr int AT_BQ = 128;                         // query rows per tile (tensor-memory lanes)
constexpr int AT_BKV = 64;                         // keys per block
constexpr int AT_STAGES = 4;
constexpr int AT_Q_BOX = AT_BQ * 64 * 2;           // 16 KB: 128 rows x 64 dims
constexpr int AT_KV_BOX = AT_BKV * 64 * 2;         // 8 KB: 64 keys x 64 dims
constexpr int AT_Q_BYTES = 2 * AT_Q_BOX;
constexpr int AT_STAGE_BYTES = 4 * AT_KV_BOX;      // K (two boxes), then V (two boxes)
constexpr int AT_P_BYTES = AT_BQ * AT_BKV * 2;     // 16 KB: 128 rows x 64 keys bf16
constexpr int AT_SMEM = AT_Q_BYTES + AT_STAGES * AT_STAGE_BYTES + 2 * AT_P_BYTES + 1024;
constexpr int AT_THREADS = 192;
constexpr uint32_t AT_S_COL = 0;                   // S buffers: columns 0..63 and 64..127
constexpr uint32_t AT_O_COL = 128;                 // O buffers: 128..255 and 256..383
constexpr uint32_t AT_TMEM_COLS = 512;
static_assert(AT_SMEM <= 227 * 1024, "shared memory");

// One query tile: up to 128 consecutive queries of one request.
struct AttnTile {
    int q0;     // token index of the tile's first query in q and o
    int kv0;    // token index of the request's first key in k and v
    int pos0;   // context position of the tile's first query
    int rows;   // queries in the tile (1..128)
};
constexpr int kAttnMaxTiles = 512;                 // tiles per launch (8 KB of kernel parameters)
struct AttnTable {
    AttnTile t[kAttnMaxTiles];
};

__host__ __device__ constexpr int attn_blocks(int pos0, int rows) { return (pos0 + rows - 1) / AT_BKV + 1; }

// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle
// as TMA lays it out from [keys][64 dims] boxes: along N (the head
// dimension) 64 contiguous elements per 128-byte row and the next 64 in the
// next box (leading byte offset = one box, 8 KB); along K (keys) rows of
// 128 bytes, 8-row atoms 1024 bytes apart (stride byte offset).  A 16-key
// step of K adds two atoms (2048 bytes) to the start address.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((uint32_t)AT_KV_BOX >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__global__ void __launch_bounds__(AT_THREADS, 1)
attn_prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ AttnTable tab,
                    __nv_bfloat16 *__restrict__ O, float *__restrict__ lse, int n_heads, int group, float c,
                    unsigned int *err)
{
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_bar, kv_full[AT_STAGES], kv_empty[AT_STAGES], s_full[2], s_empty[2],
        p_full[2], o_full[2], o_empty[2];
    __shared__ uint32_t tmem_base_sh;
    uint8_t *smem = smem_align1024(smem_raw);
    uint8_t *sq = smem, *skv = smem + AT_Q_BYTES, *sp = skv + AT_STAGES * AT_STAGE_BYTES;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ti = blockIdx.x / n_heads, h = blockIdx.x % n_heads, hk = h / group;
    const AttnTile tile = tab.t[ti];
    const int nb = attn_blocks(tile.pos0, tile.rows);

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        mbar_init(&q_bar, 1);
        for (int s = 0; s < AT_STAGES; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_empty[b], 4);
            mbar_init(&p_full[b], 4);
            mbar_init(&o_full[b], 1);
            mbar_init(&o_empty[b], 4);
        }
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(&tmem_base_sh, AT_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_sh;

    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {   // TMA producer
            mbar_arrive_expect_tx(&q_bar, (uint32_t)AT_Q_BYTES);
            tma_load_3d(sq, &tmq, &q_bar, 0, h, tile.q0);
            tma_load_3d(sq + AT_Q_BOX, &tmq, &q_bar, 64, h, tile.q0);
            for (int b = 0; b < nb; ++b) {
                const int st = b % AT_STAGES;
                const uint32_t ph = (uint32_t)(b / AT_STAGES) & 1u;
                mbar_wait(&kv_empty[st], ph ^ 1u, err, 0x61);
                uint8_t *dst = skv + st * AT_STAGE_BYTES;
                const int key = tile.kv0 + b * AT_BKV;
                mbar_arrive_expect_tx(&kv_full[st], (uint32_t)AT_STAGE_BYTES);
                tma_load_3d(dst, &tmk, &kv_full[st], 0, hk, key);
                tma_load_3d(dst + AT_KV_BOX, &tmk, &kv_full[st], 64, hk, key);
                tma_load_3d(dst + 2 * AT_KV_BOX, &tmv, &kv_full[st], 0, hk, key);
                tma_load_3d(dst + 3 * AT_KV_BOX, &tmv, &kv_full[st], 64, hk, key);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {   // MMA issuer
            const uint32_t id_s = idesc_n(AT_BKV), id_o = idesc_n(AT_D) | (1u << 16);   // B of PV MN-major
            mbar_wait(&q_bar, 0, err, 0x62);
            tc_fence_after();
            const uint32_t qa = smem_u32(sq);
            for (int b = 0; b <= nb; ++b) {
                if (b < nb) {   // S_b = Q K_b^T
                    const int st = b % AT_STAGES;
                    const uint32_t sb = (uint32_t)b & 1u, use = ((uint32_t)b >> 1) & 1u;
                    mbar_wait(&kv_full[st], (uint32_t)(b / AT_STAGES) & 1u, err, 0x63);
                    mbar_wait(&s_empty[sb], use ^ 1u, err, 0x64);
                    tc_fence_after();
                    const uint32_t ka = smem_u32(skv + st * AT_STAGE_BYTES);
                    const uint32_t d = tmem_base + AT_S_COL + sb * AT_BKV;
#pragma unroll
                    for (int half = 0; half < 2; ++half)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_bf16(d, sw128_desc(qa + half * AT_Q_BOX + k * 32),
                                      sw128_desc(ka + half * AT_KV_BOX + k * 32), id_s, (half | k) != 0 ? 1u : 0u);
                    umma_commit(&s_full[sb]);
                }
                if (b >= 1) {   // O_{b-1} = P_{b-1} V_{b-1}
                    const int pb = b - 1, st = pb % AT_STAGES;
                    const uint32_t ob = (uint32_t)pb & 1u, use = ((uint32_t)pb >> 1) & 1u;
                    mbar_wait(&p_full[ob], use, err, 0x65);
                    mbar_wait(&o_empty[ob], use ^ 1u, err, 0x66);
                    tc_fence_after();
                    const uint32_t pa = smem_u32(sp + ob * AT_P_BYTES);
                    const uint32_t va = smem_u32(skv + st * AT_STAGE_BYTES + 2 * AT_KV_BOX);
                    const uint32_t d = tmem_base + AT_O_COL + ob * AT_D;
#pragma unroll
                    for (int k = 0; k < AT_BKV / 16; ++k)
                        umma_bf16(d, sw128_desc(pa + k * 32), sw128_mn_desc(va + k * 2048), id_o, k != 0 ? 1u : 0u);
                    umma_commit(&o_full[ob]);
                    umma_commit(&kv_empty[st]);   // K and V of block pb no longer read
                }
            }
        }
    } else {
        // softmax and correction: warp w may read tensor-memory lanes 32*(w%4) .. +31
        const int quad = warp & 3, row = quad * 32 + lane;
        const int pos = tile.pos0 + row;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        float m = -INFINITY, l = 0.f, a_prev = 0.f;
        float acc[AT_D];
#pragma unroll
        for (int i = 0; i < AT_D; ++i) acc[i] = 0.f;

        auto correct = [&](int cb, float a) {
            const uint32_t ob = (uint32_t)cb & 1u, use = ((uint32_t)cb >> 1) & 1u;
            mbar_wait(&o_full[ob], use, err, 0x67);
            tc_fence_after();
#pragma unroll
            for (int ch = 0; ch < AT_D / 32; ++ch) {
                uint32_t r[32];
                tmem_ld32(tmem_base + lane_off + AT_O_COL + ob * AT_D + ch * 32, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[ch * 32 + i] = fmaf(acc[ch * 32 + i], a, __uint_as_float(r[i]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&o_empty[ob]);
        };

#pragma unroll 1
        for (int b = 0; b < nb; ++b) {
            const uint32_t sb = (uint32_t)b & 1u, use = ((uint32_t)b >> 1) & 1u;
            mbar_wait(&s_full[sb], use, err, 0x68);
            tc_fence_after();
            uint32_t s[AT_BKV];
            tmem_ld32(tmem_base + lane_off + AT_S_COL + sb * AT_BKV, *reinterpret_cast<uint32_t(*)[32]>(&s[0]));
            tmem_ld32(tmem_base + lane_off + AT_S_COL + sb * AT_BKV + 32, *reinterpret_cast<uint32_t(*)[32]>(&s[32]));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[sb]);

            const int nvis = pos - b * AT_BKV + 1;        // keys of this block the row sees (clamped below)
            float bm = -INFINITY;
#pragma unroll
            for (int j = 0; j < AT_BKV; ++j)
                if (j < nvis) bm = fmaxf(bm, __uint_as_float(s[j]));
            const float m_new = fmaxf(m, bm * c);
            const float mu = m_new == -INFINITY ? 0.f : m_new;
            const float a = exp2f(m - mu);

            // P_b as bf16, and the pairwise sum of the rounded values
            uint32_t pk[AT_BKV / 2];
#pragma unroll
            for (int j = 0; j < AT_BKV; j += 2) {
                const float p0 = j < nvis ? exp2f(fmaf(__uint_as_float(s[j]), c, -mu)) : 0.f;
                const float p1 = j + 1 < nvis ? exp2f(fmaf(__uint_as_float(s[j + 1]), c, -mu)) : 0.f;
                pk[j / 2] = pack_bf16x2(__float_as_uint(p0), __float_as_uint(p1));
            }
            float t[AT_BKV / 2];
#pragma unroll
            for (int i = 0; i < AT_BKV / 2; ++i) t[i] = bf16lo(pk[i]) + bf16hi(pk[i]);
#pragma unroll
            for (int w = AT_BKV / 4; w >= 1; w >>= 1)
#pragma unroll
                for (int i = 0; i < w; ++i) t[i] = t[2 * i] + t[2 * i + 1];
            l = fmaf(l, a, t[0]);
            m = m_new;

            // P_b into shared memory: row `row`, 16-byte chunk q of the
            // 128-byte row at chunk position q ^ (row % 8) (128-byte swizzle)
            const uint32_t prow = smem_u32(sp + sb * AT_P_BYTES) + (uint32_t)row * 128u;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                st_shared_v4(prow + (uint32_t)((q ^ (row & 7)) << 4), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                             pk[4 * q + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[sb]);

            if (b >= 1) correct(b - 1, a_prev);
            a_prev = a;
        }
        correct(nb - 1, a_prev);

        if (row < tile.rows) {
            const size_t orow = (size_t)(tile.q0 + row) * (size_t)n_heads + (size_t)h;
            uint4 *dst = reinterpret_cast<uint4 *>(O + orow * AT_D);
#pragma unroll
            for (int g = 0; g < AT_D / 8; ++g) {
                uint4 v;
                v.x = pack_bf16x2(__float_as_uint(__fdiv_rn(acc[8 * g + 0], l)), __float_as_uint(__fdiv_rn(acc[8 * g + 1], l)));
                v.y = pack_bf16x2(__float_as_uint(__fdiv_rn(acc[8 * g + 2], l)), __float_as_uint(__fdiv_rn(acc[8 * g + 3], l)));
                v.z = pack_bf16x2(__float_as_uint(__fdiv_rn(acc[8 * g + 4], l)), __float_as_uint(__fdiv_rn(acc[8 * g + 5], l)));
                v.w = pack_bf16x2(__float_as_uint(__fdiv_rn(acc[8 * g + 6], l)), __float_as_uint(__fdiv_rn(acc[8 * g + 7], l)));
                dst[g] = v;
            }
            if (lse) lse[orow] = (m + log2f(l)) * 0.693147180559945309f;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, AT_TMEM_COLS);
}

}  // namespace
}  // namespace bi

using namespace bi;

extern "C" bi_status bi_attention_prefill(const void *q, const void *k, const void *v, int32_t n_req,
                                          const int32_t *q_offsets, const int32_t *kv_offsets, int32_t n_heads,
                                          int32_t n_kv_heads, int32_t head_dim, float scale, void *o, float *lse,
                                          bi_stream s)
{
    if (n_req < 0 || n_heads <= 0 || n_kv_heads <= 0) return BI_ERR_INVALID_ARG;
    if (n_req > 0 && (!q_offsets || !kv_offsets)) return BI_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return BI_ERR_INVALID_ARG;
    if (n_heads % n_kv_heads != 0) return BI_ERR_INVALID_ARG;
    if (head_dim != AT_D) return BI_ERR_UNSUPPORTED_SHAPE;
    if (n_heads > BI_ATTN_MAX_HEADS) return BI_ERR_UNSUPPORTED_SHAPE;
    if (n_req == 0) return BI_OK;
    if (q_offsets[0] != 0 || kv_offsets[0] != 0) return BI_ERR_INVALID_ARG;
    for (int r = 0; r < n_req; ++r) {
        const int32_t ql = q_offsets[r + 1] - q_offsets[r], kl = kv_offsets[r + 1] - kv_offsets[r];
        if (ql < 0 || kl < 0 || ql > kl) return BI_ERR_INVALID_ARG;
    }
    const int64_t Tq = q_offsets[n_req], Tkv = kv_offsets[n_req];
    if (Tq == 0) return BI_OK;
    if (!q || !k || !v || !o) return BI_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return BI_ERR_MISALIGNED;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return BI_ERR_MISALIGNED;

    Device *d = nullptr;
    bi_status st = current_device(&d);
    if (st != BI_OK) return st;

    // The query tiles, longest (most key blocks) first so that the CTAs
    // that take longest start first; the order changes no result.
    std::vector<AttnTile> tiles;
    for (int r = 0; r < n_req; ++r) {
        const int ql = q_offsets[r + 1] - q_offsets[r], kl = kv_offsets[r + 1] - kv_offsets[r];
        for (int t0 = 0; t0 < ql; t0 += AT_BQ)
            tiles.push_back({q_offsets[r] + t0, kv_offsets[r], kl - ql + t0, std::min(AT_BQ, ql - t0)});
    }
    std::stable_sort(tiles.begin(), tiles.end(), [](const AttnTile &x, const AttnTile &y) {
        return attn_blocks(x.pos0, x.rows) > attn_blocks(y.pos0, y.rows);
    });

    alignas(64) CUtensorMap tmq, tmk, tmv;
    {
        const uint64_t dims[3] = {(uint64_t)AT_D, (uint64_t)n_heads, (uint64_t)Tq};
        const uint64_t strides[2] = {(uint64_t)AT_D * 2, (uint64_t)n_heads * AT_D * 2};
        const uint32_t box[3] = {64, 1, (uint32_t)AT_BQ};
        if ((st = encode_tiled(&tmq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B)) != BI_OK)
            return st;
    }
    for (int which = 0; which < 2; ++which) {
        const uint64_t dims[3] = {(uint64_t)AT_D, (uint64_t)n_kv_heads, (uint64_t)Tkv};
        const uint64_t strides[2] = {(uint64_t)AT_D * 2, (uint64_t)n_kv_heads * AT_D * 2};
        const uint32_t box[3] = {64, 1, (uint32_t)AT_BKV};
        if ((st = encode_tiled(which ? &tmv : &tmk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, which ? v : k, dims,
                               strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) != BI_OK)
            return st;
    }
    if ((st = set_smem_once(d, KID_ATTN, attn_prefill_kernel, AT_SMEM)) != BI_OK) return st;

    const float c = scale * 1.44269504088896340736f;
    static_assert(sizeof(AttnTable) <= 8192, "kernel parameter space");
    AttnTable tab;
    for (size_t first = 0; first < tiles.size(); first += kAttnMaxTiles) {
        const int n = (int)std::min<size_t>(kAttnMaxTiles, tiles.size() - first);
        std::copy(tiles.begin() + first, tiles.begin() + first + n, tab.t);
        st = launch_pdl(attn_prefill_kernel, dim3((unsigned)(n * n_heads)), dim3(AT_THREADS), (size_t)AT_SMEM,
                        reinterpret_cast<cudaStream_t>(s), tmq, tmk, tmv, tab, static_cast<__nv_bfloat16 *>(o),
                        lse, (int)n_heads, (int)(n_heads / n_kv_heads), c, d->err);
        if (st != BI_OK) return st;
    }
    return BI_OK;
}
