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
// request in blocks of 128 at fixed absolute key positions (block b holds
// keys 128b .. 128b+127 of the context), from block 0 up to the block
// holding the row's own position, and does the same arithmetic on each
// block:
//
//   s_j  = q . k_j                 f32 on the tensor cores: the 128
//                                  dimensions as eight 16-deep steps, in
//                                  increasing order; invisible keys -> -inf
//   t    = c * max_j s_j           c = scale * log2(e) (max: order-free)
//   if t > m + 8:                  the reference maximum moves (always on
//                                  the first block, where m = -inf)
//       a = 2^(m - t);  l = l * a;  O = O * a  (in tensor memory);  m = t
//   p_j  = 2^(fmaf(s_j, c, -m))    ex2.approx.ftz, <= 2^8
//   l    = l + (E + D)             E, D: pairwise trees over the 64 even-
//                                  and the 64 odd-position p_j of the block
//   O    = O + sum_j bf16_rne(p_j) v_j   f32 on the tensor cores: eight
//                                  16-deep steps over the block's keys in
//                                  increasing order, added to O in place
//
// and finally o = bf16_rne(O * (1/l)), lse = (m + log2f(l)) * ln(2).  The
// reference maximum only moves when a block's maximum exceeds it by more
// than 2^8 in the exponent, so the rescaling is rare after the first block;
// whether it moves depends only on the row's own scores.  A block that holds
// no key the row can see changes nothing (its maximum is -inf, its p_j are
// 0, its products with V are zeros added to O), so a row's bits are the same
// whichever query tile it falls in, whatever tile boundaries the batch, a
// cached prefix or a chunked prefill put around it, and whatever else is in
// the launch.
//
// Keys also come in chunks of 8192 (64 blocks) at fixed positions.  A row
// below position 8192 is exactly the above; a later row runs the above on
// each of its chunks c = 0 .. pos/8192 from a fresh state, giving (m_c, l_c,
// O_c), and these are merged in chunk order (merge_weights).  The chunk
// boundaries depend on the position alone, so the bits still do not depend
// on the batch, while one tile's chunks can run on several SMs at once.
//
// Structure: one CTA per query tile of 128 rows and NT query heads of one
// key/value head.  Warpgroup t (warps 4t .. 4t+3) is head t's softmax, one
// thread per query row; after them a TMA producer warp (the NT Q tiles once,
// then K and V of each key block into a ring of 64 KB stages, shared by the
// heads) and an MMA warp, whose one lane issues S = Q K^T and O += P V (A = P
// read from tensor memory, B = V from shared memory):
//   NT = 2   (the call bound by its total work; the heads per key/value head
//            even): 384 threads, a third warpgroup of producer, MMA and two
//            idle warps giving registers to the softmax warpgroups through
//            setmaxnreg.  Per head one S buffer; per block O += P V and then
//            the next block's S into the same columns, head after head, so
//            each head's softmax runs while the tensor cores serve the
//            other head.
//   NT = 1   (the call bound by its longest tile, or an odd group): 192
//            threads, two S buffers: S of block b+2 goes into the buffer
//            block b's P leaves, so the scores of block b+1 are ready while
//            block b's softmax runs, and a tile's chain of blocks runs in
//            about 0.55 of the time two paired heads take.
// Shared memory carries only Q, K and V: P never leaves tensor memory, and
// V is read by the P V product straight from its TMA box as an MN-major
// operand (keys along K, head dimension contiguous).  The next block's
// S = Q K^T overwrites the columns that held this block's P: the tensor
// core executes one thread's tcgen05.mma operations in issue order, and the
// S product is issued after the P V product that reads them.  Every wait on
// an mbarrier is bounded (about 2 s); on expiry the kernel records
// BI_ERR_TIMEOUT in the device error word, the producer and MMA threads
// issue nothing more and wait (bounded) for their own copies and products,
// the softmax warps carry on, and the block frees its tensor memory.
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
constexpr int AT_BKV = 128;                        // keys per block
constexpr float AT_TAU = 8.0f;                     // the reference maximum moves past this growth
constexpr int AT_Q_BOX = AT_BQ * 64 * 2;           // 16 KB: 128 rows x 64 dims
constexpr int AT_KV_BOX = AT_BKV * 64 * 2;         // 16 KB: 128 keys x 64 dims
constexpr int AT_Q_BYTES = 2 * AT_Q_BOX;
constexpr int AT_STAGE_BYTES = 4 * AT_KV_BOX;      // K (two boxes), then V (two boxes)

// Warp roles: warpgroup t (warps 4t .. 4t+3) is head t's softmax; then the
// TMA producer warp and the MMA warp.  With two heads the block has a third,
// whole warpgroup (producer, MMA, two idle warps) so that setmaxnreg can move
// registers from it to the two softmax warpgroups: launched at 168 a thread,
// 200 for the softmax, 96 for the rest.
constexpr int AT_REGS_SOFTMAX = 200, AT_REGS_OTHER = 96;
// Tensor memory (512 columns either way; S is 128 x 128 f32, P its first 64
// columns as bf16 pairs, O 128 x 128 f32):
//   NT = 2: head t's S at columns 256t .. 256t+127, its O at 256t+128 ..
//   NT = 1: two S buffers at 0 and 128 (block b in buffer b % 2), O at 256
template <int NT>
struct AttnCfg {
    static constexpr int PRODUCER_WARP = 4 * NT, MMA_WARP = 4 * NT + 1;
    static constexpr int THREADS = NT == 2 ? 384 : 192;
    static constexpr int STAGES = NT == 2 ? 2 : 3;       // K/V blocks in flight
    static constexpr int KV_OFF = NT * AT_Q_BYTES;
    static constexpr int SMEM = KV_OFF + STAGES * AT_STAGE_BYTES + 1024;
    static constexpr uint32_t TMEM_COLS = 512;
    __device__ static constexpr uint32_t s_col(int t, int buf) { return NT == 2 ? 256u * t : 128u * buf; }
    __device__ static constexpr uint32_t o_col(int t) { return NT == 2 ? 256u * t + 128u : 256u; }
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(NT == 1 || 2 * 128 * AT_REGS_SOFTMAX + 128 * AT_REGS_OTHER <= THREADS * 168, "register split");
};

// Keys are cut into chunks of 64 blocks (8192 keys) at fixed positions.  A
// row whose context fits the first chunk is computed in one pass; a longer
// row's chunks are computed from fresh softmax states, each into a partial
// (m, l, O), and merged in chunk order (merge_weights below).
constexpr int AT_CHUNK_BLOCKS = 64;
constexpr int AT_CHUNK_KEYS = AT_CHUNK_BLOCKS * AT_BKV;
constexpr int AT_PART_STRIDE = 132;                // floats per partial row: O[128], m, l, two spare

// One work entry: key blocks [kb0, kb1) of a query tile (up to 128
// consecutive queries of one request) -- the whole tile, or one chunk of it.
struct AttnTile {
    int q0;     // token index of the tile's first query in q and o
    int kv0;    // token index of the request's first key in k and v
    int pos0;   // context position of the tile's first query
    int rows;   // queries in the tile (1..128)
    int kb0;    // first key block (a multiple of AT_CHUNK_BLOCKS)
    int kb1;    // one past the last key block
    int part;   // the tile's scratch slot (mode 0, tiles past the first chunk), chunk's partial slot (mode 1), or -1
    int mode;   // 0: one CTA walks the tile, merging chunk by chunk; 1: one chunk, its partial for the merge kernel
};
constexpr int kAttnMaxTiles = 256;                 // entries per launch (8 KB of kernel parameters)
struct AttnTable {
    AttnTile t[kAttnMaxTiles];
};

__host__ __device__ constexpr int attn_blocks(int pos0, int rows) { return (pos0 + rows - 1) / AT_BKV + 1; }


// Shared-memory descriptor of an MN-major operand with the 128-byte swizzle
// as TMA lays it out from [keys][64 dims] boxes: along N (the head
// dimension) 64 contiguous elements per 128-byte row and the next 64 in the
// next box (leading byte offset = one box); along K (keys) rows of 128
// bytes, 8-row atoms 1024 bytes apart (stride byte offset).  A 16-key step
// of K adds two atoms (2048 bytes) to the start address.
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

// D (tensor memory) (+)= A (tensor memory, K-major: row i in lane i, 16-bit
// elements packed two to a 32-bit column) . B (shared memory descriptor).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 2^x by the multi-function unit (flushes subnormal results to zero; 2^-inf = 0)
__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Merge of a row's chunk c >= 1 (m, l, O) into its running state (M, L, N)
// (which starts as chunk 0's (m, l, O) unchanged): with M' = max(M, m),
// a = 2^(M - M') and b = 2^(m - M') (each exactly 1 where its maximum is
// M'), L = fmaf(L, a, l b) and N_d = fmaf(N_d, a, O_d b), every product
// rounded once.
struct MergeWeights {
    float a, b;
};
__device__ __forceinline__ MergeWeights merge_weights(float &M, float &L, float m, float l)
{
    const float Mn = fmaxf(M, m);
    MergeWeights w;
    w.a = M == Mn ? 1.f : ex2(M - Mn);
    w.b = m == Mn ? 1.f : ex2(m - Mn);
    L = fmaf(L, w.a, __fmul_rn(l, w.b));
    M = Mn;
    return w;
}

// Two independent f32 fused multiply-adds (each rounded once) in one instruction.
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0, float b1, float c0, float c1)
{
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// 32 lanes x 32 consecutive f32 columns without waiting (pair with tmem_ld_wait).
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t *r)
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns from registers (thread t writes lane t).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *r)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Chunk c of a row ends (its block's P V products done).  A row with keys
// in chunk c:
//   c == 0 and its context ends there: o from O (o = O / l)
//   mode 0: chunk 0 starts its merged state (N = O in its scratch row, M = m,
//           L = l); a later chunk merges into it (merge_weights), finishing
//           the row in its last chunk
//   mode 1: chunk c's (O, m, l) into the partial slot
// Returns the merged (M, L).  Kept out of line: it runs once a chunk, and
// inlined its registers would weigh on the block loop.  Every lane of the
// warp calls it (the tensor-memory loads are warp-wide).
__device__ __noinline__ float2 attn_chunk_end(int c, float m, float l, float M, float L, uint32_t otaddr, int lc,
                                              bool valid, int mode, uint4 *dst, float4 *srow, float *lse_elem)
{
    const bool seq = mode == 0, has = valid && lc >= c;
    const bool direct = has && c == 0 && lc == 0;
    const bool merge = seq && has && c >= 1;
    const bool merged_out = merge && c == lc;
    const bool keep = (seq && has && lc > c) || (!seq && has && lc >= 1);
    MergeWeights w = {1.f, 0.f};
    if (merge) w = merge_weights(M, L, m, l);
    else if (seq && has && c == 0 && lc >= 1) { M = m; L = l; }
    const float rl = direct ? __frcp_rn(l) : (merged_out ? __frcp_rn(L) : 0.f);
#pragma unroll 1
    for (int ch = 0; ch < AT_D / 32; ++ch) {             // columns 32 ch .. 32 ch + 31
        uint32_t r[32];
        tmem_ld32_nowait(otaddr + ch * 32, r);
        tmem_ld_wait();
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(r[i]);
        if (merge) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 n4 = srow[ch * 8 + i];
                x[4 * i] = fmaf(n4.x, w.a, __fmul_rn(x[4 * i], w.b));
                x[4 * i + 1] = fmaf(n4.y, w.a, __fmul_rn(x[4 * i + 1], w.b));
                x[4 * i + 2] = fmaf(n4.z, w.a, __fmul_rn(x[4 * i + 2], w.b));
                x[4 * i + 3] = fmaf(n4.w, w.a, __fmul_rn(x[4 * i + 3], w.b));
            }
        }
        if (direct || merged_out) {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                uint4 v;
                v.x = pack_bf16x2(__float_as_uint(x[8 * g + 0] * rl), __float_as_uint(x[8 * g + 1] * rl));
                v.y = pack_bf16x2(__float_as_uint(x[8 * g + 2] * rl), __float_as_uint(x[8 * g + 3] * rl));
                v.z = pack_bf16x2(__float_as_uint(x[8 * g + 4] * rl), __float_as_uint(x[8 * g + 5] * rl));
                v.w = pack_bf16x2(__float_as_uint(x[8 * g + 6] * rl), __float_as_uint(x[8 * g + 7] * rl));
                dst[ch * 4 + g] = v;
            }
        }
        if (keep) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                srow[ch * 8 + i] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
        }
    }
    if (lse_elem && direct) *lse_elem = (m + log2f(l)) * 0.693147180559945309f;
    if (lse_elem && merged_out) *lse_elem = (M + log2f(L)) * 0.693147180559945309f;
    if (!seq && has && lc >= 1) srow[AT_D / 4] = make_float4(m, l, 0.f, 0.f);
    return make_float2(M, L);
}

template <int NT>
__global__ void __launch_bounds__(AttnCfg<NT>::THREADS, 1)
attn_prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                    const __grid_constant__ CUtensorMap tmv, const __grid_constant__ AttnTable tab,
                    __nv_bfloat16 *__restrict__ O, float *__restrict__ lse, float *__restrict__ part, int n_heads,
                    int group, float c, unsigned int *err)
{
    using Cfg = AttnCfg<NT>;
    constexpr int NS = Cfg::STAGES;
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_bar, kv_full[NS], kv_empty[NS], s_full[2], p_full[NT], o_done[NT][2], drain_bar;
    __shared__ uint32_t tmem_base_sh;
    uint8_t *smem = smem_align1024(smem_raw);
    uint8_t *sq = smem, *skv = smem + Cfg::KV_OFF;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pairs = n_heads / NT;
    const int ti = blockIdx.x / pairs, h0 = (blockIdx.x % pairs) * NT, hk = h0 / group;
    const AttnTile tile = tab.t[ti];
    const int kb0 = tile.kb0, nb = tile.kb1 - tile.kb0;   // this CTA's key blocks: kb0 + 0 .. nb-1

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmq);
        prefetch_tmap(&tmk);
        prefetch_tmap(&tmv);
        mbar_init(&q_bar, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) mbar_init(&s_full[t], 1);    // per head (NT = 2) or per S buffer (NT = 1)
        for (int t = 0; t < NT; ++t) {
            mbar_init(&p_full[t], 4);
            mbar_init(&o_done[t][0], 1);   // P V of even blocks
            mbar_init(&o_done[t][1], 1);   // of odd blocks
        }
        mbar_init(&drain_bar, 1);
        mbar_init_fence();
    }
    if (warp == Cfg::MMA_WARP) tmem_alloc(&tmem_base_sh, Cfg::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_base_sh;

    // each role under its own register budget: ptxas allocates a region after
    // setmaxnreg to that count
    if (warp >= Cfg::PRODUCER_WARP) {
        if constexpr (NT == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(AT_REGS_OTHER));
        pdl_wait();
        if (warp == Cfg::PRODUCER_WARP) {
            if (lane == 0) {   // TMA producer
                mbar_arrive_expect_tx(&q_bar, (uint32_t)(NT * AT_Q_BYTES));
                for (int t = 0; t < NT; ++t) {
                    tma_load_3d(sq + t * AT_Q_BYTES, &tmq, &q_bar, 0, h0 + t, tile.q0);
                    tma_load_3d(sq + t * AT_Q_BYTES + AT_Q_BOX, &tmq, &q_bar, 64, h0 + t, tile.q0);
                }
                // a stage is released only by the MMA thread, after it saw
                // the stage full (it stops at its first wait that gives up),
                // so a stage is never refilled before its last load landed;
                // after a wait has given up nothing more is issued
                int issued = 0;
                for (; issued < nb; ++issued) {
                    const int b = issued, st = b % NS;
                    const uint32_t ph = (uint32_t)(b / NS) & 1u;
                    if (!mbar_wait(&kv_empty[st], ph ^ 1u, err, 0x61)) break;
                    uint8_t *dst = skv + st * AT_STAGE_BYTES;
                    const int key = tile.kv0 + (kb0 + b) * AT_BKV;
                    mbar_arrive_expect_tx(&kv_full[st], (uint32_t)AT_STAGE_BYTES);
                    tma_load_3d(dst, &tmk, &kv_full[st], 0, hk, key);
                    tma_load_3d(dst + AT_KV_BOX, &tmk, &kv_full[st], 64, hk, key);
                    tma_load_3d(dst + 2 * AT_KV_BOX, &tmv, &kv_full[st], 0, hk, key);
                    tma_load_3d(dst + 3 * AT_KV_BOX, &tmv, &kv_full[st], 64, hk, key);
                }
                // the block outlives its copies (free in a healthy pipeline:
                // the MMA thread waits for the same loads)
                mbar_drain(&q_bar, 0);
                drain_ring(kv_full, NS, issued);
            }
        } else if (warp == Cfg::MMA_WARP) {
            if (lane == 0) {   // MMA issuer
                // S: A = Q, B = K (both K-major, shared memory); O: A = P (tensor
                // memory), B = V (MN-major, shared memory)
                const uint32_t id_s = idesc_n(AT_BKV), id_o = idesc_n(AT_D) | (1u << 16);
                // S into head t's columns (NT = 2) or into buffer buf (NT = 1)
                auto issue_s = [&](int t, int buf, int st, uint64_t *bar) {
                    const uint32_t qa = smem_u32(sq + t * AT_Q_BYTES), ka = smem_u32(skv + st * AT_STAGE_BYTES);
                    const uint32_t d = tmem_base + Cfg::s_col(t, buf);
#pragma unroll
                    for (int half = 0; half < 2; ++half)
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_bf16(d, sw128_desc(qa + half * AT_Q_BOX + k * 32),
                                      sw128_desc(ka + half * AT_KV_BOX + k * 32), id_s, (half | k) != 0 ? 1u : 0u);
                    umma_commit(bar);
                };
                // O += P V for block b of head t, P read from the columns S of block b left
                auto issue_pv = [&](int t, int b, int buf, int st) {
                    const uint32_t va = smem_u32(skv + st * AT_STAGE_BYTES + 2 * AT_KV_BOX);
                    const uint32_t pa = tmem_base + Cfg::s_col(t, buf);
                    const uint32_t d = tmem_base + Cfg::o_col(t);
#pragma unroll
                    for (int k = 0; k < AT_BKV / 16; ++k)
                        umma_bf16_ts(d, pa + k * 8, sw128_mn_desc(va + k * 2048), id_o,
                                     ((kb0 + b) % AT_CHUNK_BLOCKS | k) != 0 ? 1u : 0u);   // O restarts with every chunk
                };
                // every wait that completes is followed by a fence; the
                // thread stops at the first one that gives up (it then
                // issues and releases nothing more)
                auto wait = [&](uint64_t *bar, uint32_t parity, unsigned int where) {
                    const bool done = mbar_wait(bar, parity, err, where);
                    tc_fence_after();
                    return done;
                };
                auto wait_kv = [&](int b) { return wait(&kv_full[b % NS], (uint32_t)(b / NS) & 1u, 0x63); };
                bool run = wait(&q_bar, 0, 0x62) && wait_kv(0);
                if constexpr (NT == 2) {
                    // per block: O += P V, then the next block's S into the same
                    // columns, head 0 then head 1 (each head's softmax overlaps
                    // the other head's products)
                    if (run)
                        for (int t = 0; t < NT; ++t) issue_s(t, 0, 0, &s_full[t]);
                    for (int b = 0; run && b < nb; ++b) {
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            if (!(run = wait(&p_full[t], (uint32_t)b & 1u, 0x65))) break;
                            issue_pv(t, b, 0, b % NS);
                            umma_commit(&o_done[t][b & 1]);
                            if (t == NT - 1) umma_commit(&kv_empty[b % NS]);   // K and V of block b no longer read
                            if (b + 1 < nb) {   // the next block's scores, into the columns P V has just read
                                if (t == 0 && !(run = wait_kv(b + 1))) break;
                                issue_s(t, 0, (b + 1) % NS, &s_full[t]);
                            }
                        }
                    }
                } else {
                    // two S buffers: S of blocks 0 and 1 first; then per block b,
                    // O += P_b V_b and S of block b+2 into the buffer P_b was in,
                    // so the scores of block b+1 are ready while block b's
                    // softmax runs
                    if (run) issue_s(0, 0, 0, &s_full[0]);
                    if (run && nb > 1 && (run = wait_kv(1))) issue_s(0, 1, 1, &s_full[1]);
                    for (int b = 0; run && b < nb; ++b) {
                        if (!(run = wait(&p_full[0], (uint32_t)b & 1u, 0x65))) break;
                        issue_pv(0, b, b & 1, b % NS);
                        umma_commit(&o_done[0][b & 1]);
                        umma_commit(&kv_empty[b % NS]);
                        if (b + 2 < nb) {
                            if (!(run = wait_kv(b + 2))) break;
                            issue_s(0, b & 1, (b + 2) % NS, &s_full[b & 1]);
                        }
                    }
                }
                // every product issued is complete before the tensor memory is
                // freed (free in a healthy pipeline: the softmax waits for the
                // last of them)
                umma_drain(&drain_bar);
            }
        }
    } else {
        if constexpr (NT == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(AT_REGS_SOFTMAX));
        pdl_wait();
        // softmax: warpgroup t = head h0 + t; warp w may access tensor-memory
        // lanes 32*(w%4) .. +31
        const int t = warp >> 2, quad = warp & 3, row = quad * 32 + lane;
        const int pos = tile.pos0 + row;
        const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16);
        const uint32_t ocol = Cfg::o_col(t);
        float m = -INFINITY, l = 0.f;   // the current chunk's reference maximum and sum
        float M = 0.f, L = 0.f;         // a row past the first chunk: its merged state (mode 0)

        // P V of this CTA's block n done: block n's completion is phase n/2
        // of barrier n%2; the caller has already seen the scores of a later
        // block, so the product of block n-2 is complete and neither barrier
        // is ever two phases from the one awaited.
        auto wait_pv = [&](int n) {
            mbar_wait(&o_done[t][n & 1], ((uint32_t)n >> 1) & 1u, err, 0x67);
            tc_fence_after();
        };
        const int lc = pos / AT_CHUNK_KEYS;             // the row's last chunk
        const bool valid = row < tile.rows;
        const size_t orow = (size_t)(tile.q0 + (valid ? row : 0)) * (size_t)n_heads + (size_t)(h0 + t);
        uint4 *dst = reinterpret_cast<uint4 *>(O + orow * AT_D);
        float4 *srow = tile.part >= 0 ? reinterpret_cast<float4 *>(
                           part + (((size_t)tile.part * n_heads + (h0 + t)) * AT_BQ + row) * AT_PART_STRIDE)
                                      : nullptr;

        auto chunk_end = [&](int c, int bl) {
            wait_pv(bl);
            const float2 ML = attn_chunk_end(c, m, l, M, L, tbase + ocol, lc, valid, tile.mode, dst, srow,
                                             lse ? lse + orow : nullptr);
            M = ML.x;
            L = ML.y;
        };

        // blocks 0 .. nb-1, then b == nb closes the last chunk (one call site
        // of chunk_end keeps the loop's code small)
#pragma unroll 1
        for (int b = 0;; ++b) {
            // block b's scores: head t's columns (NT = 2), buffer b % 2 (NT = 1)
            const int sb = NT == 2 ? t : (b & 1);
            const uint32_t scol = Cfg::s_col(t, b & 1);
            if (b < nb) {
                mbar_wait(&s_full[sb], NT == 2 ? ((uint32_t)b & 1u) : (((uint32_t)b >> 1) & 1u), err, 0x68);
                tc_fence_after();
            }
            const bool chunk_start = (kb0 + b) % AT_CHUNK_BLOCKS == 0;
            if (b == nb && tile.part < 0) {             // a tile within the first chunk: o = O / l
                wait_pv(b - 1);
                const float rl = __frcp_rn(l);
#pragma unroll 1
                for (int ch = 0; ch < AT_D / 32; ++ch) {
                    uint32_t r[32];
                    tmem_ld32_nowait(tbase + ocol + ch * 32, r);
                    tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            uint4 v;
                            v.x = pack_bf16x2(__float_as_uint(__uint_as_float(r[8 * g + 0]) * rl),
                                              __float_as_uint(__uint_as_float(r[8 * g + 1]) * rl));
                            v.y = pack_bf16x2(__float_as_uint(__uint_as_float(r[8 * g + 2]) * rl),
                                              __float_as_uint(__uint_as_float(r[8 * g + 3]) * rl));
                            v.z = pack_bf16x2(__float_as_uint(__uint_as_float(r[8 * g + 4]) * rl),
                                              __float_as_uint(__uint_as_float(r[8 * g + 5]) * rl));
                            v.w = pack_bf16x2(__float_as_uint(__uint_as_float(r[8 * g + 6]) * rl),
                                              __float_as_uint(__uint_as_float(r[8 * g + 7]) * rl));
                            dst[ch * 4 + g] = v;
                        }
                    }
                }
                if (valid && lse) lse[orow] = (m + log2f(l)) * 0.693147180559945309f;
                break;
            }
            if (b == nb || (b > 0 && chunk_start)) {    // a chunk ends with block b-1
                chunk_end((kb0 + b - 1) / AT_CHUNK_BLOCKS, b - 1);
                if (b == nb) break;
                m = -INFINITY;
                l = 0.f;
            }
            // The block's 128 scores (one tensor-memory wait), the keys the row
            // cannot see set to -inf, and the block maximum (eight chains; the
            // maximum is exact in any order).
            const int nvis = pos - (kb0 + b) * AT_BKV + 1;   // keys of this block the row sees
            float s[AT_BKV];
#pragma unroll
            for (int ch = 0; ch < AT_BKV / 32; ++ch)
                tmem_ld32_nowait(tbase + scol + ch * 32, reinterpret_cast<uint32_t *>(&s[ch * 32]));
            tmem_ld_wait();
            if (nvis < AT_BKV) {
#pragma unroll
                for (int j = 0; j < AT_BKV; ++j)
                    if (j >= nvis) s[j] = -INFINITY;
            }
            float mx[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
            for (int j = 8; j < AT_BKV; ++j) mx[j & 7] = fmaxf(mx[j & 7], s[j]);
            const float bmc = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                    fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * c;
            const bool move = bmc > m + AT_TAU;

            // Before O is rescaled it must hold the chunk's blocks before b:
            // wait for block b-1's P V product (at a chunk's first block O is
            // about to restart, so there is nothing to rescale).  The
            // tensor-memory loads and stores are warp-wide (.sync.aligned):
            // every lane of the warp takes them, a lane whose maximum stays
            // with a = 1 (its O row is rewritten with the same bits).
            if (__any_sync(0xFFFFFFFFu, move)) {
                float a = 1.f;
                if (move) {
                    a = ex2(m - bmc);
                    l *= a;
                    m = bmc;
                }
                if (!chunk_start) {                      // a new chunk's O starts from zero
                    wait_pv(b - 1);
#pragma unroll 1
                    for (int ch = 0; ch < AT_D / 32; ++ch) {
                        uint32_t r[32];
                        tmem_ld32_nowait(tbase + ocol + ch * 32, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * a);
                        tmem_st32(tbase + ocol + ch * 32, r);
                    }
                }
            }

            // p_j as bf16 pairs, 64 keys at a time (the P operand, written over
            // the score columns, all of them already in registers: keys 64h ..
            // 64h+63 go to columns 32h .. 32h+31) and l.  l adds two pairwise
            // trees, over the block's even- and odd-position p_j, each built
            // leaf by leaf from the pairs (p_2i, p_2i+1) (a subtree is closed
            // as soon as its sibling is complete); the two halves' 32-leaf
            // subtrees meet at the root.
            float re[2], ro[2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[32];
                float te[6], to[6];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x0, x1;
                    ffma2(x0, x1, s[half * 64 + 2 * i], s[half * 64 + 2 * i + 1], c, c, -m, -m);
                    float e = ex2(x0), o = ex2(x1);
                    pk[i] = pack_bf16x2(__float_as_uint(e), __float_as_uint(o));
                    int lv = 0;
#pragma unroll
                    for (; lv < 5 && ((i >> lv) & 1); ++lv) ffma2(e, o, te[lv], to[lv], 1.f, 1.f, e, o);
                    te[lv] = e;
                    to[lv] = o;
                }
                re[half] = te[5];
                ro[half] = to[5];
                tmem_st32(tbase + scol + half * 32, pk);
            }
            float se, so;
            ffma2(se, so, re[0], ro[0], 1.f, 1.f, re[1], ro[1]);
            l += se + so;

            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[t]);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == Cfg::MMA_WARP) tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
}

// The rows of split tiles whose context runs past the first chunk: merge
// their chunks' partials in chunk order (merge_weights), then o and lse as
// in one pass.  One warp per (tile, head, row), four columns a lane.
struct AttnSplit {
    int q0, pos0, rows, slot0;   // the tile's first query, its position and rows; chunk c's partial slot = slot0 + c
};
constexpr int kAttnMaxSplits = 512;
struct AttnSplitTable {
    AttnSplit t[kAttnMaxSplits];
};

__global__ void __launch_bounds__(256)
attn_combine_kernel(const __grid_constant__ AttnSplitTable tab, int n_split, const float *__restrict__ part,
                    __nv_bfloat16 *__restrict__ O, float *__restrict__ lse, int n_heads)
{
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const long long per_split = (long long)n_heads * AT_BQ;
    if (w >= (long long)n_split * per_split) return;
    const AttnSplit sp = tab.t[w / per_split];
    const int h = (int)((w % per_split) / AT_BQ), row = (int)(w % AT_BQ);
    if (row >= sp.rows) return;
    const int pos = sp.pos0 + row, lc = pos / AT_CHUNK_KEYS;
    if (lc == 0) return;                               // finished by its chunk-0 CTA
    auto prow = [&](int ck) {
        return part + (((size_t)(sp.slot0 + ck) * n_heads + h) * AT_BQ + row) * AT_PART_STRIDE;
    };
    const float *p0 = prow(0);
    float M = p0[AT_D], L = p0[AT_D + 1];
    float4 N = reinterpret_cast<const float4 *>(p0)[lane];
    for (int ck = 1; ck <= lc; ++ck) {
        const float *pc = prow(ck);
        const MergeWeights mw = merge_weights(M, L, pc[AT_D], pc[AT_D + 1]);
        const float4 Oc = reinterpret_cast<const float4 *>(pc)[lane];
        N.x = fmaf(N.x, mw.a, __fmul_rn(Oc.x, mw.b));
        N.y = fmaf(N.y, mw.a, __fmul_rn(Oc.y, mw.b));
        N.z = fmaf(N.z, mw.a, __fmul_rn(Oc.z, mw.b));
        N.w = fmaf(N.w, mw.a, __fmul_rn(Oc.w, mw.b));
    }
    const float rl = __frcp_rn(L);
    const size_t orow = (size_t)(sp.q0 + row) * (size_t)n_heads + (size_t)h;
    uint2 v;
    v.x = pack_bf16x2(__float_as_uint(N.x * rl), __float_as_uint(N.y * rl));
    v.y = pack_bf16x2(__float_as_uint(N.z * rl), __float_as_uint(N.w * rl));
    reinterpret_cast<uint2 *>(O + orow * AT_D)[lane] = v;
    if (lane == 0 && lse) lse[orow] = (M + log2f(L)) * 0.693147180559945309f;
}

}  // namespace
}  // namespace bi

using namespace bi;

// The work of one call.  A query tile whose context ends within the first
// chunk is one entry.  A longer tile is either one entry whose CTA walks its
// chunks in turn, merging each into the tile's scratch slot (mode 0: the
// call is bound by its total work), or an entry per chunk, each leaving its
// partial in a slot for the merge kernel (mode 1: the call is bound by its
// longest tile, and the chunks of a long tile then run on other SMs at the
// same time).  The arithmetic, and so every bit of the result, is the same.
// Longest entries first: the CTAs that run longest start first.
struct AttnPlan {
    std::vector<AttnTile> entries;
    std::vector<AttnSplit> splits;
    long long slots = 0;
};

// Workspace: the slots, [slot][head][row][AT_PART_STRIDE] f32 (the split
// plan's count bounds the other's).
static size_t attn_workspace_size(const AttnPlan &pl, int n_heads)
{
    return (size_t)pl.slots * (size_t)n_heads * AT_BQ * AT_PART_STRIDE * sizeof(float);
}

static bool attn_plan(int n_req, const int32_t *q_offsets, const int32_t *kv_offsets, bool split, AttnPlan &pl)
{
    for (int r = 0; r < n_req; ++r) {
        const int ql = q_offsets[r + 1] - q_offsets[r], kl = kv_offsets[r + 1] - kv_offsets[r];
        for (int t0 = 0; t0 < ql; t0 += AT_BQ) {
            const int rows = std::min(AT_BQ, ql - t0), pos0 = kl - ql + t0;
            const int nb = attn_blocks(pos0, rows);
            if (nb <= AT_CHUNK_BLOCKS) {
                pl.entries.push_back({q_offsets[r] + t0, kv_offsets[r], pos0, rows, 0, nb, -1, 0});
                continue;
            }
            const int nch = (nb + AT_CHUNK_BLOCKS - 1) / AT_CHUNK_BLOCKS;
            if (pl.slots + nch > INT32_MAX) return false;
            if (!split) {
                pl.entries.push_back({q_offsets[r] + t0, kv_offsets[r], pos0, rows, 0, nb, (int)pl.slots, 0});
                pl.slots += 1;
                continue;
            }
            pl.splits.push_back({q_offsets[r] + t0, pos0, rows, (int)pl.slots});
            for (int ck = 0; ck < nch; ++ck)
                pl.entries.push_back({q_offsets[r] + t0, kv_offsets[r], pos0, rows, ck * AT_CHUNK_BLOCKS,
                                      std::min(nb, (ck + 1) * AT_CHUNK_BLOCKS), (int)pl.slots + ck, 1});
            pl.slots += nch;
        }
    }
    std::stable_sort(pl.entries.begin(), pl.entries.end(),
                     [](const AttnTile &x, const AttnTile &y) { return x.kb1 - x.kb0 > y.kb1 - y.kb0; });
    return true;
}

// Whether a call is bound by its longest tile: the tile's key blocks times
// the SMs against 1.2 times the call's key blocks times head pairs.
static bool attn_longest_bound(long long longest, long long work_pairs, int sm_count)
{
    return longest * sm_count * 5 > work_pairs * 6;
}

static bi_status attn_check_offsets(int32_t n_req, const int32_t *q_offsets, const int32_t *kv_offsets)
{
    if (n_req > 0 && (!q_offsets || !kv_offsets)) return BI_ERR_INVALID_ARG;
    if (n_req == 0) return BI_OK;
    if (q_offsets[0] != 0 || kv_offsets[0] != 0) return BI_ERR_INVALID_ARG;
    for (int r = 0; r < n_req; ++r) {
        const int64_t ql = (int64_t)q_offsets[r + 1] - q_offsets[r], kl = (int64_t)kv_offsets[r + 1] - kv_offsets[r];
        if (ql < 0 || kl < 0 || ql > kl) return BI_ERR_INVALID_ARG;
    }
    return BI_OK;
}

extern "C" size_t bi_attention_workspace_bytes(int32_t n_req, const int32_t *q_offsets, const int32_t *kv_offsets,
                                              int32_t n_heads)
{
    if (n_req < 0 || n_heads <= 0 || attn_check_offsets(n_req, q_offsets, kv_offsets) != BI_OK) return 0;
    AttnPlan pl;
    if (!attn_plan(n_req, q_offsets, kv_offsets, true, pl)) return 0;
    return attn_workspace_size(pl, n_heads);
}

extern "C" bi_status bi_attention_prefill(const void *q, const void *k, const void *v, int32_t n_req,
                                          const int32_t *q_offsets, const int32_t *kv_offsets, int32_t n_heads,
                                          int32_t n_kv_heads, int32_t head_dim, float scale, void *o, float *lse,
                                          void *workspace, size_t workspace_bytes, bi_stream s)
{
    if (n_req < 0 || n_heads <= 0 || n_kv_heads <= 0) return BI_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return BI_ERR_INVALID_ARG;
    if (n_heads % n_kv_heads != 0) return BI_ERR_INVALID_ARG;
    if (head_dim != AT_D) return BI_ERR_UNSUPPORTED_SHAPE;
    if (n_heads > BI_ATTN_MAX_HEADS) return BI_ERR_UNSUPPORTED_SHAPE;
    bi_status st = attn_check_offsets(n_req, q_offsets, kv_offsets);
    if (st != BI_OK) return st;
    if (n_req == 0) return BI_OK;
    const int64_t Tq = q_offsets[n_req], Tkv = kv_offsets[n_req];
    if (Tq == 0) return BI_OK;
    if (!q || !k || !v || !o) return BI_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return BI_ERR_MISALIGNED;
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return BI_ERR_MISALIGNED;

    AttnPlan bound;                                    // the workspace the caller was told to provide
    if (!attn_plan(n_req, q_offsets, kv_offsets, true, bound)) return BI_ERR_UNSUPPORTED_SHAPE;
    const size_t need = attn_workspace_size(bound, n_heads);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return BI_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return BI_ERR_MISALIGNED;
    }

    Device *d = nullptr;
    if ((st = current_device(&d)) != BI_OK) return st;
    // split long tiles into chunk CTAs where the call is bound by its longest tile
    long long work = 0, longest = 0;
    for (int r = 0; r < n_req; ++r) {
        const int ql = q_offsets[r + 1] - q_offsets[r], kl = kv_offsets[r + 1] - kv_offsets[r];
        for (int t0 = 0; t0 < ql; t0 += AT_BQ) {
            const long long nb = attn_blocks(kl - ql + t0, std::min(AT_BQ, ql - t0));
            work += nb * std::max(1, n_heads / 2);
            longest = std::max(longest, nb);
        }
    }
    AttnPlan pl;
    if (!attn_plan(n_req, q_offsets, kv_offsets, attn_longest_bound(longest, work, d->sm_count), pl))
        return BI_ERR_UNSUPPORTED_SHAPE;
    const std::vector<AttnTile> &tiles = pl.entries;
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
    const int group = n_heads / n_kv_heads;
    // Two heads of one key/value head per CTA share the K/V ring and keep the
    // tensor cores busiest, which wins where the call is bound by the
    // average work of an SM; one head per CTA (two score buffers) runs a
    // tile's chain of blocks in about 0.55 of the time, which wins where the
    // longest tile bounds the call.  The per-head arithmetic is the same
    // either way.
    int NT = 1;
    if (group % 2 == 0) {
        long long work = 0;                        // key blocks x head pairs
        for (const AttnTile &t : tiles) work += (long long)(t.kb1 - t.kb0) * (n_heads / 2);
        const long long longest = tiles[0].kb1 - tiles[0].kb0;
        if (!attn_longest_bound(longest, work, d->sm_count)) NT = 2;
    }
    const float c = scale * 1.44269504088896340736f;
    static_assert(sizeof(AttnTable) <= 8192, "kernel parameter space");
    auto launch = [&](auto kernel, int smem, int threads, int kid) -> bi_status {
        bi_status e = set_smem_once(d, kid, kernel, smem);
        if (e != BI_OK) return e;
        AttnTable tab;
        for (size_t first = 0; first < tiles.size(); first += kAttnMaxTiles) {
            const int n = (int)std::min<size_t>(kAttnMaxTiles, tiles.size() - first);
            std::copy(tiles.begin() + first, tiles.begin() + first + n, tab.t);
            e = launch_pdl(kernel, dim3((unsigned)(n * (n_heads / NT))), dim3(threads), (size_t)smem,
                           reinterpret_cast<cudaStream_t>(s), tmq, tmk, tmv, tab, static_cast<__nv_bfloat16 *>(o),
                           lse, static_cast<float *>(workspace), (int)n_heads, group, c, d->err);
            if (e != BI_OK) return e;
        }
        return BI_OK;
    };
    st = NT == 2 ? launch(attn_prefill_kernel<2>, AttnCfg<2>::SMEM, AttnCfg<2>::THREADS, KID_ATTN + 1)
                 : launch(attn_prefill_kernel<1>, AttnCfg<1>::SMEM, AttnCfg<1>::THREADS, KID_ATTN);
    if (st != BI_OK || pl.splits.empty()) return st;
    if ((st = set_smem_once(d, KID_ATTN + 2, attn_combine_kernel, 0)) != BI_OK) return st;
    AttnSplitTable stab;
    for (size_t first = 0; first < pl.splits.size(); first += kAttnMaxSplits) {
        const int n = (int)std::min<size_t>(kAttnMaxSplits, pl.splits.size() - first);
        std::copy(pl.splits.begin() + first, pl.splits.begin() + first + n, stab.t);
        const long long warps = (long long)n * n_heads * AT_BQ;
        st = launch_pdl(attn_combine_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0,
                        reinterpret_cast<cudaStream_t>(s), stab, n, static_cast<const float *>(workspace),
                        static_cast<__nv_bfloat16 *>(o), lse, (int)n_heads);
        if (st != BI_OK) return st;
    }
    return BI_OK;
}
