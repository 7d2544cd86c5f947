// bi_gemm.cu -- bi_gemm_bf16: M-invariant bf16 projection C = A . B^T on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Source page: "The Illusion of Determinism in Disaggregated Inference",
// sections "The low-level math of tile shapes" (a GEMM library picks the
// tile shape, and with it the K-reduction tree, from M) and "The arithmetic
// cost of batch-invariant kernels" (one static reduction tree for every M,
// small batches padded up to the fixed tile, no shape heuristics).
//
// Invariance by construction: one tile shape (128 x 256) and one K schedule
// for every M and N.  Output element (m, n) is accumulated in f32 in tensor
// memory over K in blocks of 64, in increasing order, each block as four
// 16-deep tensor-core steps; nothing is split across thread blocks and there
// are no atomics.  Rows past M and columns past N are zero-filled by TMA and
// never stored.  The result is rounded to bf16 (nearest even) once.
//
// Structure (one persistent block per SM, 192 threads):
//   warp 0      TMA producer: A [128 x 64] and B [256 x 64] boxes per stage,
//               128-byte swizzle, a ring of 4 stages (48 KB each)
//   warp 1      allocates 512 tensor-memory columns (two 128 x 256 f32
//               accumulators); one lane issues tcgen05.mma and commits
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, bf16 pack,
//               16-byte global stores; releases the accumulator buffer
// Double-buffered accumulators let the epilogue of tile t overlap the MMAs
// of tile t+1.  Tiles are numbered N-fastest, so the blocks running at once
// spread over many B tiles instead of all reading the same few (same-box
// timings: 90.4 against 92.7 us at M = 4096, 162 against 173 us at 8192).  Tiles can be cut along N into 2, 4 or 8 pieces (N = 128, 64
// or 32 tensor-core steps) without changing any element's arithmetic: each
// output element still gets the same 16-deep steps in the same K order.
// Pieces serve two cases: when the tiles are more than one wave but do not
// fill the last one, the tiles of that last partial wave run as halves, so
// it takes about half the time of a full wave; and when there are fewer
// tiles than SMs (small M: one 128-row tile holds up to 128 tokens), every
// tile is cut into the most pieces that still fit one per SM, so that
// 8 times as many SMs stream the weight matrix.  Every wait on an mbarrier
// is bounded (about 2 s); on expiry the kernel records BI_ERR_TIMEOUT in the
// device error word, the producer and MMA threads issue nothing more and
// wait (bounded) for their own copies and products, the epilogue carries
// on, and the block frees its tensor memory.
#include <cuda_bf16.h>

#include "bi_device.cuh"
#include "bi_internal.h"
#include "bi_tcgen05.cuh"

namespace bi {
namespace {


__global__ void __launch_bounds__(GEMM_THREADS, 1)
gemm_bf16_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                 const __grid_constant__ CUtensorMap tmb_piece, __nv_bfloat16 *__restrict__ C, int M, int N,
                 int K, long long ldc, int n_full, int lg_s, int a_rows, unsigned int *err)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES], tfull_bar[2], tempty_bar[2], drain_bar;
    __shared__ uint32_t tmem_base_sh;
    uint8_t *smem = smem_align1024(smem_raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (M + BM - 1) / BM, n_tiles = (N + BN - 1) / BN;
    const int num_tiles = m_tiles * n_tiles, kblocks = K / BK;
    const int num_items = n_full + ((num_tiles - n_full) << lg_s);
    const int pn = BN >> lg_s;                           // columns of a piece
    const int a_bytes = a_rows * BK * 2;                 // A rows staged per K block (BM, or fewer for small M)

    if (threadIdx.x == 0) {
        prefetch_tmap(&tma);
        prefetch_tmap(&tmb);
        prefetch_tmap(&tmb_piece);
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

    if (warp == 0) {
        if (lane == 0) {   // TMA producer
            // a stage is released only by the MMA thread, after it saw the
            // stage full (it stops at its first wait that gives up), so a
            // stage is never refilled before its last load landed; after a
            // wait has given up nothing more is issued
            uint32_t s = 0, ph = 0;          // ring slot and its phase parity, advanced per K block
            int issued = 0;                  // ring steps issued
            bool run = true;
            for (int item = blockIdx.x; run && item < num_items; item += gridDim.x) {
                int piece;
                const int tile = item_tile(item, n_full, lg_s, piece);
                const int mt = tile / n_tiles, nt = tile % n_tiles;
                const int n0 = nt * BN + (piece > 0 ? piece * pn : 0);
                for (int kb = 0; kb < kblocks; ++kb, ++issued) {
                    if (!(run = mbar_wait(&empty_bar[s], ph ^ 1u, err, 0x21))) break;
                    uint8_t *st = smem + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full_bar[s], (uint32_t)a_bytes + (piece < 0 ? B_BYTES : (B_BYTES >> lg_s)));
                    tma_load_2d(st, &tma, &full_bar[s], kb * BK, mt * BM);
                    tma_load_2d(st + a_bytes, piece < 0 ? &tmb : &tmb_piece, &full_bar[s], kb * BK, n0);
                    if (++s == (uint32_t)STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // the block outlives its copies (free in a healthy pipeline: the
            // MMA thread waits for the same loads)
            drain_ring(full_bar, STAGES, issued);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // MMA issuer
            // stops at its first wait that gives up: it then issues and
            // releases nothing more
            uint32_t s = 0, ph = 0, tc = 0;
            bool run = true;
            for (int item = blockIdx.x; run && item < num_items; item += gridDim.x, ++tc) {
                const uint32_t idesc = item < n_full ? IDESC : idesc_n(pn);
                const uint32_t b = tc & 1u, tph = (tc >> 1) & 1u;
                if (!(run = mbar_wait(&tempty_bar[b], tph ^ 1u, err, 0x22))) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * ACC_COLS;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!(run = mbar_wait(&full_bar[s], ph, err, 0x23))) break;
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t b_addr = a_addr + a_bytes;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        umma_bf16(d_tmem, sw128_desc(a_addr + k * UMMA_K * 2),
                                  sw128_desc(b_addr + k * UMMA_K * 2), idesc, (kb | k) != 0 ? 1u : 0u);
                    umma_commit(&empty_bar[s]);       // stage reusable once these MMAs finish
                    if (++s == (uint32_t)STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!run) break;
                umma_commit(&tfull_bar[b]);           // accumulator ready for the epilogue
            }
            // every product issued is complete before the tensor memory is
            // freed (free in a healthy pipeline: the epilogue waits for the
            // last of them)
            umma_drain(&drain_bar);
        }
    } else {
        // epilogue: warp w may read tensor-memory lanes 32*(w%4) .. +31
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        uint32_t tc = 0;
        for (int item = blockIdx.x; item < num_items; item += gridDim.x, ++tc) {
            int piece;
            const int tile = item_tile(item, n_full, lg_s, piece);
            const int mt = tile / n_tiles, nt = tile % n_tiles;
            const int nbase = nt * BN + (piece > 0 ? piece * pn : 0), nchunks = piece < 0 ? BN / 32 : pn / 32;
            const uint32_t b = tc & 1u, tph = (tc >> 1) & 1u;
            mbar_wait(&tfull_bar[b], tph, err, 0x24);
            tc_fence_after();
            const int m = mt * BM + row;
            __nv_bfloat16 *crow = C + (size_t)(m < M ? m : 0) * (size_t)ldc;
#pragma unroll 1
            for (int chunk = 0; chunk < nchunks; ++chunk) {
                uint32_t r[32];
                tmem_ld32(tmem_base + ((uint32_t)(quad * 32) << 16) + b * ACC_COLS + chunk * 32, r);
                const int n0 = nbase + chunk * 32;
                if (m < M) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (n0 + 8 * g < N) {
                            uint4 v;
                            v.x = pack_bf16x2(r[8 * g + 0], r[8 * g + 1]);
                            v.y = pack_bf16x2(r[8 * g + 2], r[8 * g + 3]);
                            v.z = pack_bf16x2(r[8 * g + 4], r[8 * g + 5]);
                            v.w = pack_bf16x2(r[8 * g + 6], r[8 * g + 7]);
                            *reinterpret_cast<uint4 *>(crow + n0 + 8 * g) = v;
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

}  // namespace
}  // namespace bi

using namespace bi;

extern "C" bi_status bi_gemm_bf16(const void *A, const void *B, void *C, int32_t M, int32_t N, int32_t K,
                                  int64_t lda, int64_t ldb, int64_t ldc, bi_stream s)
{
    if (M < 0 || N <= 0 || K <= 0) return BI_ERR_INVALID_ARG;
    if (lda < K || ldb < K || ldc < N) return BI_ERR_INVALID_ARG;
    if ((K % BK) != 0 || (N % 16) != 0) return BI_ERR_UNSUPPORTED_SHAPE;
    if ((lda % 8) != 0 || (ldb % 8) != 0 || (ldc % 8) != 0) return BI_ERR_MISALIGNED;
    if (M == 0) return BI_OK;
    if (!A || !B || !C) return BI_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return BI_ERR_MISALIGNED;

    Device *d = nullptr;
    bi_status st = current_device(&d);
    if (st != BI_OK) return st;

    // A single M tile of fewer than BM rows stages only its rows rounded up to
    // a whole 8-row swizzle atom: the tile's other rows of A in shared memory
    // then hold whatever the stage held before, which only reaches output
    // rows past M, and those are never stored (an output row's value is a
    // function of its own A row and B alone).
    const int a_rows = M < BM ? (M + 7) / 8 * 8 : BM;
    alignas(64) CUtensorMap tma, tmb;
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)lda * 2};
        const uint32_t box[2] = {(uint32_t)BK, (uint32_t)a_rows};
        if ((st = encode_tiled(&tma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B)) != BI_OK)
            return st;
    }
    // The work plan (any plan gives the same bits):
    //  - fewer tiles than SMs: every tile cut into 2^lg_s pieces, the most
    //    (at most 8) that still give each piece an SM of its own;
    //  - otherwise whole tiles for every full wave, and the tiles of a last
    //    partial wave as halves when that keeps them to one round
    //    (2 * rest <= blocks).
    const long long tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    if (tiles > (1ll << 30)) return BI_ERR_UNSUPPORTED_SHAPE;
    long long n_full, items;
    int lg_s = 1;
    if (tiles < d->sm_count) {
        lg_s = 0;
        while (lg_s < 3 && (tiles << (lg_s + 1)) <= d->sm_count) ++lg_s;
        n_full = lg_s == 0 ? tiles : 0;
        items = tiles << lg_s;
    } else {
        const long long rest = tiles % d->sm_count;
        n_full = (rest != 0 && 2 * rest <= d->sm_count) ? tiles - rest : tiles;
        items = n_full + 2 * (tiles - n_full);
    }
    if (lg_s == 0) lg_s = 1;             // no pieces in this launch; the piece map is then unused
    const int grid = (int)(items < d->sm_count ? items : d->sm_count);
    alignas(64) CUtensorMap tmb_piece;
    for (int h = 0; h < 2; ++h) {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
        const uint64_t strides[1] = {(uint64_t)ldb * 2};
        const uint32_t box[2] = {(uint32_t)BK, (uint32_t)(h ? BN >> lg_s : BN)};
        if ((st = encode_tiled(h ? &tmb_piece : &tmb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B)) != BI_OK)
            return st;
    }
    if ((st = set_smem_once(d, KID_GEMM, gemm_bf16_kernel, GEMM_SMEM)) != BI_OK) return st;
    return launch_pdl(gemm_bf16_kernel, dim3(grid), dim3(GEMM_THREADS), (size_t)GEMM_SMEM,
                      reinterpret_cast<cudaStream_t>(s), tma, tmb, tmb_piece, static_cast<__nv_bfloat16 *>(C),
                      (int)M, (int)N, (int)K, (long long)ldc, (int)n_full, lg_s, a_rows, d->err);
}
