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
// of tile t+1.  When the tiles are more than one wave but do not fill the
// last one, the tiles of that last partial wave are done as two 128 x 128
// halves each (N = 128 tensor-core steps), so it takes about half the time
// of a full wave; each output element still gets the same 16-deep steps in
// the same K order.  Every wait on an mbarrier is bounded (about 2 s); on
// expiry the kernel records BI_ERR_TIMEOUT in the device error word and
// carries on.
#include <cuda_bf16.h>

#include "bi_device.cuh"
#include "bi_internal.h"

namespace bi {
namespace {

constexpr int BM = kGemmTileM, BN = kGemmTileN, BK = kGemmBlockK, UMMA_K = kGemmMmaK, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int B_BYTES = BN * BK * 2;             // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;   // 48 KB
constexpr int GEMM_SMEM = STAGES * STAGE_BYTES + 1024;
constexpr int GEMM_THREADS = 192;
constexpr uint32_t ACC_COLS = BN;                // f32 columns per accumulator
constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;     // 512: the whole tensor memory

// Instruction descriptor, kind::f16: D f32 (bits 4-5 = 1), A bf16 (bits 7-9
// = 1), B bf16 (bits 10-12 = 1), A and B K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t idesc_n(int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
constexpr uint32_t IDESC = idesc_n(BN), IDESC_HALF = idesc_n(BN / 2);

// Work item i of a launch: items below n_full are whole tiles (tile = i);
// the rest are halves of the tiles from n_full on.  Returns the tile and
// sets `half` to -1 for a whole tile, else 0 or 1 (which 128 columns).
__device__ __forceinline__ int item_tile(int i, int n_full, int &half)
{
    if (i < n_full) {
        half = -1;
        return i;
    }
    half = (i - n_full) & 1;
    return n_full + ((i - n_full) >> 1);
}

// Shared-memory matrix descriptor for a K-major operand laid out by TMA with
// the 128-byte swizzle: rows of 64 bf16 (128 B), 8-row atoms 1024 B apart
// (stride byte offset), fixed version bits 46-47 = 1, layout type 2
// (128-byte swizzle) in bits 61-63.  Stepping K by 16 elements inside the
// 128-byte row adds 32 bytes to the start address (the swizzle is applied
// on absolute address bits, and every tile base is 1024-byte aligned).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;      // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024u >> 4) << 32;    // stride byte offset
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive f32 columns: thread t gets row (lane) t.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
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
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
    return *reinterpret_cast<const uint32_t *>(&v);
}

__global__ void __launch_bounds__(GEMM_THREADS, 1)
gemm_bf16_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                 const __grid_constant__ CUtensorMap tmb_half, __nv_bfloat16 *__restrict__ C, int M, int N,
                 int K, long long ldc, int n_full, unsigned int *err)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[STAGES], empty_bar[STAGES], tfull_bar[2], tempty_bar[2];
    __shared__ uint32_t tmem_base_sh;
    uint8_t *smem = smem_align1024(smem_raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m_tiles = (M + BM - 1) / BM, n_tiles = (N + BN - 1) / BN;
    const int num_tiles = m_tiles * n_tiles, kblocks = K / BK;
    const int num_items = n_full + 2 * (num_tiles - n_full);

    if (threadIdx.x == 0) {
        prefetch_tmap(&tma);
        prefetch_tmap(&tmb);
        prefetch_tmap(&tmb_half);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull_bar[b], 1);
            mbar_init(&tempty_bar[b], 4);
        }
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
            uint32_t it = 0;
            for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
                int half;
                const int tile = item_tile(item, n_full, half);
                const int mt = tile % m_tiles, nt = tile / m_tiles;
                const int n0 = nt * BN + (half > 0 ? BN / 2 : 0);
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    mbar_wait(&empty_bar[s], ph ^ 1u, err, 0x21);
                    uint8_t *st = smem + s * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full_bar[s], half < 0 ? STAGE_BYTES : A_BYTES + B_BYTES / 2);
                    tma_load_2d(st, &tma, &full_bar[s], kb * BK, mt * BM);
                    tma_load_2d(st + A_BYTES, half < 0 ? &tmb : &tmb_half, &full_bar[s], kb * BK, n0);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {   // MMA issuer
            uint32_t it = 0, tc = 0;
            for (int item = blockIdx.x; item < num_items; item += gridDim.x, ++tc) {
                const uint32_t idesc = item < n_full ? IDESC : IDESC_HALF;
                const uint32_t b = tc & 1u, tph = (tc >> 1) & 1u;
                mbar_wait(&tempty_bar[b], tph ^ 1u, err, 0x22);
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + b * ACC_COLS;
                for (int kb = 0; kb < kblocks; ++kb, ++it) {
                    const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                    mbar_wait(&full_bar[s], ph, err, 0x23);
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + s * STAGE_BYTES);
                    const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k)
                        umma_bf16(d_tmem, sw128_desc(a_addr + k * UMMA_K * 2),
                                  sw128_desc(b_addr + k * UMMA_K * 2), idesc, (kb | k) != 0 ? 1u : 0u);
                    umma_commit(&empty_bar[s]);       // stage reusable once these MMAs finish
                }
                umma_commit(&tfull_bar[b]);           // accumulator ready for the epilogue
            }
        }
    } else {
        // epilogue: warp w may read tensor-memory lanes 32*(w%4) .. +31
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        uint32_t tc = 0;
        for (int item = blockIdx.x; item < num_items; item += gridDim.x, ++tc) {
            int half;
            const int tile = item_tile(item, n_full, half);
            const int mt = tile % m_tiles, nt = tile / m_tiles;
            const int nbase = nt * BN + (half > 0 ? BN / 2 : 0), nchunks = half < 0 ? BN / 32 : BN / 64;
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

    alignas(64) CUtensorMap tma, tmb;
    {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)M};
        const uint64_t strides[1] = {(uint64_t)lda * 2};
        const uint32_t box[2] = {(uint32_t)BK, (uint32_t)BM};
        if ((st = encode_tiled(&tma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B)) != BI_OK)
            return st;
    }
    alignas(64) CUtensorMap tmb_half;
    for (int h = 0; h < 2; ++h) {
        const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
        const uint64_t strides[1] = {(uint64_t)ldb * 2};
        const uint32_t box[2] = {(uint32_t)BK, (uint32_t)(h ? BN / 2 : BN)};
        if ((st = encode_tiled(h ? &tmb_half : &tmb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, dims, strides, box,
                               CU_TENSOR_MAP_SWIZZLE_128B)) != BI_OK)
            return st;
    }
    if ((st = set_smem_once(d, KID_GEMM, gemm_bf16_kernel, GEMM_SMEM)) != BI_OK) return st;

    // whole tiles for every full wave; the tiles of a last partial wave go
    // as halves when that keeps them to one round (2 * rest <= blocks)
    const long long tiles = (long long)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    if (tiles > (1ll << 30)) return BI_ERR_UNSUPPORTED_SHAPE;
    const int grid = (int)(tiles < d->sm_count ? tiles : d->sm_count);
    const long long rest = tiles % grid;
    const long long n_full = (tiles > grid && rest != 0 && 2 * rest <= grid) ? tiles - rest : tiles;
    return launch_pdl(gemm_bf16_kernel, dim3(grid), dim3(GEMM_THREADS), (size_t)GEMM_SMEM,
                      reinterpret_cast<cudaStream_t>(s), tma, tmb, tmb_half, static_cast<__nv_bfloat16 *>(C),
                      (int)M, (int)N, (int)K, (long long)ldc, (int)n_full, d->err);
}
