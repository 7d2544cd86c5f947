// bi_tcgen05.cuh -- the pieces of the tcgen05 GEMM shared by the dense
// projection (bi_gemm.cu) and the grouped expert GEMM (bi_moe.cu): the tile
// constants of the numeric contract, the instruction and shared-memory
// descriptors, tensor-memory allocation, the MMA issue/commit and the
// accumulator read-back.
#pragma once

#include <cuda_bf16.h>

#include "bi_device.cuh"
#include "bi_internal.h"

namespace bi {

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
constexpr uint32_t IDESC = idesc_n(BN);

// Work item i of a launch: items below n_full are whole tiles (tile = i);
// the rest are pieces of the tiles from n_full on, each tile cut into
// 2^lg_s pieces of BN >> lg_s columns.  Returns the tile and sets `piece` to
// -1 for a whole tile, else the piece's index within its tile.
__device__ __forceinline__ int item_tile(int i, int n_full, int lg_s, int &piece)
{
    if (i < n_full) {
        piece = -1;
        return i;
    }
    piece = (i - n_full) & ((1 << lg_s) - 1);
    return n_full + ((i - n_full) >> lg_s);
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

// After a wait has given up: every tcgen05 operation this thread issued is
// complete (bounded) before the block frees its tensor memory.
__device__ __forceinline__ void umma_drain(uint64_t *bar)
{
    umma_commit(bar);
    mbar_drain(bar, 0);
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

}  // namespace bi
