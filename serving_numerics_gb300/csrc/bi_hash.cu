// bi_hash.cu -- bi_route_trace_hash: 64-bit FNV-1a over the selected expert
// sets of ranges of token rows ("diag(MODEL-MM-QWEN4-EXP): the MoE expert
// selections DIFFER ...", section "Why a value tap could never have said
// this": one FNV-1a value per call over the tokens' sorted id lists).
//
// FNV-1a is one sequential chain over bytes, so a range is walked by one
// warp: the 32 lanes each load and sort one row (an odd-even transposition
// network on registers, ids beyond k padded with INT_MAX), then every lane
// folds the 32 sorted rows into the same chain, receiving each id by
// shuffle, and lane 0 stores the result.  The chain's critical path is one
// xor and one wide multiply per byte.  Ranges (requests) are hashed in
// parallel, one warp each.
//
// Per byte: h ^= byte; h *= 0x100000001b3 (mod 2^64).  Per row: the k ids
// in ascending order, each as 4 little-endian bytes.
#include <limits.h>

#include "bi_device.cuh"
#include "bi_internal.h"

namespace bi {
namespace {

struct HashRanges {
    int32_t off[BI_MAX_HASH_RANGES + 1];
};

constexpr int kHashWarps = 4;

// One FNV-1a byte step on the hash held as two 32-bit halves:
// h = (h ^ byte) * (2^40 + 0x1b3) mod 2^64.  With l = lo ^ byte, the product
// is l*0x1b3 (64-bit) + (hi*0x1b3 + (l << 8)) * 2^32, keeping the dependent
// chain at one xor and one wide multiply per byte.
__device__ __forceinline__ void fnv_step(uint32_t &lo, uint32_t &hi, uint32_t byte)
{
    const uint32_t l = lo ^ byte;
    const uint64_t p = (uint64_t)l * 0x1B3u;
    lo = (uint32_t)p;
    hi = hi * 0x1B3u + (uint32_t)(p >> 32) + (l << 8);
}

template <int KMAX>
__global__ void __launch_bounds__(32 * kHashWarps)
route_hash_kernel(const int32_t *__restrict__ ids, int k, HashRanges rr, int n_ranges,
                  const uint64_t *basis, uint64_t *out)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int r = blockIdx.x * kHashWarps + (threadIdx.x >> 5);
    if (r >= n_ranges) return;                        // warp-uniform
    const uint64_t h0 = basis ? basis[r] : 0xCBF29CE484222325ull;
    uint32_t hlo = (uint32_t)h0, hhi = (uint32_t)(h0 >> 32);
    const int b = rr.off[r], e = rr.off[r + 1];
    for (int row0 = b; row0 < e; row0 += 32) {
        const int row = row0 + lane;
        int32_t v[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) v[j] = (row < e && j < k) ? ids[(size_t)row * k + j] : INT_MAX;
        // odd-even transposition sort: KMAX rounds make any KMAX values ascending
#pragma unroll
        for (int round = 0; round < KMAX; ++round) {
#pragma unroll
            for (int j = round & 1; j + 1 < KMAX; j += 2) {
                const int32_t lo = min(v[j], v[j + 1]), hi = max(v[j], v[j + 1]);
                v[j] = lo;
                v[j + 1] = hi;
            }
        }
        const int nrows = min(32, e - row0);
        for (int t = 0; t < nrows; ++t) {
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                const uint32_t u = (uint32_t)__shfl_sync(0xFFFFFFFFu, v[j], t);
                if (j < k) {
                    fnv_step(hlo, hhi, u & 0xFFu);
                    fnv_step(hlo, hhi, (u >> 8) & 0xFFu);
                    fnv_step(hlo, hhi, (u >> 16) & 0xFFu);
                    fnv_step(hlo, hhi, u >> 24);
                }
            }
        }
    }
    if (lane == 0) out[r] = ((uint64_t)hhi << 32) | hlo;
}

template <int KMAX>
bi_status launch_hash(Device *d, const int32_t *ids, int k, const HashRanges &rr, int n, const uint64_t *basis,
                      uint64_t *out, cudaStream_t s)
{
    const int kid = KID_HASH + (KMAX == 4 ? 0 : KMAX == 8 ? 1 : KMAX == 16 ? 2 : 3);
    bi_status st = set_smem_once(d, kid, route_hash_kernel<KMAX>, 0);
    if (st != BI_OK) return st;
    return launch_pdl(route_hash_kernel<KMAX>, dim3((n + kHashWarps - 1) / kHashWarps),
                      dim3(32 * kHashWarps), 0, s, ids, k, rr, n, basis, out);
}

}  // namespace
}  // namespace bi

using namespace bi;

extern "C" bi_status bi_route_trace_hash(const int32_t *ids, int32_t M, int32_t k,
                                         const int32_t *row_offsets, int32_t n_ranges,
                                         const uint64_t *basis, uint64_t *hash_out, bi_stream s)
{
    if (M < 0 || k <= 0 || n_ranges <= 0 || !row_offsets || !hash_out) return BI_ERR_INVALID_ARG;
    if (k > BI_MAX_K || n_ranges > BI_MAX_HASH_RANGES) return BI_ERR_UNSUPPORTED_SHAPE;
    HashRanges rr;
    for (int r = 0; r <= n_ranges; ++r) {
        const int32_t o = row_offsets[r];
        if (o < 0 || o > M || (r > 0 && o < row_offsets[r - 1])) return BI_ERR_INVALID_ARG;
        rr.off[r] = o;
    }
    if (M > 0 && !ids) return BI_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ids) & 3u) || (reinterpret_cast<uintptr_t>(basis) & 7u) ||
        (reinterpret_cast<uintptr_t>(hash_out) & 7u))
        return BI_ERR_MISALIGNED;
    Device *d = nullptr;
    bi_status st = current_device(&d);
    if (st != BI_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    if (k <= 4) return launch_hash<4>(d, ids, k, rr, n_ranges, basis, hash_out, cs);
    if (k <= 8) return launch_hash<8>(d, ids, k, rr, n_ranges, basis, hash_out, cs);
    if (k <= 16) return launch_hash<16>(d, ids, k, rr, n_ranges, basis, hash_out, cs);
    return launch_hash<32>(d, ids, k, rr, n_ranges, basis, hash_out, cs);
}
