// bi_hash.cu -- bi_route_trace_hash: 64-bit FNV-1a over the selected expert
// sets of ranges of token rows ("diag(MODEL-MM-QWEN4-EXP): the MoE expert
// selections DIFFER ...", section "Why a value tap could never have said
// this": per call, an FNV-1a hash of every token's sorted id list).
//
// FNV-1a is a sequential chain over bytes, so one thread walks one range;
// ranges (requests) are hashed in parallel.  Per row: the k ids are sorted
// ascending (the set, not the ranking), then their little-endian int32 bytes
// are folded in: h ^= byte; h *= 0x100000001b3 (mod 2^64).
#include "bi_device.cuh"
#include "bi_internal.h"

namespace bi {
namespace {

struct HashRanges {
    int32_t off[BI_MAX_HASH_RANGES + 1];
};

__global__ void route_hash_kernel(const int32_t *__restrict__ ids, int k, HashRanges rr, int n_ranges,
                                  const uint64_t *basis, uint64_t *out)
{
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n_ranges) return;
    uint64_t h = basis ? basis[r] : 0xCBF29CE484222325ull;
    int32_t srt[BI_MAX_K];
    for (int row = rr.off[r]; row < rr.off[r + 1]; ++row) {
        const int32_t *p = ids + (size_t)row * k;
        for (int a = 0; a < k; ++a) {                 // insertion sort
            const int32_t v = p[a];
            int b = a - 1;
            while (b >= 0 && srt[b] > v) {
                srt[b + 1] = srt[b];
                --b;
            }
            srt[b + 1] = v;
        }
        for (int a = 0; a < k; ++a) {
            uint32_t u = (uint32_t)srt[a];
#pragma unroll
            for (int byte = 0; byte < 4; ++byte) {
                h ^= (uint64_t)(u & 0xFFu);
                h *= 0x00000100000001B3ull;
                u >>= 8;
            }
        }
    }
    out[r] = h;
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
    return launch_pdl(route_hash_kernel, dim3((n_ranges + 127) / 128), dim3(128), 0,
                      reinterpret_cast<cudaStream_t>(s), ids, (int)k, rr, (int)n_ranges, basis, hash_out);
}
