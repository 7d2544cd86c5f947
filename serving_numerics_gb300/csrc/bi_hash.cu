// bi_hash.cu -- bi_route_trace_hash: 64-bit FNV-1a over the selected expert
// sets of ranges of token rows ("diag(MODEL-MM-QWEN4-EXP): the MoE expert
// selections DIFFER ...", section "Why a value tap could never have said
// this": one FNV-1a value per call over the tokens' sorted id lists).
//
// FNV-1a is one sequential chain over bytes, so a range is walked by one
// warp: the 32 lanes each load and sort one row (an odd-even transposition
// network on registers, ids beyond k padded with INT_MAX); then every lane
// folds the rows into the same chain, receiving each row's ids by shuffle
// one row ahead of the fold, and lane 0 stores the result.  Ranges
// (requests) are hashed in parallel, one warp each; with one warp per
// scheduler the fold's dependent chain is the kernel's whole cost.
//
// Per byte: h ^= byte; h *= 0x100000001b3 (mod 2^64).  Per row: the k ids
// in ascending order, each as 4 little-endian bytes.  A zero byte leaves
// h ^ byte = h, so the three steps of an id's zero high bytes are plain
// multiplications by the prime and fold into the step of its low byte: an
// id in [0, 256) is one step, h = (h ^ id) * prime^4 (mod 2^64, the same
// value).  A row whose ids all lie in [0, 256) takes that path; any other
// row takes the four byte steps per id.
#include <limits.h>

#include "bi_device.cuh"
#include "bi_internal.h"

namespace bi {
namespace {

struct HashRanges {
    int32_t off[BI_MAX_HASH_RANGES + 1];
};

constexpr int kHashWarps = 4;
constexpr uint64_t kFnvPrime = 0x100000001B3ull;

constexpr uint64_t prime_pow(int n) { return n == 0 ? 1ull : kFnvPrime * prime_pow(n - 1); }

// h = (h with its low half replaced by l) * c mod 2^64, on 32-bit halves;
// the chain through lo is one multiply per step
__device__ __forceinline__ void fnv_mul(uint32_t &lo, uint32_t &hi, uint32_t l, uint64_t c)
{
    const uint32_t clo = (uint32_t)c, chi = (uint32_t)(c >> 32);
    hi = hi * clo + __umulhi(l, clo) + l * chi;
    lo = l * clo;
}

// (lo, hi) <- (lo ^ x) * c when `on`, else unchanged; no branch, so the
// chain never waits on branch resolution
__device__ __forceinline__ void fnv_step_sel(uint32_t &lo, uint32_t &hi, uint32_t x, uint64_t c, bool on)
{
    uint32_t nlo = lo, nhi = hi;
    fnv_mul(nlo, nhi, lo ^ x, c);
    lo = on ? nlo : lo;
    hi = on ? nhi : hi;
}

template <int KMAX>
__device__ __forceinline__ void fold_row(uint32_t &lo, uint32_t &hi, const uint32_t (&u)[KMAX], int k,
                                         bool one_byte)
{
    if (one_byte) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j) fnv_step_sel(lo, hi, u[j], prime_pow(4), j < k);
    } else {
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            fnv_step_sel(lo, hi, u[j] & 0xFFu, kFnvPrime, j < k);
            fnv_step_sel(lo, hi, (u[j] >> 8) & 0xFFu, kFnvPrime, j < k);
            fnv_step_sel(lo, hi, (u[j] >> 16) & 0xFFu, kFnvPrime, j < k);
            fnv_step_sel(lo, hi, u[j] >> 24, kFnvPrime, j < k);
        }
    }
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
    // each lane's row of the next 32 is loaded while the current 32 fold
    int32_t v[KMAX], vn[KMAX];
#pragma unroll
    for (int j = 0; j < KMAX; ++j) vn[j] = (b + lane < e && j < k) ? ids[(size_t)(b + lane) * k + j] : INT_MAX;
    for (int row0 = b; row0 < e; row0 += 32) {
        const int nrow = row0 + 32 + lane;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
            v[j] = vn[j];
            vn[j] = (nrow < e && j < k) ? ids[(size_t)nrow * k + j] : INT_MAX;
        }
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
        // rows whose ids all lie in [0, 256): sorted, so the ends decide
        int32_t last = v[0];
#pragma unroll
        for (int j = 1; j < KMAX; ++j)
            if (j < k) last = v[j];
        const uint32_t one_byte = __ballot_sync(0xFFFFFFFFu, v[0] >= 0 && last < 256);
        const int nrows = min(32, e - row0);
        uint32_t cur[KMAX], nxt[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) cur[j] = (uint32_t)__shfl_sync(0xFFFFFFFFu, v[j], 0);
        for (int t = 0; t < nrows; ++t) {
            const int tn = t + 1 < nrows ? t + 1 : t;         // the next row's ids travel meanwhile
#pragma unroll
            for (int j = 0; j < KMAX; ++j) nxt[j] = (uint32_t)__shfl_sync(0xFFFFFFFFu, v[j], tn);
            fold_row<KMAX>(hlo, hhi, cur, k, (one_byte >> t) & 1u);
#pragma unroll
            for (int j = 0; j < KMAX; ++j) cur[j] = nxt[j];
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
