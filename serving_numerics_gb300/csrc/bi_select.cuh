// bi_select.cuh -- the per-token selection shared by the router kernels: top-k
// under (value descending, index ascending), softmax over the selected k in
// rank order, and the routing margin as a value and in ULPs of the logit
// dtype under the sign-magnitude order.
//
// Source pages: "batch changed the model's mind" ("m-scan: the staircase":
// top_k(8 of 256) after the router GEMV); "diag(MODEL-MM-QWEN4-EXP): the MoE
// expert selections DIFFER ..." (intro: exact ties go to the lowest index;
// "Why a value tap could never have said this": the margin between the
// smallest selected and the largest rejected logit, in bf16 ULPs ordered by
// sign and then magnitude; the softmax denominator as an f32 sum in the
// device's order).
#pragma once
#include <limits.h>
#include <stdint.h>

namespace bi {

// Order key of an f32 value: larger key = ranks higher.  NaN ranks above
// everything; -0 is folded onto +0 so the two compare equal.  Key 0 is below
// every real value (the smallest, -inf, maps to 0x007FFFFF) and marks a
// taken expert.
__device__ __forceinline__ uint32_t rank_key(float x)
{
    uint32_t u = __float_as_uint(x);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0xFFFFFFFFu;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sign-magnitude ordinal of a logit-dtype pattern (+0 and -0 both 0).
__device__ __forceinline__ long long sm_ord(float x, int bf16)
{
    uint32_t u = __float_as_uint(x);
    if (bf16) {
        const uint32_t b = u >> 16;
        return (b & 0x8000u) ? -(long long)(b & 0x7FFFu) : (long long)b;
    }
    return (u & 0x80000000u) ? -(long long)(u & 0x7FFFFFFFu) : (long long)u;
}

// One warp selects for one token.  v[i] holds the logit of expert lane + 32 i
// for i < epl (already in the logit dtype's values); the rest are ignored.
// Writes ids[m, 0..k) in rank order, and (where the pointers are not NULL)
// weights[m, 0..k), margin[m], ulps[m].  k < E is assumed (checked by the
// host).  Every lane of the warp must call it.
template <int EPLM>
__device__ __forceinline__ void warp_select(float (&v)[EPLM], int lane, int epl, int k, int logit_bf16, size_t m,
                                            int32_t *__restrict__ ids, float *__restrict__ weights,
                                            float *__restrict__ margin, int32_t *__restrict__ ulps)
{
    // each lane sorts its (key, index) pairs once, best first (ascending
    // index among equal keys); a round then only compares lane heads
    uint32_t key[EPLM];
    int idx[EPLM];
#pragma unroll
    for (int i = 0; i < EPLM; ++i) {
        key[i] = i < epl ? rank_key(v[i]) : 0u;
        idx[i] = lane + 32 * i;
    }
#pragma unroll
    for (int a = 0; a < EPLM; ++a) {            // odd-even transposition network
#pragma unroll
        for (int i = a & 1; i + 1 < EPLM; i += 2) {
            const bool sw = key[i + 1] > key[i];    // equal keys keep the lower index first
            const uint32_t k0 = sw ? key[i + 1] : key[i], k1 = sw ? key[i] : key[i + 1];
            const int i0 = sw ? idx[i + 1] : idx[i], i1 = sw ? idx[i] : idx[i + 1];
            const float v0 = sw ? v[i + 1] : v[i], v1 = sw ? v[i] : v[i + 1];
            key[i] = k0; key[i + 1] = k1; idx[i] = i0; idx[i + 1] = i1; v[i] = v0; v[i + 1] = v1;
        }
    }

    float l0 = 0.0f, my_v = 0.0f, v_sel_min = 0.0f, v_rej_max = 0.0f;
    int my_id = 0;
    for (int r = 0; r <= k; ++r) {
        const uint32_t bk = key[0];
        const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, bk);
        const uint32_t holders = __ballot_sync(0xFFFFFFFFu, bk == mk);
        // one lane holds the maximum key: its head wins (its index and value
        // read in parallel); several (equal values in different lanes): the
        // lowest index among them wins
        int wl = __ffs(holders) - 1;
        uint32_t win = (uint32_t)__shfl_sync(0xFFFFFFFFu, idx[0], wl);
        float wv = __shfl_sync(0xFFFFFFFFu, v[0], wl);
        if ((holders & (holders - 1u)) != 0u) {
            win = __reduce_min_sync(0xFFFFFFFFu, bk == mk ? (uint32_t)idx[0] : 0xFFFFFFFFu);
            wl = (int)(win & 31u);
            wv = __shfl_sync(0xFFFFFFFFu, v[0], wl);
        }
        if (lane == wl) {                       // pop the head
#pragma unroll
            for (int i = 0; i + 1 < EPLM; ++i) {
                key[i] = key[i + 1];
                idx[i] = idx[i + 1];
                v[i] = v[i + 1];
            }
            key[EPLM - 1] = 0u;
        }
        if (r == k) {
            v_rej_max = wv;
            break;
        }
        if (r == 0) l0 = wv;
        if (lane == r) {                     // lane r keeps rank r
            my_v = wv;
            my_id = (int)win;
        }
        v_sel_min = wv;
    }
    // softmax over the selected: each of lanes 0..k-1 takes its rank's
    // exponential once; the denominator adds them in rank order
    const float my_e = lane < k ? expf(my_v - l0) : 0.0f;
    float den = 0.0f;
    for (int r = 0; r < k; ++r) den += __shfl_sync(0xFFFFFFFFu, my_e, r);
    if (lane < k) {
        ids[m * k + lane] = my_id;
        if (weights) weights[m * k + lane] = my_e / den;
    }
    if (lane == 0) {
        if (margin) margin[m] = v_sel_min - v_rej_max;
        if (ulps) {
            long long d = sm_ord(v_sel_min, logit_bf16) - sm_ord(v_rej_max, logit_bf16);
            if (d > INT_MAX) d = INT_MAX;
            if (d < INT_MIN) d = INT_MIN;
            ulps[m] = (int32_t)d;
        }
    }
}

}  // namespace bi
