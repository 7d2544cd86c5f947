/*
 * contract.c -- CPU restatement of the reduction order the library commits
 * to for its router projection and shared gate.
 *
 * TEST INFRASTRUCTURE ONLY, like oracle.c: only the test suite loads it.  It
 * shares no code with the CUDA library; it is written from the contract as
 * the library's header states it, so that a GPU test can hold the kernels to
 * that order bit for bit (the oracle proper, oracle.c, computes the exact
 * value in double and the parity tests use a tolerance).
 *
 * The contract (the pages' fix, "batch changed the model's mind", section
 * "The fix: m-invariant twins": one fixed reduction order per output,
 * whatever the number of rows in the launch; the order itself is this
 * library's choice):
 *   h is cut into slabs of 128 and each slab into 16 blocks of 8;
 *   partition q (0..15) owns block q of every slab and runs one f32 fused
 *   multiply-add chain from +0 over the h < H it owns, h increasing;
 *   the 16 partial sums are added by the pairwise tree (0+1), (2+3), ...,
 *   then pairs of those: four levels, in f32.
 * fmaf from the C library is the correctly rounded f32 fused multiply-add.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { SLAB = 128, BLOCK = 8, PARTITIONS = 16 };

static float bf16_widen(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static float contract_dot(const float *x, const float *w, int64_t H)
{
    float part[PARTITIONS];
    for (int q = 0; q < PARTITIONS; ++q) part[q] = 0.0f;
    for (int64_t slab = 0; slab * SLAB < H; ++slab)
        for (int q = 0; q < PARTITIONS; ++q)
            for (int i = 0; i < BLOCK; ++i) {
                const int64_t h = slab * SLAB + (int64_t)q * BLOCK + i;
                if (h < H) part[q] = fmaf(x[h], w[h], part[q]);
            }
    for (int d = 1; d < PARTITIONS; d *= 2)
        for (int q = 0; q + d < PARTITIONS; q += 2 * d) part[q] = part[q] + part[q + d];
    return part[0];
}

/* out[m*E + e] = contract dot of row m of X [M,H] and row e of W [E,H]. */
void ctr_router_f32in(const float *X, const float *W, int64_t M, int64_t E, int64_t H, float *out)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t e = 0; e < E; ++e) out[m * E + e] = contract_dot(X + m * H, W + e * H, H);
}

/* The same for bf16 inputs (widened to f32 exactly; products of two bf16
 * values are exact in f32, so each step still rounds once). */
void ctr_router_bf16in(const uint16_t *X, const uint16_t *W, int64_t M, int64_t E, int64_t H, float *out,
                       float *xs, float *ws)
{
    /* xs [H] and ws [E*H] are caller-provided scratch for the widened rows */
    for (int64_t i = 0; i < E * H; ++i) ws[i] = bf16_widen(W[i]);
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t h = 0; h < H; ++h) xs[h] = bf16_widen(X[m * H + h]);
        for (int64_t e = 0; e < E; ++e) out[m * E + e] = contract_dot(xs, ws + e * H, H);
    }
}
