/*
 * oracle.c -- plain, slow CPU reference for the batch-invariant MoE router
 * and the M-invariant bf16 projection GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only through seeded inputs.
 *
 * Every sum here is taken in double precision in plain index order.  The
 * oracle does not try to reproduce the GPU's reduction order: it computes
 * the value the method defines, and the tests compare the GPU against it
 * within a stated tolerance (or bit-exactly where the arithmetic is exact).
 *
 * Sources, cited by page title and section:
 *  [P1] "batch changed the model's mind" (blog) -- sections "m-scan: the
 *       staircase", "16% of routing decisions", "The fix: m-invariant twins".
 *  [P3] "The Illusion of Determinism in Disaggregated Inference" -- sections
 *       "The engineering cost of determinism", "The low-level math of tile
 *       shapes", "The arithmetic cost of batch-invariant kernels".
 *  [P4] "diag(MODEL-MM-QWEN4-EXP): the MoE expert selections DIFFER, and a
 *       third of the boundaries are exact bf16 ties" -- intro, "Why a value
 *       tap could never have said this", "Why it is not a defect".
 *
 * Every function is pinned by the CPU test suite (tests/pins.py) against
 * closed forms, brute force, exact integer arithmetic or published test
 * vectors, and each pin is shown to catch planted mistakes
 * (tests/test_oracle_mutations.py).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32 pattern. */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static uint32_t f32_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/*
 * Round a double to the nearest bf16 value, ties to the even significand
 * (round-to-nearest-even; the rounding a bf16 store of an f32 accumulator
 * performs in [P3] "The low-level math of tile shapes": accumulate in FP32,
 * store as BF16).
 *
 * Written from the definition: find the spacing q of bf16 values at |v|
 * (8 significant bits, subnormal spacing 2^-133), scale |v| to units of q,
 * pick the nearer integer (the even one on an exact half), scale back.
 */
uint16_t orc_double_to_bf16_rne(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    if (isinf(a))
        return sign | 0x7F80;
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);           /* a = f * 2^e, 0.5 <= f < 1 */
    int qexp = e - 8;             /* 8 significant bits in [2^(e-1), 2^e) */
    if (qexp < -133)
        qexp = -133;              /* subnormal spacing */
    double n = ldexp(a, -qexp);   /* exact: scaling by a power of two */
    double r = floor(n);
    double frac = n - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    double out = ldexp(r, qexp);
    if (out >= ldexp(1.0, 128))   /* beyond the largest finite bf16 */
        return sign | 0x7F80;
    float of = (float)out;        /* exact: out has at most 8 significant bits */
    return sign | (uint16_t)(f32_bits(of) >> 16);
}

/* Round a double to binary32 (the C conversion rounds to nearest even). */
float orc_double_to_f32(double v) { return (float)v; }

/*
 * Sign-magnitude total order on raw bit patterns ([P4] "Why a value tap
 * could never have said this": the margin is also reported as a count of
 * representable steps, ordering patterns by sign and magnitude).  Positive patterns map to themselves,
 * negative ones to minus their magnitude, so +0 and -0 both map to 0 and
 * adjacent representable values differ by exactly 1.
 */
int64_t orc_ord_bf16(uint16_t b)
{
    return (b & 0x8000u) ? -(int64_t)(b & 0x7FFFu) : (int64_t)b;
}

int64_t orc_ord_f32(uint32_t b)
{
    return (b & 0x80000000u) ? -(int64_t)(b & 0x7FFFFFFFu) : (int64_t)b;
}

/* ------------------------------------------------------------------ */
/* Router projection  ([P1] "m-scan: the staircase": the MoE prefill   */
/* router is an F32 GEMV, logits = X . W_gate^T, one output per expert) */
/* ------------------------------------------------------------------ */

/* X f32 [M][H] (row stride ldx), W f32 [E][H] (row stride ldw). */
void orc_router_logits_f32in(const float *X, int64_t ldx, const float *W, int64_t ldw,
                             int64_t M, int64_t H, int64_t E, double *out)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t e = 0; e < E; ++e) {
            double s = 0.0;
            for (int64_t h = 0; h < H; ++h)
                s += (double)X[m * ldx + h] * (double)W[e * ldw + h];
            out[m * E + e] = s;
        }
}

/* bf16 inputs ([P4] "Why it is not a defect": the gate is a plain bf16
 * linear layer; products of bf16 values are exact in double). */
void orc_router_logits_bf16in(const uint16_t *X, int64_t ldx, const uint16_t *W, int64_t ldw,
                              int64_t M, int64_t H, int64_t E, double *out)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t e = 0; e < E; ++e) {
            double s = 0.0;
            for (int64_t h = 0; h < H; ++h)
                s += orc_bf16_to_double(X[m * ldx + h]) * orc_bf16_to_double(W[e * ldw + h]);
            out[m * E + e] = s;
        }
}

/* Sum of |x_h * w_h| per logit: the scale the F32 tolerance is stated on. */
void orc_router_absdot_f32in(const float *X, int64_t ldx, const float *W, int64_t ldw,
                             int64_t M, int64_t H, int64_t E, double *out)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t e = 0; e < E; ++e) {
            double s = 0.0;
            for (int64_t h = 0; h < H; ++h)
                s += fabs((double)X[m * ldx + h] * (double)W[e * ldw + h]);
            out[m * E + e] = s;
        }
}

/* ------------------------------------------------------------------ */
/* Top-k selection with the lowest-index tie-break                     */
/* ([P1] "m-scan": top_k(8 of 256); [P4] intro: at an exact tie the    */
/* the selection at an exact tie falls to the lower index)                       */
/* ------------------------------------------------------------------ */

/* a ranks strictly above b?  NaN ranks above every number (and NaNs
 * tie among themselves); -0 and +0 compare equal. */
static int ranks_above(double a, double b)
{
    if (isnan(a))
        return !isnan(b);
    if (isnan(b))
        return 0;
    return a > b;
}

/*
 * Sequential selection: k passes; each pass scans e = 0..E-1 and keeps the
 * first strict maximum among the experts not yet chosen.  Because a later
 * equal value never replaces the current best, exact ties go to the lowest
 * index.  ids come out in rank order (value descending, index ascending).
 */
void orc_topk_row(const double *row, int32_t E, int32_t k, int32_t *ids)
{
    unsigned char taken[4096];
    memset(taken, 0, (size_t)E);
    for (int32_t j = 0; j < k; ++j) {
        int32_t best = -1;
        for (int32_t e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            if (best < 0 || ranks_above(row[e], row[best]))
                best = e;
        }
        ids[j] = best;
        taken[best] = 1;
    }
}

/* Row-wise driver over an [M][E] matrix of logits (already in the logit
 * dtype, widened to double). */
void orc_topk(const double *logits, int64_t M, int32_t E, int32_t k, int32_t *ids)
{
    for (int64_t m = 0; m < M; ++m)
        orc_topk_row(logits + m * E, E, k, ids + m * k);
}

/* ------------------------------------------------------------------ */
/* Softmax renormalised over the selected k                            */
/* ([P1] "16% of routing decisions": the selection reweights the       */
/* mixture; [P4] "Why a value tap ...": the softmax denominator is an  */
/* f32 reduction over the selected logits)                             */
/* ------------------------------------------------------------------ */

/* w_j = exp(l_j - l_top) / sum_i exp(l_i - l_top), i over the selected,
 * l_top the rank-0 logit.  Subtracting l_top changes nothing in exact
 * arithmetic and keeps exp() in range. */
void orc_softmax_selected_row(const double *row, const int32_t *ids, int32_t k, double *w)
{
    double top = row[ids[0]];
    double den = 0.0;
    for (int32_t j = 0; j < k; ++j)
        den += exp(row[ids[j]] - top);
    for (int32_t j = 0; j < k; ++j)
        w[j] = exp(row[ids[j]] - top) / den;
}

void orc_softmax_selected(const double *logits, int64_t M, int32_t E, int32_t k,
                          const int32_t *ids, double *w)
{
    for (int64_t m = 0; m < M; ++m)
        orc_softmax_selected_row(logits + m * E, ids + m * k, k, w + m * k);
}

/* ------------------------------------------------------------------ */
/* Routing margin ([P1] "16% of routing decisions": routing margins;   */
/* [P4] "Why a value tap ...": smallest selected minus largest         */
/* rejected logit, and the same gap counted in ULPs of the logit dtype */
/* ordered by sign and then magnitude)                               */
/* ------------------------------------------------------------------ */

static void margin_endpoints(const double *row, int32_t E, const int32_t *ids, int32_t k,
                             int32_t *sel_min, int32_t *rej_max)
{
    unsigned char sel[4096];
    memset(sel, 0, (size_t)E);
    for (int32_t j = 0; j < k; ++j)
        sel[ids[j]] = 1;
    int32_t smin = -1, rmax = -1;
    for (int32_t e = 0; e < E; ++e) {
        if (sel[e]) {
            if (smin < 0 || row[e] < row[smin])
                smin = e;
        } else {
            if (rmax < 0 || row[e] > row[rmax])
                rmax = e;
        }
    }
    *sel_min = smin;
    *rej_max = rmax;
}

/* F32 logits.  margin = sel_min - rej_max in double; ulps = ord difference
 * of the raw binary32 patterns (int64; the library saturates at INT32_MAX).
 * With no rejected expert (k == E) margin = +inf and ulps = INT64_MAX. */
void orc_margin_f32(const float *logits, int64_t M, int32_t E, int32_t k, const int32_t *ids,
                    double *margin, int64_t *ulps, int32_t *sel_min_id, int32_t *rej_max_id)
{
    double row[4096];
    for (int64_t m = 0; m < M; ++m) {
        for (int32_t e = 0; e < E; ++e)
            row[e] = (double)logits[m * E + e];
        int32_t smin, rmax;
        margin_endpoints(row, E, ids + m * k, k, &smin, &rmax);
        if (sel_min_id) sel_min_id[m] = smin;
        if (rej_max_id) rej_max_id[m] = rmax;
        if (rmax < 0) {
            margin[m] = INFINITY;
            ulps[m] = INT64_MAX;
            continue;
        }
        margin[m] = row[smin] - row[rmax];
        ulps[m] = orc_ord_f32(f32_bits(logits[m * E + smin])) -
                  orc_ord_f32(f32_bits(logits[m * E + rmax]));
    }
}

/* bf16 logits: the same on 16-bit patterns. */
void orc_margin_bf16(const uint16_t *logits, int64_t M, int32_t E, int32_t k, const int32_t *ids,
                     double *margin, int64_t *ulps, int32_t *sel_min_id, int32_t *rej_max_id)
{
    double row[4096];
    for (int64_t m = 0; m < M; ++m) {
        for (int32_t e = 0; e < E; ++e)
            row[e] = orc_bf16_to_double(logits[m * E + e]);
        int32_t smin, rmax;
        margin_endpoints(row, E, ids + m * k, k, &smin, &rmax);
        if (sel_min_id) sel_min_id[m] = smin;
        if (rej_max_id) rej_max_id[m] = rmax;
        if (rmax < 0) {
            margin[m] = INFINITY;
            ulps[m] = INT64_MAX;
            continue;
        }
        margin[m] = row[smin] - row[rmax];
        ulps[m] = orc_ord_bf16(logits[m * E + smin]) - orc_ord_bf16(logits[m * E + rmax]);
    }
}

/* ------------------------------------------------------------------ */
/* Shared-expert gate ([P1] "m-scan": the one-output shared-expert     */
/* gate dot; "The fix": sigmoid_dot_rows)                              */
/* ------------------------------------------------------------------ */

void orc_shared_gate(const float *X, int64_t ldx, const float *w, int64_t M, int64_t H,
                     double *dot, double *sig)
{
    for (int64_t m = 0; m < M; ++m) {
        double s = 0.0;
        for (int64_t h = 0; h < H; ++h)
            s += (double)X[m * ldx + h] * (double)w[h];
        dot[m] = s;
        sig[m] = 1.0 / (1.0 + exp(-s));
    }
}

/* ------------------------------------------------------------------ */
/* bf16 projection GEMM ([P3] "The low-level math of tile shapes":     */
/* C = A.B with FP32 accumulation stored as BF16)                      */
/* ------------------------------------------------------------------ */

/* A bf16 [M][K] (lda), B bf16 [N][K] (ldb, the [out,in] weight of a
 * linear layer), exact double sum in k order.  acc [M][N] receives the
 * double value, C [M][N] (ldc) its bf16 rounding; absacc the sum of
 * |a*b| (the scale for the near-zero floor).  Any output may be NULL. */
void orc_gemm_bf16(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                   int64_t M, int64_t N, int64_t K,
                   double *acc, double *absacc, uint16_t *C, int64_t ldc)
{
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0, sa = 0.0;
            for (int64_t kk = 0; kk < K; ++kk) {
                double p = orc_bf16_to_double(A[m * lda + kk]) * orc_bf16_to_double(B[n * ldb + kk]);
                s += p;
                sa += fabs(p);
            }
            if (acc) acc[m * N + n] = s;
            if (absacc) absacc[m * N + n] = sa;
            if (C) C[m * ldc + n] = orc_double_to_bf16_rne(s);
        }
}

/* ------------------------------------------------------------------ */
/* Route-trace hash ([P4] "Why a value tap ...": one FNV-1a value per  */
/* call over the tokens' expert lists, each sorted first)              */
/* ------------------------------------------------------------------ */

/* 64-bit FNV-1a (Fowler/Noll/Vo): for each byte, xor it into the hash,
 * then multiply by the 64-bit FNV prime modulo 2^64.  The caller passes
 * the starting value: the FNV offset basis, or an earlier hash to chain. */
#define ORC_FNV64_PRIME 0x00000100000001B3ull
#define ORC_FNV64_BASIS 0xCBF29CE484222325ull

uint64_t orc_fnv64_basis(void) { return ORC_FNV64_BASIS; }

uint64_t orc_fnv1a64(const uint8_t *bytes, size_t n, uint64_t h)
{
    for (size_t i = 0; i < n; ++i) {
        h ^= (uint64_t)bytes[i];
        h *= ORC_FNV64_PRIME;
    }
    return h;
}

/* Rows [row_begin, row_end) of ids [M][k]: each row's ids sorted ascending
 * (the selected SET, order-free), serialised as little-endian int32 bytes,
 * rows in order, no separator; hashed starting from `basis`. */
uint64_t orc_route_hash(const int32_t *ids, int32_t k, int64_t row_begin, int64_t row_end,
                        uint64_t basis)
{
    uint64_t h = basis;
    int32_t srt[64];
    for (int64_t m = row_begin; m < row_end; ++m) {
        for (int32_t j = 0; j < k; ++j)
            srt[j] = ids[m * k + j];
        for (int32_t a = 1; a < k; ++a) {           /* insertion sort */
            int32_t v = srt[a], b = a - 1;
            while (b >= 0 && srt[b] > v) {
                srt[b + 1] = srt[b];
                --b;
            }
            srt[b + 1] = v;
        }
        for (int32_t j = 0; j < k; ++j) {
            uint32_t u = (uint32_t)srt[j];
            uint8_t le[4] = {(uint8_t)(u & 0xFF), (uint8_t)((u >> 8) & 0xFF),
                             (uint8_t)((u >> 16) & 0xFF), (uint8_t)((u >> 24) & 0xFF)};
            h = orc_fnv1a64(le, 4, h);
        }
    }
    return h;
}

/* ------------------------------------------------------------------ */
/* Array forms of the conversions above (plain loops).                 */
/* ------------------------------------------------------------------ */

void orc_round_bf16_array(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_double_to_bf16_rne(v[i]);
}

void orc_round_f32_array(const double *v, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_double_to_f32(v[i]);
}

void orc_bf16_to_double_array(const uint16_t *b, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_bf16_to_double(b[i]);
}
