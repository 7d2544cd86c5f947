/*
 * bi.h -- C ABI of libbi, a batch-invariant (M-invariant) MoE prefill
 * numerics library for one NVIDIA GB300 (sm_103a).
 *
 * Every result row computed here is a function of that row's inputs and of
 * the problem's fixed sizes (H, E, k, N, K) only: never of the total token
 * count M, of the row's position in the batch, or of what else shares the
 * call.  That is the property the source pages turn on:
 *
 *  [P1] "batch changed the model's mind" (blog): "m-scan: the staircase"
 *       (a router GEMV whose library picks its reduction order by M moves a
 *       request's logits when co-arrivals change M), "16% of routing
 *       decisions" (top-k turns that drift into different expert sets),
 *       "The fix: m-invariant twins" (one fixed reduction order per row,
 *       whatever the number of rows in the launch).
 *  [P3] "The Illusion of Determinism in Disaggregated Inference": "The
 *       engineering cost of determinism" (cache hit vs miss runs the GEMM at
 *       another M), "The low-level math of tile shapes" (tile shape chosen by
 *       M changes the K-reduction tree), "The arithmetic cost of
 *       batch-invariant kernels" (a static reduction tree for every shape).
 *  [P4] "diag(MODEL-MM-QWEN4-EXP): the MoE expert selections DIFFER, and a
 *       third of the boundaries are exact bf16 ties": intro (lowest-index
 *       tie-break), "Why a value tap could never have said this" (sorted ids,
 *       margin in ULPs under the sign-magnitude order, FNV-1a per call),
 *       "Why it is not a defect" (bf16 gate, f32 widening inside top-k).
 *
 * Conventions for every call
 *  - All pointers are DEVICE pointers of the current CUDA device unless a
 *    parameter says otherwise.  The caller owns every buffer.
 *  - Calls are asynchronous on stream `s` (NULL = the legacy default
 *    stream) and never synchronise the host.
 *  - Arguments are validated on the host before anything is launched; an
 *    invalid call returns an error and leaves every output untouched.
 *  - A launch failure reported by the runtime returns BI_ERR_CUDA.  Faults
 *    detected on the device (a bounded wait that ran out, an expert id out
 *    of range) set a sticky device word read by bi_get_last_device_error();
 *    the first report stands until it is read.  After a wait has run out,
 *    every kernel's later waits give up at once, each block still lets its
 *    own bulk copies and tensor-core operations finish before it frees its
 *    tensor memory and exits, and the outputs of calls made before the word
 *    is read are unspecified; the context stays usable.  An id out of range
 *    affects only the slots that hold it.
 *  - There is no CPU fallback: an unsupported shape is an error.
 *  - Data-pointer alignment: 16 bytes.  Layouts are row-major.
 *  - bf16 means IEEE binary32 with the low 16 bits dropped (bfloat16).
 */
#ifndef BI_H
#define BI_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define BI_API __attribute__((visibility("default")))
#else
#define BI_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BI_OK = 0,
    BI_ERR_INVALID_ARG = 1,       /* null pointer, negative size, k >= E ... */
    BI_ERR_UNSUPPORTED_SHAPE = 2, /* a size outside the limits below */
    BI_ERR_MISALIGNED = 3,        /* a pointer or stride breaks the 16-byte rule */
    BI_ERR_CUDA = 4,              /* the CUDA runtime reported an error */
    BI_ERR_TIMEOUT = 5            /* a device-side bounded wait ran out */
} bi_status;

typedef enum { BI_F32 = 0, BI_BF16 = 1 } bi_dtype;

/* Same type as cudaStream_t. */
typedef struct CUstream_st *bi_stream;

/* Limits checked by every call. */
#define BI_MAX_E 1024          /* experts per router call */
#define BI_MAX_K 32            /* experts selected per token */
#define BI_MAX_H 32768         /* router hidden size */
#define BI_MAX_HASH_RANGES 256 /* row ranges per route-hash call */

/*
 * bi_router_topk -- MoE router for one prefill call: projection, top-k,
 * softmax over the selected, routing margin.
 *
 * Defined by [P1] "m-scan: the staircase" (logits = X . W_gate^T, then
 * top_k(8 of 256)), [P1] "16% of routing decisions" (the selected set and
 * its ranking), [P4] intro and "Why it is not a defect" (bf16-logit gate,
 * lowest-index tie-break), [P4] "Why a value tap could never have said
 * this" (margin = smallest selected minus largest rejected logit, also in
 * ULPs of the logit dtype ordered by sign and then magnitude).
 *
 *   x           [M, H]  in_dtype   token hidden states
 *   w_gate      [E, H]  in_dtype   router weight (one row per expert)
 *   in_dtype    BI_F32 or BI_BF16
 *   logit_dtype BI_F32, or BI_BF16: the f32 dot is rounded to bf16
 *               (nearest, ties to even) and selection runs on those values
 *   logits_out  [M, E]  logit_dtype  required
 *   ids_out     [M, k]  int32    required; rank order: value descending,
 *               exact ties by ascending expert index
 *   weights_out [M, k]  f32      optional (NULL): w_j = exp(l_j - l_0) /
 *               sum_{i<k} exp(l_i - l_0), summed in rank order
 *   margin_out  [M]     f32      optional: l_(k-1) - l_(k), the smallest
 *               selected minus the largest rejected logit (>= 0)
 *   margin_ulps_out [M] int32    optional: the same gap counted in ULPs of
 *               the logit dtype under the sign-magnitude order (+0 == -0),
 *               saturated at INT32_MAX; 0 means an exact tie at the boundary
 *
 * Reduction order (the invariance contract): h is cut into slabs of 128;
 * each slab into 16 blocks of 8.  Partition q (0..15) takes block q of every
 * slab and runs ONE fused multiply-add chain in f32 from +0 over the h < H
 * it owns, in increasing order.  The 16 partial sums are added by a fixed
 * pairwise tree: (0+1),(2+3),... then pairs of those, four levels.  This
 * order depends on H alone.
 *
 * Limits: 1 <= H <= BI_MAX_H, H % 8 == 0; 32 <= E <= BI_MAX_E, E % 32 == 0;
 * 1 <= k <= BI_MAX_K, k < E; M >= 0 (M == 0 returns BI_OK and does nothing).
 * Logits must be finite for the weights and margins to be meaningful (a
 * NaN ranks above every number and ties other NaNs by index).
 *
 * Work and memory.  Batches of at most 112 rows run as ONE launch: thread
 * block clusters in which each block computes the logits of a slice of the
 * experts and sends them, through distributed shared memory, to the block
 * that selects their token.  Larger batches run the projection as 32 x 64
 * tiles whose 16 partitions may be spread over several thread blocks; their
 * group sums meet in `workspace` and the selection kernel adds them.  From
 * one 64 x 64 x 8-partition item per SM on, a persistent kernel gives every
 * SM the same number of steps: where that cuts an item between two blocks,
 * the second continues the first's FMA chains from accumulators handed over
 * in `workspace` (the same operations in the same order).  The library
 * allocates nothing: the caller passes the workspace, and its contents
 * before a call do not matter (no clearing is needed, before the first call
 * or between calls: the hand-off flags carry a per-call epoch that the call
 * itself advances).
 *   workspace        device buffer, 16-byte aligned, owned by the caller; may
 *                    be NULL when workspace_bytes is 0
 *   workspace_bytes  its size; must be at least bi_router_workspace_bytes(M, E)
 *                    (0 for M <= 112 and E <= 512), else BI_ERR_INVALID_ARG
 *                    before anything is launched
 * Calls that could run at the same time on the GPU (different streams with
 * no event between them) need workspaces that do not overlap; calls queued
 * on one stream may share one.  BI_ERR_UNSUPPORTED_SHAPE is returned (before
 * any launch) only on a GPU that cannot place clusters of 8 blocks, for a
 * call of at most 112 rows given less workspace than its tiled plan needs.
 *
 * Ordering: the kernels start streaming w_gate before they wait for the
 * preceding kernel in the stream (programmatic dependent launch); x is read
 * only after that wait.  So w_gate must not be written by a kernel on `s`
 * that releases its dependents early (griddepcontrol.launch_dependents) and
 * may still be running; ordinary kernels, copies and this library's own
 * kernels are safe.
 */
BI_API bi_status bi_router_topk(const void *x, const void *w_gate, bi_dtype in_dtype,
                         bi_dtype logit_dtype, int32_t M, int32_t H, int32_t E, int32_t k,
                         void *logits_out, int32_t *ids_out, float *weights_out,
                         float *margin_out, int32_t *margin_ulps_out, void *workspace,
                         size_t workspace_bytes, bi_stream s);

/*
 * bi_router_workspace_bytes -- the workspace bi_router_topk and
 * bi_router_gate_topk need for M rows and E experts, on any GPU: 0 for
 * M <= 112 with E <= 512 (the one-launch cluster router); where some GPU may
 * take the persistent projection (at least 128 items of 64 x 64 x 8
 * partitions, 8*M*E at most 64 MiB), 16 KB + 160 * 130 KB (epoch, hand-off
 * flags and accumulators of up to 160 blocks) + 8*M*E + 8*M (the two halves'
 * group sums of the logits and of the gate); otherwise the largest
 * group-sum area any of the tiled plans may use, 8*M*E bytes while that is
 * at most 64 MiB, never less than min(64*M*E, 16 MiB) and never more than
 * 64 MiB.  Host-only: touches no GPU.  Returns 0 for M <= 0.
 */
BI_API size_t bi_router_workspace_bytes(int32_t M, int32_t E);

/*
 * bi_router_plan -- how bi_router_topk (and bi_router_gate_topk) would cut
 * the work for M rows and E experts on the current device.  For the
 * one-launch cluster router (M <= 112): *m_split = M, *C = minus the number
 * of blocks per cluster, *launches = 1.  For the persistent projection
 * (large batches, one CTA per SM, each with the same number of steps):
 * *m_split = minus the number of CTAs, *C = 2 (each tile's partitions as two
 * halves), *launches = 2.  Otherwise the rows below *m_split run as whole
 * tiles and the rest with each tile's partitions split over *C blocks, and
 * *launches counts the projection launches plus the selection.
 * Introspection only (any plan gives the same bits); it launches nothing.
 * Returns BI_ERR_INVALID_ARG for NULL outputs or bad sizes, BI_ERR_CUDA when
 * no device is current.
 */
BI_API bi_status bi_router_plan(int32_t M, int32_t E, int32_t *m_split, int32_t *C, int32_t *launches);

/*
 * bi_router_gate_topk -- bi_router_topk and bi_shared_gate in one call: the
 * same router outputs, plus the shared-expert gate of every row computed in
 * the selection kernel from the rows of X the projection just read (one
 * launch and one pass over X from device memory fewer than the two calls).
 * The gate follows the router's reduction contract (above) with w_sg as one
 * more gate row that never enters the top-k; its dot and sigmoid are
 * byte-identical to bi_shared_gate's for f32 inputs, and for bf16 inputs it
 * is the same contract on the widened values (exact products, one rounding
 * per step).
 *
 *   x, w_gate, ...   as bi_router_topk
 *   w_sg             [H] in in_dtype, 16-byte aligned
 *   gate_dot_out     [M] f32: the dot of each row with w_sg
 *   gate_sigmoid_out [M] f32, optional (NULL): 1 / (1 + exp(-dot))
 *   workspace, workspace_bytes  as bi_router_topk
 * Errors: as bi_router_topk; BI_ERR_INVALID_ARG for a NULL w_sg or
 * gate_dot_out when M > 0.
 */
BI_API bi_status bi_router_gate_topk(const void *x, const void *w_gate, const void *w_sg, bi_dtype in_dtype,
                              bi_dtype logit_dtype, int32_t M, int32_t H, int32_t E, int32_t k,
                              void *logits_out, int32_t *ids_out, float *weights_out,
                              float *margin_out, int32_t *margin_ulps_out, float *gate_dot_out,
                              float *gate_sigmoid_out, void *workspace, size_t workspace_bytes,
                              bi_stream s);

/*
 * bi_shared_gate -- the one-output shared-expert gate: dot = X[m,:] . w_sg,
 * gate = 1 / (1 + exp(-dot)).
 *
 * Defined by [P1] "m-scan: the staircase" (a single-output dot product per
 * token that gates the shared expert) and [P1] "The fix: m-invariant twins"
 * (sigmoid_dot_rows, reducing each row in one fixed order).  Same reduction order as bi_router_topk.
 *
 *   x            [M, H] f32;  w_sg [H] f32
 *   dot_out      [M] f32 required;  sigmoid_out [M] f32 optional (NULL)
 * Limits: 1 <= H <= BI_MAX_H, H % 8 == 0; M >= 0.
 */
BI_API bi_status bi_shared_gate(const float *x, const float *w_sg, int32_t M, int32_t H,
                         float *dot_out, float *sigmoid_out, bi_stream s);

/*
 * bi_gemm_bf16 -- M-invariant projection C = A . B^T on the tensor cores.
 *
 * Defined by [P3] "The low-level math of tile shapes" (bf16 GEMM with FP32
 * accumulation stored as BF16; a K-reduction tree chosen by M is what makes
 * rows differ) and [P3] "The arithmetic cost of batch-invariant kernels"
 * (one static reduction tree for every M, small batches padded to the fixed
 * tile, no shape heuristics, no split-K).
 *
 *   A [M, K] bf16, row stride lda (elements)
 *   B [N, K] bf16, row stride ldb: the [out, in] weight of a linear layer
 *   C [M, N] bf16, row stride ldc; C = round_bf16(sum_k A[m,k] B[n,k]),
 *     f32 accumulation in a fixed K order (blocks of 64 in order, 16 per
 *     tensor-core step), one tile shape (128 x 256) for every M.
 * Limits: M >= 0 (0 is a no-op), 1 <= N, N % 16 == 0, 64 <= K, K % 64 == 0,
 * lda >= K, ldb >= K, ldc >= N, each a multiple of 8; M, N <= 2^31 - 1.
 */
BI_API bi_status bi_gemm_bf16(const void *A, const void *B, void *C, int32_t M, int32_t N, int32_t K,
                       int64_t lda, int64_t ldb, int64_t ldc, bi_stream s);

/*
 * bi_route_trace_hash -- per-request route hash: 64-bit FNV-1a over the
 * selected expert SETS of a range of token rows.
 *
 * Defined by [P4] "Why a value tap could never have said this": one FNV-1a
 * value per call over the tokens' sorted id lists, so that two runs compare
 * with a single equality test (the combine over the k slots ignores their
 * order, so the set, not the ranking, is what is compared).
 *
 *   ids          [M, k] int32 (device), as written by bi_router_topk
 *   row_offsets  HOST array [n_ranges + 1], non-decreasing, 0 <= . <= M:
 *                range r covers rows [row_offsets[r], row_offsets[r+1])
 *   basis        device [n_ranges] start values, or NULL for the FNV-1a
 *                64 offset basis 0xcbf29ce484222325 (pass the previous
 *                layer's hashes to chain layers; may alias hash_out)
 *   hash_out     device [n_ranges]
 * For each row of a range: its k ids sorted ascending, serialised as
 * little-endian int32 bytes, rows in order, no separator; each byte is
 * xor-ed into the hash, which is then multiplied by 0x100000001b3 mod 2^64.
 * Ranges are hashed in parallel; an empty range returns its basis.
 * Limits: 1 <= k <= BI_MAX_K; 1 <= n_ranges <= BI_MAX_HASH_RANGES.
 */
BI_API bi_status bi_route_trace_hash(const int32_t *ids, int32_t M, int32_t k,
                              const int32_t *row_offsets, int32_t n_ranges,
                              const uint64_t *basis, uint64_t *hash_out, bi_stream s);

/*
 * bi_router_topk_noalloc -- bi_router_topk for callers that must not
 * allocate device memory, with the same arguments and bit-identical results.
 *
 * No counterpart on the source pages: it exists for the caller, not for the
 * method.  bi_router_topk needs a device workspace from its caller for
 * batches of more than 112 rows or with E = 1024.  Some callers cannot
 * provide one: a plugin or an embedded runtime that is handed device pointers for its inputs and
 * outputs but owns no device memory and has no allocator to call, or code
 * that must not let device memory be reserved on its behalf at all.  This
 * entry point instead uses a fixed device array of BI_NOALLOC_SCRATCH_BYTES
 * compiled into the library (held by every GPU that loads the library until
 * the process exits) and never calls cudaMalloc, cudaFree or any allocating
 * routine.
 *
 * It always spreads each 32x64 tile's 16 partitions over 16 thread blocks,
 * needing 16*M*E*4 bytes of the array, so it serves M*E <=
 * BI_NOALLOC_SCRATCH_BYTES / 64 (M <= 64 at E = 256, M <= 32 at E = 512,
 * M <= 16 at E = 1024); larger problems return BI_ERR_UNSUPPORTED_SHAPE.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current): make that first call
 * before any stream capture.  Every call shares the one array, whose
 * contents persist between calls; each call overwrites all of the scratch
 * it reads before reading it, so nothing needs clearing.  Calls that overlap
 * on the GPU (on different streams, or from different host threads) race on
 * the array and must be serialised by the caller.  The cached address is
 * only valid for the CUDA context it was looked up in: do not use the
 * library across a cudaDeviceReset.
 */
#define BI_NOALLOC_SCRATCH_BYTES (1u << 20)
BI_API bi_status bi_router_topk_noalloc(const void *x, const void *w_gate, bi_dtype in_dtype,
                                        bi_dtype logit_dtype, int32_t M, int32_t H, int32_t E,
                                        int32_t k, void *logits_out, int32_t *ids_out,
                                        float *weights_out, float *margin_out,
                                        int32_t *margin_ulps_out, bi_stream s);

/* Human-readable name of a status code (static string). */
BI_API const char *bi_status_string(bi_status st);

/*
 * Reads and clears the sticky device-side error word of the current device
 * (BI_OK if no kernel reported a fault).  Synchronises the device.
 */
BI_API bi_status bi_get_last_device_error(void);

/*
 * Self-test of the device-side failure path (no counterpart on the source
 * pages): launches one thread that waits on a barrier nothing ever completes,
 * with a wait bound of limit_us microseconds (1 .. 2,000,000).  The wait gives
 * up, records BI_ERR_TIMEOUT in the sticky device error word and the kernel
 * returns normally: bi_get_last_device_error() then reports BI_ERR_TIMEOUT and
 * the context stays usable.  No kernel of this library traps or spins
 * without a bound; this is how that property is checked on a GPU.
 */
BI_API bi_status bi_selftest_wait_timeout(uint32_t limit_us, bi_stream s);

/*
 * bi_rmsnorm -- batch-invariant RMSNorm of every row:
 *
 *   r[m]    = 1 / sqrt( (sum_h x[m,h]^2) / H + eps )
 *   y[m, h] = bf16_rne( (x[m, h] * r[m]) * w[h] )
 *
 * [P3] "The physics of the cascade": one root-mean-square over the whole
 * hidden state divides every element of the row, so the order of that one
 * reduction decides all of the row's outputs.  The sum of squares follows
 * the router's reduction contract (above: 16 partitions, one f32 fused
 * multiply-add chain each, pairwise tree); the division, the square root
 * and the two products are each rounded once (nearest even), in that order.
 *
 *   x        [M, H] in dtype (BI_F32 or BI_BF16), 16-byte aligned
 *   w        [H] in dtype, 16-byte aligned
 *   eps      >= 0, finite
 *   y_out    [M, H] bf16, 16-byte aligned
 *   rstd_out [M] f32: r[m], optional (NULL)
 * Limits: 1 <= H <= BI_MAX_H, H % 8 == 0.  M == 0 returns BI_OK.
 */
BI_API bi_status bi_rmsnorm(const void *x, const void *w, bi_dtype dtype, int32_t M, int32_t H, float eps,
                     void *y_out, float *rstd_out, bi_stream s);

/*
 * bi_attention_prefill -- batch-invariant causal attention for one prefill
 * call over ragged requests (bf16 in, bf16 out, f32 arithmetic):
 *
 *   request r: queries q[q_offsets[r] .. q_offsets[r+1]), keys and values
 *   k, v[kv_offsets[r] .. kv_offsets[r+1]); its q_len queries are the last
 *   q_len positions of its kv_len-token context (a cached prefix, if any,
 *   comes first), and query i (position kv_len - q_len + i) attends to keys
 *   0 .. that position of its own request:
 *
 *     o[i, h]   = sum_j softmax_j( scale * q[i, h] . k[j, h / g] ) v[j, h / g]
 *     lse[i, h] = log sum_j exp( scale * q[i, h] . k[j, h / g] )
 *
 *   with g = n_heads / n_kv_heads query heads per key/value head.
 *
 * [P3] "The physics of the cascade": the softmax's exponential stretches a
 * one-ULP difference in the scores and the product with V spreads it over
 * every feature, so attention is the next operation on the cascade path
 * that must give a row the same bits whatever the batch.
 *
 * Invariance contract: each query row walks its own context in blocks of
 * 128 keys at fixed positions (block b = keys 128b .. 128b+127), in
 * increasing order, up to the block holding its own position.  Per block:
 * the scores s_j as f32 tensor-core dot products over the 128 dimensions in
 * 16-deep steps, in increasing order (keys the row cannot see: -inf); with
 * c = scale * log2(e) rounded to f32 and t = c * max_j s_j, when t exceeds
 * the row's reference maximum m by more than 8 (always on the first block)
 * the accumulators are rescaled by a = 2^(m - t) and m = t; then
 * p_j = 2^fmaf(s_j, c, -m) (ex2.approx.ftz); l += E + D, where E and D are
 * pairwise trees over the block's 64 even- and 64 odd-position f32 p_j; and
 * O += sum_j bf16_rne(p_j) v_j as f32 tensor-core sums over the block's keys
 * in 16-deep steps, in increasing order.  Finally o = bf16_rne(O * (1/l))
 * and lse = (m + log2f(l)) * ln 2.  Keys come in chunks of 8192 (64
 * blocks) at fixed positions: a row whose position is below 8192 is exactly
 * the above; a later row's chunks c = 0 .. pos/8192 each run the above from
 * a fresh state (m = -inf, l = 0, O = 0), giving (m_c, l_c, O_c), which are
 * merged in chunk order: (M, L, N) = (m_0, l_0, O_0), then for c >= 1 with
 * M' = max(M, m_c), a = 2^(M - M') and b = 2^(m_c - M') (each exactly 1
 * where its maximum is M'), L = fmaf(L, a, l_c b), N = fmaf(N, a, O_c b),
 * M = M' (products rounded once); o = bf16_rne(N * (1/L)), lse =
 * (M + log2f(L)) * ln 2.  So a row's bits depend only on its own query, its
 * position and its request's keys and values: not on the other requests,
 * on how many of its request's queries are in the call (a cached prefix, a
 * chunked prefill), or on which query tile it falls in.
 *
 *   q           [Tq, n_heads, 128] bf16, Tq = q_offsets[n_req]
 *   k, v        [Tkv, n_kv_heads, 128] bf16, Tkv = kv_offsets[n_req]
 *   n_req       requests, >= 0
 *   q_offsets   HOST [n_req + 1] int32: 0, then running sums of q_len
 *   kv_offsets  HOST [n_req + 1] int32: 0, then running sums of kv_len;
 *               0 <= q_len <= kv_len for every request (a request with
 *               q_len == 0 is skipped)
 *   n_heads, n_kv_heads  >= 1, n_heads a multiple of n_kv_heads,
 *               n_heads <= BI_ATTN_MAX_HEADS
 *   head_dim    must be 128 (else BI_ERR_UNSUPPORTED_SHAPE)
 *   scale       finite, > 0 (usually 1 / sqrt(head_dim))
 *   o           [Tq, n_heads, 128] bf16 output
 *   lse         [Tq, n_heads] f32 natural-log sum of exponentials, or NULL
 *   workspace, workspace_bytes  caller-owned device buffer, 256-byte
 *               aligned, at least bi_attention_workspace_bytes(n_req,
 *               q_offsets, kv_offsets, n_heads) bytes: the chunks' partials of
 *               the query tiles whose context runs past 8192 keys (0 bytes,
 *               and NULL allowed, when none does); its contents do not
 *               matter; nothing is allocated by the call.
 *               Two calls that could overlap on the GPU must not share it.
 * All inputs must be finite.  Key and value rows past a request's end but
 * inside the tensors are read (they belong to the next request) and get
 * weight zero.  Tq == 0 returns BI_OK.  The offsets are read before the
 * call returns.
 */
#define BI_ATTN_MAX_HEADS 256
BI_API size_t bi_attention_workspace_bytes(int32_t n_req, const int32_t *q_offsets, const int32_t *kv_offsets,
                                          int32_t n_heads);
BI_API bi_status bi_attention_prefill(const void *q, const void *k, const void *v, int32_t n_req,
                                      const int32_t *q_offsets, const int32_t *kv_offsets, int32_t n_heads,
                                      int32_t n_kv_heads, int32_t head_dim, float scale, void *o, float *lse,
                                      void *workspace, size_t workspace_bytes, bi_stream s);

/*
 * bi_moe_expert_gemm -- the grouped expert projection that consumes the
 * router's choice: every token-slot (m, j) is one row through its expert,
 *
 *   Y[m, j, n] = bf16_rne( sum_k X[m, k] * W[ids[m, j], n, k] )
 *   out[m, n]  = bf16_rne( sum_{j<k} weights[m, j] * Y[m, j, n] )
 *
 * [P4] "Why a value tap could never have said this": the assembled per-slot
 * expert outputs, and the grouped expert GEMM -- whose per-expert row counts
 * change with the batch -- as the amplifier of run-to-run differences.  The
 * pages' experts are quantised; here they are bf16.
 *
 * Invariance contract: each Y row is accumulated in f32 over K in blocks of
 * 64, in increasing order, each block as four 16-deep tensor-core steps,
 * and rounded to bf16 once -- the schedule of bi_gemm_bf16, whatever the
 * number of rows its expert receives and wherever the row lands in its
 * expert's group.  out is one f32 fused multiply-add chain over j = 0..k-1
 * (rank order, the order ids come in), rounded once.
 *
 *   X        [M, K] bf16 (16-byte aligned)
 *   ids      [M, k] int32 expert of each slot, in [0, E); an id outside
 *            that range sets BI_ERR_INVALID_ARG in the device error word and
 *            its slot's outputs are left unwritten
 *   weights  [M, k] f32, needed when out is requested, else may be NULL
 *   W        [E, N, K] bf16: expert e's [N, K] projection (16-byte aligned)
 *   Y_out    [M, k, N] bf16 per-slot outputs, or NULL (then they live in
 *            the workspace)
 *   out      [M, N] bf16 combined rows, or NULL; at least one of Y_out, out
 *   workspace, workspace_bytes  caller-owned device buffer, 256-byte
 *            aligned, at least bi_moe_workspace_bytes(M, k, E, N, K) bytes;
 *            nothing is allocated by the call.  Two calls that could overlap
 *            on the GPU must not share a workspace.
 * Limits: 1 <= k <= BI_MAX_K, 1 <= E <= BI_MAX_E, K % 64 == 0, N % 16 == 0,
 * K, N <= 65536, M * k <= 2^24.  M == 0 returns BI_OK.
 */
BI_API size_t bi_moe_workspace_bytes(int32_t M, int32_t k, int32_t E, int32_t N, int32_t K);
BI_API bi_status bi_moe_expert_gemm(const void *X, const int32_t *ids, const float *weights, const void *W,
                             int32_t M, int32_t k, int32_t E, int32_t N, int32_t K, void *Y_out,
                             void *out, void *workspace, size_t workspace_bytes, bi_stream s);

/*
 * bi_get_config -- the numeric contract as data, so that a caller (or a
 * checker comparing two deployments) can verify that two libraries reduce
 * in the same order before trusting byte equality across them.  [P3] "The
 * arithmetic cost of batch-invariant kernels" asks for exactly this: one
 * static reduction tree, fixed accumulator precision and block size, named
 * rather than chosen by a heuristic.  Host-only: touches no GPU.
 *
 *   out       host pointer to a bi_config the caller owns
 *   out_size  sizeof(bi_config) as the caller compiled it; the library fills
 *             min(out_size, its own size) bytes (fields are only appended in
 *             later versions), and struct_size reports its own size
 * Returns BI_ERR_INVALID_ARG for a NULL `out` or an out_size smaller than
 * the first two fields.
 */
typedef enum { BI_TREE_PAIRWISE = 1 } bi_tree;

typedef struct {
    int32_t struct_size;            /* sizeof(bi_config) in this library */
    int32_t abi_version;            /* BI_ABI_VERSION */
    /* router projection and shared gate (bi_router_topk, bi_shared_gate) */
    int32_t router_slab;            /* 128: h is cut into slabs of this many */
    int32_t router_block;           /* 8: each slab into blocks of this many */
    int32_t router_partitions;      /* 16: partition q owns block q of every slab */
    int32_t router_partition_order; /* 1: one fused multiply-add chain from +0, h increasing */
    int32_t router_tree;            /* BI_TREE_PAIRWISE over the 16 partials, 4 levels */
    int32_t router_accum;           /* BI_F32 */
    /* bf16 projection (bi_gemm_bf16) */
    int32_t gemm_tile_m, gemm_tile_n; /* 128 x 256 output tile (the last partial wave as 128 x 128) */
    int32_t gemm_block_k;           /* 64: K consumed in blocks of this many, increasing */
    int32_t gemm_mma_k;             /* 16: each block as four tensor-core steps of this depth */
    int32_t gemm_accum;             /* BI_F32, rounded to bf16 (nearest even) once */
    int32_t gemm_split_k;           /* 0: K is never split across thread blocks */
    /* selection */
    int32_t topk_tie_rule;          /* 1: equal values rank by ascending expert index */
    int32_t softmax_sum_order;      /* 1: denominators summed in rank order */
} bi_config;

BI_API bi_status bi_get_config(bi_config *out, size_t out_size);

/*
 * bi_prefix_split -- which rows a prefix-cache hit recomputes.  [P3] "The
 * engineering cost of determinism": a request of N tokens runs at M = N on
 * a cache miss, but on a hit the engine keeps the block-aligned prefix and
 * runs only the suffix, M = N mod block_size.  When N is a multiple of the
 * block size that suffix is empty; the plainest reading kept here is that
 * the last full block is recomputed (so every request yields rows to
 * compare), and a request shorter than one block is recomputed whole.
 * Host-only: touches no GPU.
 *
 *   lengths            host [n_requests] int32, each >= 0
 *   block              KV block size in tokens, >= 1
 *   cached_out         host [n_requests]: tokens kept from the cache (a
 *                      multiple of block); request r recomputes its rows
 *                      [cached_out[r], lengths[r])
 *   suffix_offsets_out host [n_requests + 1]: the recomputed rows packed
 *                      request after request (offset 0, then running sums),
 *                      ready to pass as row offsets to bi_route_trace_hash
 * Returns BI_ERR_INVALID_ARG for NULL pointers, n_requests < 0, block < 1,
 * a negative length, or a total above INT32_MAX (outputs untouched).
 */
BI_API bi_status bi_prefix_split(const int32_t *lengths, int32_t n_requests, int32_t block,
                                 int32_t *cached_out, int32_t *suffix_offsets_out);

/*
 * bi_selftest_fma_rate -- measurement aid: launches a kernel of 8 blocks of
 * 256 threads per SM, each thread running 8 independent f32 fused
 * multiply-add chains for iters x 16 steps, and reports the floating-point
 * operations it performs in *flops_launched (2 per FMA).  Timing it with
 * events on `s` gives the FP32 FMA rate this GPU sustains, the ceiling the
 * router projection (pure FMA chains) is measured against.
 *   iters   1 .. 2^20
 *   packed  0: scalar f32 FMAs; 1: each chain a pair of lanes of the two-wide
 *           f32 FMA instruction (two independent FMAs, each rounded once)
 *   sink    device memory for at least 8 * SMs floats (written only in a
 *           case that does not occur, to keep the work live)
 */
BI_API bi_status bi_selftest_fma_rate(int32_t iters, int32_t packed, float *sink, bi_stream s,
                                      double *flops_launched);

/* ABI version of this header: bumps on any incompatible change (2: the
 * router calls take a caller-owned workspace). */
/*
 * bi_selftest_dependent_floor -- measurement aid (no counterpart on the
 * source pages): launches one thread-block cluster shaped like the
 * one-launch router's at a single token (16 blocks, or 8 where 16 cannot be
 * placed) whose blocks wait for the preceding kernel in the stream (the same
 * programmatic dependent launch as the router), read in[block], pass two
 * cluster barriers and write out[block] = in[block] + 1.  Timing a chain of
 * these calls (each reading the previous call's out) gives the fixed cost of
 * a dependent one-launch call with no arithmetic: the floor under the
 * router's time at small M.
 *   in, out  device arrays of at least 16 floats
 * Returns BI_ERR_INVALID_ARG for NULL pointers, BI_ERR_UNSUPPORTED_SHAPE on
 * a GPU that cannot place the cluster.
 */
BI_API bi_status bi_selftest_dependent_floor(const float *in, float *out, bi_stream s);

#define BI_ABI_VERSION 2
BI_API int32_t bi_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* BI_H */
