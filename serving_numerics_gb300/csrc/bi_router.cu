// bi_router.cu -- bi_router_topk: M-invariant MoE router projection on CUDA
// cores (f32 FMA, never TF32), then top-k with the lowest-index tie-break,
// softmax over the selected and the routing margin.
//
// Source pages: "batch changed the model's mind" ("m-scan: the staircase",
// "The fix: m-invariant twins"); "diag(MODEL-MM-QWEN4-EXP): the MoE expert
// selections DIFFER ..." (intro, "Why a value tap could never have said
// this", "Why it is not a defect").
//
// Reduction contract (depends on H only).  h is cut into slabs of 128 and
// each slab into 16 blocks of 8.  Partition q in 0..15 owns block q of every
// slab; its partial sum is ONE f32 fused multiply-add chain from +0 over the
// h < H it owns, in increasing h.  The 16 partials are added by the pairwise
// tree (0+1),(2+3),...,(14+15), then (01+23),..., four levels.
//
// Work decomposition (free to depend on M, since it never changes the
// order): one tile shape for every M, 32 tokens x 64 experts.  A tile's 16
// partitions are split over C thread blocks (C = 1, 2, 4, 8 or 16; 16/C
// warps each, one warp per partition).  A block adds its partitions with the
// lower levels of the tree; with C > 1 the C group sums meet in library
// scratch and the selection kernel adds them with the remaining upper
// levels.  The plan (plan_split below) picks C from M; batches of at most 64
// rows take the matrix-vector twin instead.
//
// Data path: the X and W_gate blocks of a slab are staged by TMA into
// shared memory in boxes of 4 (f32) or 8 (bf16) partition blocks, 128-byte
// rows with the 128-byte swizzle, a ring of stages deep.  Lane (tg, eg) of a warp owns tokens
// tg + 4j and experts eg + 8i (j, i < 8): 64 accumulators.  A 128-bit
// shared load moves 512 bytes whatever the lanes share, so the shared-memory
// path delivers 32 lane-floats per clock against 128 FMAs per clock; an
// 8 x 8 thread tile (64 FMAs per 16 floats loaded) is the smallest that
// keeps the FMA pipe, not the shared-memory pipe, the limit.
#include <cuda_bf16.h>
#include <limits.h>

#include <algorithm>

#include "bi_device.cuh"
#include "bi_internal.h"
#include "bi_select.cuh"

namespace bi {
namespace {

constexpr int kTileM = 32, kTileE = 64, kSlab = kRouterSlab, kBlk = kRouterBlock, kParts = kRouterParts;

// SHALLOW: a 96 KB ring instead of 192 KB, so that two blocks share an SM
// (used with C = 2 when the tiles fill the SMs: one block computes while the
// other starts up or adds its partition tree).
template <typename InT, int C, bool SHALLOW = false>
struct ProjCfg {
    static constexpr int ES = (int)sizeof(InT);
    static constexpr int NPL = kParts / C;                       // partitions (= warps) per block
    static constexpr int THREADS = 32 * NPL;
    // one TMA box covers PB adjacent partition blocks of a slab: rows of
    // P = PB * 8 * ES bytes (at most 128), swizzled over their whole width
    static constexpr int PB0 = 128 / (kBlk * ES);
    static constexpr int PB = NPL < PB0 ? NPL : PB0;
    static constexpr int P = PB * kBlk * ES;
    static constexpr int NB = NPL / PB;                          // boxes per operand per stage
    static constexpr int XBOX = kTileM * P, WBOX = kTileE * P;
    static constexpr int XOP = XBOX * NB, WOP = WBOX * NB;       // per stage
    static constexpr int STAGE_BYTES = XOP + WOP;
    static constexpr int NST_RAW = ((SHALLOW ? 96 : 192) * 1024) / STAGE_BYTES;
    static constexpr int NST = NST_RAW > 16 ? 16 : (NST_RAW < 2 ? 2 : NST_RAW);
    static constexpr int TREE_BYTES = NPL * 64 * 33 * 4;           // every warp's 64 partials
    static constexpr int BODY0 = NST * STAGE_BYTES;
    static constexpr int BODY = BODY0 > TREE_BYTES ? BODY0 : TREE_BYTES;
    static constexpr int SMEM = BODY + 1024;                      // + alignment slack
    static_assert(P == 16 || P == 32 || P == 64 || P == 128, "TMA swizzle span");
};

// Layout of a staged box: P-byte rows with the P-byte TMA swizzle, so
// 16-byte chunk `ch` of row r sits at r * P + 16 * (ch ^ sx(r)), where
// sx(r) is bits [7, 7+log2(P/16)) of r * P (every box starts 1024-byte
// aligned; P = 16 is unswizzled).  For the rows a thread reads it depends on
// little: x rows tg + 4j (tg < 4)
// give sx(tg + 4 (j & 1)), and gate rows eg + 8i (eg < 8) give sx(eg) for
// every i.  So each half-block needs three base addresses, and the row
// steps 4P (x) and 8P (w) become immediate offsets of the loads.
template <int P>
__device__ __forceinline__ int sx(int r)
{
    return P == 16 ? 0 : ((r * P) >> 7) & (P / 16 - 1);
}

// One 8-wide block of the chain for the 8x8 thread tile, f32 inputs.  The
// block is chunks 2*pc and 2*pc+1 of each row of its box.
template <int P>
__device__ __forceinline__ void block_f32(float (&acc)[8][8], const uint8_t *xs, const uint8_t *ws,
                                          int pc, int tg, int eg)
{
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
        const int ch = 2 * pc + c;
        const uint8_t *xe = xs + tg * P + 16 * (ch ^ sx<P>(tg));       // rows tg + 4j, j even
        const uint8_t *xo = xs + tg * P + 16 * (ch ^ sx<P>(tg + 4));   // j odd
        const uint8_t *wb = ws + eg * P + 16 * (ch ^ sx<P>(eg));        // rows eg + 8i
        float4 xv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            xv[j] = *reinterpret_cast<const float4 *>((j & 1 ? xo : xe) + 4 * j * P);
        float4 wn = *reinterpret_cast<const float4 *>(wb);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 wv = wn;       // this expert's four values; the next one loads meanwhile
            if (i + 1 < 8) wn = *reinterpret_cast<const float4 *>(wb + 8 * (i + 1) * P);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float a = acc[j][i];
                a = __fmaf_rn(xv[j].x, wv.x, a);
                a = __fmaf_rn(xv[j].y, wv.y, a);
                a = __fmaf_rn(xv[j].z, wv.z, a);
                a = __fmaf_rn(xv[j].w, wv.w, a);
                acc[j][i] = a;
            }
        }
    }
}

// The same for bf16 inputs: the block is chunk pc of each row; it is used
// in two halves of four values (8-byte loads).  Products of two bf16 values
// are exact in f32, so each step rounds once, as in f32.
template <int P>
__device__ __forceinline__ void block_bf16(float (&acc)[8][8], const uint8_t *xs, const uint8_t *ws,
                                           int pc, int tg, int eg)
{
    const uint8_t *xe = xs + tg * P + 16 * (pc ^ sx<P>(tg));
    const uint8_t *xo = xs + tg * P + 16 * (pc ^ sx<P>(tg + 4));
    const uint8_t *wb = ws + eg * P + 16 * (pc ^ sx<P>(eg));
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
        uint2 xr[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            xr[j] = *reinterpret_cast<const uint2 *>((j & 1 ? xo : xe) + 4 * j * P + 8 * c);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint2 wr = *reinterpret_cast<const uint2 *>(wb + 8 * i * P + 8 * c);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float a = acc[j][i];
                a = __fmaf_rn(bf16lo(xr[j].x), bf16lo(wr.x), a);
                a = __fmaf_rn(bf16hi(xr[j].x), bf16hi(wr.x), a);
                a = __fmaf_rn(bf16lo(xr[j].y), bf16lo(wr.y), a);
                a = __fmaf_rn(bf16hi(xr[j].y), bf16hi(wr.y), a);
                acc[j][i] = a;
            }
        }
    }
}

enum OutMode : int { OUT_F32 = 0, OUT_BF16 = 1, OUT_PARTIAL = 2 };

template <typename InT, int C, bool SHALLOW>
__global__ void __launch_bounds__(ProjCfg<InT, C, SHALLOW>::THREADS, C)     // 16 warps per SM in every split
router_proj_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                   int M, int m_base, int E, int H, int out_mode, void *__restrict__ out,
                   unsigned int *err)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    using Cfg = ProjCfg<InT, C, SHALLOW>;
    constexpr int NPL = Cfg::NPL, NST = Cfg::NST;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[NST];
    __shared__ int released[NST];          // warps done with the slot's current slab
    __shared__ int last_step[NST];         // the last slab issued into each slot
    __shared__ int ring_stop;              // set once a refill was skipped: nothing more is issued
    uint8_t *smem = smem_align1024(smem_raw);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int e_tile = blockIdx.x / C, g = blockIdx.x % C;
    const int m0 = m_base + blockIdx.y * kTileM, e0 = e_tile * kTileE, q0 = g * NPL;
    const int ns = (H + kSlab - 1) / kSlab;
    const int tg = lane & 3, eg = lane >> 2;

    if (tid == 0) {
        prefetch_tmap(&tmx);
        prefetch_tmap(&tmw);
#pragma unroll
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full_bar[s], 1);
            released[s] = 0;
            last_step[s] = s < ns ? s : -1;
        }
        ring_stop = 0;
        mbar_init_fence();
    }
    __syncthreads();

    // producer step: stage slab s into ring slot `slot` (valid blocks only);
    // after the prologue, whichever warp releases a slot last refills it
    auto issue = [&](int s, int slot) {
        uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
        int nvalid = 0;        // boxes starting before H (a box may run past H: TMA fills zeros)
#pragma unroll
        for (int bx = 0; bx < Cfg::NB; ++bx) nvalid += (kSlab * s + kBlk * (q0 + bx * Cfg::PB) < H) ? 1 : 0;
        mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)(nvalid * (Cfg::XBOX + Cfg::WBOX)));
#pragma unroll
        for (int bx = 0; bx < Cfg::NB; ++bx) {
            const int h0 = kSlab * s + kBlk * (q0 + bx * Cfg::PB);
            if (h0 < H) {
                tma_load_2d(st + bx * Cfg::XBOX, &tmx, &full_bar[slot], h0, m0);
                tma_load_2d(st + Cfg::XOP + bx * Cfg::WBOX, &tmw, &full_bar[slot], h0, e0);
            }
        }
    };

    // prologue: the gate boxes of the first stages are weights, not the
    // preceding kernel's output, so they stream before the dependency wait;
    // the X boxes follow it
    const int nst = ns < NST ? ns : NST;
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            uint8_t *st = smem + s * Cfg::STAGE_BYTES;
            int nvalid = 0;
#pragma unroll
            for (int bx = 0; bx < Cfg::NB; ++bx) nvalid += (kSlab * s + kBlk * (q0 + bx * Cfg::PB) < H) ? 1 : 0;
            mbar_arrive_expect_tx(&full_bar[s], (uint32_t)(nvalid * (Cfg::XBOX + Cfg::WBOX)));
#pragma unroll
            for (int bx = 0; bx < Cfg::NB; ++bx) {
                const int h0 = kSlab * s + kBlk * (q0 + bx * Cfg::PB);
                if (h0 < H) tma_load_2d(st + Cfg::XOP + bx * Cfg::WBOX, &tmw, &full_bar[s], h0, e0);
            }
        }
    }
    pdl_wait();       // X may be the preceding kernel's output
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            uint8_t *st = smem + s * Cfg::STAGE_BYTES;
#pragma unroll
            for (int bx = 0; bx < Cfg::NB; ++bx) {
                const int h0 = kSlab * s + kBlk * (q0 + bx * Cfg::PB);
                if (h0 < H) tma_load_2d(st + bx * Cfg::XBOX, &tmx, &full_bar[s], h0, m0);
            }
        }
    }

    float acc[8][8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;

    // a warp whose four token rows are all past M has nothing to compute
    const bool live = tg < M - m0;
    bool ok = true;        // every wait of this thread completed
    int slot = 0;
    uint32_t phase = 0;
    for (int s = 0; s < ns; ++s) {
        ok &= mbar_wait(&full_bar[slot], phase, err, 0x11);
        if (live && kSlab * s + kBlk * (q0 + warp) < H) {
            const uint8_t *st = smem + slot * Cfg::STAGE_BYTES;
            const int bx = warp / Cfg::PB, pc = warp % Cfg::PB;
            const uint8_t *xs = st + bx * Cfg::XBOX, *ws = st + Cfg::XOP + bx * Cfg::WBOX;
            if constexpr (sizeof(InT) == 4)
                block_f32<Cfg::P>(acc, xs, ws, pc, tg, eg);
            else
                block_bf16<Cfg::P>(acc, xs, ws, pc, tg, eg);
        }
        // release the slot without a block-wide barrier: the last warp to
        // finish with it stages slab s + NST into it
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&released[slot], 1) == NPL - 1) {
                released[slot] = 0;
                if (s + NST < ns) {
                    // slab s must have landed (always so unless a wait gave
                    // up; then this and every later refill is skipped)
                    volatile int *stop = &ring_stop;
                    if (*stop == 0 && ring_slot_free(full_bar, NST, s + NST)) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue(s + NST, slot);
                        last_step[slot] = s + NST;
                    } else {
                        *stop = 1;
                    }
                }
            }
        }
        if (++slot == NST) {
            slot = 0;
            phase ^= 1u;
        }
    }
    if (__syncthreads_or(!ok)) {                           // every warp is done with the ring
        // a wait gave up: the slabs still landing finish before the ring's
        // memory is reused
        if (tid == 0)
            for (int sl = 0; sl < NST; ++sl)
                if (last_step[sl] >= 0) mbar_drain(&full_bar[sl], (uint32_t)(last_step[sl] / NST) & 1u);
        __syncthreads();
    }

    // partition tree: every warp parks its 64 partial sums (value v of lane L
    // at part[(warp * 64 + v) * 33 + L], padded rows); after one barrier each
    // thread adds the NPL partials of its outputs with the lower levels of the
    // pairwise tree, in registers, and stores them row-coalesced
    float *part = reinterpret_cast<float *>(smem);
#pragma unroll
    for (int v = 0; v < 64; ++v) part[(warp * 64 + v) * 33 + lane] = acc[v >> 3][v & 7];
    __syncthreads();
    for (int idx = tid; idx < kTileM * kTileE; idx += Cfg::THREADS) {
        const int t = idx >> 6, e = idx & 63, m = m0 + t;
        // output (t, e) is value 8*(t/4) + e/8 of lane (t%4) + 4*(e%8)
        const int v = 8 * (t >> 2) + (e >> 3), L = (t & 3) + 4 * (e & 7);
        float p[NPL];
#pragma unroll
        for (int w = 0; w < NPL; ++w) p[w] = part[(w * 64 + v) * 33 + L];
#pragma unroll
        for (int d = 1; d < NPL; d *= 2)
#pragma unroll
            for (int w = 0; w + d < NPL; w += 2 * d) p[w] = p[w] + p[w + d];
        if (m < M && e0 + e < E) {
            const size_t o = (size_t)m * E + e0 + e;
            if (out_mode == OUT_F32)
                static_cast<float *>(out)[o] = p[0];
            else if (out_mode == OUT_BF16)
                static_cast<__nv_bfloat16 *>(out)[o] = __float2bfloat16_rn(p[0]);
            else        // group sums of rows [m_base, M), group-major
                static_cast<float *>(out)[((size_t)g * (M - m_base) + (m - m_base)) * E + e0 + e] = p[0];
        }
    }
}

constexpr int kSelWarps = 8;
constexpr size_t kGateStageMax = 96 * 1024;   // shared memory for the staged gate rows (2 blocks per SM)

// The shared-expert gate fused into the selection: the optional inputs of
// bi_router_gate_topk (NULL gx = no gate).
struct GateArgs {
    const void *gx = nullptr;   // X again ([M, H], the input dtype)
    const void *gw = nullptr;   // w_sg [H]
    const float *gsum = nullptr;   // or the gate's two group sums [2][M], from the persistent projection
    int bf16 = 0;
    int staged = 0;             // the block's X rows and w_sg are copied to shared memory first
    float *dot = nullptr, *sig = nullptr;
    unsigned int *err = nullptr;   // the library's device error word (bounded wait on the copies)
};

__device__ __forceinline__ void load8(const float *p, float (&v)[8])
{
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8])
{
    const uint4 r = *reinterpret_cast<const uint4 *>(p);
    v[0] = bf16lo(r.x); v[1] = bf16hi(r.x); v[2] = bf16lo(r.y); v[3] = bf16hi(r.y);
    v[4] = bf16lo(r.z); v[5] = bf16hi(r.z); v[6] = bf16lo(r.w); v[7] = bf16hi(r.w);
}

// Partition q's chain of the gate dot for one row (the router's contract:
// block q of every slab, one FMA chain from +0, h increasing), with the
// loads of two slabs in flight at a time.
template <typename InT>
__device__ __forceinline__ float gate_partition(const InT *xr, const InT *w, int H, int q)
{
    float acc = 0.0f;
    const int ns = (H + kSlab - 1) / kSlab;
    for (int s0 = 0; s0 < ns; s0 += 2) {
        float xv[2][8], wv[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int h0 = kSlab * (s0 + u) + kBlk * q;
            if (h0 < H) {
                load8(xr + h0, xv[u]);
                load8(w + h0, wv[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int h0 = kSlab * (s0 + u) + kBlk * q;
            if (h0 < H) {
#pragma unroll
                for (int i = 0; i < 8; ++i) acc = __fmaf_rn(xv[u][i], wv[u][i], acc);
            }
        }
    }
    return acc;
}

// The top log2(CC) levels of the pairwise tree for a split row: lane's
// logits i (experts lane + 32 i) from the CC group sums (group-major planes
// gs floats apart), loaded about 32 at a time before their adds.
template <int EPLM, int CC>
__device__ __forceinline__ void group_tree(const float *__restrict__ part, size_t gs, size_t prow, int epl,
                                           float (&v)[EPLM])
{
    constexpr int IB0 = 32 / CC > 0 ? 32 / CC : 1;
    constexpr int IB = IB0 < EPLM ? IB0 : EPLM;      // logits per batch of loads
#pragma unroll
    for (int i0 = 0; i0 < EPLM; i0 += IB) {
        float p[IB][CC];
#pragma unroll
        for (int u = 0; u < IB; ++u)
#pragma unroll
            for (int q = 0; q < CC; ++q)
                p[u][q] = i0 + u < epl ? part[(size_t)q * gs + prow + 32 * (i0 + u)] : 0.0f;
#pragma unroll
        for (int u = 0; u < IB; ++u) {
#pragma unroll
            for (int d = 1; d < CC; d *= 2)
#pragma unroll
                for (int q = 0; q + d < CC; q += 2 * d) p[u][q] = p[u][q] + p[u][q + d];
            v[i0 + u] = p[u][0];
        }
    }
}

// One warp per token: finish the tree (C > 1), round to the logit dtype,
// then k+1 rounds of warp arg-max (value desc, index asc).  Round k yields
// the largest rejected logit for the margin.  Rows below m_split already
// have their logits (the projection ran whole for them); rows from m_split
// on have C group sums in `part`, laid out group-major over those rows.
// Blocks per SM the register budget is set for: E <= 256 keeps four blocks
// (three with the gate's 72 KB of staged rows each); larger E is left free.
template <int EPLM, bool GATE>
constexpr int sel_min_blocks() { return EPLM <= 8 ? (GATE ? 3 : 4) : 1; }

// TWO: the instantiation for split rows with two group sums (or none), with
// a run-time-C loop as its general case; the other instantiation adds 4, 8
// or 16 sums with trees unrolled at compile time.  (Same-box timings: the
// compile-time trees in the two-sum kernel cost it 1.5 us per call at
// M = 4096; in their own kernel they take 2 us off the calls at M = 128-256.)
template <int EPLM, bool GATE, bool TWO>
__global__ void __launch_bounds__(32 * kSelWarps, sel_min_blocks<EPLM, GATE>())
router_select_kernel(const float *__restrict__ part, int C, int m_split, void *logits, int logit_bf16,
                     int M, int E, int k, int32_t *__restrict__ ids, float *__restrict__ weights,
                     float *__restrict__ margin, int32_t *__restrict__ ulps, GateArgs gate, int H,
                     unsigned int *epoch)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    extern __shared__ __align__(16) uint8_t gate_rows[];   // staged gate: kSelWarps rows of X, then w_sg
    __shared__ __align__(8) uint64_t gate_bar;
    const bool staged = GATE && gate.staged;
    const uint32_t row_bytes = (uint32_t)H * (gate.bf16 ? 2u : 4u);
    if (staged) {
        if (threadIdx.x == 0) {
            mbar_init(&gate_bar, 1);
            mbar_init_fence();
        }
        __syncthreads();
    }
    pdl_wait();
    // the persistent projection's call epoch: advanced once that projection
    // is complete (its hand-off flags of this call then never match again)
    if (epoch && blockIdx.x == 0 && threadIdx.x == 0) atomicAdd(epoch, 1u);
    if (staged && threadIdx.x == 0) {
        // the rows land while the selection below runs
        const int m0 = blockIdx.x * kSelWarps, rows = M - m0 < kSelWarps ? M - m0 : kSelWarps;
        mbar_arrive_expect_tx(&gate_bar, (uint32_t)(rows + 1) * row_bytes);
        bulk_load(gate_rows + kSelWarps * row_bytes, gate.gw, row_bytes, &gate_bar);
        for (int r = 0; r < rows; ++r)
            bulk_load(gate_rows + r * row_bytes, static_cast<const uint8_t *>(gate.gx) + (size_t)(m0 + r) * row_bytes,
                      row_bytes, &gate_bar);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m = blockIdx.x * kSelWarps + warp;
    if (m >= M) return;     // warp 0's row always exists, so the block outlives its copies
    const int epl = E >> 5;

    // gather this lane's logits (experts lane + 32 i), all loads issued first
    float v[EPLM];
    const size_t row = (size_t)m * E + lane;
    if (m < m_split) {
        if (logit_bf16) {
            const __nv_bfloat16 *lp = static_cast<const __nv_bfloat16 *>(logits) + row;
#pragma unroll
            for (int i = 0; i < EPLM; ++i) v[i] = i < epl ? __bfloat162float(lp[32 * i]) : 0.0f;
        } else {
            const float *lp = static_cast<const float *>(logits) + row;
#pragma unroll
            for (int i = 0; i < EPLM; ++i) v[i] = i < epl ? lp[32 * i] : 0.0f;
        }
    } else {
        // finish the pairwise tree over the C group sums, then round to the
        // logit dtype and store the logits
        const size_t gs = (size_t)(M - m_split) * E;
        const size_t prow = (size_t)(m - m_split) * E + lane;
        if constexpr (TWO) {
            if (C == 2) {      // the common split (two-block tiles): the tree's top level only
                const float *p0 = part + prow, *p1 = part + gs + prow;
                float a[EPLM], b[EPLM];
#pragma unroll
                for (int i = 0; i < EPLM; ++i) {
                    a[i] = i < epl ? p0[32 * i] : 0.0f;
                    b[i] = i < epl ? p1[32 * i] : 0.0f;
                }
#pragma unroll
                for (int i = 0; i < EPLM; ++i) v[i] = a[i] + b[i];
            } else {           // any C, with C taken at run time
#pragma unroll
                for (int i = 0; i < EPLM; ++i) {
                    float p[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        p[q] = (i < epl && q < C) ? part[(size_t)q * gs + prow + 32 * i] : 0.0f;
#pragma unroll
                    for (int d = 1; d < 16; d *= 2)
                        if (d < C) {
#pragma unroll
                            for (int q = 0; q + d < 16; q += 2 * d) p[q] = p[q] + p[q + d];
                        }
                    v[i] = p[0];
                }
            }
        } else if (C == 4) {   // a split row of the general instantiation has 4, 8 or 16 group sums
            group_tree<EPLM, 4>(part, gs, prow, epl, v);
        } else if (C == 8) {
            group_tree<EPLM, 8>(part, gs, prow, epl, v);
        } else {
            group_tree<EPLM, 16>(part, gs, prow, epl, v);
        }
#pragma unroll
        for (int i = 0; i < EPLM; ++i) {
            if (i < epl) {
                if (logit_bf16) {
                    const __nv_bfloat16 b = __float2bfloat16_rn(v[i]);
                    static_cast<__nv_bfloat16 *>(logits)[row + 32 * i] = b;
                    v[i] = __bfloat162float(b);
                } else {
                    static_cast<float *>(logits)[row + 32 * i] = v[i];
                }
            }
        }
    }

    warp_select<EPLM>(v, lane, epl, k, logit_bf16, (size_t)m, ids, weights, margin, ulps);

    // the gate from the persistent projection: its top tree level
    if (gate.gsum && lane == 0) {
        const float g = gate.gsum[m] + gate.gsum[(size_t)M + m];
        gate.dot[m] = g;
        if (gate.sig) gate.sig[m] = 1.0f / (1.0f + expf(-g));
    }

    // the shared gate (bi_router_gate_topk): lanes 0..15 are the 16
    // partitions; the butterfly with offsets 1, 2, 4, 8 is the pairwise tree
    // (each pair's lanes hold the same sum: fp addition commutes), as in
    // bi_shared_gate, so the two give the same bytes
    if (GATE) {
        float g = 0.0f;
        if (staged) {
            // warp 0 outlives the copies: after a wait that gave up it
            // still lets them land
            if (!mbar_wait(&gate_bar, 0, gate.err, 0x40) && warp == 0) mbar_drain(&gate_bar, 0);
            if (lane < 16) {
                const uint8_t *xr = gate_rows + warp * row_bytes, *wr = gate_rows + kSelWarps * row_bytes;
                g = gate.bf16 ? gate_partition(reinterpret_cast<const __nv_bfloat16 *>(xr),
                                               reinterpret_cast<const __nv_bfloat16 *>(wr), H, lane)
                              : gate_partition(reinterpret_cast<const float *>(xr),
                                               reinterpret_cast<const float *>(wr), H, lane);
            }
        } else if (lane < 16) {
            g = gate.bf16 ? gate_partition(static_cast<const __nv_bfloat16 *>(gate.gx) + (size_t)m * H,
                                           static_cast<const __nv_bfloat16 *>(gate.gw), H, lane)
                          : gate_partition(static_cast<const float *>(gate.gx) + (size_t)m * H,
                                           static_cast<const float *>(gate.gw), H, lane);
        }
#pragma unroll
        for (int d = 1; d < 16; d *= 2) g = g + __shfl_xor_sync(0xFFFFFFFFu, g, d);
        if (lane == 0) {
            gate.dot[m] = g;
            if (gate.sig) gate.sig[m] = 1.0f / (1.0f + expf(-g));
        }
    }
}

template <typename InT, int C, bool SHALLOW = false>
bi_status launch_proj(Device *d, const void *x, const void *w, int M, int m_base, int m_end, int E, int H,
                      int out_mode, void *out, cudaStream_t s, int kid)
{
    using Cfg = ProjCfg<InT, C, SHALLOW>;
    auto kern = router_proj_kernel<InT, C, SHALLOW>;
    bi_status st = set_smem_once(d, kid, kern, Cfg::SMEM);
    if (st != BI_OK) return st;
    const CUtensorMapDataType dt = sizeof(InT) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle sw = Cfg::P == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : Cfg::P == 64  ? CU_TENSOR_MAP_SWIZZLE_64B
                                : Cfg::P == 32  ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_NONE;
    const uint64_t strides[1] = {(uint64_t)H * sizeof(InT)};
    alignas(64) CUtensorMap tmx, tmw;
    {
        const uint64_t dims[2] = {(uint64_t)H, (uint64_t)M};
        const uint32_t box[2] = {(uint32_t)(Cfg::PB * kBlk), (uint32_t)kTileM};
        if ((st = encode_tiled(&tmx, dt, 2, x, dims, strides, box, sw)) != BI_OK) return st;
    }
    {
        const uint64_t dims[2] = {(uint64_t)H, (uint64_t)E};
        const uint32_t box[2] = {(uint32_t)(Cfg::PB * kBlk), (uint32_t)kTileE};
        if ((st = encode_tiled(&tmw, dt, 2, w, dims, strides, box, sw)) != BI_OK) return st;
    }
    // rows [m_base, m_end); the tensor maps span all M rows, and a tile
    // never crosses m_end because m_end is M or a multiple of the tile
    dim3 grid(((E + kTileE - 1) / kTileE) * C, (m_end - m_base + kTileM - 1) / kTileM);
    return launch_pdl(kern, grid, dim3(Cfg::THREADS), (size_t)Cfg::SMEM, s, tmx, tmw, M, m_base, E, H,
                      out_mode, out, d->err);
}

template <typename InT>
bi_status launch_proj_c(Device *d, int C, const void *x, const void *w, int M, int m_base, int m_end, int E,
                        int H, int out_mode, void *out, cudaStream_t s, bool shallow = false)
{
    const int base = KID_ROUTER_PROJ + (sizeof(InT) == 4 ? 0 : 5);
    if (shallow)   // only C = 2 has the shallow ring
        return launch_proj<InT, 2, true>(d, x, w, M, m_base, m_end, E, H, out_mode, out, s,
                                         KID_ROUTER_PROJ_SHALLOW + (sizeof(InT) == 4 ? 0 : 1));
    switch (C) {
    case 1: return launch_proj<InT, 1>(d, x, w, M, m_base, m_end, E, H, out_mode, out, s, base + 0);
    case 2: return launch_proj<InT, 2>(d, x, w, M, m_base, m_end, E, H, out_mode, out, s, base + 1);
    case 4: return launch_proj<InT, 4>(d, x, w, M, m_base, m_end, E, H, out_mode, out, s, base + 2);
    case 8: return launch_proj<InT, 8>(d, x, w, M, m_base, m_end, E, H, out_mode, out, s, base + 3);
    default: return launch_proj<InT, 16>(d, x, w, M, m_base, m_end, E, H, out_mode, out, s, base + 4);
    }
}

template <int EPLM>
bi_status launch_select1(Device *d, dim3 grid, dim3 block, cudaStream_t cs, const float *pp, int C,
                         int m_split, void *logits, int lbf, int M, int E, int k, int32_t *ids, float *w, float *mg,
                         int32_t *mu, const GateArgs &gate, int H, unsigned int *epoch)
{
    const bool two = C <= 2;
    const int kid = (gate.gx ? (two ? KID_SELECT_GATE : KID_SELECT_GATE_GENERAL)
                             : (two ? KID_SELECT : KID_SELECT_GENERAL)) +
                    (EPLM == 4 ? 0 : EPLM == 8 ? 1 : EPLM == 16 ? 2 : 3);
    auto kern = gate.gx ? (two ? router_select_kernel<EPLM, true, true> : router_select_kernel<EPLM, true, false>)
                        : (two ? router_select_kernel<EPLM, false, true> : router_select_kernel<EPLM, false, false>);
    bi_status st = set_smem_once(d, kid, kern, gate.gx ? kGateStageMax : 0);
    if (st != BI_OK) return st;
    GateArgs g = gate;
    size_t smem = 0;
    if (g.gx) {
        g.err = d->err;
        smem = (size_t)(kSelWarps + 1) * H * (g.bf16 ? 2 : 4);
        g.staged = smem <= kGateStageMax ? 1 : 0;     // larger rows are read from device memory directly
        if (!g.staged) smem = 0;
    }
    return launch_pdl(kern, grid, block, smem, cs, pp, C, m_split, logits, lbf, M, E, k, ids, w, mg, mu, g, H,
                      epoch);
}

bi_status launch_select(Device *d, int epl, dim3 grid, dim3 block, cudaStream_t cs, const float *pp, int C,
                        int m_split, void *logits, int lbf, int M, int E, int k, int32_t *ids, float *w,
                        float *mg, int32_t *mu, const GateArgs &g = GateArgs(), int H = 0,
                        unsigned int *epoch = nullptr)
{
    if (epl <= 4)
        return launch_select1<4>(d, grid, block, cs, pp, C, m_split, logits, lbf, M, E, k, ids, w, mg, mu, g, H,
                                 epoch);
    if (epl <= 8)
        return launch_select1<8>(d, grid, block, cs, pp, C, m_split, logits, lbf, M, E, k, ids, w, mg, mu, g, H,
                                 epoch);
    if (epl <= 16)
        return launch_select1<16>(d, grid, block, cs, pp, C, m_split, logits, lbf, M, E, k, ids, w, mg, mu, g, H,
                                  epoch);
    return launch_select1<32>(d, grid, block, cs, pp, C, m_split, logits, lbf, M, E, k, ids, w, mg, mu, g, H,
                              epoch);
}

// How the projection's work is cut for a batch of more than kClusterMaxM rows
// (any plan gives the same bits; plans differ only in how well the work fills
// the SMs, and each rule below was the fastest measured in its range):
//  - at least one two-block tile half per SM: every tile's 16 partitions as
//    two blocks of 8 (C = 2) with the shallow 96 KB ring, up to two blocks to
//    an SM, so one block's start-up and partition tree overlap the other's
//    arithmetic; the selection adds the two group sums (2*M*E*4 bytes of
//    them).  (Same-box timings at M = 768 and 1024, where whole tiles had
//    been used: 38.4 and 42.6 us against 43.8 and 44.2.)
//  - fewer tiles than SMs: C = the largest power of two (at most 16) that
//    still gives every block an SM of its own (tiles * C <= SMs), deep rings;
//  - batches whose group sums would pass 64 MiB: rows [0, m_split) in whole
//    tiles (all 16 partitions in one block, logits written directly) for as
//    many full waves as they fill, and the tail rows split as in the
//    previous rule, within 16 MiB of group sums.
// The group sums live in the caller's workspace; router_workspace_bytes
// bounds what any of these plans needs on any GPU.
struct SplitPlan {
    int m_split, C;
    bool shallow;
};

constexpr long long kSplitAllMax = 64ll << 20, kSplitTailMax = 16ll << 20;

SplitPlan plan_split(int M, int E, int sms)
{
    const long long n_et = (E + kTileE - 1) / kTileE, tiles_m = (M + kTileM - 1) / kTileM;
    // at least a tile half per SM: every tile as two 8-partition blocks with
    // the shallow ring, up to two blocks to an SM (their start-up and tree
    // phases then overlap the other's arithmetic)
    if (tiles_m * n_et * 2 >= sms && 2ll * M * E * 4 <= kSplitAllMax) return {0, 2, true};
    const long long waves = tiles_m * n_et / sms;
    const long long head_tm = waves * sms / n_et;
    if (head_tm >= tiles_m) return {M, 1, false};
    const long long tail = (tiles_m - head_tm) * n_et, tail_rows = M - head_tm * kTileM;
    int c = 1;
    while (c < 16 && tail * 2 * c <= sms && 2ll * c * tail_rows * E * 4 <= kSplitTailMax) c *= 2;
    if (c == 1) return {M, 1, false};
    return {(int)(head_tm * kTileM), c, false};
}

// Bytes of group sums any tiled plan above may need for M rows and E experts,
// whatever the GPU's SM count: the two-block plan's 8*M*E when it is within
// its 64 MiB cap, and the tail plan's at most min(64*M*E, 16 MiB).
size_t tiled_workspace_bound(long long M, long long E)
{
    const long long two = 8 * M * E;
    const long long tail = std::min(64 * M * E, kSplitTailMax);
    return (size_t)(two <= kSplitAllMax ? std::max(two, tail) : tail);
}

// Calls of at most kClusterMaxM rows with E <= kClusterMaxE take the cluster
// router (clusters of 16 blocks, or of 8 where 16 cannot be placed: at most
// 64 experts per block either way) and need no workspace.
size_t router_workspace_bound(long long M, long long E)
{
    if (M <= 0 || (M <= kClusterMaxM && E <= kClusterMaxE)) return 0;
    size_t need = tiled_workspace_bound(M, E);
    // the persistent projection (bi_router_persist.cu) wherever some GPU may
    // choose it: enough items for its smallest grid, group sums within its cap
    const long long n_items = ((M + 63) / 64) * ((E + 63) / 64) * 2;
    if (n_items >= kPersistMinItems && 8 * M * E <= kPersistSumsMax)
        need = std::max(need, persist_workspace_bytes(M, E));
    return need;
}

}  // namespace
}  // namespace bi

using namespace bi;

namespace bi {
namespace {

// bi_router_topk and bi_router_gate_topk: validation, work plan, launches.
bi_status router_call(const void *x, const void *w_gate, bi_dtype in_dtype, bi_dtype logit_dtype, int32_t M,
                      int32_t H, int32_t E, int32_t k, void *logits_out, int32_t *ids_out, float *weights_out,
                      float *margin_out, int32_t *margin_ulps_out, const GateArgs &gate, void *workspace,
                      size_t workspace_bytes, bi_stream s)
{
    if ((in_dtype != BI_F32 && in_dtype != BI_BF16) || (logit_dtype != BI_F32 && logit_dtype != BI_BF16))
        return BI_ERR_INVALID_ARG;
    if (M < 0 || H <= 0 || E <= 0 || k <= 0 || k >= E) return BI_ERR_INVALID_ARG;
    if (H > BI_MAX_H || (H % 8) != 0 || E < 32 || E > BI_MAX_E || (E % 32) != 0 || k > BI_MAX_K)
        return BI_ERR_UNSUPPORTED_SHAPE;
    if (M > (1 << 21)) return BI_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return BI_OK;
    if (!x || !w_gate || !logits_out || !ids_out) return BI_ERR_INVALID_ARG;
    const size_t need = router_workspace_bound(M, E);
    if (workspace_bytes < need || (need > 0 && !workspace)) return BI_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_gate) || (workspace && !aligned16(workspace))) return BI_ERR_MISALIGNED;
    const uintptr_t lal = logit_dtype == BI_F32 ? 3u : 1u;
    if ((reinterpret_cast<uintptr_t>(logits_out) & lal) || (reinterpret_cast<uintptr_t>(ids_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(weights_out) & 3u) || (reinterpret_cast<uintptr_t>(margin_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(margin_ulps_out) & 3u))
        return BI_ERR_MISALIGNED;
    if (gate.gx && (!aligned16(gate.gw) || (reinterpret_cast<uintptr_t>(gate.dot) & 3u) ||
                    (reinterpret_cast<uintptr_t>(gate.sig) & 3u)))
        return BI_ERR_MISALIGNED;

    Device *d = nullptr;
    bi_status st = current_device(&d);
    if (st != BI_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);
    const bool f32in = in_dtype == BI_F32;
    const int lbf = logit_dtype == BI_BF16 ? 1 : 0;

    // small batches: projection and selection in one cluster launch
    const ClusterPlan cp = cluster_plan(d, M, E, H, f32in ? 4 : 2, gate.gx != nullptr);
    if (cp.ok)
        return router_cluster_call(d, cp, x, w_gate, f32in, lbf, M, H, E, k, logits_out, ids_out, weights_out,
                                   margin_out, margin_ulps_out, gate.gx ? gate.gw : nullptr, gate.dot, gate.sig,
                                   cs);

    const int epl = E / 32;
    dim3 grid((M + kSelWarps - 1) / kSelWarps), block(32 * kSelWarps);
    GateArgs g = gate;
    g.bf16 = f32in ? 0 : 1;

    // large batches: the persistent projection, every SM the same share of
    // the steps, then the selection adds the two halves' group sums
    const PersistPlan pp = persist_plan(d, M, E, f32in, gate.gx != nullptr);
    if (pp.ok) {
        if (!workspace || workspace_bytes < persist_workspace_bytes(M, E)) return BI_ERR_UNSUPPORTED_SHAPE;
        st = launch_persist(d, pp, f32in, x, w_gate, gate.gx ? gate.gw : nullptr, M, E, H, workspace, cs);
        if (st != BI_OK) return st;
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        const float *sums = reinterpret_cast<const float *>(ws + kPersistGroupSumsOffset);
        GateArgs pg;                         // the gate needs only its two group sums here
        if (gate.gx) {
            pg.gsum = sums + (size_t)2 * M * E;
            pg.dot = gate.dot;
            pg.sig = gate.sig;
        }
        return launch_select(d, epl, grid, block, cs, sums, 2, 0, logits_out, lbf, M, E, k, ids_out, weights_out,
                             margin_out, margin_ulps_out, pg, H, reinterpret_cast<unsigned int *>(ws));
    }

    const SplitPlan plan = plan_split(M, E, d->sm_count);
    void *part = nullptr;
    if (plan.m_split < M) {
        // a workspace within the bound always holds the plan's group sums;
        // below it only a call that expected the cluster router lands here
        if ((size_t)plan.C * (size_t)(M - plan.m_split) * (size_t)E * sizeof(float) > workspace_bytes ||
            !workspace)
            return BI_ERR_UNSUPPORTED_SHAPE;
        part = workspace;
    }
    // the tail goes first: it is the shorter launch, and the whole tiles
    // queue behind it on the SMs it leaves free
    if (plan.m_split < M) {
        st = f32in ? launch_proj_c<float>(d, plan.C, x, w_gate, M, plan.m_split, M, E, H, OUT_PARTIAL, part, cs,
                                          plan.shallow)
                   : launch_proj_c<__nv_bfloat16>(d, plan.C, x, w_gate, M, plan.m_split, M, E, H, OUT_PARTIAL,
                                                  part, cs, plan.shallow);
        if (st != BI_OK) return st;
    }
    if (plan.m_split > 0) {
        const int om = lbf ? OUT_BF16 : OUT_F32;
        st = f32in ? launch_proj_c<float>(d, 1, x, w_gate, M, 0, plan.m_split, E, H, om, logits_out, cs)
                   : launch_proj_c<__nv_bfloat16>(d, 1, x, w_gate, M, 0, plan.m_split, E, H, om, logits_out, cs);
        if (st != BI_OK) return st;
    }

    return launch_select(d, epl, grid, block, cs, static_cast<const float *>(part), plan.C, plan.m_split,
                         logits_out, lbf, M, E, k, ids_out, weights_out, margin_out, margin_ulps_out, g, H);
}

}  // namespace
}  // namespace bi

extern "C" size_t bi_router_workspace_bytes(int32_t M, int32_t E)
{
    return router_workspace_bound(M, E);
}

extern "C" bi_status bi_router_plan(int32_t M, int32_t E, int32_t *m_split, int32_t *C, int32_t *launches)
{
    if (M < 0 || E <= 0 || !m_split || !C || !launches) return BI_ERR_INVALID_ARG;
    Device *d = nullptr;
    if (current_device(&d) != BI_OK) return BI_ERR_CUDA;
    if (M == 0) {
        *m_split = 0;
        *C = 1;
        *launches = 0;
        return BI_OK;
    }
    // the f32 shape of the call decides; the bf16 one gives the same cut
    const ClusterPlan cp = cluster_plan(d, M, E, kRouterSlab, 4, false);
    if (cp.ok) {
        *m_split = M;
        *C = -cp.CS;          // negative: a cluster of this many blocks, one launch
        *launches = 1;
        return BI_OK;
    }
    const PersistPlan pp = persist_plan(d, M, E, true, false);
    if (pp.ok) {      // the persistent projection: minus its CTA count, two halves per tile
        *m_split = -pp.G;
        *C = 2;
        *launches = 2;
        return BI_OK;
    }
    const SplitPlan p = plan_split(M, E, d->sm_count);
    *m_split = p.m_split;
    *C = p.C;
    // projection launches (a split part and/or a whole-tile part) plus the selection
    *launches = (p.m_split < M ? 1 : 0) + (p.m_split > 0 ? 1 : 0) + 1;
    return BI_OK;
}

extern "C" bi_status bi_router_topk(const void *x, const void *w_gate, bi_dtype in_dtype,
                                    bi_dtype logit_dtype, int32_t M, int32_t H, int32_t E, int32_t k,
                                    void *logits_out, int32_t *ids_out, float *weights_out,
                                    float *margin_out, int32_t *margin_ulps_out, void *workspace,
                                    size_t workspace_bytes, bi_stream s)
{
    return router_call(x, w_gate, in_dtype, logit_dtype, M, H, E, k, logits_out, ids_out, weights_out, margin_out,
                       margin_ulps_out, GateArgs(), workspace, workspace_bytes, s);
}

extern "C" bi_status bi_router_gate_topk(const void *x, const void *w_gate, const void *w_sg, bi_dtype in_dtype,
                                         bi_dtype logit_dtype, int32_t M, int32_t H, int32_t E, int32_t k,
                                         void *logits_out, int32_t *ids_out, float *weights_out,
                                         float *margin_out, int32_t *margin_ulps_out, float *gate_dot_out,
                                         float *gate_sigmoid_out, void *workspace, size_t workspace_bytes,
                                         bi_stream s)
{
    if (M > 0 && (!w_sg || !gate_dot_out)) return BI_ERR_INVALID_ARG;
    GateArgs g;
    g.gx = M > 0 ? x : nullptr;
    g.gw = w_sg;
    g.dot = gate_dot_out;
    g.sig = gate_sigmoid_out;
    return router_call(x, w_gate, in_dtype, logit_dtype, M, H, E, k, logits_out, ids_out, weights_out, margin_out,
                       margin_ulps_out, g, workspace, workspace_bytes, s);
}

// ---------------------------------------------------------------------------
// bi_router_topk_noalloc: the same router for callers that cannot provide
// any device memory beyond their inputs and outputs.  The partial sums of the
// 16 partition groups live in a fixed array compiled into the library
// instead of the caller's workspace of bi_router_topk.  Host code must not
// pass the array's name to a kernel (that is a host-side stand-in); its
// device address is looked up once per device with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------
#include <mutex>

static __device__ __align__(256) float g_noalloc_partials[BI_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace bi {
namespace {
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64];

// Device address of g_noalloc_partials on the current device (looked up on
// the first call per device).
bi_status noalloc_scratch(const Device *d, void **out)
{
    if (d->ordinal < 0 || d->ordinal >= 64) return BI_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[d->ordinal]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || !p) return BI_ERR_CUDA;
        g_noalloc_ptr[d->ordinal] = p;
    }
    *out = g_noalloc_ptr[d->ordinal];
    return BI_OK;
}
}  // namespace
}  // namespace bi

extern "C" bi_status bi_router_topk_noalloc(const void *x, const void *w_gate, bi_dtype in_dtype,
                                            bi_dtype logit_dtype, int32_t M, int32_t H, int32_t E,
                                            int32_t k, void *logits_out, int32_t *ids_out,
                                            float *weights_out, float *margin_out,
                                            int32_t *margin_ulps_out, bi_stream s)
{
    if ((in_dtype != BI_F32 && in_dtype != BI_BF16) || (logit_dtype != BI_F32 && logit_dtype != BI_BF16))
        return BI_ERR_INVALID_ARG;
    if (M < 0 || H <= 0 || E <= 0 || k <= 0 || k >= E) return BI_ERR_INVALID_ARG;
    if (H > BI_MAX_H || (H % 8) != 0 || E < 32 || E > BI_MAX_E || (E % 32) != 0 || k > BI_MAX_K)
        return BI_ERR_UNSUPPORTED_SHAPE;
    constexpr int C = 16;                                   // always the 16-way split
    if ((size_t)C * (size_t)M * (size_t)E * sizeof(float) > (size_t)BI_NOALLOC_SCRATCH_BYTES)
        return BI_ERR_UNSUPPORTED_SHAPE;                    // beyond the fixed array
    if (M == 0) return BI_OK;
    if (!x || !w_gate || !logits_out || !ids_out) return BI_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_gate)) return BI_ERR_MISALIGNED;
    const uintptr_t lal = logit_dtype == BI_F32 ? 3u : 1u;
    if ((reinterpret_cast<uintptr_t>(logits_out) & lal) || (reinterpret_cast<uintptr_t>(ids_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(weights_out) & 3u) || (reinterpret_cast<uintptr_t>(margin_out) & 3u) ||
        (reinterpret_cast<uintptr_t>(margin_ulps_out) & 3u))
        return BI_ERR_MISALIGNED;

    Device *d = nullptr;
    bi_status st = current_device(&d);
    if (st != BI_OK) return st;
    void *part = nullptr;
    if ((st = noalloc_scratch(d, &part)) != BI_OK) return st;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(s);

    const bool f32in = in_dtype == BI_F32;
    const int lbf = logit_dtype == BI_BF16 ? 1 : 0;
    st = f32in ? launch_proj_c<float>(d, C, x, w_gate, M, 0, M, E, H, OUT_PARTIAL, part, cs)
               : launch_proj_c<__nv_bfloat16>(d, C, x, w_gate, M, 0, M, E, H, OUT_PARTIAL, part, cs);
    if (st != BI_OK) return st;
    const int epl = E / 32;
    dim3 grid((M + kSelWarps - 1) / kSelWarps), block(32 * kSelWarps);
    const float *pp = static_cast<const float *>(part);
    return launch_select(d, epl, grid, block, cs, pp, C, 0, logits_out, lbf, M, E, k, ids_out, weights_out,
                         margin_out, margin_ulps_out);
}
