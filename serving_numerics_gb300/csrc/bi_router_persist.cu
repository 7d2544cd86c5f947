// bi_router_persist.cu -- the router projection for large batches as a
// persistent kernel: one CTA per SM, every CTA the same number of steps.
//
// Source pages: "batch changed the model's mind" ("The fix: m-invariant
// twins": the router's batched twin keeps each output's reduction order
// fixed whatever the batch); "The Illusion of Determinism ..." ("The
// engineering cost of determinism": a fixed order costs throughput unless the
// kernel is built around it).
//
// Reduction contract (the same as every router kernel, bi_router.cu): h in
// slabs of 128 and blocks of 8; partition q owns block q of every slab; its
// partial is ONE f32 FMA chain from +0 in increasing h; the 16 partials are
// added by the pairwise tree (0+1),(2+3),..., then (01+23),..., four levels.
//
// Work.  Tiles of 64 tokens x 64 experts; the 16 partitions of a tile as two
// halves of 8, an "item" (8 warps, one partition each).  Lane (tg, eg) of a
// warp holds outputs (tokens tg + 4j, experts eg + 8i), j < 16, i < 8: 128
// accumulators, so each 16-byte shared load feeds 32 FMAs and the shared-
// memory path needs three quarters of the FMA rate, not all of it.
//
// Balance.  The items' slabs, item-major, form one sequence of
// n_items * ns steps, cut into G equal contiguous ranges (G = one CTA per
// SM).  A range starts and ends inside items, so neighbouring CTAs share an
// item: CTA b computes slabs [0, s) of its last item FIRST (its head), stores
// the raw chain accumulators and raises a flag; CTA b+1 computes the slabs
// [s, ns) of that item LAST (its continuation), its chains starting from
// those accumulators instead of +0.  A continued chain takes the same FMAs in
// the same order, so the bits do not depend on where an item was cut (nor on
// G).  Flags carry a value derived from an epoch word that the selection
// kernel of the same call advances once the projection is complete, so a
// flag from an earlier call never matches and the workspace needs no
// clearing, before the first call or between calls.
//
// Epilogue.  An item's 8 partials meet in shared memory by the lower three
// levels of the pairwise tree and are stored as that half's group sum; the
// selection kernel adds the two halves (the top level) as for every split
// plan with two group sums.
#include <cuda_bf16.h>

#include "bi_device.cuh"
#include "bi_internal.h"

namespace bi {
namespace {

constexpr int kSlab = kRouterSlab, kBlk = kRouterBlock;
constexpr int PT_M = 64, PT_E = 64;          // tile
constexpr int PT_WARPS = 8;                  // partitions per item
constexpr int PT_VALS = 128;                 // accumulators per thread (16 x 8)
constexpr int PT_SLOT = PT_VALS * 32;        // floats per warp in the tree / hand-off

template <typename InT, bool GATE>
struct PersistCfg {
    static constexpr int ES = (int)sizeof(InT);
    static constexpr int PB = 128 / (kBlk * ES);   // partition blocks per 128-byte box row: 4 (f32), 8 (bf16)
    static constexpr int P = 128;
    static constexpr int NB = PT_WARPS / PB;       // boxes per operand per stage: 2 (f32), 1 (bf16)
    static constexpr int XBOX = PT_M * P, WBOX = PT_E * P;
    static constexpr int XOP = XBOX * NB, WOP = WBOX * NB;
    static constexpr int STAGE = XOP + WOP;        // 32 KB (f32), 16 KB (bf16)
    static constexpr int NST = (160 * 1024) / STAGE;
    static constexpr int TREE = 4 * PT_SLOT * 4;   // 8 warps x 64 partials: 64 KB
    static constexpr int WSG = PT_WARPS * kBlk * ES;   // GATE: w_sg's slice of a step (the half's 8 blocks)
    static constexpr int SMEM = NST * STAGE + TREE + (GATE ? NST * WSG : 0) + 1024;
};

// 16-byte chunk `ch` of row r of a 128-byte-swizzled box sits at
// r * 128 + 16 * (ch ^ (r & 7)).  Rows tg + 4j give (tg + 4 (j & 1)) & 7
// and rows eg + 8i give eg, so three base addresses serve a lane.
__device__ __forceinline__ int sw8(int r) { return r & 7; }

// One partition block (8 h) of the chains for the 16 x 8 thread tile, f32:
// chunks 2 pc and 2 pc + 1 of each row; the chunk's 8 experts are held, the
// 16 tokens streamed.  (Loading the second chunk's experts during the first
// chunk's arithmetic measured slower.)
__device__ __forceinline__ void pblock_f32(float (&acc)[16][8], const uint8_t *xs, const uint8_t *ws, int pc,
                                           int tg, int eg)
{
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
        const int ch = 2 * pc + c;
        const uint8_t *xe = xs + tg * 128 + 16 * (ch ^ sw8(tg));
        const uint8_t *xo = xs + tg * 128 + 16 * (ch ^ sw8(tg + 4));
        const uint8_t *wb = ws + eg * 128 + 16 * (ch ^ sw8(eg));
        float4 wv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) wv[i] = *reinterpret_cast<const float4 *>(wb + 8 * i * 128);
        float4 xn = *reinterpret_cast<const float4 *>(xe);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float4 x = xn;      // token tg + 4j; the next one loads meanwhile
            if (j + 1 < 16) xn = *reinterpret_cast<const float4 *>(((j + 1) & 1 ? xo : xe) + 4 * (j + 1) * 128);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float a = acc[j][i];
                a = __fmaf_rn(x.x, wv[i].x, a);
                a = __fmaf_rn(x.y, wv[i].y, a);
                a = __fmaf_rn(x.z, wv[i].z, a);
                a = __fmaf_rn(x.w, wv[i].w, a);
                acc[j][i] = a;
            }
        }
    }
}

// The same for bf16 inputs: the block is chunk pc of each row, used in two
// halves of four values.  A product of two bf16 values is exact in f32, so
// each step rounds once, as in f32.
__device__ __forceinline__ void pblock_bf16(float (&acc)[16][8], const uint8_t *xs, const uint8_t *ws, int pc,
                                            int tg, int eg)
{
    const uint8_t *xe = xs + tg * 128 + 16 * (pc ^ sw8(tg));
    const uint8_t *xo = xs + tg * 128 + 16 * (pc ^ sw8(tg + 4));
    const uint8_t *wb = ws + eg * 128 + 16 * (pc ^ sw8(eg));
#pragma unroll 1
    for (int c = 0; c < 2; ++c) {
        uint2 wr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) wr[i] = *reinterpret_cast<const uint2 *>(wb + 8 * i * 128 + 8 * c);
        uint2 xn = *reinterpret_cast<const uint2 *>(xe + 8 * c);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const uint2 x = xn;
            if (j + 1 < 16) xn = *reinterpret_cast<const uint2 *>(((j + 1) & 1 ? xo : xe) + 4 * (j + 1) * 128 + 8 * c);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float a = acc[j][i];
                a = __fmaf_rn(bf16lo(x.x), bf16lo(wr[i].x), a);
                a = __fmaf_rn(bf16hi(x.x), bf16hi(wr[i].x), a);
                a = __fmaf_rn(bf16lo(x.y), bf16lo(wr[i].y), a);
                a = __fmaf_rn(bf16hi(x.y), bf16hi(wr[i].y), a);
                acc[j][i] = a;
            }
        }
    }
}

// The shared gate (GATE): lane L of gate warp q owns token row t = 32 q + L
// of the tile and runs w_sg's chains of the half's 8 partitions through the
// same staged rows, one FMA each in increasing h (the router's contract,
// w_sg being one more gate row); w_sg's slice of the step (wsl) is staged
// with the step.  One row a lane keeps the shared loads free
// of bank conflicts; the tree over the 8 partitions then needs no exchange.
template <typename Cfg, typename InT>
__device__ __forceinline__ void gate_rows_step(float (&gp)[8], const uint8_t *st, int t, int s, int g,
                                               const uint8_t *wsl, int H)
{
#pragma unroll
    for (int p = 0; p < PT_WARPS; ++p) {
        const int hw = kSlab * s + kBlk * (8 * g + p);
        if (hw < H) {
            const uint8_t *xs = st + (p / Cfg::PB) * Cfg::XBOX + t * 128;
            const int pc = p % Cfg::PB;
            float c = gp[p];
            if constexpr (sizeof(InT) == 4) {
                const float4 w0 = *reinterpret_cast<const float4 *>(wsl + p * 32);
                const float4 w1 = *reinterpret_cast<const float4 *>(wsl + p * 32 + 16);
                const float4 a0 = *reinterpret_cast<const float4 *>(xs + 16 * ((2 * pc) ^ sw8(t)));
                const float4 a1 = *reinterpret_cast<const float4 *>(xs + 16 * ((2 * pc + 1) ^ sw8(t)));
                c = __fmaf_rn(a0.x, w0.x, c); c = __fmaf_rn(a0.y, w0.y, c);
                c = __fmaf_rn(a0.z, w0.z, c); c = __fmaf_rn(a0.w, w0.w, c);
                c = __fmaf_rn(a1.x, w1.x, c); c = __fmaf_rn(a1.y, w1.y, c);
                c = __fmaf_rn(a1.z, w1.z, c); c = __fmaf_rn(a1.w, w1.w, c);
            } else {
                const uint4 w = *reinterpret_cast<const uint4 *>(wsl + p * 16);
                const uint4 x = *reinterpret_cast<const uint4 *>(xs + 16 * (pc ^ sw8(t)));
                c = __fmaf_rn(bf16lo(x.x), bf16lo(w.x), c); c = __fmaf_rn(bf16hi(x.x), bf16hi(w.x), c);
                c = __fmaf_rn(bf16lo(x.y), bf16lo(w.y), c); c = __fmaf_rn(bf16hi(x.y), bf16hi(w.y), c);
                c = __fmaf_rn(bf16lo(x.z), bf16lo(w.z), c); c = __fmaf_rn(bf16hi(x.z), bf16hi(w.z), c);
                c = __fmaf_rn(bf16lo(x.w), bf16lo(w.w), c); c = __fmaf_rn(bf16hi(x.w), bf16hi(w.w), c);
            }
            gp[p] = c;
        }
    }
}

// The flag value that marks a head finished in the call with this epoch: a
// bijective scramble of epoch + 1, so that neither the previous call's flags
// nor the float data another plan may have left in the workspace match it
// except by a 2^-32 chance (and a CTA scrubs such a match from its own flags
// before it starts).
__device__ __forceinline__ unsigned int head_done(unsigned int epoch)
{
    return (epoch + 1u) * 2654435761u ^ 0x5A17C0DEu;
}

// A store that L2 gives up first when it needs room: the hand-off lines are
// read once, at the end of the next CTA's range, and must not push out the
// token rows that the selection kernel's shared gate reads again next.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void st_evict_first(float *p, float v, uint64_t pol)
{
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(v), "l"(pol) : "memory");
}

__device__ __forceinline__ void named_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned int *p, unsigned int v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Rows j in [J0, J0 + NJ) of the thread tile to / from a warp's region of
// the tree (value (j, i) of lane L at [(j - J0) * 8 + i][L]): compile-time
// ranges keep the array in registers.
template <int J0, int NJ>
__device__ __forceinline__ void park(const float (&acc)[16][8], float *r, int lane)
{
#pragma unroll
    for (int j = J0; j < J0 + NJ; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) r[((j - J0) * 8 + i) * 32 + lane] = acc[j][i];
}

template <int J0, int NJ>
__device__ __forceinline__ void add_parked(float (&acc)[16][8], const float *r, int lane)
{
#pragma unroll
    for (int j = J0; j < J0 + NJ; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[j][i] = acc[j][i] + r[((j - J0) * 8 + i) * 32 + lane];
}

// Levels 1-3 of the pairwise tree over an item's 8 partitions (warp w holds
// partition w of the half) as a reduce-scatter: at each level a warp and its
// partner (w ^ 1, then w ^ 2, then w ^ 4) hold the same rows; each keeps half
// of them, takes the partner's partial for that half and adds it.  Every add
// is one node of the pairwise tree, (p0 + p1), (p01 + p23), (p0123 + p4567)
// and so on (the two operands' order does not change an f32 sum), so after
// three levels warp w holds the half's group sum for tile rows j in
// [2 w', 2 w' + 2), w' = 4 (w & 1) + 2 ((w >> 1) & 1) + (w >> 2), and stores
// them.  W is the warp index as a template argument, so every row range is
// known at compile time.  The second barrier of a level keeps the next
// write to a warp's region (the next level's, or the next item's) out of it
// while the partner may still read it: every read of region w in a tree is
// done once warp w has passed its own three levels, so no block-wide
// barrier is needed between items.
template <int W>
__device__ __forceinline__ void tree_and_store(float (&acc)[16][8], float *tree, int lane, float *__restrict__ part,
                                               int M, int E, int m0, int e0, int tg, int eg)
{
    constexpr int H1 = W & 1, Q2 = (W >> 1) & 1, Q3 = (W >> 2) & 1;
    constexpr int K1 = 8 * H1, K2 = K1 + 4 * Q2, K3 = K2 + 2 * Q3;   // first kept row per level
    float *mine = tree + W * PT_SLOT / 2;                             // 8 KB per warp
    // level 1 (w, w ^ 1): keep rows [K1, K1 + 8)
    park<8 - K1, 8>(acc, mine, lane);
    named_sync(2 + (W >> 1), 64);
    add_parked<K1, 8>(acc, tree + (W ^ 1) * PT_SLOT / 2, lane);
    named_sync(2 + (W >> 1), 64);
    // level 2 (w, w ^ 2): keep rows [K2, K2 + 4)
    park<K1 + 4 - 4 * Q2, 4>(acc, mine, lane);
    named_sync(6 + (W & 1) + 2 * (W >> 2), 64);
    add_parked<K2, 4>(acc, tree + (W ^ 2) * PT_SLOT / 2, lane);
    named_sync(6 + (W & 1) + 2 * (W >> 2), 64);
    // level 3 (w, w ^ 4): keep rows [K3, K3 + 2)
    park<K2 + 2 - 2 * Q3, 2>(acc, mine, lane);
    named_sync(10 + (W & 3), 64);
    add_parked<K3, 2>(acc, tree + (W ^ 4) * PT_SLOT / 2, lane);
    named_sync(10 + (W & 3), 64);
#pragma unroll
    for (int j = K3; j < K3 + 2; ++j) {
        const int m = m0 + tg + 4 * j;
        if (m < M) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = e0 + eg + 8 * i;
                if (e < E) part[(size_t)m * E + e] = acc[j][i];
            }
        }
    }
}

// The producer's walk over a CTA's steps in processing order: the head
// (slabs [0, h_len) of item `last`), whole items [f0, f1), then the
// continuation (slabs [sa, ns) of item `first`).
struct Cursor {
    int item, slab, s_end, piece;      // piece: 0 head, 1 whole items, 2 continuation
    __device__ void start(int h_len, int last, int f0, int f1, int first, int sa, int ns)
    {
        if (h_len > 0) {
            item = last; slab = 0; s_end = h_len; piece = 0;
        } else if (f0 < f1) {
            item = f0; slab = 0; s_end = ns; piece = 1;
        } else {
            item = first; slab = sa; s_end = ns; piece = 2;
        }
    }
    __device__ void advance(int f0, int f1, int first, int sa, int ns)
    {
        if (++slab < s_end) return;
        if (piece == 1 && item + 1 < f1) {
            ++item;
            slab = 0;
        } else if (piece == 0 && f0 < f1) {
            item = f0; slab = 0; s_end = ns; piece = 1;
        } else {
            item = first; slab = sa; s_end = ns; piece = 2;    // past the continuation: never used
        }
    }
};

// The boxes of one step (item, slab) into stage `st` (which: 1 = gate rows,
// 2 = token rows, 3 = both; expect: arm the barrier with the step's bytes).
// A box that starts past H is not loaded: its partition has no data there.
// With `wsl` (the gate's kernel, items of the first expert tile), w_sg's
// slice of the step goes there too: the half's 8 blocks, cut at H.
template <typename Cfg>
__device__ __forceinline__ void load_boxes(uint8_t *st, uint64_t *bar, const CUtensorMap *tmx, const CUtensorMap *tmw,
                                           int item, int slab, const PersistArgs &a, int which, bool expect,
                                           uint8_t *wsl = nullptr)
{
    const int g = item & 1, tile = item >> 1;
    const int m0 = (tile / a.n_et) * PT_M, e0 = (tile % a.n_et) * PT_E;
    const int hs = kSlab * slab + kBlk * 8 * g;                                // the slice's first h
    const bool gate = wsl != nullptr && tile % a.n_et == 0 && hs < a.H && (which & 1);
    const uint32_t wsg_bytes = gate ? (uint32_t)((a.H - hs < 8 * kBlk ? a.H - hs : 8 * kBlk) * Cfg::ES) : 0u;
    if (expect) {
        int nvalid = 0;
#pragma unroll
        for (int bx = 0; bx < Cfg::NB; ++bx) nvalid += (kSlab * slab + kBlk * (8 * g + bx * Cfg::PB) < a.H) ? 1 : 0;
        mbar_arrive_expect_tx(bar, (uint32_t)(nvalid * (Cfg::XBOX + Cfg::WBOX)) + wsg_bytes);
    }
    if (gate) bulk_load(wsl, static_cast<const uint8_t *>(a.w_sg) + (size_t)hs * Cfg::ES, wsg_bytes, bar);
#pragma unroll
    for (int bx = 0; bx < Cfg::NB; ++bx) {
        const int h0 = kSlab * slab + kBlk * (8 * g + bx * Cfg::PB);
        if (h0 < a.H) {
            if (which & 1) tma_load_2d(st + Cfg::XOP + bx * Cfg::WBOX, tmw, bar, h0, e0);
            if (which & 2) tma_load_2d(st + bx * Cfg::XBOX, tmx, bar, h0, m0);
        }
    }
}

// Register split: the block is launched as three warpgroups at 168
// registers a thread (12 warps x 32 x 168 = 64,512); the two compute
// warpgroups raise theirs to 224 and the producer warpgroup (the TMA
// producer and the gate warps) lowers its to 56
// (2 x 128 x 224 + 128 x 56 = 64,512: the same total, so the raise never
// waits on registers nobody releases).  Each SM sub-partition has a quarter
// of the register file, so a ninth warp at full width would not fit.
constexpr int PT_THREADS = (PT_WARPS + 4) * 32;
constexpr int PT_REGS_COMPUTE = 224, PT_REGS_PRODUCER = 56;
static_assert(2 * 128 * PT_REGS_COMPUTE + 128 * PT_REGS_PRODUCER <= PT_THREADS * 168, "register split");

// GATE: also the shared gate (bi_router_gate_topk), on two warps of the
// producer warpgroup: on every item of the first expert tile they run w_sg's
// chains for the tile's 64 token rows from the same staged stages, add each
// half's 8 partials by the lower tree levels into a.gpart[g][M], and the
// selection kernel adds the two halves.  (Run on the compute warps instead,
// the gate's few extra loads and FMAs cost those warps' main loop about 5 %.)
template <typename InT, bool GATE>
__global__ void __launch_bounds__(PT_THREADS, 1)
router_proj_persist_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                           PersistArgs a)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    using Cfg = PersistCfg<InT, GATE>;
    constexpr int NST = Cfg::NST;
    constexpr int RELEASERS = PT_WARPS + (GATE ? 2 : 0);   // warps that read every stage
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[NST];    // stage landed (TMA bytes)
    __shared__ __align__(8) uint64_t empty_bar[NST];   // every warp that reads stages is done with it
    uint8_t *smem = smem_align1024(smem_raw);
    float *tree = reinterpret_cast<float *>(smem + NST * Cfg::STAGE);
    uint8_t *wsg_ring = smem + NST * Cfg::STAGE + Cfg::TREE;    // GATE: w_sg's slice of each stage

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, tg = lane & 3, eg = lane >> 2;
    const int b = blockIdx.x, G = gridDim.x, ns = a.ns;

    // this CTA's steps [u0, u1) of the item-major sequence, as pieces in
    // processing order: the head (slabs [0, h_len) of item `last`), whole
    // items [f0, f1), the continuation (slabs [sa, ns) of item `first`)
    const long long U = (long long)a.n_items * ns;
    const long long u0 = U * b / G, u1 = U * (b + 1) / G;
    const int first = (int)(u0 / ns), sa = (int)(u0 % ns);
    const int last = (int)((u1 - 1) / ns), se = (int)((u1 - 1) % ns) + 1;
    const int h_len = se < ns ? se : 0;
    const int f0 = sa > 0 ? first + 1 : first, f1 = se < ns ? last : last + 1;
    const int T = (int)(u1 - u0);

    if (tid == 0) {
        prefetch_tmap(&tmx);
        prefetch_tmap(&tmw);
#pragma unroll
        for (int s = 0; s < NST; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&empty_bar[s], RELEASERS);
        }
        mbar_init_fence();
    }
    __syncthreads();

    // the waits on a hand-off flag (bounded; the flag of the previous CTA)
    auto wait_flag = [&](const unsigned int *fl, unsigned int done, unsigned int where) {
        if (ld_acquire(fl) == done) return;
        const uint64_t t0 = global_ns();
        while (ld_acquire(fl) != done) {
            if ((load_volatile(a.err) & 0xFFu) == kErrTimeout) return;
            if (global_ns() - t0 > kWaitLimitNs) {
                report_error(a.err, kErrTimeout, where);
                return;
            }
            __nanosleep(256);
        }
    };

    if (warp >= PT_WARPS) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(PT_REGS_PRODUCER));
        // the producer: one thread walks the steps in order, each into the
        // next ring slot once the stage's readers have released it
        if (warp == PT_WARPS && lane == 0) {
            Cursor c;
            c.start(h_len, last, f0, f1, first, sa, ns);
            const int npro = T < NST ? T : NST;
            int pro_item[NST], pro_slab[NST];
            // the gate boxes of the first steps are weights, not a preceding
            // kernel's output: they stream before the dependency wait
            for (int t = 0; t < npro; ++t) {
                pro_item[t] = c.item;
                pro_slab[t] = c.slab;
                load_boxes<Cfg>(smem + t * Cfg::STAGE, &full_bar[t], &tmx, &tmw, c.item, c.slab, a, 1, true,
                                GATE ? wsg_ring + t * Cfg::WSG : nullptr);
                c.advance(f0, f1, first, sa, ns);
            }
            pdl_wait();
            for (int t = 0; t < npro; ++t)
                load_boxes<Cfg>(smem + t * Cfg::STAGE, &full_bar[t], &tmx, &tmw, pro_item[t], pro_slab[t], a, 2, false);
            int slot = 0;
            uint32_t parity = 0;        // of the release that step t waits for: round t / NST - 1
            int t = npro;               // steps issued
            for (; t < T; ++t) {
                // after a wait has given up, nothing more is issued
                if (!mbar_wait(&empty_bar[slot], parity, a.err, 0x16) || !ring_slot_free(full_bar, NST, t)) break;
                load_boxes<Cfg>(smem + slot * Cfg::STAGE, &full_bar[slot], &tmx, &tmw, c.item, c.slab, a, 3, true,
                                GATE ? wsg_ring + slot * Cfg::WSG : nullptr);
                c.advance(f0, f1, first, sa, ns);
                if (++slot == NST) {
                    slot = 0;
                    parity ^= 1u;
                }
            }
            // the block outlives its copies: the producer stays until the
            // last steps it issued have landed (the readers wait for them
            // too, so this costs nothing unless a wait gave up)
            drain_ring(full_bar, NST, t);
        } else if (GATE && (warp == PT_WARPS + 1 || warp == PT_WARPS + 2)) {
            // the shared gate: lane L of gate warp q owns token row 32 q + L
            // of the tile and all 8 partition chains of the half for it, on
            // the items of the first expert tile; it reads every stage, so it
            // releases every stage
            const int q = warp - PT_WARPS - 1, t = 32 * q + lane;
            pdl_wait();
            const unsigned int done = head_done(load_volatile(a.epoch));
            unsigned int *my_flag = a.flags + (size_t)b * kPersistFlagsPerCta + PT_WARPS + q;
            if (h_len > 0 && lane == 0 && load_volatile(my_flag) == done) *my_flag = ~done;
            float gp[PT_WARPS];
            int slot = 0;
            uint32_t phase = 0;
            auto run_g = [&](int item, int s_begin, int s_end) {
                const int g = item & 1, tile = item >> 1;
                const bool gitem = tile % a.n_et == 0 && (tile / a.n_et) * PT_M + 32 * q < a.M;
                // (a stage of a first-expert-tile item carries the w_sg slice
                // whatever this warp's rows; rows past M only skip the work)
                for (int s = s_begin; s < s_end; ++s) {
                    mbar_wait(&full_bar[slot], phase, a.err, 0x17);
                    if (gitem)
                        gate_rows_step<Cfg, InT>(gp, smem + slot * Cfg::STAGE, t, s, g, wsg_ring + slot * Cfg::WSG, a.H);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty_bar[slot]);
                    if (++slot == NST) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            };
            auto zero_g = [&]() {
#pragma unroll
                for (int p = 0; p < PT_WARPS; ++p) gp[p] = 0.0f;
            };
            // levels 1-3 of the pairwise tree over the half's partitions
            auto store_g = [&](int item) {
                const int g = item & 1, tile = item >> 1;
                const int m = (tile / a.n_et) * PT_M + t;
                if (tile % a.n_et == 0 && m < a.M)
                    a.gpart[(size_t)g * a.M + m] = ((gp[0] + gp[1]) + (gp[2] + gp[3])) + ((gp[4] + gp[5]) + (gp[6] + gp[7]));
            };
            float *gho = a.ghandoff + ((size_t)b * 2 + q) * (PT_WARPS * 32);
            if (h_len > 0) {
                zero_g();
                run_g(last, 0, h_len);
                if ((last >> 1) % a.n_et == 0) {
                    const uint64_t pol = l2_evict_first_policy();
#pragma unroll
                    for (int p = 0; p < PT_WARPS; ++p) st_evict_first(gho + p * 32 + lane, gp[p], pol);
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) st_release(my_flag, done);
                }
            }
            for (int it = f0; it < f1; ++it) {
                zero_g();
                run_g(it, 0, ns);
                store_g(it);
            }
            if (sa > 0) {
                const bool gcont = (first >> 1) % a.n_et == 0;
                const float *gprev = a.ghandoff + ((size_t)(b - 1) * 2 + q) * (PT_WARPS * 32);
                zero_g();
                if (gcont) {
                    wait_flag(a.flags + (size_t)(b - 1) * kPersistFlagsPerCta + PT_WARPS + q, done, 0x18);
#pragma unroll
                    for (int p = 0; p < PT_WARPS; ++p) gp[p] = __ldcg(gprev + p * 32 + lane);
                }
                run_g(first, sa, ns);
                store_g(first);
                if (gcont && (reinterpret_cast<uintptr_t>(gprev) & 127u) == 0 && lane < PT_WARPS)
                    asm volatile("discard.global.L2 [%0], 128;" ::"l"(gprev + lane * 32) : "memory");
            }
        }
        return;
    }

    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(PT_REGS_COMPUTE));
    pdl_wait();   // the epoch word and the workspace: the preceding kernel is complete

    // the epoch of this call; a flag equal to head_done(epoch) marks a
    // finished head
    const unsigned int done = head_done(load_volatile(a.epoch));
    unsigned int *my_flag = a.flags + (size_t)b * kPersistFlagsPerCta + warp;
    if (h_len > 0 && lane == 0 && load_volatile(my_flag) == done)
        *my_flag = ~done;      // left over, and happens to match: not this call's

    float acc[16][8];
    int slot = 0;
    uint32_t phase = 0;
    // the slabs [s_begin, s_end) of `item` into acc
    auto run = [&](int item, int s_begin, int s_end) {
        const int g = item & 1, tile = item >> 1;
        const bool live = tg < a.M - (tile / a.n_et) * PT_M;   // some of this lane's tokens exist
        for (int s = s_begin; s < s_end; ++s) {
            mbar_wait(&full_bar[slot], phase, a.err, 0x14);
            if (live && kSlab * s + kBlk * (8 * g + warp) < a.H) {
                const uint8_t *st = smem + slot * Cfg::STAGE;
                const int bx = warp / Cfg::PB, pc = warp % Cfg::PB;
                if constexpr (sizeof(InT) == 4)
                    pblock_f32(acc, st + bx * Cfg::XBOX, st + Cfg::XOP + bx * Cfg::WBOX, pc, tg, eg);
                else
                    pblock_bf16(acc, st + bx * Cfg::XBOX, st + Cfg::XOP + bx * Cfg::WBOX, pc, tg, eg);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_bar[slot]);
            if (++slot == NST) {
                slot = 0;
                phase ^= 1u;
            }
        }
    };
    auto zero = [&]() {
#pragma unroll
        for (int j = 0; j < 16; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;
    };
    // the item's group sums for its half of the partitions
    auto finish = [&](int item) {
        const int g = item & 1, tile = item >> 1;
        const int m0 = (tile / a.n_et) * PT_M, e0 = (tile % a.n_et) * PT_E;
        float *part = a.part + (size_t)g * a.M * a.E;
        switch (warp) {
        case 0: tree_and_store<0>(acc, tree, lane, part, a.M, a.E, m0, e0, tg, eg); break;
        case 1: tree_and_store<1>(acc, tree, lane, part, a.M, a.E, m0, e0, tg, eg); break;
        case 2: tree_and_store<2>(acc, tree, lane, part, a.M, a.E, m0, e0, tg, eg); break;
        case 3: tree_and_store<3>(acc, tree, lane, part, a.M, a.E, m0, e0, tg, eg); break;
        case 4: tree_and_store<4>(acc, tree, lane, part, a.M, a.E, m0, e0, tg, eg); break;
        case 5: tree_and_store<5>(acc, tree, lane, part, a.M, a.E, m0, e0, tg, eg); break;
        case 6: tree_and_store<6>(acc, tree, lane, part, a.M, a.E, m0, e0, tg, eg); break;
        default: tree_and_store<7>(acc, tree, lane, part, a.M, a.E, m0, e0, tg, eg); break;
        }
    };

    if (h_len > 0) {                     // the head: its chains go to the next CTA
        zero();
        run(last, 0, h_len);
        float *ho = a.handoff + ((size_t)b * PT_WARPS + warp) * PT_SLOT;
        const uint64_t pol = l2_evict_first_policy();
#pragma unroll
        for (int j = 0; j < 16; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) st_evict_first(ho + (j * 8 + i) * 32 + lane, acc[j][i], pol);
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release(my_flag, done);
    }
    for (int it = f0; it < f1; ++it) {
        zero();
        run(it, 0, ns);
        finish(it);
    }
    if (sa > 0) {                        // the continuation of the previous CTA's head
        wait_flag(a.flags + (size_t)(b - 1) * kPersistFlagsPerCta + warp, done, 0x15);
        const float *ho = a.handoff + ((size_t)(b - 1) * PT_WARPS + warp) * PT_SLOT;
#pragma unroll
        for (int j = 0; j < 16; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[j][i] = __ldcg(ho + (j * 8 + i) * 32 + lane);
        run(first, sa, ns);
        finish(first);
        // every value read from the hand-off has been used by now: drop its
        // lines from L2 without writing them back to device memory (they are
        // dead; each call's heads write them anew), 128-byte lines only
        if ((reinterpret_cast<uintptr_t>(ho) & 127u) == 0) {
#pragma unroll
            for (int r = 0; r < PT_VALS / 32; ++r)
                asm volatile("discard.global.L2 [%0], 128;" ::"l"(ho + (r * 32 + lane) * 32) : "memory");
        }
    }
}

}  // namespace

size_t persist_workspace_bytes(long long M, long long E)
{
    return kPersistGroupSumsOffset + (size_t)(2 * M * E + 2 * M) * sizeof(float);
}

namespace {
// One block (12 warps, about 225 KB of shared memory) per SM
// is what the kernel is built for; ask the runtime once per device.
constexpr int persist_kid(bool f32in, bool gate) { return KID_ROUTER_PERSIST + (f32in ? 0 : 1) + (gate ? 2 : 0); }

template <typename InT, bool GATE>
bool persist_fits(Device *d)
{
    std::atomic<int> &f = d->persist_fits[(sizeof(InT) == 4 ? 0 : 1) + (GATE ? 2 : 0)];
    int v = f.load(std::memory_order_acquire);
    if (v >= 0) return v == 1;
    auto kern = router_proj_persist_kernel<InT, GATE>;
    int blocks = 0;
    const bool ok = set_smem_once(d, persist_kid(sizeof(InT) == 4, GATE), kern, PersistCfg<InT, GATE>::SMEM) == BI_OK &&
                    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kern, PT_THREADS,
                                                                  PersistCfg<InT, GATE>::SMEM) == cudaSuccess &&
                    blocks >= 1;
    f.store(ok ? 1 : 0, std::memory_order_release);
    return ok;
}
}  // namespace

PersistPlan persist_plan(Device *d, int M, int E, bool f32in, bool gate)
{
    PersistPlan p = {};
    const long long n_mt = (M + PT_M - 1) / PT_M, n_et = (E + PT_E - 1) / PT_E;
    const long long n_items = n_mt * n_et * 2;
    const int G = d->sm_count < kPersistMaxCtas ? d->sm_count : kPersistMaxCtas;
    // every CTA needs at least one item's worth of steps (so that a head and
    // a continuation never fall in the same item), and the group sums must
    // fit the cap of the split plans
    if (n_items < kPersistMinItems || n_items < G || 8ll * M * E > kPersistSumsMax) return p;
    const bool fits = f32in ? (gate ? persist_fits<float, true>(d) : persist_fits<float, false>(d))
                            : (gate ? persist_fits<__nv_bfloat16, true>(d) : persist_fits<__nv_bfloat16, false>(d));
    if (!fits) return p;
    p.ok = true;
    p.G = G;
    p.n_et = (int)n_et;
    p.n_items = (int)n_items;
    return p;
}

template <typename InT, bool GATE>
bi_status launch_persist_t(Device *d, const PersistPlan &p, const void *x, const void *w, const void *w_sg, int M,
                           int E, int H, void *workspace, cudaStream_t s)
{
    using Cfg = PersistCfg<InT, GATE>;
    auto kern = router_proj_persist_kernel<InT, GATE>;
    bi_status st = set_smem_once(d, persist_kid(sizeof(InT) == 4, GATE), kern, Cfg::SMEM);
    if (st != BI_OK) return st;
    const CUtensorMapDataType dt = sizeof(InT) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t strides[1] = {(uint64_t)H * sizeof(InT)};
    const uint32_t box[2] = {(uint32_t)(Cfg::PB * kBlk), (uint32_t)PT_M};
    alignas(64) CUtensorMap tmx, tmw;
    {
        const uint64_t dims[2] = {(uint64_t)H, (uint64_t)M};
        if ((st = encode_tiled(&tmx, dt, 2, x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) != BI_OK) return st;
    }
    {
        const uint64_t dims[2] = {(uint64_t)H, (uint64_t)E};
        if ((st = encode_tiled(&tmw, dt, 2, w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B)) != BI_OK) return st;
    }
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    PersistArgs a;
    a.M = M;
    a.E = E;
    a.H = H;
    a.n_et = p.n_et;
    a.ns = (H + kSlab - 1) / kSlab;
    a.n_items = p.n_items;
    a.part = reinterpret_cast<float *>(ws + kPersistGroupSumsOffset);
    a.epoch = reinterpret_cast<unsigned int *>(ws);
    a.flags = reinterpret_cast<unsigned int *>(ws + kPersistFlagsOffset);
    a.handoff = reinterpret_cast<float *>(ws + kPersistHandoffOffset);
    a.w_sg = w_sg;
    a.gpart = reinterpret_cast<float *>(ws + kPersistGroupSumsOffset + (size_t)2 * M * E * sizeof(float));
    a.ghandoff = reinterpret_cast<float *>(ws + kPersistGateHandoffOffset);
    a.err = d->err;
    return launch_pdl(kern, dim3(p.G), dim3(PT_THREADS), (size_t)Cfg::SMEM, s, tmx, tmw, a);
}

bi_status launch_persist(Device *d, const PersistPlan &p, bool f32in, const void *x, const void *w,
                         const void *w_sg, int M, int E, int H, void *workspace, cudaStream_t s)
{
    if (w_sg)
        return f32in ? launch_persist_t<float, true>(d, p, x, w, w_sg, M, E, H, workspace, s)
                     : launch_persist_t<__nv_bfloat16, true>(d, p, x, w, w_sg, M, E, H, workspace, s);
    return f32in ? launch_persist_t<float, false>(d, p, x, w, nullptr, M, E, H, workspace, s)
                 : launch_persist_t<__nv_bfloat16, false>(d, p, x, w, nullptr, M, E, H, workspace, s);
}

}  // namespace bi
