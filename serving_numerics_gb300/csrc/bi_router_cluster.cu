// bi_router_cluster.cu -- the router for small batches (M <= 128): projection,
// top-k, softmax and margin in ONE launch, with no scratch memory.
//
// Source pages: "batch changed the model's mind" ("m-scan: the staircase":
// a 256-output F32 GEMV followed by top_k(8 of 256); "The fix: m-invariant
// twins": the decode router, router_gemv, reduces each row in one fixed
// order whatever the number of rows in the launch); "diag(MODEL-MM-QWEN4-
// EXP) ..." (lowest-index tie-break; margin in ULPs).
//
// Same reduction contract as every router kernel of the library: h is cut
// into slabs of 128 and each slab into 16 blocks of 8; partition q owns
// block q of every slab and runs ONE f32 fused multiply-add chain from +0
// over its h < H in increasing order; the 16 partials are added by the
// pairwise tree (0+1),(2+3),... four levels.  Lanes q and 16 + q of a warp
// run partition q for two different experts, so a token's 16 partials sit
// in one half-warp and the butterfly with offsets 1, 2, 4, 8 is exactly
// that tree (after each level lanes q and q^d hold the same sum, as fp
// addition is commutative).
//
// Decomposition.  A thread-block cluster of CS blocks (16, or 8 where the
// GPU cannot place 16) covers all E experts of TM tokens: block b owns the
// E/CS experts [b E/CS, (b+1) E/CS) and computes their logits for the
// cluster's tokens.  Each logit is then stored into the shared memory of
// the block that selects its token (block t mod CS for token t of the
// cluster) -- distributed shared memory, no device scratch -- and after one
// cluster barrier every token's top-k runs in the block that received its
// E logits.  The top-k of a token needs all E logits, and a cluster is the
// largest group of blocks whose shared memory can meet them inside one
// launch; a batch of M tokens runs as ceil(M / TM) clusters with TM chosen
// so that the clusters fill the GPU.
//
// Data path.  Per slab (128 values of h), the block's gate rows (E/CS rows),
// the cluster's X rows and, for the fused shared gate, the slab of w_sg are
// staged by TMA (one 2-D box per operand and stage, 512-byte rows for f32)
// into a ring of shared-memory stages; the weight rows of every stage the
// ring holds stream in before the dependency wait (weights are never the
// preceding kernel's output), the X rows after it.  Reading partition q's
// 8 values as two 16-byte loads would put lanes q and q + 4 on the same
// banks (their blocks are 128 bytes apart), so lanes with bit 2 of q set
// load their second half first and swap the two in registers: each quarter-
// warp's load then meets every bank once, and the fused multiply-adds still
// run in h order.  (bf16 blocks are 16 bytes: lane q reads 16 q.)
//
// Work per block: a half-warp owns NE experts and TJ of the cluster's tokens
// (2 x NT for up to 4 tokens per cluster, 4 x 4 at 8, 4 x 8 at 16); lane q
// runs partition q's NE x TJ chains.  One warp per scheduler is all the
// parallelism a block has at these sizes, so the shapes trade operand reuse
// (fewer shared-memory loads per multiply-add) against independent chains
// and warps; each was the fastest of those measured at its token count.  The block's logits are gathered
// in its own shared memory first, then pushed to the selecting blocks one
// contiguous run of E/CS values per token (a remote store whose lanes all
// go to one block is one transaction).
#include <cuda_bf16.h>

#include <mutex>

#include "bi_device.cuh"
#include "bi_internal.h"
#include "bi_select.cuh"

namespace bi {
namespace {

constexpr int kSlab = kRouterSlab, kBlk = kRouterBlock;
constexpr int kCluMaxStages = 32;
constexpr int kCluMaxWarps = 16;
// The half-warp job for NT tokens per cluster: NE experts x TJ tokens, the
// fastest shape measured for each NT at 16 experts per block (all give four
// warps there): 2 x NT up to 4 tokens, 4 x 4 at 8, 4 x 8 at 16.
constexpr int clu_ne(int NT) { return NT <= 4 ? 2 : 4; }
constexpr int clu_tj(int NT) { return NT <= 4 ? NT : NT == 8 ? 4 : 8; }
constexpr int kCluEbAlign = 4;                    // gate rows per block padded to a multiple of this
constexpr size_t kCluSmemMax = 226 * 1024;        // the per-block opt-in maximum less static shared memory

struct CluArgs {
    const void *x, *w;
    int M, E, H, k, logit_bf16;
    int Eb4;                 // gate rows per block, rounded up to a multiple of kCluEbAlign
    int nst, stage_bytes, x_off, g_off, gather_off, tile_off;
    void *logits;
    int32_t *ids;
    float *weights, *margin;
    int32_t *ulps;
    const void *gw;          // w_sg, or NULL (no shared gate)
    float *gdot, *gsig;
    unsigned int *err;
};

__device__ __forceinline__ uint32_t mapa_u32(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Partition q's 8 values of a staged row (h increasing).  f32 rows are 512
// bytes, block q at 32 q; lanes with bit 2 of q set load the block's second
// half first (see the data path above) and swap.
// Bitwise select (no branch): m all ones picks b, all zeros picks a.
__device__ __forceinline__ float pick(float a, float b, uint32_t m)
{
    return __uint_as_float((__float_as_uint(a) & ~m) | (__float_as_uint(b) & m));
}

__device__ __forceinline__ void load_block(const uint8_t *row, int q, float (&v)[8], float)
{
    const int sw = (q >> 2) & 1;
    const uint32_t m = 0u - (uint32_t)sw;
    const float4 a = *reinterpret_cast<const float4 *>(row + 32 * q + 16 * sw);
    const float4 b = *reinterpret_cast<const float4 *>(row + 32 * q + 16 * (sw ^ 1));
    v[0] = pick(a.x, b.x, m); v[1] = pick(a.y, b.y, m); v[2] = pick(a.z, b.z, m); v[3] = pick(a.w, b.w, m);
    v[4] = pick(b.x, a.x, m); v[5] = pick(b.y, a.y, m); v[6] = pick(b.z, a.z, m); v[7] = pick(b.w, a.w, m);
}

__device__ __forceinline__ void load_block(const uint8_t *row, int q, float (&v)[8], __nv_bfloat16)
{
    const uint4 r = *reinterpret_cast<const uint4 *>(row + 16 * q);
    v[0] = bf16lo(r.x); v[1] = bf16hi(r.x); v[2] = bf16lo(r.y); v[3] = bf16hi(r.y);
    v[4] = bf16lo(r.z); v[5] = bf16hi(r.z); v[6] = bf16lo(r.w); v[7] = bf16hi(r.w);
}

__device__ __forceinline__ float chain8(const float (&x)[8], const float (&w)[8], float a)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) a = __fmaf_rn(x[i], w[i], a);
    return a;
}

// One token's selection from the E logits gathered in this block.
template <int EPLM>
__device__ __forceinline__ void select_gathered(const float *g, int lane, const CluArgs &a, size_t m)
{
    const int epl = a.E >> 5;
    float v[EPLM];
#pragma unroll
    for (int i = 0; i < EPLM; ++i) v[i] = i < epl ? g[lane + 32 * i] : 0.0f;
    warp_select<EPLM>(v, lane, epl, a.k, a.logit_bf16, m, a.ids, a.weights, a.margin, a.ulps);
}

// NT: tokens per cluster (1, 2, 4, 8 or 16); a half-warp takes TJ of them.
template <typename InT, int NT>
__global__ void __launch_bounds__(32 * kCluMaxWarps, 1)
router_cluster_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw, CluArgs a)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    constexpr int ES = (int)sizeof(InT);
    constexpr int ROW = kSlab * ES;                         // bytes of one staged slab row
    constexpr int NE = clu_ne(NT), TJ = clu_tj(NT);         // a half-warp's experts and tokens
    constexpr int TG = NT / TJ;                             // token groups
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kCluMaxStages];
    uint8_t *smem = smem_align1024(smem_raw);

    const int CS = gridDim.x, b = blockIdx.x;               // the cluster spans gridDim.x: rank = blockIdx.x
    const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5, lane = tid & 31, q = lane & 15;
    const int nwarps = nthreads >> 5;
    const int Eb = a.E / CS, e0 = b * Eb, EG = a.Eb4 / NE;
    const int m0 = blockIdx.y * NT;
    const int nt = min(NT, a.M - m0);                       // >= 1 by the grid
    const int H = a.H, ns = (H + kSlab - 1) / kSlab, NST = a.nst;
    const bool gate_here = a.gw != nullptr && b < nt;       // block b computes the gate of its token b
    const int job = 2 * warp + (lane >> 4);
    const bool active = job < EG * TG;
    const int eg = job % EG, tg = job / EG;                 // experts NE eg .., tokens TJ tg ..
    float *gather = reinterpret_cast<float *>(smem + a.gather_off);
    float *tile = reinterpret_cast<float *>(smem + a.tile_off);     // this block's logits [NT][Eb4]

    if (tid == 0) {
        prefetch_tmap(&tmx);
        prefetch_tmap(&tmw);
        for (int s = 0; s < NST; ++s) mbar_init(&full_bar[s], 1);
        mbar_init_fence();
    }
    __syncthreads();
    // every block of the cluster has started once all have arrived; waited
    // for just before the first store into another block's shared memory
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    auto stage_tx = [&](int s) -> uint32_t {
        uint32_t tx = (uint32_t)(Eb + NT) * ROW;
        if (gate_here) tx += (uint32_t)min(kSlab, H - kSlab * s) * ES;
        return tx;
    };
    auto issue_w = [&](int s, int slot) {
        uint8_t *st = smem + slot * a.stage_bytes;
        tma_load_2d(st, &tmw, &full_bar[slot], kSlab * s, e0);
        if (gate_here)
            bulk_load(st + a.g_off, static_cast<const InT *>(a.gw) + (size_t)kSlab * s,
                      (uint32_t)min(kSlab, H - kSlab * s) * ES, &full_bar[slot]);
    };
    auto issue_x = [&](int s, int slot) {
        tma_load_2d(smem + slot * a.stage_bytes + a.x_off, &tmx, &full_bar[slot], kSlab * s, m0);
    };

    const int nst = ns < NST ? ns : NST;
    if (tid == 0)
        for (int s = 0; s < nst; ++s) {
            mbar_arrive_expect_tx(&full_bar[s], stage_tx(s));
            issue_w(s, s);
        }
    pdl_wait();       // X may be the preceding kernel's output
    if (tid == 0)
        for (int s = 0; s < nst; ++s) issue_x(s, s);

    float acc[NE][TJ];
#pragma unroll
    for (int j = 0; j < NE; ++j)
#pragma unroll
        for (int t = 0; t < TJ; ++t) acc[j][t] = 0.0f;
    float gacc = 0.0f;

    // one slab of the partition chains from ring slot `slot`
    auto slab = [&](int s, int slot) {
        if (kSlab * s + kBlk * q >= H) return;
        const uint8_t *st = smem + slot * a.stage_bytes;
        const uint8_t *xs = st + a.x_off + (size_t)(tg * TJ) * ROW;
        if (active) {
            float w[NE][8];
#pragma unroll
            for (int j = 0; j < NE; ++j) load_block(st + (NE * eg + j) * ROW, q, w[j], InT());
#pragma unroll
            for (int t = 0; t < TJ; ++t) {
                float x[8];
                load_block(xs + t * ROW, q, x, InT());
                // each chain is h-ordered; the NE chains of a token advance
                // together (independent multiply-adds)
#pragma unroll
                for (int i = 0; i < 8; ++i)
#pragma unroll
                    for (int j = 0; j < NE; ++j) acc[j][t] = __fmaf_rn(x[i], w[j][i], acc[j][t]);
            }
        }
        if (gate_here && job == 0) {
            float x[8], gv[8];
            load_block(st + a.x_off + b * ROW, q, x, InT());
            if constexpr (ES == 4) {      // the w_sg slab is a plain bulk copy: block q at 32 q
                const float4 g0 = *reinterpret_cast<const float4 *>(st + a.g_off + 32 * q);
                const float4 g1 = *reinterpret_cast<const float4 *>(st + a.g_off + 32 * q + 16);
                gv[0] = g0.x; gv[1] = g0.y; gv[2] = g0.z; gv[3] = g0.w;
                gv[4] = g1.x; gv[5] = g1.y; gv[6] = g1.z; gv[7] = g1.w;
            } else {
                load_block(st + a.g_off, q, gv, InT());
            }
            gacc = chain8(x, gv, gacc);
        }
    };

    bool ok = true;          // every wait of this thread completed
    int issued = nst;        // slabs issued (by thread 0)
    if (ns <= NST) {
        // the ring holds all of H: every stage is waited for up front, and
        // the loop has no waits in it, so that the loads of one slab can be
        // scheduled under the arithmetic of the previous one
        for (int s = 0; s < ns; ++s) ok &= mbar_wait(&full_bar[s], 0, a.err, 0x1C);
#pragma unroll 2
        for (int s = 0; s < ns; ++s) slab(s, s);
    } else {
        int slot = 0;
        uint32_t phase = 0;
        for (int s = 0; s < ns; ++s) {
            ok &= mbar_wait(&full_bar[slot], phase, a.err, 0x1C);
            slab(s, slot);
            if (s + NST < ns) {          // refill the slot once every warp is done with it
                __syncthreads();
                // slabs are issued in order while each slot's previous slab
                // has landed (always so unless a wait gave up)
                if (tid == 0 && issued == s + NST && ring_slot_free(full_bar, NST, s + NST)) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive_expect_tx(&full_bar[slot], stage_tx(s + NST));
                    issue_w(s + NST, slot);
                    issue_x(s + NST, slot);
                    ++issued;
                }
            }
            if (++slot == NST) {
                slot = 0;
                phase ^= 1u;
            }
        }
    }
    // thread 0 waited for every slab it issued; if one of those waits gave
    // up, the slabs still landing finish before the block goes on
    if (tid == 0 && !ok) drain_ring(full_bar, NST, issued);

    // the pairwise tree over the 16 partitions of every (expert, token), then
    // the block's logits (in the logit dtype's values) into its own tile
#pragma unroll
    for (int d = 1; d < 16; d *= 2) {         // one tree level at a time: its shuffles are independent
        float o[NE][TJ];
#pragma unroll
        for (int j = 0; j < NE; ++j)
#pragma unroll
            for (int t = 0; t < TJ; ++t) o[j][t] = __shfl_xor_sync(0xFFFFFFFFu, acc[j][t], d);
#pragma unroll
        for (int j = 0; j < NE; ++j)
#pragma unroll
            for (int t = 0; t < TJ; ++t) acc[j][t] = acc[j][t] + o[j][t];
    }
#pragma unroll
    for (int d = 1; d < 16; d *= 2) gacc = gacc + __shfl_xor_sync(0xFFFFFFFFu, gacc, d);
    if (active && q == 0) {              // every lane of the half-warp holds the sums
#pragma unroll
        for (int j = 0; j < NE; ++j)
#pragma unroll
            for (int t = 0; t < TJ; ++t) {
                const float v = acc[j][t];
                tile[(tg * TJ + t) * a.Eb4 + NE * eg + j] =
                    a.logit_bf16 ? __bfloat162float(__float2bfloat16_rn(v)) : v;
            }
    }
    __syncthreads();

    // every block of the cluster is running: each token's run of Eb logits
    // goes to the block that selects the token (the barrier's release then
    // waits for these remote stores only; this call's global outputs are
    // written after it)
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    const uint32_t gbase = smem_u32(gather);
    for (int t = warp; t < nt; t += nwarps) {
        const uint32_t dst = mapa_u32(gbase + 4u * (uint32_t)((t / CS) * a.E + e0), (uint32_t)(t % CS));
        for (int e = lane; e < Eb; e += 32) st_cluster_f32(dst + 4u * (uint32_t)e, tile[t * a.Eb4 + e]);
    }
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

    for (int t = warp; t < nt; t += nwarps) {
        const size_t orow = (size_t)(m0 + t) * a.E + e0;
        for (int e = lane; e < Eb; e += 32) {
            const float v = tile[t * a.Eb4 + e];
            if (a.logit_bf16)
                static_cast<__nv_bfloat16 *>(a.logits)[orow + e] = __float2bfloat16_rn(v);
            else
                static_cast<float *>(a.logits)[orow + e] = v;
        }
    }
    if (gate_here && tid == 0) {
        a.gdot[m0 + b] = gacc;
        if (a.gsig) a.gsig[m0 + b] = 1.0f / (1.0f + expf(-gacc));
    }

    // the tokens whose logits this block received: t = r * CS + b
    const int epl = a.E >> 5;
    for (int r = warp; r * CS + b < nt; r += nwarps) {
        const float *gr = gather + r * a.E;
        const size_t m = (size_t)(m0 + r * CS + b);
        if (epl <= 4)
            select_gathered<4>(gr, lane, a, m);
        else if (epl <= 8)
            select_gathered<8>(gr, lane, a, m);
        else
            select_gathered<16>(gr, lane, a, m);      // E <= 512 on this path
    }
}

// Per-device choice of the cluster size and how many clusters fit at once
// (queried once, for a block of the largest shared-memory footprint).
struct CluDevice {
    int cs = 0;        // 16 or 8; 0 = not yet queried; -1 = no cluster can be placed
    int max_active = 0;
};
std::mutex g_clu_mu;
CluDevice g_clu[64];

template <typename InT, int NT>
bi_status set_cluster_attrs(Device *d, int kid)
{
    auto kern = router_cluster_kernel<InT, NT>;
    return set_attr_once(d, kid, [&]() -> bool {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCluSmemMax) == cudaSuccess &&
               cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
               cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    (int)cudaSharedmemCarveoutMaxShared) == cudaSuccess;
    });
}

constexpr int kid_cluster(int es, int NT)
{
    return KID_ROUTER_CLUSTER + (es == 4 ? 0 : 5) + (NT == 1 ? 0 : NT == 2 ? 1 : NT == 4 ? 2 : NT == 8 ? 3 : 4);
}

bi_status cluster_device(Device *d, CluDevice *out)
{
    std::lock_guard<std::mutex> lk(g_clu_mu);
    CluDevice &c = g_clu[d->ordinal];
    if (c.cs == 0) {
        bi_status st = set_cluster_attrs<float, 16>(d, kid_cluster(4, 16));
        if (st != BI_OK) return st;
        auto kern = router_cluster_kernel<float, 16>;
        c.cs = -1;
        for (int cs : {16, 8}) {
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(cs, 64);
            cfg.blockDim = dim3(32 * 4);
            cfg.dynamicSmemBytes = kCluSmemMax;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = cs;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
                (void)cudaGetLastError();
                n = 0;
            }
            if (n > 0) {
                c.cs = cs;
                c.max_active = n;
                break;
            }
        }
    }
    *out = c;
    return BI_OK;
}

}  // namespace

// The cluster plan of one call: ok = false when this path does not apply
// (then the tiled kernels run).  Tokens per cluster: the smallest power of
// two (at most 16) whose clusters all fit the GPU at once.
ClusterPlan cluster_plan(Device *d, int M, int E, int H, int es, bool gate)
{
    ClusterPlan p = {};
    if (M < 1 || M > kClusterMaxM) return p;
    CluDevice cd;
    if (cluster_device(d, &cd) != BI_OK || cd.cs <= 0) return p;
    // E <= 512: a token's selection keeps at most 16 logits per lane in
    // registers (the 32-wide one would spill at this kernel's thread count)
    const int CS = cd.cs, Eb = E / CS;
    if (E > kClusterMaxE || E % CS != 0 || Eb < 2) return p;
    int NT = 1;
    while (NT < 16 && (M + NT - 1) / NT > cd.max_active) NT *= 2;
    const int Eb4 = (Eb + kCluEbAlign - 1) / kCluEbAlign * kCluEbAlign;
    const int jobs = (Eb4 / clu_ne(NT)) * (NT / clu_tj(NT));
    const int warps = (jobs + 1) / 2;
    if (warps > kCluMaxWarps) return p;
    const int ROW = kSlab * es, ns = (H + kSlab - 1) / kSlab;
    p.CS = CS;
    p.TM = NT;
    p.NT = NT;
    p.NC = (M + NT - 1) / NT;
    p.warps = warps;
    p.Eb4 = Eb4;
    p.x_off = Eb4 * ROW;
    p.g_off = p.x_off + NT * ROW;
    p.stage_bytes = p.g_off + (gate ? ROW : 0);
    const int gather = ((NT + CS - 1) / CS) * E * 4;
    const int tile = NT * Eb4 * 4;
    const long budget = (long)kCluSmemMax - 1024 - gather - tile;
    long nst = budget / p.stage_bytes;
    if (nst > kCluMaxStages) nst = kCluMaxStages;
    if (nst > ns) nst = ns;
    if (nst < (ns < 2 ? ns : 2)) return p;
    p.nst = (int)nst;
    p.gather_off = p.nst * p.stage_bytes;
    p.tile_off = p.gather_off + gather;
    p.smem = p.tile_off + tile + 1024;
    p.ok = true;
    return p;
}

namespace {

template <typename InT, int NT>
bi_status launch_cluster(Device *d, const ClusterPlan &p, const CluArgs &args, cudaStream_t s)
{
    bi_status st = set_cluster_attrs<InT, NT>(d, kid_cluster((int)sizeof(InT), NT));
    if (st != BI_OK) return st;
    const CUtensorMapDataType dt = sizeof(InT) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t strides[1] = {(uint64_t)args.H * sizeof(InT)};
    alignas(64) CUtensorMap tmx, tmw;
    {
        const uint64_t dims[2] = {(uint64_t)args.H, (uint64_t)args.M};
        const uint32_t box[2] = {(uint32_t)kSlab, (uint32_t)NT};
        if ((st = encode_tiled(&tmx, dt, 2, args.x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)) != BI_OK)
            return st;
    }
    {
        const uint64_t dims[2] = {(uint64_t)args.H, (uint64_t)args.E};
        const uint32_t box[2] = {(uint32_t)kSlab, (uint32_t)(args.E / p.CS)};
        if ((st = encode_tiled(&tmw, dt, 2, args.w, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE)) != BI_OK)
            return st;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.CS, p.NC);
    cfg.blockDim = dim3(32 * p.warps);
    cfg.dynamicSmemBytes = (size_t)p.smem;
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = p.CS;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return from_cuda(cudaLaunchKernelEx(&cfg, router_cluster_kernel<InT, NT>, tmx, tmw, args));
}

template <typename InT>
bi_status launch_cluster_nt(Device *d, const ClusterPlan &p, const CluArgs &args, cudaStream_t s)
{
    switch (p.NT) {
    case 1: return launch_cluster<InT, 1>(d, p, args, s);
    case 2: return launch_cluster<InT, 2>(d, p, args, s);
    case 4: return launch_cluster<InT, 4>(d, p, args, s);
    case 8: return launch_cluster<InT, 8>(d, p, args, s);
    default: return launch_cluster<InT, 16>(d, p, args, s);
    }
}

}  // namespace

bi_status router_cluster_call(Device *d, const ClusterPlan &p, const void *x, const void *w_gate, bool f32in,
                              int logit_bf16, int M, int H, int E, int k, void *logits, int32_t *ids,
                              float *weights, float *margin, int32_t *ulps, const void *w_sg, float *gdot,
                              float *gsig, cudaStream_t s)
{
    CluArgs a;
    a.x = x;
    a.w = w_gate;
    a.M = M;
    a.E = E;
    a.H = H;
    a.k = k;
    a.logit_bf16 = logit_bf16;
    a.Eb4 = p.Eb4;
    a.nst = p.nst;
    a.stage_bytes = p.stage_bytes;
    a.x_off = p.x_off;
    a.g_off = p.g_off;
    a.gather_off = p.gather_off;
    a.tile_off = p.tile_off;
    a.logits = logits;
    a.ids = ids;
    a.weights = weights;
    a.margin = margin;
    a.ulps = ulps;
    a.gw = w_sg;
    a.gdot = gdot;
    a.gsig = gsig;
    a.err = d->err;
    return f32in ? launch_cluster_nt<float>(d, p, a, s) : launch_cluster_nt<__nv_bfloat16>(d, p, a, s);
}

}  // namespace bi

// ---------------------------------------------------------------------------
// Measurement aid: the fixed cost of one dependent cluster launch.  A cluster
// of CS blocks (the router's shape at M <= TM) whose threads start, release
// their dependents, wait for the preceding kernel in the stream, read one
// word it wrote, pass a cluster barrier and write one word: no projection,
// no selection.  Back-to-back launches of it (each reading the previous
// one's word) time the floor under any one-launch router call that reads
// its input after the preceding kernel finishes.
// ---------------------------------------------------------------------------
namespace bi {
namespace {
__global__ void __launch_bounds__(128, 1) dependent_floor_kernel(const float *in, float *out)
{
    pdl_trigger();
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    pdl_wait();
    float v = 0.0f;
    if (threadIdx.x == 0) v = in[blockIdx.x] + 1.0f;
    __syncwarp();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (threadIdx.x == 0) out[blockIdx.x] = v;
}
}  // namespace
}  // namespace bi

extern "C" bi_status bi_selftest_dependent_floor(const float *in, float *out, bi_stream s)
{
    if (!in || !out) return BI_ERR_INVALID_ARG;
    bi::Device *d = nullptr;
    bi_status st = bi::current_device(&d);
    if (st != BI_OK) return st;
    bi::CluDevice cd;
    if ((st = bi::cluster_device(d, &cd)) != BI_OK) return st;
    if (cd.cs <= 0) return BI_ERR_UNSUPPORTED_SHAPE;
    st = bi::set_attr_once(d, bi::KID_FLOOR, [&]() -> bool {
        return cudaFuncSetAttribute(bi::dependent_floor_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
               cudaSuccess;
    });
    if (st != BI_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cd.cs);
    cfg.blockDim = dim3(128);
    cfg.stream = reinterpret_cast<cudaStream_t>(s);
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = cd.cs;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return bi::from_cuda(cudaLaunchKernelEx(&cfg, bi::dependent_floor_kernel, in, out));
}
