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
// Data path.  Per slab (128 values of h), the block's gate rows (E/CS rows,
// padded to a multiple of 4), the cluster's X rows (TM rows) and, for the
// fused shared gate, the slab of w_sg are copied into a ring of shared-
// memory stages with 16-byte asynchronous copies (cp.async), the weight rows
// of every stage the ring holds before the dependency wait (weights are
// never the preceding kernel's output), the X rows after it; each thread's
// completion arrives on the stage's mbarrier.  Within a staged f32 row the
// first halves of the 16 partition blocks come first, then the second
// halves, so lane q reads its 8 values as two 16-byte loads at 16 q and at
// 256 + 16 q: each quarter-warp's load covers 128 contiguous bytes, every
// bank once.  (bf16 blocks are 16 bytes: lane q reads 16 q.)
//
// Work per block: a half-warp owns 4 experts and up to 8 of the cluster's
// tokens; lane q runs partition q's 32 chains (4 experts x 8 tokens), which
// reuse each loaded value 4 or 8 times and keep 32 independent fused
// multiply-add chains in flight per lane.
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
constexpr int kCluNE = 4;                         // experts per half-warp
constexpr int kCluTokJob = 8;                     // tokens per half-warp at most
constexpr size_t kCluSmemMax = 226 * 1024;        // the per-block opt-in maximum less static shared memory

struct CluArgs {
    const void *x, *w;
    int M, E, H, k, logit_bf16;
    int Eb4;                 // gate rows per block, rounded up to a multiple of kCluNE
    int nst, stage_bytes, x_off, g_off, gather_off;
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

// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

// The barrier's phase gets one arrival from this thread once every
// cp.async it issued so far has landed.
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One slab-row of `src` (row pointer, h0 = start of the slab) into a staged
// row: f32 as [half][block][4 values], bf16 as [block][8 values].  Copies
// chunk i of the row's CPR chunks; values past H are zero-filled.
template <typename InT>
__device__ __forceinline__ void copy_chunk(uint32_t row_dst, const InT *row_src, int h0, int H, int i, bool valid)
{
    if constexpr (sizeof(InT) == 4) {
        const int q = i >> 1, h = i & 1;                      // global order: block q, half h
        const int hh = h0 + 8 * q + 4 * h;
        const bool in = valid && hh < H;
        cp_async16(row_dst + 16u * (uint32_t)(16 * h + q), in ? row_src + hh : row_src, in ? 16u : 0u);
    } else {
        const int hh = h0 + 8 * i;
        const bool in = valid && hh < H;
        cp_async16(row_dst + 16u * (uint32_t)i, in ? row_src + hh : row_src, in ? 16u : 0u);
    }
}

// Partition q's 8 values of a staged row (h increasing).
__device__ __forceinline__ void load_block(const uint8_t *row, int q, float (&v)[8], float)
{
    const float4 a = *reinterpret_cast<const float4 *>(row + 16 * q);
    const float4 b = *reinterpret_cast<const float4 *>(row + 256 + 16 * q);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
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
__global__ void __launch_bounds__(32 * kCluMaxWarps, 1) router_cluster_kernel(CluArgs a)
{
    pdl_trigger();   // dependents may launch now; each waits before reading our outputs
    constexpr int ES = (int)sizeof(InT);
    constexpr int ROW = kSlab * ES;                         // bytes of one staged slab row
    constexpr int CPR = ROW / 16;                           // 16-byte chunks per row
    constexpr int TJ = NT < kCluTokJob ? NT : kCluTokJob;   // tokens per half-warp
    constexpr int TG = NT / TJ;                             // token groups
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kCluMaxStages];
    uint8_t *smem = smem_align1024(smem_raw);

    const int CS = gridDim.x, b = blockIdx.x;               // the cluster spans gridDim.x: rank = blockIdx.x
    const int tid = threadIdx.x, nthreads = blockDim.x, warp = tid >> 5, lane = tid & 31, q = lane & 15;
    const int Eb = a.E / CS, e0 = b * Eb, EG = a.Eb4 / kCluNE;
    const int m0 = blockIdx.y * NT;
    const int nt = min(NT, a.M - m0);                       // >= 1 by the grid
    const int H = a.H, ns = (H + kSlab - 1) / kSlab, NST = a.nst;
    const bool gate_here = a.gw != nullptr && b < nt;       // block b computes the gate of its token b
    const int job = 2 * warp + (lane >> 4);
    const bool active = job < EG * TG;
    const int eg = job % EG, tg = job / EG;                 // experts 4 eg .. 4 eg + 3, tokens TJ tg ..
    const InT *X = static_cast<const InT *>(a.x), *W = static_cast<const InT *>(a.w);
    float *gather = reinterpret_cast<float *>(smem + a.gather_off);
    const uint32_t sbase = smem_u32(smem);

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) mbar_init(&full_bar[s], (uint32_t)nthreads);
        mbar_init_fence();
    }
    __syncthreads();
    // every block of the cluster has started once all have arrived; waited
    // for just before the first store into another block's shared memory
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    auto issue_w = [&](int s, int slot) {
        const uint32_t st = sbase + (uint32_t)(slot * a.stage_bytes);
        for (int i = tid; i < Eb * CPR; i += nthreads) {
            const int r = i / CPR;
            copy_chunk<InT>(st + (uint32_t)(r * ROW), W + (size_t)(e0 + r) * H, kSlab * s, H, i % CPR, true);
        }
        if (gate_here)
            for (int i = tid; i < CPR; i += nthreads)
                copy_chunk<InT>(st + (uint32_t)a.g_off, static_cast<const InT *>(a.gw), kSlab * s, H, i, true);
    };
    auto issue_x = [&](int s, int slot) {
        const uint32_t st = sbase + (uint32_t)(slot * a.stage_bytes + a.x_off);
        for (int i = tid; i < NT * CPR; i += nthreads) {
            const int t = i / CPR;
            const bool in = t < nt;
            copy_chunk<InT>(st + (uint32_t)(t * ROW), X + (size_t)(in ? m0 + t : 0) * H, kSlab * s, H, i % CPR, in);
        }
    };

    const int nst = ns < NST ? ns : NST;
    for (int s = 0; s < nst; ++s) issue_w(s, s);
    pdl_wait();       // X may be the preceding kernel's output
    for (int s = 0; s < nst; ++s) {
        issue_x(s, s);
        cp_async_arrive(&full_bar[s]);
    }

    float acc[kCluNE][TJ];
#pragma unroll
    for (int j = 0; j < kCluNE; ++j)
#pragma unroll
        for (int t = 0; t < TJ; ++t) acc[j][t] = 0.0f;
    float gacc = 0.0f;
    int slot = 0;
    uint32_t phase = 0;
    for (int s = 0; s < ns; ++s) {
        mbar_wait(&full_bar[slot], phase, a.err, 0x1C);
        if (kSlab * s + kBlk * q < H) {
            const uint8_t *st = smem + slot * a.stage_bytes;
            const uint8_t *xs = st + a.x_off + (size_t)(tg * TJ) * ROW;
            if (active) {
                float w[kCluNE][8];
#pragma unroll
                for (int j = 0; j < kCluNE; ++j) load_block(st + (kCluNE * eg + j) * ROW, q, w[j], InT());
#pragma unroll
                for (int t = 0; t < TJ; ++t) {
                    float x[8];
                    load_block(xs + t * ROW, q, x, InT());
#pragma unroll
                    for (int j = 0; j < kCluNE; ++j) acc[j][t] = chain8(x, w[j], acc[j][t]);
                }
            }
            if (gate_here && job == 0) {
                float gv[8], x[8];
                load_block(st + a.g_off, q, gv, InT());
                load_block(st + a.x_off + b * ROW, q, x, InT());
                gacc = chain8(x, gv, gacc);
            }
        }
        if (s + NST < ns) {              // refill the slot once every warp is done with it
            __syncthreads();
            issue_w(s + NST, slot);
            issue_x(s + NST, slot);
            cp_async_arrive(&full_bar[slot]);
        }
        if (++slot == NST) {
            slot = 0;
            phase ^= 1u;
        }
    }

    // the pairwise tree over the 16 partitions of every (expert, token)
#pragma unroll
    for (int j = 0; j < kCluNE; ++j)
#pragma unroll
        for (int t = 0; t < TJ; ++t)
#pragma unroll
            for (int d = 1; d < 16; d *= 2) acc[j][t] = acc[j][t] + __shfl_xor_sync(0xFFFFFFFFu, acc[j][t], d);
#pragma unroll
    for (int d = 1; d < 16; d *= 2) gacc = gacc + __shfl_xor_sync(0xFFFFFFFFu, gacc, d);

    // every block of the cluster is running: logits go to this call's output
    // and to the shared memory of the block that selects their token
    __syncwarp();
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (active) {
        const uint32_t gbase = smem_u32(gather);
#pragma unroll
        for (int j = 0; j < kCluNE; ++j)
#pragma unroll
            for (int t = 0; t < TJ; ++t) {
                const int el = kCluNE * eg + j, tt = tg * TJ + t;
                if (((j * TJ + t) & 15) == q && el < Eb && tt < nt) {
                    float v = acc[j][t];
                    const int e = e0 + el;
                    const size_t o = (size_t)(m0 + tt) * a.E + e;
                    if (a.logit_bf16) {
                        const __nv_bfloat16 r = __float2bfloat16_rn(v);
                        static_cast<__nv_bfloat16 *>(a.logits)[o] = r;
                        v = __bfloat162float(r);
                    } else {
                        static_cast<float *>(a.logits)[o] = v;
                    }
                    const uint32_t dst = gbase + 4u * (uint32_t)((tt / CS) * a.E + e);
                    st_cluster_f32(mapa_u32(dst, (uint32_t)(tt % CS)), v);
                }
            }
    }
    if (gate_here && tid == 0) {
        a.gdot[m0 + b] = gacc;
        if (a.gsig) a.gsig[m0 + b] = 1.0f / (1.0f + expf(-gacc));
    }
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

    // the tokens whose logits this block received: t = r * CS + b
    const int epl = a.E >> 5, nwarps = nthreads >> 5;
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
    const int Eb4 = (Eb + kCluNE - 1) / kCluNE * kCluNE;
    const int TJ = NT < kCluTokJob ? NT : kCluTokJob;
    const int jobs = (Eb4 / kCluNE) * (NT / TJ);
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
    const long budget = (long)kCluSmemMax - 1024 - gather;
    long nst = budget / p.stage_bytes;
    if (nst > kCluMaxStages) nst = kCluMaxStages;
    if (nst > ns) nst = ns;
    if (nst < (ns < 2 ? ns : 2)) return p;
    p.nst = (int)nst;
    p.gather_off = p.nst * p.stage_bytes;
    p.smem = p.gather_off + gather + 1024;
    p.ok = true;
    return p;
}

namespace {

template <typename InT, int NT>
bi_status launch_cluster(Device *d, const ClusterPlan &p, const CluArgs &args, cudaStream_t s)
{
    bi_status st = set_cluster_attrs<InT, NT>(d, kid_cluster((int)sizeof(InT), NT));
    if (st != BI_OK) return st;
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
    return from_cuda(cudaLaunchKernelEx(&cfg, router_cluster_kernel<InT, NT>, args));
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
