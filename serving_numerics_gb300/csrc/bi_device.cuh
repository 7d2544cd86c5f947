// bi_device.cuh -- device-side helpers: bounded mbarrier waits, TMA loads,
// programmatic-dependent-launch controls, the sticky error word.
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace bi {

// error word layout: low byte = bi_status, next bytes = where it happened;
// the first report stands until the host reads the word
constexpr unsigned int kErrTimeout = 5u;   // BI_ERR_TIMEOUT: a bounded wait ran out

__device__ __forceinline__ void report_error(unsigned int *err, unsigned int code, unsigned int where)
{
    atomicCAS(err, 0u, code | (where << 8));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The first 1024-byte aligned byte of a dynamic shared-memory array.  The
// offset is added to the __shared__ pointer itself (never through an
// integer round trip), so the compiler still knows the result is shared
// memory and emits shared loads for it rather than generic ones.
__device__ __forceinline__ uint8_t *smem_align1024(uint8_t *smem_raw)
{
    return smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch.  Every kernel of the library triggers its
// dependents at entry (so the next kernel in the stream can be resident and
// stream its weights early) and calls pdl_wait() before it reads anything a
// preceding kernel may have written or writes anything it may still read.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned int load_volatile(const unsigned int *p)
{
    return *reinterpret_cast<const volatile unsigned int *>(p);
}

// Wait for the phase with the given parity to complete, for at most about
// two seconds.  On expiry: record BI_ERR_TIMEOUT (code 5) with `where` and
// return false; no thread is left waiting (what the caller does next is its
// kernel's failure path: carry on, or stop issuing and drain).
// Once any wait has given up (the error word holds a timeout), every later
// wait that is not already satisfied gives up at once, so a broken pipeline
// drains in milliseconds instead of two seconds per wait.  Other reports (an
// expert id out of range) leave the waits alone: the rest of the work in
// flight still completes correctly.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ bool mbar_wait_limit(uint64_t *bar, uint32_t parity, unsigned int *err,
                                                unsigned int where, uint64_t limit_ns)
{
    const uint32_t addr = smem_u32(bar);
    if (mbar_try_wait(addr, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(addr, parity)) return true;
        if ((i & 255u) == 0) {
            if ((load_volatile(err) & 0xFFu) == kErrTimeout) return false;
            if (global_ns() - t0 > limit_ns) {
                report_error(err, kErrTimeout, where);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned int *err,
                                          unsigned int where)
{
    return mbar_wait_limit(bar, parity, err, where, kWaitLimitNs);
}

// Has the phase with this parity completed?  One test, no waiting.
__device__ __forceinline__ bool mbar_done(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// After a wait has given up, a block still lets the bulk copies it issued
// land (and its tensor-core products finish) before it exits or frees
// tensor memory: no copy may still be writing the shared memory of a block
// that has gone.  This wait ignores the error word and ends after at most
// about 0.1 s.
constexpr uint64_t kDrainLimitNs = 100000000ull;

__device__ __forceinline__ bool mbar_drain(uint64_t *bar, uint32_t parity)
{
    const uint32_t addr = smem_u32(bar);
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(addr, parity)) return true;
        if ((i & 255u) == 255u && global_ns() - t0 > kDrainLimitNs) return false;
    }
}

// A ring of `stages` slots filled in order: step j goes into slot
// j % stages and completes phase j / stages of that slot's full barrier.
// A producer issues step j only once step j - stages has landed, so a
// slot's barrier is never more than one phase behind the last step issued
// into it, and drain_ring can wait for exactly those steps.  Where the one
// reader that releases a slot stops at its first wait that gives up (the
// MMA thread of the tensor-core kernels), every release follows a completed
// wait and that holds by itself; where readers carry on after a wait gave
// up, the producer tests it (ring_slot_free), a test that always passes in
// a pipeline whose waits all completed.
__device__ __forceinline__ bool ring_slot_free(uint64_t *full, int stages, int j)
{
    return j < stages || mbar_done(&full[j % stages], (uint32_t)(j / stages - 1) & 1u);
}

__device__ __forceinline__ void drain_ring(uint64_t *full, int stages, int issued)
{
    for (int j = issued > stages ? issued - stages : 0; j < issued; ++j)
        mbar_drain(&full[j % stages], (uint32_t)(j / stages) & 1u);
}

// 3-D tiled TMA load into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled TMA load into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// Untiled bulk copy global -> shared, completing on `bar`: both addresses
// 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// bf16 pattern (low or high half of a 32-bit word) widened to f32 exactly
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

}  // namespace bi
