// Device-side building blocks for the sm_103a kernels of libpi: shared-memory
// mbarriers, bulk (TMA) global->shared copies, bounded waits, the grid
// barrier of the persistent step kernel, and 16-bit float helpers.
//
// Every wait here is bounded by a globaltimer deadline.  A wait that runs out
// records PI_ERR_TIMEOUT in the device status word, raises the abort flag
// that every other wait also polls, and returns false; callers then unwind
// and the kernel exits.  Nothing traps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pi_kernels.h"

namespace pi {

// ------------------------------------------------------------------ status
static __device__ __forceinline__ void raise_error(const StepParams &p, int code)
{
    atomicCAS(p.status, 0, code);
    atomicExch(p.abort_flag, 1);
}

static __device__ __forceinline__ bool aborted(const StepParams &p)
{
    return *(volatile int *)p.abort_flag != 0;
}

static __device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ shared memory / mbarrier
static __device__ __forceinline__ uint32_t smem_u32(const void *ptr)
{
    return (uint32_t)__cvta_generic_to_shared(ptr);
}

static __device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// make initialised mbarriers visible to the async (TMA) proxy
static __device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// order this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) writes to the same bytes
static __device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

static __device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

static __device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// Non-blocking: has the phase with the given parity completed?
static __device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

static __device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity of `bar` has completed.
static __device__ __noinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const StepParams &p)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    // try_wait suspends the warp for a while by itself; the abort flag (an
    // L2 read) and the clock are looked at every 16th round only
    for (unsigned it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15) == 0) {
            if (aborted(p)) return false;
            if (globaltimer() - t0 > p.wait_ns) {
                raise_error(p, PI_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

// Bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is counted on `bar`.
static __device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

static __device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// c + a.lo * b.lo, then + a.hi * b.hi, for two 16-bit values (f16 or bf16)
// packed in each 32-bit word, with an fp32 accumulator.  The mixed-precision
// fma of sm_100+ multiplies the exactly widened operands and rounds once, so
// each step equals fmaf(float(a), float(b), c) and no conversion is issued.
template <typename T>
__device__ __forceinline__ float fma_pair(uint32_t a, uint32_t b, float c);

template <>
__device__ __forceinline__ float fma_pair<__half>(uint32_t a, uint32_t b, float c)
{
    asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;"
        " fma.rn.f32.f16 %0, al, bl, %0; fma.rn.f32.f16 %0, ah, bh, %0; }"
        : "+f"(c)
        : "r"(a), "r"(b));
    return c;
}

template <>
__device__ __forceinline__ float fma_pair<__nv_bfloat16>(uint32_t a, uint32_t b, float c)
{
    asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;"
        " fma.rn.f32.bf16 %0, al, bl, %0; fma.rn.f32.bf16 %0, ah, bh, %0; }"
        : "+f"(c)
        : "r"(a), "r"(b));
    return c;
}

// Eight 16-bit products of a chunk, in element order, onto c.
template <typename T>
__device__ __forceinline__ float fma_chunk(const uint4 &w, const uint4 &x, float c)
{
    c = fma_pair<T>(w.x, x.x, c);
    c = fma_pair<T>(w.y, x.y, c);
    c = fma_pair<T>(w.z, x.z, c);
    return fma_pair<T>(w.w, x.w, c);
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint16_t ld_shared_u16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// named barrier over the consumer warps only (the producer warps never join)
static __device__ __forceinline__ void cons_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// ------------------------------------------------------------------ epoch-tagged words
// A tagged word is one naturally aligned 64-bit store (single-copy atomic):
// epoch in the high half, the 32-bit value in the low half.  Strong relaxed
// accesses at gpu scope: the writer needs no fence, the reader sees either
// the old word or the new one, never a mix.
__device__ __forceinline__ void st_tagged(uint64_t *a, unsigned epoch, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(a), "l"(((uint64_t)epoch << 32) | v) : "memory");
}

__device__ __forceinline__ uint64_t ld_tagged(const uint64_t *a)
{
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}

// Two adjacent tagged words (a 16-byte aligned), one vector access; each
// word is still atomic on its own.
__device__ __forceinline__ void st_tagged2(uint64_t *a, unsigned epoch, uint32_t v0, uint32_t v1)
{
    const uint64_t hi = (uint64_t)epoch << 32;
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(a), "l"(hi | v0), "l"(hi | v1) : "memory");
}

__device__ __forceinline__ void ld_tagged2(const uint64_t *a, uint64_t &v0, uint64_t &v1)
{
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(v0), "=l"(v1) : "l"(a) : "memory");
}

__device__ __forceinline__ bool tag_is(uint64_t v, unsigned epoch) { return (unsigned)(v >> 32) == epoch; }

// Wait for a set of tagged words.  `reload` re-reads the caller's words
// (they stay in its registers: this is inline on purpose) and returns the
// address of one that does not carry `epoch` yet, or nullptr when all do.
// While a word is stale only that word is polled (8 bytes per round, with a
// short sleep), then the whole set is read again; re-reading the whole set
// every round floods L2 while the last writers are still at work.  Bounded by
// the wait limit; on a timeout or an abort it sets the CTA's failure word.
template <typename F>
__device__ __forceinline__ bool poll_tags(const StepParams &p, volatile int *fail, unsigned epoch,
                                          const uint64_t *stale, F reload)
{
    if (!stale) return true; // (the clock is read only once a word has to be polled)
    const uint64_t t0 = globaltimer();
    unsigned it = 0;
    while (stale) {
        while (!tag_is(ld_tagged(stale), epoch)) {
            __nanosleep(64);
            if (*fail) return false;
            if ((++it & 15) == 0) {
                if (aborted(p)) {
                    *fail = 1;
                    return false;
                }
                if (globaltimer() - t0 > p.wait_ns) {
                    raise_error(p, PI_DEV_TIMEOUT);
                    *fail = 1;
                    return false;
                }
            }
        }
        stale = reload();
    }
    return true;
}

// Bulk prefetch of [src, src+bytes) into L2 (no shared memory, no completion).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes, uint64_t policy)
{
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src), "r"(bytes),
                 "l"(policy)
                 : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_normal()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Wait until the shared counter reaches `target` (bounded; polls the abort flag).
static __device__ __noinline__ bool wait_counter(volatile int *ctr, int target, const StepParams &p)
{
    if (*ctr >= target) return true;
    const uint64_t t0 = globaltimer();
    for (unsigned it = 1;; ++it) {
        if (*ctr >= target) return true;
        if ((it & 15) == 0) {
            if (aborted(p)) return false;
            if (globaltimer() - t0 > p.wait_ns) {
                raise_error(p, PI_DEV_TIMEOUT);
                return false;
            }
        }
        __nanosleep(64);
    }
}

// Consumer-side wait on an mbarrier phase.  A failed wait (timeout or abort)
// sets the CTA's shared failure word; the warp then skips the rest of its
// work but keeps meeting the consumer barriers, after which every consumer
// thread sees the word and the CTA unwinds as a whole (a warp that left
// early would leave the others blocked on a named barrier).
static __device__ __forceinline__ bool wait_cta(uint64_t *bar, uint32_t parity, const StepParams &p, volatile int *fail,
                                         bool &ok)
{
    if (!ok) return false;
    if (mbar_try_wait(bar, parity)) return true; // fast path, no call
    if (*fail || !mbar_wait(bar, parity, p)) {
        *fail = 1;
        ok = false;
    }
    return ok;
}

static __device__ __forceinline__ bool cons_sync_ok(volatile int *fail)
{
    cons_sync();
    return *fail == 0;
}

// ------------------------------------------------------------------ 16-bit floats
template <typename T> struct F16T;

template <> struct F16T<__half> {
    static __device__ __forceinline__ float2 pair(uint32_t u)
    {
        __half2 h;
        memcpy(&h, &u, 4);
        return __half22float2(h);
    }
    static __device__ __forceinline__ float one(uint16_t u) { return __half2float(__ushort_as_half(u)); }
    static __device__ __forceinline__ uint16_t round(float f) { return __half_as_ushort(__float2half_rn(f)); }
};

template <> struct F16T<__nv_bfloat16> {
    static __device__ __forceinline__ float2 pair(uint32_t u)
    {
        return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
    static __device__ __forceinline__ float one(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }
    static __device__ __forceinline__ uint16_t round(float f)
    {
        return __bfloat16_as_ushort(__float2bfloat16_rn(f));
    }
};

// ------------------------------------------------------------------ slices
static __device__ __forceinline__ int slice_lo(long long total, int c, int G)
{
    return (int)((total * (long long)c) / G);
}

} // namespace pi
