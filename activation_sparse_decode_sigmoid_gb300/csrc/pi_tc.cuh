// Device helpers shared by the tensor-core kernels of libpi (tcgen05 MMAs with
// accumulators in tensor memory, TMA loads, bounded mbarrier waits): the
// 16-bit FFN (pi_mma.cu) and the Q4_0 FFN that dequantises its rows in
// shared memory (pi_mma_q4.cu).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pi_kernels.h"

namespace pi {
namespace {

constexpr int kBK = 64;       // K elements per stage (one 128-byte row)

template <typename T> struct H16;
template <> struct H16<__half> {
    static __device__ __forceinline__ float one(uint16_t u) { return __half2float(__ushort_as_half(u)); }
    static __device__ __forceinline__ uint16_t round(float f) { return __half_as_ushort(__float2half_rn(f)); }
    static constexpr uint32_t fmt = 0; // instruction-descriptor operand format: F16
};
template <> struct H16<__nv_bfloat16> {
    static __device__ __forceinline__ float one(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }
    static __device__ __forceinline__ uint16_t round(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }
    static constexpr uint32_t fmt = 1; // BF16
};

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void fail(const MmaParams &p, int code)
{
    atomicCAS(p.status, 0, code);
    atomicExch(p.abort_flag, 1);
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count)
{
    asm volatile("mbarrier.init.shared.b64 [%0], %1;" ::"r"(smem_addr(b)), "r"(count));
}
__device__ __forceinline__ void mbar_init1(uint64_t *b) { mbar_init(b, 1); }


__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{ .reg .pred q; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 q, [%1], %2; "
                 "selp.u32 %0, 1, 0, q; }"
                 : "=r"(ok)
                 : "r"(smem_addr(b)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// bounded wait for the phase of the given parity; false after the wait limit
// or an abort.  A phase that has completed costs one try_wait.  Once the
// wait has to spin, the clock is read after every try_wait (each may suspend
// the thread for a while, so the limit holds however short it is) and the
// abort flag, an L2 read, after every 16th.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *b, uint32_t parity, const MmaParams &p)
{
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = gtimer();
    for (unsigned it = 1;; ++it) {
        if (mbar_try(b, parity)) return true;
        if (gtimer() - t0 > p.wait_ns) {
            fail(p, PI_DEV_TIMEOUT);
            return false;
        }
        if ((it & 15) == 0 && *(volatile int *)p.abort_flag) return false;
    }
}

// Bounded wait that ignores the abort flag: a CTA lets its own copies land
// before it exits, even after a failure elsewhere.  Copies land within
// microseconds; the limit only guards against a device that stopped.
constexpr unsigned long long kDrainNs = 100000000ull; // 100 ms

__device__ __forceinline__ bool mbar_drain(uint64_t *b, uint32_t parity, unsigned long long ns)
{
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = gtimer();
    for (;;) {
        if (mbar_try(b, parity)) return true;
        if (gtimer() - t0 > ns) return false;
    }
}

// Wait for `done` (committed by the MMA lane after its last MMA of a pass,
// whatever happened before): ignores the abort flag, so tensor memory is
// never read or freed while an MMA runs; a timeout past the MMA lane's own
// bounded waits is reported.
__device__ __forceinline__ bool mbar_settle(uint64_t *b, uint32_t parity, const MmaParams &p)
{
    if (mbar_drain(b, parity, p.wait_ns + kDrainNs)) return true;
    fail(p, PI_DEV_TIMEOUT);
    return false;
}

// End of a kernel, producer lanes (iss >= 0, lane 0): complete every round of
// the full barriers (count NP each, one per producer; nst slots) up to the
// furthest stage any producer issued, then wait for the last round of each
// slot.  pub [NP] is shared memory; `gp` = the stages this producer issued.
// Every thread of the CTA must call it (it holds a CTA barrier).
template <int NP>
__device__ __forceinline__ void settle_producers(uint64_t *full, int nst, int *pub, int iss, int lane, uint32_t gp)
{
    if (iss >= 0 && lane == 0) pub[iss] = (int)gp;
    __syncthreads();
    if (iss < 0 || lane != 0) return;
    uint32_t gmax = 0;
    for (int i = 0; i < NP; ++i) gmax = max(gmax, (uint32_t)pub[i]);
    for (uint32_t g = gp; g < gmax; ++g) {
        const uint32_t st = g % (uint32_t)nst, r = g / (uint32_t)nst;
        // this producer saw round r - 2 of the slot complete (it issued or
        // filled in stage g - nst after it), so a parity wait here is exact
        if (r > 0) mbar_drain(full + st, (r - 1) & 1, kDrainNs);
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(full + st)) : "memory");
    }
    for (uint32_t g = gmax > (uint32_t)nst ? gmax - nst : 0u; g < gmax; ++g)
        mbar_drain(full + g % (uint32_t)nst, (g / (uint32_t)nst) & 1, kDrainNs);
}

// a = hi + lo to about twice the 16-bit precision: hi = round(a), lo =
// round(a - hi) (the difference is exact in fp32)
template <typename H>
__device__ __forceinline__ void split16(float a, uint16_t &hi, uint16_t &lo)
{
    hi = H::round(a);
    lo = H::round(a - H::one(hi));
}

// Position in a ring of n slots: slot s, and the parity ph of the slot's
// current round.  Advancing is an add and a compare; the role loops need no
// division per step.
struct Cur {
    uint32_t s, ph;
    __device__ __forceinline__ Cur(uint32_t g, uint32_t n) : s(g % n), ph((g / n) & 1u) {}
    __device__ __forceinline__ void next(uint32_t n)
    {
        if (++s == n) s = 0, ph ^= 1u;
    }
};

// shared-memory matrix descriptor, 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// instruction descriptor, kind::f16 with fp32 accumulation
__device__ __forceinline__ uint32_t idesc(uint32_t fmt, uint32_t a_mn, uint32_t b_mn, uint32_t M, uint32_t N)
{
    return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t acc)
{
    asm volatile("{ .reg .pred q; setp.ne.b32 q, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, q; }" ::"r"(
                     d_tmem),
                 "l"(a), "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t *b)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(b))
                 : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// TMEM columns: warp 0 allocates, everyone reads the base address after a barrier
__device__ __forceinline__ uint32_t tmem_alloc(uint32_t *slot, uint32_t ncols)
{
    if (threadIdx.x < 32) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
                     "r"(ncols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_before();
    __syncthreads();
    tc_after();
    return *(volatile uint32_t *)slot;
}

__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols)
{
    tc_before();
    __syncthreads();
    tc_after();
    if (threadIdx.x < 32)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

__device__ __forceinline__ int slice_at(int m, int c, int G) { return (int)(((long long)m * c) / G); }

__device__ __forceinline__ int list_len(const MmaParams &p, int n)
{
    int m = p.count ? *(volatile const int *)p.count : n;
    if (m < 0 || m > n) {
        if (threadIdx.x == 0) fail(p, PI_DEV_FLAG);
        m = 0;
    }
    return m;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void mbar_expect(uint64_t *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(b)), "r"(bytes) : "memory");
}

// rows r0..r3 (tensor-map row indices; out-of-range rows read as zeros) x 64
// columns from column `col` into 4 consecutive 128-byte rows at dst, swizzled
__device__ __forceinline__ void gather4(uint32_t dst, const CUtensorMap *tm, int col, int r0, int r1, int r2, int r3,
                                        uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
                 "l"(tm), "r"(smem_addr(bar)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

// a box of 64 columns x box-rows rows at (col, row)
__device__ __forceinline__ void tile_load(uint32_t dst, const CUtensorMap *tm, int col, int row, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
                     dst),
                 "l"(tm), "r"(smem_addr(bar)), "r"(col), "r"(row)
                 : "memory");
}

} // namespace
} // namespace pi
