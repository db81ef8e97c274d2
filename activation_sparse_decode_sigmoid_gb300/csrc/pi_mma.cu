// Tensor-core (tcgen05) path of the sparse FFN for batches of 8 to 64 tokens.
//
// PowerInfer (blog.csdn.net QbitAI/IPADS article, section "CPU/GPU混合推理设计";
// arXiv 2312.12456, section 5, neuron-aware operators): a batch computes the
// union of its tokens' predicted neurons, reading only those rows of W_up
// (W_gate) and W_down.  With B tokens every row read feeds B dot products, so
// from 8 tokens up the work is a gather-GEMM:
//
//   U[i, t] = W_up[idx_i] . x_hat_t           (m x B, K = d_model)
//   A[i, t] = act(U[i, t] + b_i)  (ReGLU: relu(W_gate[idx_i] . x_hat_t + b_i) * U[i, t])
//   Y[t, :] = sum_i A[i, t] * W_down^T[idx_i, :]   (+ b_down)
//
// Two kernels, both on tcgen05 with the accumulators in tensor memory:
//   ffn_up_mma    neuron-parallel: SM c takes the equal slice [s0, s1) of the
//                 list, gathers 128 rows at a time (cp.async, 128-byte
//                 swizzle), D = W_rows (M = 128, K-major) x X_hat^T (N = B
//                 rounded up to 16, K-major), K = d_model in steps of 64;
//                 the epilogue applies the activation and writes A^T [B][m]
//                 rounded to the weights' 16-bit type (the product of a
//                 16-bit GEMM takes both operands in one type).
//   ffn_down_mma  column-parallel: SM c owns 64-column tiles of the output,
//                 D = A^T (M = 128 token rows, zero past B, K-major) x
//                 W_down^T rows (N = 64 columns, MN-major), K = the list in
//                 steps of 64 neurons; the epilogue adds b_down and writes y
//                 (16-bit) or adds into the fp32 residual x.  Every output
//                 column has one owner: no split-K partials, no merge.
// Between the two kernels A^T goes through global memory (m * B * 2 bytes,
// small next to the rows); stream order separates them.
//
// Shared-memory operand layouts are the canonical 128-byte-swizzle layouts:
// a "row" of 128 bytes (64 16-bit elements) at 128-byte pitch, 16-byte chunk
// c of row r stored at chunk c ^ (r & 7), 8-row groups at 1024 bytes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pi_kernels.h"

namespace pi {
namespace {

constexpr int kMT = 128;      // threads per CTA (4 warps: TMEM lanes 0..127)
constexpr int kStages = 4;    // pipeline depth
constexpr int kBK = 64;       // K elements per stage (one 128-byte row)
constexpr uint32_t kTileA = 16384; // 128 rows x 128 bytes
constexpr uint32_t kTileX = 8192;  // up to 64 rows x 128 bytes

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

// byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled tile
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk)
{
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((chunk ^ (row & 7u)) << 4);
}

// 16-byte global -> shared copy; n = 0 writes zeros and reads nothing
__device__ __forceinline__ void cp16(uint32_t dst, const void *src, uint32_t n)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void mbar_init1(uint64_t *b)
{
    asm volatile("mbarrier.init.shared.b64 [%0], 1;" ::"r"(smem_addr(b)));
}

// bounded wait for the phase of the given parity; false after the wait limit or an abort
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *b, uint32_t parity, const MmaParams &p)
{
    const uint64_t t0 = gtimer();
    for (unsigned it = 0;; ++it) {
        uint32_t ok;
        asm volatile("{ .reg .pred q; mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 q, [%1], %2; "
                     "selp.u32 %0, 1, 0, q; }"
                     : "=r"(ok)
                     : "r"(smem_addr(b)), "r"(parity)
                     : "memory");
        if (ok) return true;
        if ((it & 15) == 15) {
            if (*(volatile int *)p.abort_flag) return false;
            if (gtimer() - t0 > p.wait_ns) {
                fail(p, PI_DEV_TIMEOUT);
                return false;
            }
        }
    }
}

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

// ------------------------------------------------------------------ up / gate kernel
template <typename T, bool REGLU>
__global__ void __launch_bounds__(kMT, 1) ffn_up_mma(const MmaParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    using H = H16<T>;
    const LayerDev &L = *p.layer;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = L.d, n = L.n, B = p.B, Np = p.Npad;
    constexpr uint32_t kStage = kTileA * (REGLU ? 2 : 1) + kTileX;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kStages * kStage); // [kStages] MMA done per stage
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + kStages);
    int *sid = reinterpret_cast<int *>(tslot + 4); // [128] row ids of the current tile
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init1(bar + s);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const uint32_t tmem = tmem_alloc(tslot, 128); // U at columns [0, Np), gate at [Np, 2 Np)
    const int m = list_len(p, n);
    const int s0 = slice_at(m, blockIdx.x, gridDim.x), s1 = slice_at(m, blockIdx.x + 1, gridDim.x);
    const int KT = (d + kBK - 1) / kBK;
    const uint32_t base = smem_addr(smem);
    const uint32_t id_up = idesc(H::fmt, 0, 0, 128, (uint32_t)Np);
    uint32_t g = 0; // stages consumed so far by this CTA (ring position and mbarrier phase)
    bool ok = true;

    // rows padded beyond d read nothing (zeros)
    auto load = [&](uint32_t st, int kt) {
        const uint32_t sbase = base + st * kStage;
        const int col = kt * kBK;
#pragma unroll
        for (int i = 0; i < 8; ++i) { // 128 rows x 8 chunks of W_up (and W_gate)
            const int q = tid + i * kMT, r = q >> 3, ch = q & 7;
            const int id = sid[r];
            const int c = col + ch * 8;
            const bool v = id >= 0 && c < d;
            const uint8_t *src = v ? L.up + (size_t)id * L.upB + (size_t)c * 2 : L.up;
            cp16(sbase + sw128(r, ch), src, v ? 16u : 0u);
            if (REGLU) {
                const uint8_t *sg = v ? L.gate + (size_t)id * L.rowB + (size_t)c * 2 : L.gate;
                cp16(sbase + kTileA + sw128(r, ch), sg, v ? 16u : 0u);
            }
        }
        for (int q = tid; q < Np * 8; q += kMT) { // x_hat rows (tokens) x 8 chunks
            const int t = q >> 3, ch = q & 7, c = col + ch * 8;
            const bool v = t < B && c < d;
            const uint16_t *src = v ? p.xhat + (size_t)t * d + c : p.xhat;
            cp16(sbase + kTileA * (REGLU ? 2 : 1) + sw128(t, ch), src, v ? 16u : 0u);
        }
    };

    for (int r0 = s0; r0 < s1; r0 += 128) {
        const int rows = min(128, s1 - r0);
        {
            int id = -1;
            if (tid < rows) {
                id = p.idx ? p.idx[r0 + tid] : r0 + tid;
                if (id < 0 || id >= n) {
                    fail(p, PI_DEV_FLAG);
                    id = -1;
                }
            }
            sid[tid] = id;
        }
        __syncthreads();
        // prologue: stages 0 .. kStages-2
        for (int s = 0; s < kStages - 1; ++s) {
            if (s < KT) load((g + s) % kStages, s);
            cp_commit();
        }
        for (int kt = 0; kt < KT; ++kt) {
            const uint32_t st = (g + kt) % kStages;
            cp_wait<kStages - 2>(); // this thread's copies of stage kt have landed
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();        // ... and everyone's
            if (tid == 0) {
                tc_after();
                const uint32_t sb = base + st * kStage;
                const uint32_t xb = sb + kTileA * (REGLU ? 2 : 1);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k) {
                    const uint64_t bx = sdesc(xb + k * 32, 16, 1024);
                    mma(tmem, sdesc(sb + k * 32, 16, 1024), bx, id_up, (kt | k) != 0);
                    if (REGLU) mma(tmem + (uint32_t)Np, sdesc(sb + kTileA + k * 32, 16, 1024), bx, id_up, (kt | k) != 0);
                }
                mma_commit(bar + st);
            }
            // refill the stage that K-step kt-1 used, once its MMAs are done
            const int nk = kt + kStages - 1;
            if (nk < KT) {
                if (kt >= 1) {
                    const uint32_t gp = g + kt - 1;
                    if (ok && !mbar_wait_bounded(bar + gp % kStages, (gp / kStages) & 1, p)) ok = false;
                }
                load((g + nk) % kStages, nk);
            }
            cp_commit();
        }
        // the last commit covers every MMA of the tile
        {
            const uint32_t gl = g + KT - 1;
            if (ok && !mbar_wait_bounded(bar + gl % kStages, (gl / kStages) & 1, p)) ok = false;
        }
        // every stage's last use must be waited for once, so the phases stay in step
        for (int s = 0; s < kStages - 1 && s < KT - 1; ++s) {
            const uint32_t gp = g + KT - 2 - s;
            if (ok && !mbar_wait_bounded(bar + gp % kStages, (gp / kStages) & 1, p)) ok = false;
        }
        g += (uint32_t)KT;
        tc_after();
        // epilogue: thread = neuron row r of the tile (TMEM lane), 16 token columns at a time
        const int r = warp * 32 + lane;
        const int id = sid[r];
        float bias = 0.f;
        if (id >= 0)
            bias = L.bias_tail ? H::one(*reinterpret_cast<const uint16_t *>(L.up + (size_t)id * L.upB + L.rowB))
                               : H::one(L.b[id]);
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        for (int c0 = 0; c0 < Np; c0 += 16) {
            float u[16], gt[16];
            tmem_ld16(lane_addr + (uint32_t)c0, u);
            if (REGLU) tmem_ld16(lane_addr + (uint32_t)(Np + c0), gt);
            if (r < rows && ok) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int t = c0 + j;
                    if (t < B) {
                        const float a = REGLU ? fmaxf(gt[j] + bias, 0.f) * u[j] : fmaxf(u[j] + bias, 0.f);
                        p.actT[(size_t)t * p.mstride + r0 + r] = H::round(id >= 0 ? a : 0.f);
                    }
                }
            }
        }
        tc_before();
        __syncthreads(); // TMEM and sid are reused by the next tile
        tc_after();
    }
    // the list's tail up to a whole 64-neuron step reads as zeros in the down kernel
    if (blockIdx.x == gridDim.x - 1) {
        const int mp = (m + kBK - 1) / kBK * kBK;
        for (int q = tid; q < (mp - m) * B; q += kMT) {
            const int t = q / (mp - m), i = m + q % (mp - m);
            p.actT[(size_t)t * p.mstride + i] = 0;
        }
    }
    cp_wait<0>();
    tmem_free(tmem, 128);
}

// ------------------------------------------------------------------ down kernel
template <typename T>
__global__ void __launch_bounds__(kMT, 1) ffn_down_mma(const MmaParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    using H = H16<T>;
    const LayerDev &L = *p.layer;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = L.d, n = L.n, B = p.B;
    constexpr uint32_t kStage = kTileA + kTileX; // A^T rows (128 x 64 neurons) + W_down^T (64 neurons x 64 columns)
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + kStages * kStage);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + kStages);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init1(bar + s);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // token rows B..127 of every A^T stage stay zero
    for (int q = tid; q < kStages * (int)kTileA / 16; q += kMT) {
        const int s = q / ((int)kTileA / 16), o = q % ((int)kTileA / 16);
        const int row = (o * 16) / 128;
        if (row >= B) *reinterpret_cast<uint4 *>(smem + s * kStage + o * 16) = make_uint4(0, 0, 0, 0);
    }
    const uint32_t tmem = tmem_alloc(tslot, 64);
    const int m = list_len(p, n);
    const int KT = (m + kBK - 1) / kBK;
    const int ntile = (d + 63) / 64;
    const uint32_t base = smem_addr(smem);
    const uint32_t id_dn = idesc(H::fmt, 0, 1, 128, 64);
    uint32_t g = 0;
    bool ok = true;

    for (int tile = blockIdx.x; tile < ntile; tile += gridDim.x) {
        const int c0 = tile * 64;
        auto load = [&](uint32_t st, int kt) {
            const uint32_t sbase = base + st * kStage;
            const int k0 = kt * kBK;
            for (int q = tid; q < B * 8; q += kMT) { // A^T: token rows x 8 chunks of 8 neurons
                const int t = q >> 3, ch = q & 7;
                cp16(sbase + sw128(t, ch), p.actT + (size_t)t * p.mstride + k0 + ch * 8, 16u);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) { // W_down^T: 64 neuron rows x 8 chunks of 8 columns
                const int q = tid + i * kMT, j = q >> 3, ch = q & 7;
                const int pos = k0 + j, c = c0 + ch * 8;
                int id = -1;
                if (pos < m) {
                    id = p.idx ? p.idx[pos] : pos;
                    if (id < 0 || id >= n) id = -1; // flagged by the up kernel
                }
                const bool v = id >= 0 && c < d;
                const uint8_t *src = v ? L.dn + (size_t)id * L.rowB + (size_t)c * 2 : L.dn;
                cp16(sbase + kTileA + sw128(j, ch), src, v ? 16u : 0u);
            }
        };
        for (int s = 0; s < kStages - 1; ++s) {
            if (s < KT) load((g + s) % kStages, s);
            cp_commit();
        }
        for (int kt = 0; kt < KT; ++kt) {
            const uint32_t st = (g + kt) % kStages;
            cp_wait<kStages - 2>();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncthreads();
            if (tid == 0) {
                tc_after();
                const uint32_t sb = base + st * kStage;
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                    mma(tmem, sdesc(sb + k * 32, 16, 1024), sdesc(sb + kTileA + k * 16 * 128, 8192, 1024), id_dn,
                        (kt | k) != 0);
                mma_commit(bar + st);
            }
            const int nk = kt + kStages - 1;
            if (nk < KT) {
                if (kt >= 1) {
                    const uint32_t gp = g + kt - 1;
                    if (ok && !mbar_wait_bounded(bar + gp % kStages, (gp / kStages) & 1, p)) ok = false;
                }
                load((g + nk) % kStages, nk);
            }
            cp_commit();
        }
        if (KT > 0) {
            const uint32_t gl = g + KT - 1;
            if (ok && !mbar_wait_bounded(bar + gl % kStages, (gl / kStages) & 1, p)) ok = false;
            for (int s = 0; s < kStages - 1 && s < KT - 1; ++s) {
                const uint32_t gp = g + KT - 2 - s;
                if (ok && !mbar_wait_bounded(bar + gp % kStages, (gp / kStages) & 1, p)) ok = false;
            }
        }
        g += (uint32_t)KT;
        tc_after();
        // epilogue: thread = token row t (TMEM lane), 64 output columns
        const int t = warp * 32 + lane;
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        for (int j0 = 0; j0 < 64; j0 += 16) {
            float v[16];
            if (KT > 0) tmem_ld16(lane_addr + (uint32_t)j0, v);
            else
                for (int j = 0; j < 16; ++j) v[j] = 0.f;
            if (t < B && ok) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = c0 + j0 + j;
                    if (c < d) {
                        const float y = v[j] + H::one(L.bdown[c]);
                        if (p.x) p.x[(size_t)t * d + c] += y;
                        else p.y[(size_t)t * d + c] = H::round(y);
                    }
                }
            }
        }
        tc_before();
        __syncthreads();
        tc_after();
    }
    cp_wait<0>();
    tmem_free(tmem, 64);
}

template <typename T, bool REGLU>
cudaError_t launch_up(const MmaParams &p, int grid, cudaStream_t s)
{
    const int smem = kStages * (int)(kTileA * (REGLU ? 2 : 1) + kTileX) + 256 + 128 * 4;
    auto kern = ffn_up_mma<T, REGLU>;
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<grid, kMT, smem, s>>>(p);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_down(const MmaParams &p, int grid, cudaStream_t s)
{
    const int smem = kStages * (int)(kTileA + kTileX) + 256;
    auto kern = ffn_down_mma<T>;
    static bool configured = false;
    if (!configured) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    kern<<<grid, kMT, smem, s>>>(p);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_ffn_mma(const MmaParams &p, bool bf16, bool reglu, int grid, cudaStream_t s)
{
    cudaError_t e;
    if (bf16) e = reglu ? launch_up<__nv_bfloat16, true>(p, grid, s) : launch_up<__nv_bfloat16, false>(p, grid, s);
    else e = reglu ? launch_up<__half, true>(p, grid, s) : launch_up<__half, false>(p, grid, s);
    if (e != cudaSuccess) return e;
    const int ntile = (p.d + 63) / 64;
    const int gd = ntile < grid ? ntile : grid;
    return bf16 ? launch_down<__nv_bfloat16>(p, gd, s) : launch_down<__half>(p, gd, s);
}

} // namespace pi
