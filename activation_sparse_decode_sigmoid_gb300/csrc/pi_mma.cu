// Tensor-core (tcgen05) path of the sparse FFN for batches of 2 to 64 tokens.
//
// PowerInfer (blog.csdn.net QbitAI/IPADS article, section "CPU/GPU混合推理设计";
// arXiv 2312.12456, section 5, neuron-aware operators): a batch computes the
// union of its tokens' predicted neurons, reading only those rows of W_up
// (W_gate) and W_down.  With B tokens every row read feeds B dot products, so
// from a few tokens up the work is a gather-GEMM:
//
//   U[i, t] = W_up[idx_i] . x_hat_t           (m x B, K = d_model)
//   A[i, t] = act(U[i, t] + b_i)  (ReGLU: relu(W_gate[idx_i] . x_hat_t + b_i) * U[i, t])
//   Y[t, :] = sum_i A[i, t] * W_down^T[idx_i, :]   (+ b_down)
//
// Two kernels, both on tcgen05 with the accumulators in tensor memory:
//   ffn_up_mma    neuron-parallel: SM c takes the equal slice [s0, s1) of the
//                 list, up to 256 gathered rows per pass (TMA tile::gather4,
//                 128-byte swizzle), D = W_rows (two M = 128 tiles, K-major) x X_hat^T
//                 (N = B rounded up to 16, K-major), K = d_model in steps of
//                 64; the epilogue applies the activation and writes A^T
//                 [B][m] as two parts in the weights' 16-bit type, hi =
//                 round(a) and lo = round(a - hi) (the product of a 16-bit
//                 GEMM takes both operands in one type; the two parts carry a
//                 to about twice that precision).
//   ffn_down_mma  column blocks of 256 x shares of the list: D = W_down^T
//                 (M = 128 columns per tile, MN-major: 512-byte segments of
//                 the gathered rows, by gather4) x A^T (K-major: the hi rows,
//                 then the lo rows, N = 2 x B rounded up to 16, so each stage
//                 of rows is read once; the epilogue adds the two products),
//                 K = the share of the list in steps of 64 neurons; the
//                 epilogue adds b_down and writes y (16-bit) or adds into the
//                 fp32 residual x, or, when a block has several shares, fp32
//                 partials that ffn_merge adds in share order.
//   ffn_up_rows   up to 4 tokens, in place of ffn_up_mma: whole W_up / W_gate
//                 rows by bulk copy through a ring, dot products on the CUDA
//                 cores, the same A^T.
// Between the kernels A^T goes through global memory (m * B * 2 bytes, small
// next to the rows); stream order separates them.
//
// Shared-memory operand layouts are the canonical 128-byte-swizzle layouts:
// a "row" of 128 bytes (64 16-bit elements) at 128-byte pitch, 16-byte chunk
// c of row r stored at chunk c ^ (r & 7), 8-row groups at 1024 bytes.
//
// Failure handling: every wait is bounded and also gives up once another CTA
// or launch has raised the abort flag.  A CTA that gives up still lets its
// own asynchronous work finish before it exits:
//   * the MMA lane always commits `done`, which every thread waits for
//     (bounded, ignoring the flag) before tensor memory is read or freed;
//   * a stage's full barrier counts one arrival per producer, so a producer
//     that stopped early would leave it incomplete forever.  At the end the
//     producers publish how many stages they issued; each one then arrives,
//     without copies, on the stages it skipped up to the furthest any of them
//     reached (stage by stage, each after the slot's previous round has
//     completed), and finally waits (bounded, ignoring the flag) for the last
//     round of every slot.  Rounds of a slot complete in order, so every
//     copy the CTA issued has then landed.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "pi_kernels.h"
#include "pi_tc.cuh"

namespace pi {
namespace {

constexpr int kIssuers = 11;                // TMA producer warps
constexpr int kMT = 32 * (kIssuers + 1);  // + the MMA warp; warps 0..3 (TMEM lanes 0..127) run the epilogues
constexpr uint32_t kTileA = 16384; // 128 rows x 128 bytes
constexpr uint32_t kTileX = 8192;  // up to 64 rows x 128 bytes
constexpr int kUpMaxSt = 9;        // stages of the up kernel, at most
constexpr uint32_t kUpArena = 9 * (kTileA + kTileX); // its stages: 216 KB (the same for ReGLU's 3 x 72 KB)

// TMA issue is split over the producer warps (one lane each): warp 0 and
// warps 2.. take every kIssuers-th load of a stage and each posts its own
// expected bytes on the stage's full barrier (kIssuers arrivals); warp 1
// issues the MMAs.  One lane issues TMA loads at a limited rate, so several
// are needed to keep enough bytes in flight.
__device__ __forceinline__ int issuer_index(int warp) { return warp == 0 ? 0 : (warp >= 2 ? warp - 1 : -1); }

// ------------------------------------------------------------------ up / gate kernel
// Rows of the SM's slice are taken up to RP = 128 at a time (one MMA tile),
// or up to 256 (two tiles sharing each K step) when the slice holds more than
// 128: a second pass over all of K for a few rows would cost nearly as much
// as the first.  Small stages leave room for more of them in shared memory:
// nine for ReLU, five for ReGLU, whose stages carry two matrices (five and
// three of 256 rows); more stages keep more bytes in flight.
// Warp 0 (one lane) produces: per stage, gather4 loads of the rows' next 64
// columns (W_up, W_gate) and a tile load of x_hat; warp 1 (one lane) issues
// the MMAs and commits each stage back to the producer; all four warps run
// the epilogue.  Rows past the slice are gathered from row n (out of range:
// zeros) or left stale; their accumulator rows are never read.
//
// up_passes: the passes of one CTA's slice with RP rows per pass (128 or 256)
// and as many stages as the arena holds.
template <typename T, bool REGLU, int RP>
__device__ __forceinline__ void up_passes(const MmaParams &p, uint8_t *smem, uint64_t *full, uint64_t *empty,
                                          uint64_t *done, int *sid, int *pub, uint32_t tmem, int m, int s0, int s1)
{
    using H = H16<T>;
    const LayerDev &L = *p.layer;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = L.d, n = L.n, B = p.B, Np = p.Npad;
    constexpr uint32_t kW = RP / 128 * kTileA; // RP rows x 128 bytes of one weight matrix
    constexpr uint32_t kStage = kW * (REGLU ? 2 : 1) + kTileX;
    constexpr uint32_t nst = kUpArena / kStage < (uint32_t)kUpMaxSt ? kUpArena / kStage : (uint32_t)kUpMaxSt;
    const int KT = (d + kBK - 1) / kBK;
    const uint32_t base = smem_addr(smem);
    const uint32_t id_up = idesc(H::fmt, 0, 0, 128, (uint32_t)Np);
    const int iss = issuer_index(warp);
    uint32_t gp = 0, gc = 0, pass = 0; // stages produced (by this producer lane) / consumed, passes
    bool ok = true;

    for (int r0 = s0; r0 < s1; r0 += RP, ++pass) {
        const int rows = min(RP, s1 - r0);
        const int ntile = (rows + 127) / 128;
        for (int r = tid; r < RP; r += kMT) {
            int id = n; // out of range: zeros
            if (r < rows) {
                id = p.idx ? p.idx[r0 + r] : r0 + r;
                if (id < 0 || id >= n) {
                    fail(p, PI_DEV_FLAG);
                    id = n;
                }
            }
            sid[r] = id;
        }
        __syncthreads();
        if (iss >= 0 && lane == 0) {
            const int nq = (rows + 3) / 4;
            const int mine = (nq - iss + kIssuers - 1) / kIssuers; // gathers q = iss, iss + kIssuers, ...
            const uint32_t bytes = (uint32_t)mine * 512u * (REGLU ? 2u : 1u) + (iss == 0 ? (uint32_t)Np * 128u : 0u);
            Cur cp(gp, nst);
            for (int kt = 0; kt < KT && ok; ++kt, ++gp, cp.next(nst)) {
                const uint32_t st = cp.s;
                if (gp >= nst && !mbar_wait_bounded(empty + st, cp.ph ^ 1u, p)) {
                    ok = false; // (nothing issued for this stage)
                    break;
                }
                const uint32_t sb = base + st * kStage;
                uint64_t *fb = full + st;
                mbar_expect(fb, bytes);
                for (int q = iss; q < nq; q += kIssuers) {
                    const int r = 4 * q;
                    const uint32_t dst = sb + (uint32_t)(r >> 7) * kTileA + (uint32_t)(r & 127) * 128u;
                    gather4(dst, &p.tm_up, kt * kBK, sid[r], sid[r + 1], sid[r + 2], sid[r + 3], fb);
                    if (REGLU) gather4(dst + kW, &p.tm_gate, kt * kBK, sid[r], sid[r + 1], sid[r + 2], sid[r + 3], fb);
                }
                if (iss == 0) tile_load(sb + kW * (REGLU ? 2 : 1), &p.tm_x, kt * kBK, 0, fb);
            }
        } else if (warp == 1 && lane == 0) {
            // descriptors of stage 0; a byte offset o adds o / 16 (the start address field)
            const uint64_t d0 = sdesc(base, 16, 1024);
            Cur cc(gc, nst);
            for (int kt = 0; kt < KT && ok; ++kt, ++gc, cc.next(nst)) {
                if (!mbar_wait_bounded(full + cc.s, cc.ph, p)) {
                    ok = false;
                    break;
                }
                tc_after();
                const uint64_t ds = d0 + ((cc.s * kStage) >> 4);
                const uint64_t bx0 = ds + ((kW * (REGLU ? 2u : 1u)) >> 4);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k) {
                    for (int j = 0; j < ntile; ++j) {
                        const uint64_t a = ds + ((j * kTileA) >> 4) + 2 * k;
                        mma(tmem + (uint32_t)(j * Np), a, bx0 + 2 * k, id_up, (kt | k) != 0);
                        if (REGLU)
                            mma(tmem + (uint32_t)((2 + j) * Np), a + (kW >> 4), bx0 + 2 * k, id_up, (kt | k) != 0);
                    }
                }
                mma_commit(empty + cc.s);
            }
            mma_commit(done); // always: the MMAs issued so far complete before `done` flips
        }
        __syncwarp(); // (gp lives in the producer lane, gc in the MMA lane)
        const bool settled = mbar_settle(done, pass & 1, p);
        tc_after();
        // epilogue (warps 0..3): thread = row r of tile j (TMEM lane), 16 token columns at a time
        const bool live = ok && settled && !*(volatile int *)p.abort_flag;
        for (int j = 0; j < ntile && warp < 4; ++j) { // (tcgen05.ld is warp-wide: no per-thread condition here)
            const int r = j * 128 + warp * 32 + lane;
            const int id = sid[r];
            float bias = 0.f;
            if (id < n)
                bias = L.bias_tail ? H::one(*reinterpret_cast<const uint16_t *>(L.up + (size_t)id * L.upB + L.rowB))
                                   : H::one(L.b[id]);
            const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
            for (int c0 = 0; c0 < Np; c0 += 16) {
                float u[16], gt[16];
                tmem_ld16(lane_addr + (uint32_t)(j * Np + c0), u);
                if (REGLU) tmem_ld16(lane_addr + (uint32_t)((2 + j) * Np + c0), gt);
                if (r < rows && live) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int t = c0 + jj;
                        if (t < B) {
                            const float rl = fmaxf((REGLU ? gt[jj] : u[jj]) + bias, 0.f);
                            const float a = REGLU ? rl * u[jj] : (L.act == ACT_SQRELU ? rl * rl : rl);
                            uint16_t hi, lo;
                            split16<H>(id < n ? a : 0.f, hi, lo);
                            p.actT[(size_t)t * p.mstride + r0 + r] = hi;
                            p.actL[(size_t)t * p.mstride + r0 + r] = lo;
                        }
                    }
                }
            }
        }
        tc_before();
        __syncthreads(); // TMEM and sid are reused by the next pass
        tc_after();
    }
    // the list's tail up to a whole 64-neuron step reads as zeros in the down kernel
    if (blockIdx.x == gridDim.x - 1) {
        const int mp = (m + kBK - 1) / kBK * kBK;
        for (int q = tid; q < (mp - m) * B; q += kMT) {
            const int t = q / (mp - m), i = m + q % (mp - m);
            p.actT[(size_t)t * p.mstride + i] = 0;
            p.actL[(size_t)t * p.mstride + i] = 0;
        }
    }
    // no copy of this CTA may be in flight when it exits
    settle_producers<kIssuers>(full, (int)nst, pub, iss, lane, gp);
}

template <typename T, bool REGLU>
__global__ void __launch_bounds__(kMT, 1) ffn_up_mma(const __grid_constant__ MmaParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const LayerDev &L = *p.layer;
    const int tid = threadIdx.x;
    const int n = L.n;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kUpArena); // [kUpMaxSt], one arrival per producer
    uint64_t *empty = full + kUpMaxSt;
    uint64_t *done = empty + kUpMaxSt;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    int *sid = reinterpret_cast<int *>(tslot + 4); // [256] row ids of the current pass
    int *pub = sid + 256;                          // [kIssuers] stages each producer issued
    if (tid == 0) {
        for (int s = 0; s < kUpMaxSt; ++s) mbar_init(full + s, kIssuers), mbar_init1(empty + s);
        mbar_init1(done);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // TMEM: tile j (0, 1) of U at columns [j Np, (j+1) Np), of the gate at [(2+j) Np, ...)
    const uint32_t tmem = tmem_alloc(tslot, 256);
    pdl_enter(); // (the barriers and tensor memory above were set up while the list was finished)
    const int m = list_len(p, n);
    const int s0 = slice_at(m, blockIdx.x, gridDim.x), s1 = slice_at(m, blockIdx.x + 1, gridDim.x);
    // a slice of more than 128 rows runs in passes of up to 256 (two MMA tiles
    // per K step) rather than a second pass of a few rows; its stages are
    // twice as large, so fewer of them fit in the arena
    if (s1 - s0 > 128) up_passes<T, REGLU, 256>(p, smem, full, empty, done, sid, pub, tmem, m, s0, s1);
    else up_passes<T, REGLU, 128>(p, smem, full, empty, done, sid, pub, tmem, m, s0, s1);
    tmem_free(tmem, 256);
}

// ------------------------------------------------------------------ up / gate kernel, few tokens
// For a few tokens the rows are streamed whole instead: each neuron's W_up
// row (with its bias tail) and W_gate row arrive by bulk copies into one
// stage of a ring, and a consumer warp computes the neuron's dot products
// with every token's x_hat (shared memory) on the CUDA cores, then the
// activation, written to A^T (hi and lo parts) as the tensor-core kernel
// writes it.  A 4-row
// gather per TMA instruction limits that kernel at small batches; here one
// bulk copy brings a whole row and the ring holds many neurons.
// Every stage slot has one consumer warp, which takes the slot's stages in
// order, so it never waits on a slot more than one phase ahead (a parity
// wait cannot tell phase j from phase j + 2): with nst slots, W = nst warps
// when nst <= 16, else W = 16 and nst a multiple of 16; warp w takes the
// SM's neurons w, w + W, w + 2W, ...
constexpr int kRowWarps = 16;               // consumer warps
constexpr int kRowT = 32 * (kRowWarps + 1); // + the producer warp
constexpr int kRowMaxB = 4;                 // tokens up to which the row kernel runs
constexpr int kRowMinStages = 6;            // fewer stages than this: the tensor-core kernel

__device__ __forceinline__ void cp16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void bulk_row(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
                 "%4;" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_one(uint64_t *b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}

__device__ __forceinline__ uint4 lds16(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// c + the eight products of a 16-bit chunk pair, in element order (the
// mixed-precision fma multiplies the exactly widened operands, rounds once)
template <typename T> __device__ __forceinline__ float fma8(const uint4 &w, const uint4 &x, float c);
template <> __device__ __forceinline__ float fma8<__half>(const uint4 &w, const uint4 &x, float c)
{
    const uint32_t a[4] = {w.x, w.y, w.z, w.w}, b[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;"
            " fma.rn.f32.f16 %0, al, bl, %0; fma.rn.f32.f16 %0, ah, bh, %0; }"
            : "+f"(c)
            : "r"(a[i]), "r"(b[i]));
    return c;
}
template <> __device__ __forceinline__ float fma8<__nv_bfloat16>(const uint4 &w, const uint4 &x, float c)
{
    const uint32_t a[4] = {w.x, w.y, w.z, w.w}, b[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{ .reg .b16 al, ah, bl, bh; mov.b32 {al, ah}, %1; mov.b32 {bl, bh}, %2;"
            " fma.rn.f32.bf16 %0, al, bl, %0; fma.rn.f32.bf16 %0, ah, bh, %0; }"
            : "+f"(c)
            : "r"(a[i]), "r"(b[i]));
    return c;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// shared memory of the row kernel: x_hat [B][d], then nst stages of stageB, then 2 nst mbarriers
__host__ __device__ inline uint32_t row_xs_bytes(int B, int d) { return ((uint32_t)B * d * 2 + 127u) / 128u * 128u; }

template <typename T, bool REGLU>
__global__ void __launch_bounds__(kRowT, 1) ffn_up_rows(const __grid_constant__ MmaParams p, int nst, uint32_t stageB)
{
    extern __shared__ __align__(128) uint8_t smem[];
    using H = H16<T>;
    const LayerDev &L = *p.layer;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = L.d, n = L.n, B = p.B;
    const uint32_t xs = smem_addr(smem);
    const uint32_t ring = xs + row_xs_bytes(B, d);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + row_xs_bytes(B, d) + (size_t)nst * stageB);
    uint64_t *empty = full + nst;
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) mbar_init1(full + s), mbar_init1(empty + s);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_enter(); // (the barriers above were set up while the list was finished)
    const int m = list_len(p, n);
    const int s0 = slice_at(m, blockIdx.x, gridDim.x), cnt = slice_at(m, blockIdx.x + 1, gridDim.x) - s0;
    const uint32_t upB = (uint32_t)L.upB, rowB = (uint32_t)L.rowB;
    if (warp == kRowWarps) {
        // producer: the slice's rows in list order, one neuron per stage
        if (lane == 0) {
            const uint64_t pol = []() {
                uint64_t q;
                asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(q));
                return q;
            }();
            int k = 0;
            for (; k < cnt; ++k) {
                const int st = k % nst;
                if (*(volatile const int *)p.abort_flag) break; // (consumers stop waiting for stages)
                if (k >= nst && !mbar_wait_bounded(empty + st, ((k / nst) - 1) & 1, p)) break;
                const int id = p.idx ? __ldg(p.idx + s0 + k) : s0 + k;
                const bool v = id >= 0 && id < n; // (a bad id is flagged by its consumer)
                mbar_expect(full + st, v ? upB + (REGLU ? rowB : 0u) : 0u);
                if (v) {
                    const uint32_t dst = ring + (uint32_t)st * stageB;
                    bulk_row(dst, L.up + (size_t)id * upB, upB, full + st, pol);
                    if (REGLU) bulk_row(dst + upB, L.gate + (size_t)id * rowB, rowB, full + st, pol);
                }
            }
            // no copy may still be in flight when the CTA exits
            for (int j = max(0, k - nst); j < k; ++j) mbar_drain(full + j % nst, (j / nst) & 1, kDrainNs);
        }
        return;
    }
    // consumers: every token's x_hat into shared memory (rows are 16-byte multiples)
    for (int q = tid; q < B * (d >> 3); q += kRowWarps * 32) {
        const int t = q / (d >> 3), ch = q % (d >> 3);
        cp16(xs + (uint32_t)(t * d + ch * 8) * 2, p.xhat + (size_t)t * d + ch * 8, 16u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    asm volatile("bar.sync 1, %0;" ::"n"(kRowWarps * 32) : "memory");
    const int nch = d >> 3;
    const int W = nst < kRowWarps ? nst : kRowWarps; // (nst: a multiple of kRowWarps from kRowWarps up)
    for (int k = warp; k < cnt && warp < W; k += W) {
        const int st = k % nst, pos = s0 + k;
        const int id = p.idx ? __ldg(p.idx + pos) : pos;
        const bool v = id >= 0 && id < n;
        if (!v && lane == 0) fail(p, PI_DEV_FLAG);
        const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(full + st, (k / nst) & 1, p));
        float au[kRowMaxB], ag[kRowMaxB];
#pragma unroll
        for (int t = 0; t < kRowMaxB; ++t) au[t] = ag[t] = 0.f;
        const uint32_t a = ring + (uint32_t)st * stageB;
        if (ok && v) {
            for (int ch = lane; ch < nch; ch += 32) {
                const uint4 wu = lds16(a + (uint32_t)ch * 16);
                uint4 wg = make_uint4(0, 0, 0, 0);
                if (REGLU) wg = lds16(a + upB + (uint32_t)ch * 16);
#pragma unroll
                for (int t = 0; t < kRowMaxB; ++t)
                    if (t < B) {
                        const uint4 xv = lds16(xs + (uint32_t)(t * d + ch * 8) * 2);
                        au[t] = fma8<T>(wu, xv, au[t]);
                        if (REGLU) ag[t] = fma8<T>(wg, xv, ag[t]);
                    }
            }
        }
        float bias = 0.f;
        if (ok && v)
            bias = L.bias_tail ? H::one(*reinterpret_cast<const uint16_t *>(smem + (a - xs) + rowB)) : H::one(L.b[id]);
#pragma unroll
        for (int t = 0; t < kRowMaxB; ++t) {
            au[t] = warp_sum(au[t]);
            if (REGLU) ag[t] = warp_sum(ag[t]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_one(empty + st); // the stage's rows are no longer read
        if (lane < B && lane < kRowMaxB && ok) {
            float u = 0.f, g = 0.f;
#pragma unroll
            for (int t = 0; t < kRowMaxB; ++t)
                if (t == lane) u = au[t], g = ag[t];
            const float rl = fmaxf((REGLU ? g : u) + bias, 0.f);
            const float av = REGLU ? rl * u : (L.act == ACT_SQRELU ? rl * rl : rl);
            uint16_t hi, lo;
            split16<H>(v ? av : 0.f, hi, lo);
            p.actT[(size_t)lane * p.mstride + pos] = hi;
            p.actL[(size_t)lane * p.mstride + pos] = lo;
        }
    }
    // the list's tail up to a whole 64-neuron step reads as zeros in the down kernel
    if (blockIdx.x == gridDim.x - 1) {
        const int mp = (m + kBK - 1) / kBK * kBK;
        for (int q = tid; q < (mp - m) * B; q += kRowWarps * 32) {
            const int t = q / (mp - m), i = m + q % (mp - m);
            p.actT[(size_t)t * p.mstride + i] = 0;
            p.actL[(size_t)t * p.mstride + i] = 0;
        }
    }
}

// ------------------------------------------------------------------ down kernel
// Work unit u = (256-column block cb, share ks of the list).  For each of the
// block's two 128-column tiles, D[128 columns x Np tokens] = W_down^T (MN-
// major A: per stage 64 neurons x 256 columns, four 64-column atoms filled by
// gather4) x A^T (K-major B: tile loads of tokens x 64 neurons, the hi part
// then the lo part, one operand of 2 Np rows; the epilogue adds the two
// halves of the accumulator).  When the list is
// split over several shares, the units write fp32 partials that ffn_merge
// adds in share order; with one share the unit writes y or x.  A stage holds
// 32 KB of rows and 2 x Np x 128 bytes of A^T: nst stages, as many as fit.
constexpr uint32_t kDnAtom = 8192;        // 64 neurons x 64 columns (128 bytes)
constexpr uint32_t kDnW = 4 * kDnAtom;    // 64 neurons x 256 columns
__host__ __device__ constexpr uint32_t dn_stage_bytes(int Np) { return kDnW + 2u * (uint32_t)Np * 128u; }
__host__ __device__ constexpr int dn_fixed_bytes() { return 16 + kIssuers * 65 * 4; }
__host__ __device__ constexpr int dn_smem_bytes(int Np, int nst)
{
    return nst * (int)dn_stage_bytes(Np) + (2 * nst + 1) * 8 + dn_fixed_bytes();
}

template <typename T>
__global__ void __launch_bounds__(kMT, 1) ffn_down_mma(const __grid_constant__ MmaParams p, int nks, int nst)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    using H = H16<T>;
    const LayerDev &L = *p.layer;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = L.d, n = L.n, B = p.B, Np = p.Npad;
    const uint32_t kX = (uint32_t)Np * 128u; // one A^T part of a stage
    const uint32_t kStage = dn_stage_bytes(Np);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)nst * kStage); // one arrival per producer
    uint64_t *empty = full + nst;
    uint64_t *done = empty + nst;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    int *sidd = reinterpret_cast<int *>(tslot + 4); // [kIssuers][64] ids of the stage each producer is on
    int *pub = sidd + kIssuers * 64;                 // [kIssuers] stages each producer issued
    if (tid == 0) {
        for (int s = 0; s < nst; ++s) mbar_init(full + s, kIssuers), mbar_init1(empty + s);
        mbar_init1(done);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // tile j at columns [2 j Np, 2 (j+1) Np): the product with the hi rows, then with the lo rows
    const uint32_t tmem = tmem_alloc(tslot, 256);
    pdl_enter(); // (the barriers and tensor memory above were set up while the up kernel finished)
    const int m = list_len(p, n);
    const int KTall = (m + kBK - 1) / kBK;
    const int ncb = (d + 255) / 256;
    const uint32_t base = smem_addr(smem);
    // one MMA per (k, tile) against the hi and lo rows together (N = 2 Np, the
    // lo part follows the hi part in the stage), so the rows are read once
    const uint32_t id_dn = idesc(H::fmt, 1, 0, 128, 2u * (uint32_t)Np);
    const int iss = issuer_index(warp);
    // 64 gathers per stage (4 column atoms x 16 groups of 4 neurons): g = iss, iss + kIssuers, ...
    const uint32_t bytes = (uint32_t)((64 - iss + kIssuers - 1) / kIssuers) * 512u + (iss == 0 ? 2u * kX : 0u);
    int *myids = sidd + (iss < 0 ? 0 : iss) * 64;
    uint32_t gp = 0, gc = 0, pass = 0;
    bool ok = true;

    for (int u = blockIdx.x; u < ncb * nks; u += gridDim.x, ++pass) {
        const int cb = u / nks, ks = u % nks;
        const int c0 = cb * 256;
        const int k_lo = slice_at(KTall, ks, nks), KT = slice_at(KTall, ks + 1, nks) - k_lo;
        if (iss >= 0) {
            // the list entries of stage kt (two per lane), fetched three stages
            // ahead so that the gathers never wait for the list itself
            const auto fetch = [&](int kt, int h) {
                const int pos = (k_lo + kt) * kBK + lane + 32 * h;
                return kt < KT && pos < m ? (p.idx ? __ldg(p.idx + pos) : pos) : n;
            };
            int f0[2], f1[2], f2[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) f0[h] = fetch(0, h), f1[h] = fetch(1, h), f2[h] = fetch(2, h);
            Cur cp(gp, nst);
            for (int kt = 0; kt < KT; ++kt) {
                const uint32_t st = cp.s;
                const int k0 = (k_lo + kt) * kBK;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    int id = f0[h]; // past the list: n, i.e. zeros (their A^T entries are 0, but 0 x garbage could be NaN)
                    if (id < 0 || id >= n) id = n; // flagged by the up kernel
                    myids[lane + 32 * h] = id;
                    f0[h] = f1[h];
                    f1[h] = f2[h];
                    f2[h] = fetch(kt + 3, h);
                }
                __syncwarp();
                if (lane == 0 && ok) {
                    if (gp >= (uint32_t)nst && !mbar_wait_bounded(empty + st, cp.ph ^ 1u, p)) ok = false;
                    if (ok) {
                        const uint32_t sb = base + st * kStage;
                        uint64_t *fb = full + st;
                        mbar_expect(fb, bytes);
                        for (int gi = iss; gi < 64; gi += kIssuers) {
                            const int a = gi >> 4, q = gi & 15;
                            gather4(sb + (uint32_t)a * kDnAtom + (uint32_t)q * 512u, &p.tm_dn, c0 + 64 * a,
                                    myids[4 * q], myids[4 * q + 1], myids[4 * q + 2], myids[4 * q + 3], fb);
                        }
                        if (iss == 0) {
                            tile_load(sb + kDnW, &p.tm_act, k0, 0, fb);
                            tile_load(sb + kDnW + kX, &p.tm_act_lo, k0, 0, fb);
                        }
                        ++gp; // (lane 0 counts the stages it issued)
                        cp.next(nst);
                    }
                }
                __syncwarp(); // myids is rewritten for the next stage
            }
        }
        if (warp == 1 && lane == 0) {
            // descriptors of stage 0; a byte offset o adds o / 16 (the start address field)
            const uint64_t dA = sdesc(base, kDnAtom, 1024), dB = sdesc(base + kDnW, 16, 1024);
            Cur cc(gc, nst);
            for (int kt = 0; kt < KT && ok; ++kt, ++gc, cc.next(nst)) {
                if (!mbar_wait_bounded(full + cc.s, cc.ph, p)) {
                    ok = false;
                    break;
                }
                tc_after();
                const uint64_t a0 = dA + ((cc.s * kStage) >> 4), b0 = dB + ((cc.s * kStage) >> 4);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k) {
#pragma unroll
                    for (int j = 0; j < 2; ++j) { // atoms 2j, 2j+1: LBO steps from one 64-column atom to the next
                        const uint64_t a = a0 + (uint64_t)((2 * j * kDnAtom + k * 16 * 128) >> 4);
                        mma(tmem + (uint32_t)(2 * j * Np), a, b0 + 2 * k, id_dn, (kt | k) != 0);
                    }
                }
                mma_commit(empty + cc.s);
            }
            mma_commit(done); // always: the MMAs issued so far complete before `done` flips
        }
        const bool settled = mbar_settle(done, pass & 1, p);
        tc_after();
        const bool live = ok && settled && !*(volatile int *)p.abort_flag;
        // epilogue: thread = output column (TMEM lane) of tile j, 16 tokens at a time
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        for (int j = 0; j < 2 && warp < 4; ++j) { // epilogue: warps 0..3
            const int c = c0 + j * 128 + warp * 32 + lane;
            const float bd = c < d ? H::one(L.bdown[c]) : 0.f;
            for (int t0 = 0; t0 < Np; t0 += 16) {
                float v[16], vl[16];
                if (KT > 0) {
                    tmem_ld16(lane_addr + (uint32_t)(2 * j * Np + t0), v);
                    tmem_ld16(lane_addr + (uint32_t)(2 * j * Np + Np + t0), vl);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += vl[i];
                } else
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                if (c < d && live) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int t = t0 + i;
                        if (t < B) {
                            if (nks > 1) p.part[((size_t)ks * B + t) * d + c] = v[i];
                            else if (p.x) p.x[(size_t)t * d + c] += v[i] + bd;
                            else p.y[(size_t)t * d + c] = H::round(v[i] + bd);
                        }
                    }
                }
            }
        }
        tc_before();
        __syncthreads();
        tc_after();
    }
    // no copy of this CTA may be in flight when it exits
    settle_producers<kIssuers>(full, nst, pub, iss, lane, gp);
    tmem_free(tmem, 256);
}

// y (or x +=) = the shares' partials added in share order, + b_down
template <typename T>
__global__ void ffn_merge(const __grid_constant__ MmaParams p, int nks)
{
    using H = H16<T>;
    pdl_enter();
    const LayerDev &L = *p.layer;
    const int d = L.d;
    const size_t total = (size_t)p.B * d;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int k = 0; k < nks; ++k) s += p.part[(size_t)k * total + i];
        s += H::one(L.bdown[i % d]);
        if (p.x) p.x[i] += s;
        else p.y[i] = H::round(s);
    }
}

template <typename T, bool REGLU>
cudaError_t launch_up(const MmaParams &p, int grid, cudaStream_t s)
{
    // the stage arena: nine 128-row stages for ReLU, five for ReGLU (whose
    // stages carry two matrices), or five / three of 256 rows; then
    // full[kUpMaxSt], empty[kUpMaxSt], done, the TMEM slot (16 bytes), the row
    // ids [256] and the producers' stage counts [kIssuers]
    const int smem = (int)kUpArena + (2 * kUpMaxSt + 1) * 8 + 16 + 256 * 4 + kIssuers * 4;
    auto kern = ffn_up_mma<T, REGLU>;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kMT), smem, s, p);
}

// The row kernel for up to kRowMaxB tokens when its ring holds kRowMinStages
// neurons or more; returns cudaErrorNotSupported otherwise.
template <typename T, bool REGLU>
cudaError_t launch_up_rows(const MmaParams &p, int grid, int smem_optin, cudaStream_t s)
{
    if (p.B > kRowMaxB) return cudaErrorNotSupported;
    const uint32_t stageB = ((uint32_t)(p.d * 2 + 16) + (REGLU ? (uint32_t)p.d * 2 : 0u) + 127u) / 128u * 128u;
    const int fixed = (int)row_xs_bytes(p.B, p.d);
    int nst = std::min(32, (smem_optin - fixed - 2 * 32 * 8) / (int)stageB);
    if (nst < kRowMinStages) return cudaErrorNotSupported;
    if (nst > kRowWarps) nst = nst / kRowWarps * kRowWarps; // one consumer warp per slot
    const int smem = fixed + nst * (int)stageB + 2 * nst * 8;
    auto kern = ffn_up_rows<T, REGLU>;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kRowT), smem, s, p, nst, stageB);
}

template <typename T>
cudaError_t launch_down(const MmaParams &p, int grid, int smem_optin, cudaStream_t s)
{
    // as many stages as shared memory holds (at most 6): 4 at 64 tokens, 6 at 16
    int st = 6;
    while (st > 2 && dn_smem_bytes(p.Npad, st) > smem_optin) --st;
    const int smem = dn_smem_bytes(p.Npad, st);
    if (smem > smem_optin) return cudaErrorInvalidValue;
    auto kern = ffn_down_mma<T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // as many shares of the list per 256-column block as keep every SM busy with one unit
    const int ncb = (p.d + 255) / 256;
    const int nks = grid / ncb > 8 ? 8 : (grid / ncb < 1 ? 1 : grid / ncb);
    const int units = ncb * nks;
    e = launch_pdl(kern, dim3(units < grid ? units : grid), dim3(kMT), smem, s, p, nks, st);
    if (e != cudaSuccess || nks == 1) return e;
    return launch_pdl(ffn_merge<T>, dim3(grid * 4), dim3(256), 0, s, p, nks);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

} // namespace

cudaError_t encode_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                       uint32_t box_rows)
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f) return e != cudaSuccess ? e : cudaErrorNotSupported;
        fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_ffn_merge(const MmaParams &p, bool bf16, int nks, int grid, cudaStream_t s)
{
    return bf16 ? launch_pdl(ffn_merge<__nv_bfloat16>, dim3(grid * 4), dim3(256), 0, s, p, nks)
                : launch_pdl(ffn_merge<__half>, dim3(grid * 4), dim3(256), 0, s, p, nks);
}

cudaError_t launch_ffn_mma(const MmaParams &p, bool bf16, bool reglu, int grid, cudaStream_t s)
{
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    // a few tokens: whole rows on the CUDA cores, if the ring holds enough neurons
    if (bf16) e = reglu ? launch_up_rows<__nv_bfloat16, true>(p, grid, optin, s)
                        : launch_up_rows<__nv_bfloat16, false>(p, grid, optin, s);
    else e = reglu ? launch_up_rows<__half, true>(p, grid, optin, s) : launch_up_rows<__half, false>(p, grid, optin, s);
    if (e == cudaErrorNotSupported) {
        if (bf16) e = reglu ? launch_up<__nv_bfloat16, true>(p, grid, s) : launch_up<__nv_bfloat16, false>(p, grid, s);
        else e = reglu ? launch_up<__half, true>(p, grid, s) : launch_up<__half, false>(p, grid, s);
    }
    if (e != cudaSuccess) return e;
    return bf16 ? launch_down<__nv_bfloat16>(p, grid, optin, s) : launch_down<__half>(p, grid, optin, s);
}

} // namespace pi
