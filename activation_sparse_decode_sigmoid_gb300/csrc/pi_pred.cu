// Predictor of a batch of 2 to 64 tokens, as short launches per layer.
//
// PowerInfer (arXiv 2312.12456, section 5 "online predictors"; blog.csdn.net
// QbitAI/IPADS article, section "充分利用模型和硬件特点"): each layer's small
// MLP predicts which neurons a token fires, h = relu(W1 x_hat + b1) and
// neuron i active <=> sigmoid(W2 h + b2)_i > 0.5 <=> (W2 h + b2)_i > 0; a
// batch takes the union of its tokens' sets.  With B tokens every weight row
// feeds B dot products (at B = 64, 1.9 G multiply-adds per layer for the
// 29 M-weight output layer), so the work is arithmetic, not streaming: these
// kernels give each warp a register tile of R rows x TT tokens (TT = 2, 4 or
// 8 by batch size) and read every weight row from HBM once.
//
//   rmsnorm_rows  x_hat = RMSNorm(x), one CTA per token, in the step
//                 kernel's reduction order (the same bits)
//   pred_hidden   h = relu(W1 x_hat + b1), fp32 [B][r]: a CTA keeps one block
//                 of TT tokens' x_hat in shared memory; its warps stream R rows
//                 of W1 each from global memory, PD chunks ahead
//   pred_out      union mask words: a CTA owns 8R rows of W2, brought into
//                 shared memory by one bulk copy per warp, and streams the
//                 batch's h through in blocks of TT tokens; each CTA writes
//                 whole mask words (no atomics, nothing to clear first)
//   pred_compact  mask words -> ascending list + count (one CTA)
//
// Every dot product is CDOT: lane l of 32 accumulates chunks l, l+32, ... of
// 8 consecutive elements with correctly rounded fmas, then the 32 lane sums
// meet in the xor butterfly (16, 8, 4, 2, 1).  A lane here holds its lane
// sum of R x TT dot products and the warp combines them by a halving
// butterfly: each level exchanges half of the values and lane l keeps the
// half its bit selects, so every value still meets its partner lanes in the
// butterfly's order (fp32 addition is commutative): the same bits as one dot
// product per warp, and 62 shuffles instead of 320 for 64 values.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "pi_device.cuh"

namespace pi {
namespace {

constexpr int kPT = 256; // threads per CTA of the predictor kernels (8 warps)

__device__ __forceinline__ void cp16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void flag(const PredParams &p, int code)
{
    atomicCAS(p.status, 0, code);
    atomicExch(p.abort_flag, 1);
}

// bounded wait for a bulk copy; false after the wait limit or an abort (the
// clock after every try_wait that failed, the abort flag after every 16th)
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, const PredParams &p)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (unsigned it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > p.wait_ns) {
            flag(p, PI_DEV_TIMEOUT);
            return false;
        }
        if ((it & 15) == 0 && *(volatile int *)p.abort_flag) return false;
    }
}

// An earlier launch failed: read the flag once per CTA, so that every
// thread takes the same path (a CTA barrier follows).
__device__ __forceinline__ bool cta_aborted(const PredParams &p)
{
    __shared__ int a;
    if (threadIdx.x == 0) a = *(volatile int *)p.abort_flag;
    __syncthreads();
    return a != 0;
}

// Halving butterfly over the NV lane sums of a warp (NV a power of two):
// on return lane l holds the CDOT results of values base + j, j < max(NV/32, 1).
template <int C, int M, int NV>
__device__ __forceinline__ void halve(float (&v)[NV], int lane, int &base)
{
    if constexpr (M >= 1) {
        if constexpr (C > 1) {
            constexpr int H = C / 2;
            const bool hi = (lane & M) != 0;
#pragma unroll
            for (int j = 0; j < H; ++j) {
                const float keep = hi ? v[H + j] : v[j];
                const float send = hi ? v[j] : v[H + j];
                v[j] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, M));
            }
            if (hi) base += H;
            halve<H, M / 2, NV>(v, lane, base);
        } else {
            v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], M));
            halve<1, M / 2, NV>(v, lane, base);
        }
    }
}

// values a lane holds after the halving butterfly of NV values
__host__ __device__ constexpr int held(int nv) { return nv >= 32 ? nv / 32 : 1; }
// lanes that differ only in these bits hold the same values
__host__ __device__ constexpr int dup_mask(int nv) { return nv >= 32 ? 0 : 32 / nv - 1; }

// ------------------------------------------------------------------ RMSNorm
// Thread tid of 512 owns the float4 chunks tid + 512 q (q < 4) of the row;
// per-thread squares in chunk order, the warp butterfly, then the 16 warp
// sums in order: exactly the step kernel's x_hat.
template <typename T>
__global__ void __launch_bounds__(512) rmsnorm_rows(const PredParams p)
{
    using F = F16T<T>;
    __shared__ float part[16];
    __shared__ float inv_s;
    const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_enter();
    if (cta_aborted(p)) return;
    const int d = p.L.d, n4 = d / 4;
    const float4 *xr = reinterpret_cast<const float4 *>(p.x + (size_t)t * d);
    float4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int k = tid + q * 512;
        v[q] = k < n4 ? __ldcg(xr + k) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.tr_x && k < n4) reinterpret_cast<float4 *>(p.tr_x + (size_t)t * d)[k] = v[q];
    }
    float ss = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        ss = __fmaf_rn(v[q].x, v[q].x, ss);
        ss = __fmaf_rn(v[q].y, v[q].y, ss);
        ss = __fmaf_rn(v[q].z, v[q].z, ss);
        ss = __fmaf_rn(v[q].w, v[q].w, ss);
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, m));
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    if (tid == 0) {
        float tot = 0.f;
        for (int w = 0; w < 16; ++w) tot = __fadd_rn(tot, part[w]);
        inv_s = rsqrtf(__fadd_rn(__fdiv_rn(tot, (float)d), 1e-5f));
    }
    __syncthreads();
    const float inv = inv_s;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int k = tid + q * 512;
        if (k < n4) {
            const uint32_t lo = (uint32_t)F::round(__fmul_rn(v[q].x, inv)) |
                                ((uint32_t)F::round(__fmul_rn(v[q].y, inv)) << 16);
            const uint32_t hi = (uint32_t)F::round(__fmul_rn(v[q].z, inv)) |
                                ((uint32_t)F::round(__fmul_rn(v[q].w, inv)) << 16);
            reinterpret_cast<uint2 *>(p.xhat + (size_t)t * d)[k] = make_uint2(lo, hi);
        }
    }
}

// ------------------------------------------------------------------ hidden layer
// acc[rr][t] += the lane's chunks of CDOT(W1[i0 + rr], x_hat_t): rows from
// global memory, PD chunks in flight per row; x_hat of the TT tokens in
// shared memory ([8][K] 16-bit); the mixed-precision fma needs no conversion.
template <typename T, int R, int PD, int TT>
__device__ __forceinline__ void cdot_x16(const uint16_t *W, int K, int M, int i0, const uint8_t *xs, int lane,
                                         float (&acc)[R][TT])
{
    const int nch = K >> 3;
    const uint4 *wr[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) wr[rr] = reinterpret_cast<const uint4 *>(W + (size_t)min(i0 + rr, M - 1) * K);
    uint4 w[PD][R];
#pragma unroll
    for (int s = 0; s < PD; ++s)
        if (lane + 32 * s < nch)
#pragma unroll
            for (int rr = 0; rr < R; ++rr) w[s][rr] = __ldg(wr[rr] + lane + 32 * s);
    for (int c0 = lane; c0 < nch; c0 += 32 * PD) {
#pragma unroll
        for (int s = 0; s < PD; ++s) {
            const int ch = c0 + 32 * s;
            if (ch < nch) {
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    const uint4 xv = *reinterpret_cast<const uint4 *>(xs + (size_t)t * K * 2 + (size_t)ch * 16);
#pragma unroll
                    for (int rr = 0; rr < R; ++rr) acc[rr][t] = fma_chunk<T>(w[s][rr], xv, acc[rr][t]);
                }
                const int cn = ch + 32 * PD;
                if (cn < nch)
#pragma unroll
                    for (int rr = 0; rr < R; ++rr) w[s][rr] = __ldg(wr[rr] + cn);
            }
        }
    }
}

// h[t][j] = max(CDOT(W1[j], x_hat_t) + b1[j], 0).  CTA c takes token block
// c mod ntb and every ncta-th group of 8R rows.  It also clears the mask
// words, for output tiles narrower than a word.
template <typename T, int R, int PD, int TT>
__global__ void __launch_bounds__(kPT, 1) pred_hidden(const PredParams p)
{
    using F = F16T<T>;
    extern __shared__ __align__(128) uint8_t smem[];
    const LayerDev &L = p.L;
    const int d = L.d, r = L.r, B = p.B;
    const int ntb = (B + TT - 1) / TT;
    const int tb = blockIdx.x % ntb, cta = blockIdx.x / ntb;
    const int ncta = ((int)gridDim.x - tb + ntb - 1) / ntb;
    const int t0 = tb * TT, nch = d >> 3;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nrg = (r + 8 * R - 1) / (8 * R);
    // this warp's rows of every unit start for L2 now, while the previous
    // launch finishes (they do not depend on it): the loads below then wait
    // on L2, not HBM
    if (lane == 0)
        for (int rg = cta; rg < nrg; rg += ncta) {
            const int i0 = rg * 8 * R + warp * R, nr = min(R, r - i0);
            if (nr > 0) bulk_prefetch_l2(L.w1 + (size_t)i0 * d, (uint32_t)nr * d * 2, policy_evict_normal());
        }
    pdl_enter();
    if (cta_aborted(p)) return;
    for (int k = blockIdx.x * kPT + threadIdx.x; k < (L.n + 31) >> 5; k += (int)gridDim.x * kPT) p.mask[k] = 0u;
    for (int q = threadIdx.x; q < TT * nch; q += kPT) {
        const int t = q / nch, ch = q - t * nch;
        const bool v = t0 + t < B;
        cp16(smem_u32(smem) + (uint32_t)(t * d * 2 + ch * 16), v ? (const void *)(p.xhat + (size_t)(t0 + t) * d + ch * 8)
                                                                 : (const void *)p.xhat,
             v ? 16u : 0u);
    }
    cp_commit();
    cp_wait<0>();
    __syncthreads();
    constexpr int NV = R * TT;
    for (int rg = cta; rg < nrg; rg += ncta) {
        const int i0 = rg * 8 * R + warp * R;
        if (i0 >= r) continue; // warp-uniform; no CTA barrier below
        // the rows' biases, loaded now so that the epilogue does not wait for them
        const float b1r = lane < R && i0 + lane < r ? F::one(L.b1[i0 + lane]) : 0.f;
        float acc[R][TT];
#pragma unroll
        for (int rr = 0; rr < R; ++rr)
#pragma unroll
            for (int t = 0; t < TT; ++t) acc[rr][t] = 0.f;
        cdot_x16<T, R, PD, TT>(L.w1, d, r, i0, smem, lane, acc);
        float v[NV];
#pragma unroll
        for (int rr = 0; rr < R; ++rr)
#pragma unroll
            for (int t = 0; t < TT; ++t) v[rr * TT + t] = acc[rr][t];
        int base = 0;
        halve<NV, 16, NV>(v, lane, base);
#pragma unroll
        for (int j = 0; j < held(NV); ++j) {
            const int k = base + j, rr = k / TT, t = k % TT;
            const int row = i0 + rr, tok = t0 + t;
            const float b1v = __shfl_sync(0xffffffffu, b1r, rr, 32); // (every lane: a full-warp shuffle)
            if ((lane & dup_mask(NV)) == 0 && row < r && tok < B) {
                const float s1 = __fadd_rn(v[j], b1v);
                p.h[(size_t)tok * r + row] = s1 > 0.f ? s1 : 0.f;
            }
        }
    }
}

// ------------------------------------------------------------------ output layer
// Position of element i of a token's h in a block's shared-memory copy
// (tokens Kp floats apart, Kp = r rounded up to 256): the two 4-float halves
// of chunk ch = i / 8 sit 128 floats apart, so a warp's float4 load of one
// half of 32 consecutive chunks reads 512 contiguous bytes.
__device__ __forceinline__ int hpos(int ch, int hf) { return (ch >> 5) * 256 + hf * 128 + (ch & 31) * 4; }

// z = CDOT(W2[i], h_t) + b2[i] > 0, OR over the batch.  Unit u = rows
// [8R u, 8R (u+1)): warp w's R rows arrive by one bulk copy into its own part
// of the tile and stay while the batch's h passes through in blocks of 8
// tokens (two buffers).  With WS = 2 tile slots, a warp issues the copy of
// its rows of the next unit before it computes this one (small batches,
// where the rows' transfer, not the arithmetic, is the longer part).  Units
// wholly inside the layer's hot prefix are skipped: the compaction sets the
// prefix's bits.
template <typename T, int R, int WS, int TT>
__global__ void __launch_bounds__(kPT, 1) pred_out(const PredParams p)
{
    using F = F16T<T>;
    constexpr int RT = 8 * R; // rows per unit
    extern __shared__ __align__(128) uint8_t smem[];
    const LayerDev &L = p.L;
    const int r = L.r, n = L.n, B = p.B;
    const int Kp = (r + 255) & ~255, nch = r >> 3;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t wB = (uint32_t)R * r * 2; // bytes of one warp's rows
    uint8_t *wtile = smem + (size_t)warp * WS * wB;
    float *hbuf = reinterpret_cast<float *>(smem + 8 * (size_t)WS * wB);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + 8 * (size_t)WS * wB + 2 * (size_t)TT * Kp * 4);
    uint32_t *smask = reinterpret_cast<uint32_t *>(bar + 8 * WS);
    if (threadIdx.x < 8 * WS) mbar_init(bar + threadIdx.x, 1);
    if (threadIdx.x < (RT + 31) / 32) smask[threadIdx.x] = 0u;
    fence_barrier_init();
    // (an earlier launch's failure; one the hidden-layer launch raises while
    // this one starts stays in the status word.  The barrier also publishes
    // the initialised mbarriers)
    if (cta_aborted(p)) return;
    const int ntb = (B + TT - 1) / TT;
    const int nrt = (n + RT - 1) / RT;
    const int u0 = min(L.hot, n) / RT; // units wholly inside the hot prefix are not evaluated
    const int nwords = (n + 31) >> 5;
    // h block tb into buffer b (zeros past B), in the conflict-free layout
    const auto stage_h = [&](int tb, int b) {
        const int t0 = tb * TT;
        float *dst = hbuf + (size_t)b * TT * Kp;
        for (int q = threadIdx.x; q < TT * nch * 2; q += kPT) {
            const int t = q / (nch * 2), c = q - t * nch * 2, ch = c >> 1, hf = c & 1;
            const bool v = t0 + t < B;
            cp16(smem_u32(dst + (size_t)t * Kp + hpos(ch, hf)),
                 v ? (const void *)(p.h + (size_t)(t0 + t) * r + ch * 8 + hf * 4) : (const void *)p.h, v ? 16u : 0u);
        }
        cp_commit();
    };
    // copies issued into / waited for in each tile slot of this warp (warp-
    // uniform counts): at most one is outstanding per slot, and the warp
    // waits for it before the CTA exits, whatever happened
    uint32_t n_iss[2] = {0u, 0u}, n_wt[2] = {0u, 0u};
    // warp-level: bring this warp's rows of unit u into tile slot sl
    const auto load_rows = [&](int u, int sl) {
        const int i0 = u * RT + warp * R;
        const int nr = max(0, min(R, n - i0));
        if (nr > 0) {
            if (lane == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar + warp * WS + sl, (uint32_t)nr * r * 2);
                bulk_g2s(wtile + (size_t)sl * wB, L.w2 + (size_t)i0 * r, (uint32_t)nr * r * 2, bar + warp * WS + sl,
                         policy_evict_first());
            }
            ++n_iss[sl];
        }
    };
    // the first unit's rows do not depend on the hidden layer: they start
    // while it finishes
    if (u0 + (int)blockIdx.x < nrt) load_rows(u0 + blockIdx.x, 0);
    pdl_enter();
    if (ntb == 1) stage_h(0, 0); // one block serves every unit
    bool ok = true;
    uint32_t it = 0;
    for (int u = u0 + blockIdx.x; u < nrt; u += gridDim.x, ++it) {
        const int sl = WS == 2 ? (int)(it & 1) : 0;
        const uint32_t par = WS == 2 ? (it >> 1) & 1 : it & 1;
        // (after a failed wait nothing more is issued: that slot's copy may still be in flight)
        if (WS == 2) {
            if (ok && u + (int)gridDim.x < nrt) load_rows(u + gridDim.x, sl ^ 1); // slot sl ^ 1 was read by the last unit
        } else if (it > 0 && ok) {
            load_rows(u, 0);
        }
        const int i0 = u * RT + warp * R;
        const int nr = max(0, min(R, n - i0));
        const uint8_t *wt = wtile + (size_t)sl * wB;
        // the rows' biases, loaded now so that the epilogues do not wait for them
        const float b2r = lane < nr ? F::one(L.b2[i0 + lane]) : 0.f;
        if (ntb > 1) stage_h(0, 0);
        uint32_t bits = 0; // bit rr: row i0 + rr active for some token
        bool landed = nr == 0;
        for (int tb = 0; tb < ntb; ++tb) {
            if (ntb > 1 && tb + 1 < ntb) {
                stage_h(tb + 1, (tb + 1) & 1);
                cp_wait<1>();
            } else {
                cp_wait<0>();
            }
            __syncthreads();
            if (!landed) {
                // every lane waits; the warp goes on only if all saw the rows (shuffles follow)
                const bool got = ok && wait_bounded(bar + warp * WS + sl, par, p);
                ok = __all_sync(0xffffffffu, got);
                if (ok) ++n_wt[sl];
                landed = true;
            }
            if (nr > 0 && ok) {
                const float *hs = hbuf + (size_t)(ntb > 1 ? (tb & 1) : 0) * TT * Kp;
                float acc[R][TT];
#pragma unroll
                for (int rr = 0; rr < R; ++rr)
#pragma unroll
                    for (int t = 0; t < TT; ++t) acc[rr][t] = 0.f;
                for (int ch = lane; ch < nch; ch += 32) {
                    uint4 w[R];
#pragma unroll
                    for (int rr = 0; rr < R; ++rr)
                        w[rr] = *reinterpret_cast<const uint4 *>(wt + (size_t)rr * r * 2 + (size_t)ch * 16);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        float4 hv[TT];
#pragma unroll
                        for (int t = 0; t < TT; ++t)
                            hv[t] = *reinterpret_cast<const float4 *>(hs + (size_t)t * Kp + hpos(ch, hf));
#pragma unroll
                        for (int e2 = 0; e2 < 2; ++e2) { // elements 4 hf + 2 e2 and 4 hf + 2 e2 + 1
#pragma unroll
                            for (int rr = 0; rr < R; ++rr) {
                                const uint32_t word = hf == 0 ? (e2 == 0 ? w[rr].x : w[rr].y) : (e2 == 0 ? w[rr].z : w[rr].w);
                                const float2 wf = F::pair(word);
#pragma unroll
                                for (int t = 0; t < TT; ++t) {
                                    const float h0 = e2 == 0 ? hv[t].x : hv[t].z, h1 = e2 == 0 ? hv[t].y : hv[t].w;
                                    acc[rr][t] = __fmaf_rn(wf.y, h1, __fmaf_rn(wf.x, h0, acc[rr][t]));
                                }
                            }
                        }
                    }
                }
                constexpr int NV = R * TT;
                float v[NV];
#pragma unroll
                for (int rr = 0; rr < R; ++rr)
#pragma unroll
                    for (int t = 0; t < TT; ++t) v[rr * TT + t] = acc[rr][t];
                int base = 0;
                halve<NV, 16, NV>(v, lane, base);
                uint32_t mine = 0;
#pragma unroll
                for (int j = 0; j < held(NV); ++j) {
                    const int k = base + j, rr = k / TT, t = k % TT;
                    const float b2v = __shfl_sync(0xffffffffu, b2r, rr, 32);
                    if (rr < nr && tb * TT + t < B && __fadd_rn(v[j], b2v) > 0.f) mine |= 1u << rr;
                }
                bits |= __reduce_or_sync(0xffffffffu, mine);
            }
            __syncthreads(); // the buffer of block tb is free for block tb + 2
        }
        if (lane == 0 && bits) atomicOr(smask + ((warp * R) >> 5), bits << ((warp * R) & 31));
        __syncthreads();
        if (threadIdx.x < (RT + 31) / 32) {
            const int wi = u * RT / 32 + threadIdx.x;
            if constexpr (RT % 32 == 0) { // whole words: this CTA's alone
                if (wi < nwords) p.mask[wi] = smask[threadIdx.x];
            } else if (smask[threadIdx.x]) { // part of a word (cleared by the hidden-layer launch)
                atomicOr(p.mask + wi, smask[threadIdx.x] << ((u * RT) & 31));
            }
            smask[threadIdx.x] = 0u;
        }
        // (the next unit's shared-mask atomics come after the barrier of its first block)
    }
    cp_wait<0>();
    // no bulk copy of this CTA may be in flight when it exits (bounded, ignoring the abort flag)
    for (int sl = 0; sl < WS; ++sl)
        if (n_iss[sl] > n_wt[sl]) {
            const uint32_t par = (n_iss[sl] - 1) & 1;
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(bar + warp * WS + sl, par) && globaltimer() - t0 < 100000000ull) {
            }
        }
}

// ------------------------------------------------------------------ compaction
// CTA c of 256 threads owns mask words [256 c, 256 c + 256), one per thread.
// Its list offset is the popcount of all words before them (every CTA adds
// those up itself: n <= 65536 is at most 2048 words); a block scan places
// each word, then each warp writes its 32 words' ids lane-parallel, one
// word per round.
__global__ void __launch_bounds__(256) pred_compact(const PredParams p)
{
    __shared__ int red[8];
    __shared__ int wsum[8];
    pdl_enter();
    if (cta_aborted(p)) return;
    const int n = p.L.n, nwords = (n + 31) >> 5;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (p.dense) { // every neuron
        for (int k = blockIdx.x * 256 + tid; k < n; k += (int)gridDim.x * 256) {
            p.idx[k] = k;
            if (p.tr_idx) p.tr_idx[k] = k;
        }
        if (blockIdx.x == 0 && tid == 0) {
            *p.count = n;
            if (p.tr_cnt) *p.tr_cnt = n;
        }
        return;
    }
    const int w0 = blockIdx.x * 256;
    const int hot = p.L.hot; // neurons [0, hot) are on whatever their mask bits say
    int before = 0;
    for (int k = tid; k < w0; k += 256) before += __popc(p.mask[k] | hot_bits(k, hot));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    if (lane == 0) red[warp] = before;
    const int wi = w0 + tid;
    const uint32_t m = wi < nwords ? p.mask[wi] | hot_bits(wi, hot) : 0u;
    const int c = __popc(m);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int off = 0, tot = 0;
    for (int w = 0; w < 8; ++w) {
        off += w < warp ? wsum[w] : 0;
        tot += wsum[w];
    }
    int base = 0;
    for (int w = 0; w < 8; ++w) base += red[w];
    const int pos = base + off + incl - c; // list position of this word's first id
    for (int k = 0; k < 32; ++k) {
        const uint32_t mk = __shfl_sync(0xffffffffu, m, k);
        const int pk = __shfl_sync(0xffffffffu, pos, k);
        if ((mk >> lane) & 1u) {
            const int at = pk + __popc(mk & ((1u << lane) - 1u));
            const int id = (w0 + warp * 32 + k) * 32 + lane;
            p.idx[at] = id;
            if (p.tr_idx) p.tr_idx[at] = id;
        }
    }
    if (blockIdx.x == gridDim.x - 1 && tid == 0) {
        *p.count = base + tot;
        if (p.tr_cnt) *p.tr_cnt = base + tot;
    }
}

// shared memory of pred_out: WS tile slots, two h blocks of TT tokens, the mbarriers, the mask words
int out_smem(int R, int WS, int TT, int r) { return 8 * WS * R * r * 2 + 2 * TT * ((r + 255) & ~255) * 4 + 8 * WS * 8 + 16; }

int compact_grid(int n) { return std::max(1, ((n + 31) / 32 + 255) / 256); }

template <typename T, int R, int PD, int TT>
cudaError_t launch_hidden(const PredParams &p, int sms, cudaStream_t s)
{
    const int smem = TT * p.L.d * 2, ntb = (p.B + TT - 1) / TT;
    auto kern = pred_hidden<T, R, PD, TT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 1;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kPT, smem);
    if (e != cudaSuccess) return e;
    const int nrg = (p.L.r + 8 * R - 1) / (8 * R);
    int grid = std::min(ntb * nrg, std::max(1, per_sm) * sms);
    grid = std::max(ntb, grid / ntb * ntb); // every token block gets the same number of CTAs
    return launch_pdl(kern, dim3(grid), dim3(kPT), smem, s, p);
}

template <typename T, int R, int WS, int TT>
cudaError_t launch_out(const PredParams &p, int sms, cudaStream_t s)
{
    const int smem = out_smem(R, WS, TT, p.L.r);
    auto kern = pred_out<T, R, WS, TT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int nrt = (p.L.n + 8 * R - 1) / (8 * R) - std::min(p.L.hot, p.L.n) / (8 * R);
    return launch_pdl(kern, dim3(std::max(1, std::min(nrt, sms))), dim3(kPT), smem, s, p);
}

template <typename T>
cudaError_t launch_all(const PredParams &p, int sms, cudaStream_t s)
{
    const int B = p.B;
    // hidden layer: token tiles of 2, 4 (two blocks up to 8 tokens: twice the CTAs) or 8;
    // one row per warp up to 8 tokens, else two; row chunks in flight per lane: 16 for 2
    // tokens, 12 for 4 (measured, pred_hidden at 2 / 3 / 8 tokens, us: 8 in flight 17.2 /
    // 14.1 / 15.1, 12: 15.9 / 13.7 / 14.6, 16: 14.0 / 12.6 / 19.0)
    cudaError_t e = B <= 2   ? launch_hidden<T, 1, 16, 2>(p, sms, s)
                    : B <= 8 ? launch_hidden<T, 1, 12, 4>(p, sms, s)
                             : launch_hidden<T, 2, 4, 8>(p, sms, s);
    if (e != cudaSuccess) return e;
    // output layer (the tile stays within shared memory): beyond r = 1024, 2 rows per
    // warp; else for one or two token blocks 4 rows with the next unit's in flight,
    // else 8 rows; token tiles of 2, 4 or 8
    if (p.L.r > 1024) e = B <= 2 ? launch_out<T, 2, 1, 2>(p, sms, s) : launch_out<T, 2, 1, 8>(p, sms, s);
    else if (B <= 2) e = launch_out<T, 4, 2, 2>(p, sms, s);
    else if (B <= 4) e = launch_out<T, 4, 2, 4>(p, sms, s);
    else if (B <= 16) e = launch_out<T, 4, 2, 8>(p, sms, s);
    else e = launch_out<T, 8, 1, 8>(p, sms, s);
    if (e != cudaSuccess) return e;
    return launch_pdl(pred_compact, dim3(compact_grid(p.L.n)), dim3(256), 0, s, p);
}

} // namespace

cudaError_t launch_rmsnorm_rows(const PredParams &p, bool bf16, cudaStream_t s)
{
    return bf16 ? launch_pdl(rmsnorm_rows<__nv_bfloat16>, dim3(p.B), dim3(512), 0, s, p)
                : launch_pdl(rmsnorm_rows<__half>, dim3(p.B), dim3(512), 0, s, p);
}

cudaError_t launch_list_all(const PredParams &p, cudaStream_t s)
{
    PredParams q = p;
    q.dense = 1;
    return launch_pdl(pred_compact, dim3(compact_grid(p.L.n)), dim3(256), 0, s, q);
}

cudaError_t launch_predict_batch(const PredParams &p, bool bf16, int sms, cudaStream_t s)
{
    return bf16 ? launch_all<__nv_bfloat16>(p, sms, s) : launch_all<__half>(p, sms, s);
}

} // namespace pi
