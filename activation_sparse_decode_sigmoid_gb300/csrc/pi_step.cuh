// The persistent step kernel of libpi: activation predictor followed by the
// neuron-aware sparse FFN, for one layer or a whole stack, in one launch.
//
// PowerInfer (blog.csdn.net QbitAI/IPADS article, sections
// "充分利用模型和硬件特点" and "CPU/GPU混合推理设计"): a small per-layer
// routing predictor selects the neurons an input activates; only those
// neurons' rows of W_up (W_gate) and columns of W_down are read; the partial
// results of the executors are merged.  On GB300 every executor is an SM: the
// predicted list is split evenly over the SMs, each SM accumulates an fp32
// partial of the layer output, and a fixed-order split-K reduction merges
// them into the residual stream.
//
// One CTA per SM (cooperative launch), 18 warps:
//   warps 0..15  consumers: dot products, activations, partial sums, merge;
//   warp 16      static producer: streams this CTA's slice of the predictor
//                weights W1 / W2 with bulk copies (cp.async.bulk + mbarrier)
//                into nss slots of the shared ring, and, once a layer's slice
//                is issued, prefetches the next layer's slice into L2;
//   warp 17      dynamic producer: once the predicted list is known, streams
//                the rows (W_up, W_gate, W_down^T) of this CTA's share of the
//                predicted neurons into nsd stages of the same ring.
// The ring is time-shared: static slots during phases A/B, dynamic stages
// during phase C (the static producer of the next layer waits until the
// consumers have finished phase C).
// Per layer (consumers):
//   A  x_hat = RMSNorm(x) (or given); h = max(CDOT(W1, x_hat) + b1, 0)  -> global
//   B  z = CDOT(W2, h) + b2 for this CTA's rows; z > 0 sets a bit of the
//      CTA's mask words -> global bitmap
//   C  a prefix scan of the bitmap gives the ascending global list; this CTA
//      takes an equal share of it, streams those neurons' rows, computes
//      a = act(W_up x_hat + b ...) and accumulates a * W_down^T rows -> fp32
//      partial [B][d] of this CTA -> global
//   D  every CTA reduces a slice of the columns over all partials in a fixed
//      order and adds the result (+ b_down) into x (or writes y)
// Each step reads what every SM wrote in the step before (h, the mask words,
// the partials, the new x), so each hand-over is all-to-all.  There is no grid
// barrier: those four hand-overs are 64-bit words carrying the value and the
// epoch of the layer that wrote it, and the reader polls the words themselves
// until they carry its epoch (one L2 round trip when the writers are done,
// instead of a barrier's arrive, poll and then the read).  The all-to-all
// pattern also orders reuse: no SM can write layer l+1's h, mask, partials or
// x before every SM has read layer l's.
#pragma once

#include "pi_device.cuh"

namespace pi {

// ------------------------------------------------------------------ shared layout
struct Shm {
    uint8_t *ring, *hs, *xs;
    uint64_t *full_s, *empty_s, *full_d, *empty_d, *lst_full, *lst_free;
    int *info;      // [16] scalars
    float *tmp;     // [256] scratch (norm sums, scan totals)
    int *slist;     // [lcap] this CTA's neuron ids (phase C)
    float *sbias;   // [lcap] their biases
    unsigned *swords; // [wcap] predicted-mask words of this CTA's rows
    uint16_t *pb1s, *pb2s; // this CTA's b1 / b2 slices, as copied (16-byte-rounded ranges)
    uint64_t *bias_full;   // completes when a layer's bias slices have landed
    uint64_t *act_full;    // [nsd] completes when a stage's P owner warps have written their partial sums
    float *red;     // partial dot sums of the FFN stages: [nsd][npd][P][TGF][2] (nsd * npd * P <= 2 * 16 * 8)
};

enum { INFO_FLAG = 0, INFO_NCNT = 1, INFO_FAIL = 2, INFO_M = 3, INFO_REGION = 4, INFO_OWNP = 5 };

static __device__ __forceinline__ volatile int *fail_word(const Shm &S) { return S.info + INFO_FAIL; }

// debug timeline: thread 0 of each CTA stamps the globaltimer at phase ends
static __device__ __forceinline__ void mark(const StepParams &p, int ev)
{
    if (p.timeline && threadIdx.x == 0 && ev < p.tl_stride)
        p.timeline[(size_t)blockIdx.x * p.tl_stride + ev] = globaltimer();
}

static __device__ __forceinline__ int rcap_bytes(int rcap) { return (rcap * 2 + 32 + 15) & ~15; }

static __device__ __forceinline__ Shm carve(uint8_t *smem, const StepParams &p, int tgf)
{
    Shm s;
    s.ring = smem;
    s.hs = smem + p.off_h;
    s.xs = smem + p.off_xs;
    const MiscLayout m = misc_layout(p.nss, p.nsd, p.lcap, p.wcap, p.rcap, tgf);
    uint8_t *base = smem + p.off_misc;
    s.full_s = (uint64_t *)(base + m.bars);
    s.empty_s = s.full_s + p.nss;
    s.full_d = s.empty_s + p.nss;
    s.empty_d = s.full_d + p.nsd;
    s.lst_full = s.empty_d + p.nsd;
    s.lst_free = s.lst_full + 1;
    s.bias_full = s.lst_free + 1;
    s.act_full = s.bias_full + 1;
    s.info = (int *)(base + m.info);
    s.tmp = (float *)(base + m.tmp);
    s.slist = (int *)(base + m.slist);
    s.sbias = (float *)(base + m.sbias);
    s.swords = (unsigned *)(base + m.swords);
    s.pb1s = (uint16_t *)(base + m.pbias);
    s.pb2s = s.pb1s + ((rcap_bytes(p.rcap)) >> 1);
    s.red = (float *)(base + m.red);
    return s;
}

// ------------------------------------------------------------------ slices (shared by producers and consumers)
struct SliceA {
    int j0, j1, rps, nst; // W1 rows [j0,j1), rows per slot, stages per token group
};
struct SliceB {
    int i0, i1, rps, nst; // W2 rows [i0,i1) (word aligned), rows per slot, stages per token group
};

static __device__ __forceinline__ SliceA slice_a(const LayerDev &L, const StepParams &p)
{
    SliceA a;
    a.j0 = slice_lo(L.r, blockIdx.x, gridDim.x);
    a.j1 = slice_lo(L.r, blockIdx.x + 1, gridDim.x);
    a.rps = max(1, p.slotB / (L.d * 2));
    a.nst = (a.j1 - a.j0 + a.rps - 1) / a.rps;
    return a;
}

static __device__ __forceinline__ int word_row_start(int n, int c, int G)
{
    const int nw = (n + 31) >> 5;
    return min(n, 32 * slice_lo(nw, c, G));
}

// Neurons [0, hot) are active without prediction (the hot prefix); counting
// the predictor's selections for calibration evaluates every row.
static __device__ __forceinline__ int hot_rows(const LayerDev &L, const StepParams &p)
{
    return (p.mode & M_COUNTS) ? 0 : L.hot;
}

// Phase B evaluates rows [h0, n), h0 = the hot prefix rounded down to a whole
// mask word; the rows of the boundary word below the prefix are evaluated and
// then forced on.
static __device__ __forceinline__ SliceB slice_b(const LayerDev &L, const StepParams &p)
{
    SliceB b;
    const int h0 = hot_rows(L, p) & ~31;
    b.i0 = h0 + word_row_start(L.n - h0, blockIdx.x, gridDim.x);
    b.i1 = h0 + word_row_start(L.n - h0, blockIdx.x + 1, gridDim.x);
    b.rps = max(1, p.slotB / (L.r * 2));
    b.nst = (b.i1 - b.i0 + b.rps - 1) / b.rps;
    return b;
}

// One neuron in a ring stage: [W_up row (+ bias tail)][W_gate row][W_down^T row].
static __device__ __forceinline__ int neuron_bytes(const LayerDev &L)
{
    return L.upB + (L.gate ? 2 : 1) * L.rowB;
}

static __device__ __forceinline__ int neurons_per_stage(const LayerDev &L, const StepParams &p)
{
    return max(1, min(kMaxNeuronsPerStage, p.dslotB / neuron_bytes(L)));
}

// ------------------------------------------------------------------ producers
// Wait (bounded, ignoring the abort flag) until the copies of the last issued
// stages have landed, so that no bulk copy is in flight when the CTA exits.
static __device__ __forceinline__ const uint8_t *down16(const void *a)
{
    return reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(a) & ~(uintptr_t)15);
}

static __device__ __forceinline__ const uint8_t *up16(const void *a)
{
    return reinterpret_cast<const uint8_t *>((reinterpret_cast<uintptr_t>(a) + 15) & ~(uintptr_t)15);
}

// Element offset of a 16-bit array element within its 16-byte-rounded copy.
static __device__ __forceinline__ int off16(const uint16_t *a)
{
    return (int)((reinterpret_cast<uintptr_t>(a) & 15) >> 1);
}

static __device__ void drain(uint64_t *full, uint32_t issued, int nslots)
{
    const uint32_t first = issued > (uint32_t)nslots ? issued - nslots : 0;
    for (uint32_t k = first; k < issued; ++k) {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(full + (k % nslots), (k / nslots) & 1)) {
            if (globaltimer() - t0 > 100000000ull) break; // 100 ms: copies land in microseconds
        }
    }
}

// L2 prefetch of layer l's predictor slice of this CTA (W1 rows, then W2
// rows).  Mode 1 issues it all at once; mode 2 paces it (one 16 KB chunk per
// prefetch_ns) so the backlog never queues in front of latency-critical
// requests (grid-barrier atomics, bitmap reads, the first FFN rows), and stops
// early once the ring is free for the next layer (the regular loads then
// fetch the rest).
static __device__ void prefetch_predictor(const StepParams &p, const Shm &S, int l, int ready_at, uint64_t pol)
{
    const LayerDev &L = p.layers[l];
    const SliceA A = slice_a(L, p);
    const SliceB Bs = slice_b(L, p);
    const uint8_t *seg[2] = {(const uint8_t *)L.w1 + (size_t)A.j0 * L.d * 2,
                             (const uint8_t *)L.w2 + (size_t)Bs.i0 * L.r * 2};
    const size_t len[2] = {(size_t)(A.j1 - A.j0) * L.d * 2, (size_t)(Bs.i1 - Bs.i0) * L.r * 2};
    const size_t chunk = p.prefetch == 1 ? 65536 : 16384;
    uint64_t t = globaltimer();
    for (int sgi = 0; sgi < 2; ++sgi) {
        for (size_t o = 0; o < len[sgi];) {
            if (p.prefetch == 2) {
                if (*(volatile int *)(S.info + INFO_REGION) >= ready_at || aborted(p)) return;
                const uint64_t now = globaltimer();
                if (now < t) {
                    __nanosleep(200);
                    continue;
                }
                t = now + (uint64_t)p.prefetch_ns;
            }
            bulk_prefetch_l2(seg[sgi] + o, (uint32_t)min(chunk, len[sgi] - o), pol);
            o += chunk;
        }
    }
}

static __device__ void static_producer(const StepParams &p, const Shm &S)
{
    if (!(p.mode & (M_PREDICT | M_COUNTS)) || p.nss == 0) return;
    const uint64_t pol = policy_evict_first();
    const uint64_t keep = policy_evict_last();
    const uint64_t norm = policy_evict_normal();
    const bool ffn = (p.mode & M_FFN) != 0;
    uint32_t s = 0, nbias = 0;
    bool ok = true;
    for (int l = 0; l < p.L && ok; ++l) {
        // the ring holds dynamic stages during phase C of the previous layer
        // (without an FFN phase: the consumers are done with its phase B)
        if (l > 0 && !wait_counter(S.info + INFO_REGION, l, p)) break;
        const LayerDev &L = p.layers[l];
        const SliceA A = slice_a(L, p);
        const SliceB Bs = slice_b(L, p);
        {
            // this CTA's b1 and b2 slices (16-byte-rounded ranges: the
            // library pads both arrays), off the consumers' critical path
            const uint8_t *s1 = down16(L.b1 + A.j0), *e1 = up16(L.b1 + A.j1);
            const uint8_t *s2 = down16(L.b2 + Bs.i0), *e2 = up16(L.b2 + Bs.i1);
            mbar_arrive_expect_tx(S.bias_full, (uint32_t)((e1 - s1) + (e2 - s2)));
            if (e1 > s1) bulk_g2s(S.pb1s, s1, (uint32_t)(e1 - s1), S.bias_full, pol);
            if (e2 > s2) bulk_g2s(S.pb2s, s2, (uint32_t)(e2 - s2), S.bias_full, pol);
            ++nbias;
        }
        const int nga = (p.B + p.tg - 1) / p.tg;
        const int ngb = (p.B + p.tgB - 1) / p.tgB;
        for (int pass = 0; pass < 2 && ok; ++pass) {
            const int ng = pass == 0 ? nga : ngb;
            const int lo = pass == 0 ? A.j0 : Bs.i0;
            const int hi = pass == 0 ? A.j1 : Bs.i1;
            const int rps = pass == 0 ? A.rps : Bs.rps;
            const size_t rowB = pass == 0 ? (size_t)L.d * 2 : (size_t)L.r * 2;
            const uint8_t *src = (const uint8_t *)(pass == 0 ? L.w1 : L.w2);
            if (pass == 1 && p.prefetch == 3) {
                // W1's slots are issued; W2's slice (most of it beyond the
                // ring) streams into L2 while the merge, the barriers and
                // phase A run, so phase B reads it from L2
                const uint8_t *w = src + (size_t)lo * rowB;
                const size_t len = (size_t)(hi - lo) * rowB;
                for (size_t o = 0; o < len; o += 32768)
                    bulk_prefetch_l2(w + o, (uint32_t)min((size_t)32768, len - o), norm);
            }
            for (int g = 0; g < ng && ok; ++g) {
                for (int row = lo; row < hi; row += rps, ++s) {
                    const int slot = s % p.nss;
                    if (s >= (uint32_t)p.nss && !mbar_wait(S.empty_s + slot, ((s / p.nss) - 1) & 1, p)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bytes = (uint32_t)(min(rps, hi - row) * rowB);
                    mbar_arrive_expect_tx(S.full_s + slot, bytes);
                    bulk_g2s(S.ring + (size_t)slot * p.slotB, src + (size_t)row * rowB, bytes, S.full_s + slot, pol);
                }
            }
        }
        // keep HBM busy through the barriers, the merge and the next layer's
        // first phases: pull the next layer's predictor slice into L2 now
        if (ok && (p.mode & M_RESID) && (p.prefetch == 1 || p.prefetch == 2))
            prefetch_predictor(p, S, l + 1 < p.L ? l + 1 : 0, ffn ? l + 1 : 0x7fffffff, keep);
    }
    drain(S.full_s, s, p.nss);
    drain(S.bias_full, nbias, 1);
}

static __device__ void dynamic_producer(const StepParams &p, const Shm &S)
{
    if (!(p.mode & M_FFN)) return;
    const uint64_t pol = policy_evict_first();
    const uint64_t norm = policy_evict_normal();
    uint32_t sd = 0;
    for (int l = 0; l < p.L; ++l) {
        if (!mbar_wait(S.lst_full, l & 1, p)) break;
        const LayerDev &L = p.layers[l];
        const int ncnt = S.info[INFO_NCNT];
        const int nb = neuron_bytes(L);
        const int npd = neurons_per_stage(L, p);
        const int ngf = (p.B + p.tg - 1) / p.tg;
        const size_t rowB = (size_t)L.rowB, upB = (size_t)L.upB;
        bool ok = true;
        int pf = 0; // next list position to prefetch into L2
        for (int g = 0; g < ngf && ok; ++g) {
            for (int k = 0; k < ncnt; k += npd, ++sd) {
                if (g == 0 && p.rows_ahead > 0) {
                    // keep rows_ahead neurons beyond this stage on their way
                    // into L2, so HBM streams at full rate however few bytes
                    // the ring can hold
                    for (const int lim = min(ncnt, k + npd + p.rows_ahead); pf < lim; ++pf) {
                        const int id = S.slist[pf];
                        if (id < 0) continue;
                        bulk_prefetch_l2(L.up + (size_t)id * upB, (uint32_t)upB, norm);
                        if (L.gate) bulk_prefetch_l2(L.gate + (size_t)id * rowB, (uint32_t)rowB, norm);
                        bulk_prefetch_l2(L.dn + (size_t)id * rowB, (uint32_t)rowB, norm);
                    }
                }
                const int slot = sd % p.nsd;
                if (sd >= (uint32_t)p.nsd && !mbar_wait(S.empty_d + slot, ((sd / p.nsd) - 1) & 1, p)) {
                    ok = false;
                    break;
                }
                const int nn = min(npd, ncnt - k);
                uint32_t bytes = 0;
                for (int j = 0; j < nn; ++j)
                    if (S.slist[k + j] >= 0) bytes += (uint32_t)nb;
                mbar_arrive_expect_tx(S.full_d + slot, bytes);
                uint8_t *dst = S.ring + (size_t)slot * p.dslotB;
                for (int j = 0; j < nn; ++j) {
                    const int id = S.slist[k + j];
                    if (id < 0) continue;
                    uint8_t *o = dst + (size_t)j * nb;
                    bulk_g2s(o, L.up + (size_t)id * upB, (uint32_t)upB, S.full_d + slot, pol);
                    o += upB;
                    if (L.gate) {
                        bulk_g2s(o, L.gate + (size_t)id * rowB, (uint32_t)rowB, S.full_d + slot, pol);
                        o += rowB;
                    }
                    bulk_g2s(o, L.dn + (size_t)id * rowB, (uint32_t)rowB, S.full_d + slot, pol);
                }
            }
        }
        if (!ok) break;
        mbar_arrive(S.lst_free); // done reading this layer's list and count
    }
    drain(S.full_d, sd, p.nsd);
}

// ------------------------------------------------------------------ canonical dot products (CDOT)
static __device__ __forceinline__ float butterfly_sum(float a)
{
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, m));
    return a;
}

// acc[r] = CDOT(w_r, v) for NR rows w_r = w + r*rstride (16-bit, K elements,
// shared memory) and one vector v: 16-bit (x_hat, VF = false) or fp32 (h,
// VF = true), in shared memory.  The NR chains are independent: each keeps
// the canonical per-lane order, they only share the loads of v.
template <typename T, int NR, bool VF>
static __device__ __forceinline__ void cdot_rows(const uint8_t *w, size_t rstride, const void *v, int K, int lane,
                                                 float (&acc)[NR])
{
    using F = F16T<T>;
#pragma unroll
    for (int r = 0; r < NR; ++r) acc[r] = 0.f;
    const int nch = K >> 3;
    if constexpr (!VF) {
        // 16-bit vector: mixed-precision fma on the raw halves
        if constexpr (NR == 1) {
            // one chain: the next chunk's loads are in flight during this one's fmas
            int ch = lane;
            if (ch < nch) {
                uint4 wv = *reinterpret_cast<const uint4 *>(w + (size_t)ch * 16);
                uint4 xv = *reinterpret_cast<const uint4 *>((const uint8_t *)v + (size_t)ch * 16);
                for (; ch < nch; ch += 32) {
                    uint4 wn = wv, xn = xv;
                    if (ch + 32 < nch) {
                        wn = *reinterpret_cast<const uint4 *>(w + (size_t)(ch + 32) * 16);
                        xn = *reinterpret_cast<const uint4 *>((const uint8_t *)v + (size_t)(ch + 32) * 16);
                    }
                    acc[0] = fma_chunk<T>(wv, xv, acc[0]);
                    wv = wn;
                    xv = xn;
                }
            }
        } else {
            for (int ch = lane; ch < nch; ch += 32) {
                const uint4 xv = *reinterpret_cast<const uint4 *>((const uint8_t *)v + (size_t)ch * 16);
#pragma unroll
                for (int r = 0; r < NR; ++r)
                    acc[r] = fma_chunk<T>(*reinterpret_cast<const uint4 *>(w + r * rstride + (size_t)ch * 16), xv,
                                          acc[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[r] = butterfly_sum(acc[r]);
        return;
    } else {
        // fp32 vector (h): the rows are widened, the products and sums are fp32
        for (int ch = lane; ch < nch; ch += 32) {
            const float4 a = *reinterpret_cast<const float4 *>((const float *)v + (size_t)ch * 8);
            const float4 b = *reinterpret_cast<const float4 *>((const float *)v + (size_t)ch * 8 + 4);
            const float vv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const uint4 wv = *reinterpret_cast<const uint4 *>(w + r * rstride + (size_t)ch * 16);
                const float2 w0 = F::pair(wv.x), w1 = F::pair(wv.y), w2 = F::pair(wv.z), w3 = F::pair(wv.w);
                float s = acc[r];
                s = __fmaf_rn(w0.x, vv[0], s);
                s = __fmaf_rn(w0.y, vv[1], s);
                s = __fmaf_rn(w1.x, vv[2], s);
                s = __fmaf_rn(w1.y, vv[3], s);
                s = __fmaf_rn(w2.x, vv[4], s);
                s = __fmaf_rn(w2.y, vv[5], s);
                s = __fmaf_rn(w3.x, vv[6], s);
                s = __fmaf_rn(w3.y, vv[7], s);
                acc[r] = s;
            }
        }
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[r] = butterfly_sum(acc[r]);
    }
}

// acc0[r] = CDOT(w_r, v0), acc1[r] = CDOT(w_r, v1) for NR 16-bit rows and two
// fp32 vectors in shared memory: each row chunk is loaded and widened once
// for both tokens; each chain keeps the canonical per-lane order.
template <typename T, int NR>
static __device__ __forceinline__ void cdot_rows_2t(const uint8_t *w, size_t rstride, const float *v0, const float *v1,
                                                    int K, int lane, float (&acc0)[NR], float (&acc1)[NR])
{
    using F = F16T<T>;
#pragma unroll
    for (int r = 0; r < NR; ++r) acc0[r] = acc1[r] = 0.f;
    const int nch = K >> 3;
    for (int ch = lane; ch < nch; ch += 32) {
        const float4 a0 = *reinterpret_cast<const float4 *>(v0 + (size_t)ch * 8);
        const float4 b0 = *reinterpret_cast<const float4 *>(v0 + (size_t)ch * 8 + 4);
        const float4 a1 = *reinterpret_cast<const float4 *>(v1 + (size_t)ch * 8);
        const float4 b1 = *reinterpret_cast<const float4 *>(v1 + (size_t)ch * 8 + 4);
        const float x0[8] = {a0.x, a0.y, a0.z, a0.w, b0.x, b0.y, b0.z, b0.w};
        const float x1[8] = {a1.x, a1.y, a1.z, a1.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint4 wv = *reinterpret_cast<const uint4 *>(w + r * rstride + (size_t)ch * 16);
            const float2 p[4] = {F::pair(wv.x), F::pair(wv.y), F::pair(wv.z), F::pair(wv.w)};
            float s0 = acc0[r], s1 = acc1[r];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                s0 = __fmaf_rn(p[e].x, x0[2 * e], s0);
                s1 = __fmaf_rn(p[e].x, x1[2 * e], s1);
                s0 = __fmaf_rn(p[e].y, x0[2 * e + 1], s0);
                s1 = __fmaf_rn(p[e].y, x1[2 * e + 1], s1);
            }
            acc0[r] = s0, acc1[r] = s1;
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) acc0[r] = butterfly_sum(acc0[r]), acc1[r] = butterfly_sum(acc1[r]);
}

// Rows [0, nrows) of a static stage against two fp32 vectors, 4 rows at a
// time, then one by one; emit(row, acc0, acc1) gets both CDOTs of each row.
template <typename T, typename Emit>
static __device__ __forceinline__ void stage_rows_2t(const uint8_t *base, size_t rstride, int nrows, const float *v0,
                                                     const float *v1, int K, int lane, Emit emit)
{
    int r = 0;
    for (; r + 4 <= nrows; r += 4) {
        float a0[4], a1[4];
        cdot_rows_2t<T, 4>(base + (size_t)r * rstride, rstride, v0, v1, K, lane, a0, a1);
#pragma unroll
        for (int u = 0; u < 4; ++u) emit(r + u, a0[u], a1[u]);
    }
    for (; r < nrows; ++r) {
        float a0[1], a1[1];
        cdot_rows_2t<T, 1>(base + (size_t)r * rstride, rstride, v0, v1, K, lane, a0, a1);
        emit(r, a0[0], a1[0]);
    }
}

// Rows [0, nrows) of a static stage (row stride rstride), 4 independent rows
// at a time, then the remainder one by one; emit(row, acc) gets each CDOT.
template <typename T, bool VF, typename Emit>
static __device__ __forceinline__ void stage_rows(const uint8_t *base, size_t rstride, int nrows, const void *v, int K,
                                                  int lane, Emit emit)
{
    // 8 independent row chains at a time (then 4, then 1): the per-row order
    // is the canonical one, the interleaving only hides latency
    int r = 0;
    for (; r + 8 <= nrows; r += 8) {
        float acc[8];
        cdot_rows<T, 8, VF>(base + (size_t)r * rstride, rstride, v, K, lane, acc);
#pragma unroll
        for (int u = 0; u < 8; ++u) emit(r + u, acc[u]);
    }
    for (; r + 4 <= nrows; r += 4) {
        float acc[4];
        cdot_rows<T, 4, VF>(base + (size_t)r * rstride, rstride, v, K, lane, acc);
#pragma unroll
        for (int u = 0; u < 4; ++u) emit(r + u, acc[u]);
    }
    for (; r < nrows; ++r) {
        float acc[1];
        cdot_rows<T, 1, VF>(base + (size_t)r * rstride, rstride, v, K, lane, acc);
        emit(r, acc[0]);
    }
}

// ------------------------------------------------------------------ x_hat staging
// xs[t][:] = x_hat of tokens t0..t0+nt-1, either RMSNorm of the fp32 residual
// (fixed reduction order: every CTA computes bit-identical values) or a copy
// of the caller's x_hat.  One round trip to L2 per token.  CTA 0 writes the
// trace.
template <typename T>
static __device__ bool stage_xhat(const StepParams &p, const Shm &S, int l, int t0, int nt)
{
    using F = F16T<T>;
    const int d = p.d, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint16_t *xs = reinterpret_cast<uint16_t *>(S.xs);
    const int n4 = d / 4; // float4 chunks of a row; thread owns k = tid + 512 q, q < 4
    if (p.mode & M_RMSNORM) {
        for (int t = 0; t < nt; ++t) {
            float4 v[4];
            if (l == 0) {
                // the caller's residual, written before the launch
                const float4 *xr = reinterpret_cast<const float4 *>(p.x + (size_t)(t0 + t) * d);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int k = tid + q * kConsumerThreads;
                    v[q] = k < n4 ? __ldcg(xr + k) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            } else {
                // the previous layer's merge output, from its tagged words
                const uint64_t *xr = p.xx + (size_t)(t0 + t) * d;
                const unsigned ew = p.epoch + l - 1 + (unsigned)p.bar_extra;
#pragma unroll
                for (int h2 = 0; h2 < 4; h2 += 2) { // two float4 per round: fewer live registers
                    uint64_t w[2][4];
                    const auto reload = [&]() {
                        const uint64_t *stale = nullptr;
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int k = tid + (h2 + q) * kConsumerThreads;
                            if (k < n4) {
                                ld_tagged2(xr + 4 * k, w[q][0], w[q][1]);
                                ld_tagged2(xr + 4 * k + 2, w[q][2], w[q][3]);
                            } else {
                                w[q][0] = w[q][1] = w[q][2] = w[q][3] = (uint64_t)ew << 32; // zero-padded
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int k = tid + (h2 + q) * kConsumerThreads;
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (!tag_is(w[q][e], ew)) stale = xr + 4 * k + e;
                        }
                        return stale;
                    };
                    poll_tags(p, fail_word(S), ew, reload(), reload);
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        v[h2 + q] = make_float4(__uint_as_float((uint32_t)w[q][0]), __uint_as_float((uint32_t)w[q][1]),
                                                __uint_as_float((uint32_t)w[q][2]), __uint_as_float((uint32_t)w[q][3]));
                }
            }
            float ss = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                ss = __fmaf_rn(v[q].x, v[q].x, ss);
                ss = __fmaf_rn(v[q].y, v[q].y, ss);
                ss = __fmaf_rn(v[q].z, v[q].z, ss);
                ss = __fmaf_rn(v[q].w, v[q].w, ss);
            }
            ss = butterfly_sum(ss);
            if (lane == 0) S.tmp[warp] = ss;
            if (!cons_sync_ok(fail_word(S))) return false;
            if (tid == 0) {
                float tot = 0.f;
                for (int w = 0; w < kConsumerWarps; ++w) tot = __fadd_rn(tot, S.tmp[w]);
                S.tmp[128] = rsqrtf(__fadd_rn(__fdiv_rn(tot, (float)d), 1e-5f));
            }
            cons_sync();
            const float inv = S.tmp[128];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int k = tid + q * kConsumerThreads;
                if (k < n4) {
                    const uint32_t lo = (uint32_t)F::round(__fmul_rn(v[q].x, inv)) |
                                        ((uint32_t)F::round(__fmul_rn(v[q].y, inv)) << 16);
                    const uint32_t hi = (uint32_t)F::round(__fmul_rn(v[q].z, inv)) |
                                        ((uint32_t)F::round(__fmul_rn(v[q].w, inv)) << 16);
                    *reinterpret_cast<uint2 *>(xs + (size_t)t * d + 4 * k) = make_uint2(lo, hi);
                    if (p.tr_x && blockIdx.x == 0)
                        reinterpret_cast<float4 *>(p.tr_x + ((size_t)l * p.B + t0 + t) * d)[k] = v[q];
                }
            }
        }
    } else {
        for (int t = 0; t < nt; ++t) {
            const uint4 *src = reinterpret_cast<const uint4 *>(p.xhat_in + (size_t)(t0 + t) * d);
            uint4 *dst = reinterpret_cast<uint4 *>(xs + (size_t)t * d);
            for (int k = tid; k < d / 8; k += kConsumerThreads) dst[k] = src[k];
        }
    }
    cons_sync();
    if (p.tr_xhat && blockIdx.x == 0) {
        for (int t = 0; t < nt; ++t) {
            const uint4 *src = reinterpret_cast<const uint4 *>(xs + (size_t)t * d);
            uint4 *dst = reinterpret_cast<uint4 *>(p.tr_xhat + ((size_t)l * p.B + t0 + t) * d);
            for (int k = tid; k < d / 8; k += kConsumerThreads) dst[k] = src[k];
        }
    }
    return true;
}

// ------------------------------------------------------------------ phase A: h = relu(W1 x_hat + b1)
// Warp w consumes exactly the stages that land in slot w (w < nss), so each of
// its waits is one phase ahead of what it last saw (a parity wait cannot tell
// phases two apart).
template <typename T>
static __device__ bool phase_a(const StepParams &p, const Shm &S, const LayerDev &L, int l, uint32_t &ss)
{
    using F = F16T<T>;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const SliceA A = slice_a(L, p);
    bool ok = true;
    const uint16_t *b1s = S.pb1s + off16(L.b1 + A.j0); // b1[A.j0 + k] = b1s[k]
    const int nga = (p.B + p.tg - 1) / p.tg;
    for (int g = 0; g < nga; ++g) {
        const int t0 = g * p.tg, nt = min(p.tg, p.B - t0);
        if (!stage_xhat<T>(p, S, l, t0, nt)) return false; // ends with cons_sync
        wait_cta(S.bias_full, l & 1, p, fail_word(S), ok); // landed long ago: the copy is issued a layer ahead
        for (int k = 0; k < A.nst; ++k) {
            const uint32_t s = ss + k;
            const int slot = s % p.nss;
            if (slot != warp) continue;
            if (!wait_cta(S.full_s + slot, (s / p.nss) & 1, p, fail_word(S), ok)) continue;
            const uint8_t *base = S.ring + (size_t)slot * p.slotB;
            const int jr0 = A.j0 + k * A.rps, nrows = min(A.j1, jr0 + A.rps) - jr0;
            for (int t = 0; t < nt; ++t) {
                stage_rows<T, false>(base, (size_t)L.d * 2, nrows, S.xs + (size_t)t * L.d * 2, L.d, lane,
                                     [&](int r, float acc) {
                                         if (lane == 0) {
                                             const int j = jr0 + r;
                                             const float s1 = __fadd_rn(acc, F::one(b1s[j - A.j0]));
                                             st_tagged(p.hx + (size_t)(t0 + t) * L.r + j, p.epoch + l,
                                                       __float_as_uint(s1 > 0.f ? s1 : 0.f));
                                         }
                                     });
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(S.empty_s + slot);
        }
        ss += A.nst;
        if (!cons_sync_ok(fail_word(S))) return false; // xs is rewritten by the next group
    }
    return true;
}

// ------------------------------------------------------------------ phase B: z = W2 h + b2 > 0
template <typename T>
static __device__ bool phase_b(const StepParams &p, const Shm &S, const LayerDev &L, int l, uint32_t &ss)
{
    using F = F16T<T>;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const SliceB Bs = slice_b(L, p);
    const int nrows = Bs.i1 - Bs.i0;
    const int nwords = (nrows + 31) >> 5;
    for (int k = tid; k < nwords; k += kConsumerThreads) S.swords[k] = 0u;
    const uint16_t *b2s = S.pb2s + off16(L.b2 + Bs.i0); // b2[Bs.i0 + k] = b2s[k] (landed before phase A)
    float *hs = reinterpret_cast<float *>(S.hs);
    const int ngb = (p.B + p.tgB - 1) / p.tgB;
    bool ok = true;
    for (int g = 0; g < ngb; ++g) {
        const int t0 = g * p.tgB, nt = min(p.tgB, p.B - t0);
        // h of the group, straight from the writers' tagged words: the first
        // read usually finds them all; stale ones are polled until phase A of
        // every SM has written them
        {
            const uint64_t *src = p.hx + (size_t)t0 * L.r;
            const unsigned ew = p.epoch + l + (unsigned)p.bar_extra;
            const int nh = nt * L.r;
            for (int k0 = tid; k0 < nh; k0 += 4 * kConsumerThreads) {
                uint64_t v[4];
                const auto reload = [&]() {
                    const uint64_t *stale = nullptr;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int k = k0 + u * kConsumerThreads;
                        v[u] = k < nh ? ld_tagged(src + k) : ((uint64_t)ew << 32);
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (!tag_is(v[u], ew)) stale = src + k0 + u * kConsumerThreads;
                    return stale;
                };
                if (!poll_tags(p, fail_word(S), ew, reload(), reload)) break;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int k = k0 + u * kConsumerThreads;
                    if (k < nh) hs[k] = __uint_as_float((uint32_t)v[u]);
                }
            }
        }
        if (!cons_sync_ok(fail_word(S))) return false;
        for (int k = 0; k < Bs.nst; ++k) {
            const uint32_t s = ss + k;
            const int slot = s % p.nss;
            if (slot != warp) continue;
            if (!wait_cta(S.full_s + slot, (s / p.nss) & 1, p, fail_word(S), ok)) continue;
            const uint8_t *base = S.ring + (size_t)slot * p.slotB;
            const int ir0 = Bs.i0 + k * Bs.rps, nr = min(Bs.i1, ir0 + Bs.rps) - ir0;
            for (int r0 = 0; r0 < nr; r0 += 32) {
                const int nrr = min(32, nr - r0);
                unsigned bits = 0; // bit r: row ir0 + r0 + r selected for some token of the group
                const auto pick = [&](int r, float acc) {
                    if (__fadd_rn(acc, F::one(b2s[ir0 + r0 + r - Bs.i0])) > 0.f) {
                        bits |= 1u << r;
                        if (lane == 0 && (p.mode & M_COUNTS)) atomicAdd(p.counts_out + ir0 + r0 + r, 1);
                    }
                };
                if (nt == 2) { // two tokens share every row chunk's load and widening
                    stage_rows_2t<T>(base + (size_t)r0 * L.r * 2, (size_t)L.r * 2, nrr, hs, hs + L.r, L.r, lane,
                                     [&](int r, float a0, float a1) { pick(r, a0), pick(r, a1); });
                } else {
                    for (int t = 0; t < nt; ++t)
                        stage_rows<T, true>(base + (size_t)r0 * L.r * 2, (size_t)L.r * 2, nrr, hs + (size_t)t * L.r,
                                            L.r, lane, pick);
                }
                if (lane == 0 && (p.mode & M_PREDICT) && bits) {
                    const int rel = ir0 + r0 - Bs.i0; // rows relative to the word-aligned i0
                    const int w0 = rel >> 5, sh = rel & 31;
                    atomicOr(S.swords + w0, bits << sh);
                    if (sh && (bits >> (32 - sh))) atomicOr(S.swords + w0 + 1, bits >> (32 - sh));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(S.empty_s + slot);
        }
        ss += Bs.nst;
        if (!cons_sync_ok(fail_word(S))) return false; // hs is rewritten by the next group
    }
    if (p.mode & M_PREDICT)
        for (int k = tid; k < nwords; k += kConsumerThreads) st_tagged(p.bmx + (Bs.i0 >> 5) + k, p.epoch + l, S.swords[k]);
    return true;
}

// ------------------------------------------------------------------ list resolution
// This CTA's equal share [s0, s1) of the layer's neuron list -> slist/sbias.
// A predicted list comes from an exclusive prefix scan of the bitmap's
// popcounts (each thread owns a contiguous run of at most 4 words), so one
// round trip to L2 suffices.
template <typename T>
static __device__ bool resolve_list(const StepParams &p, const Shm &S, const LayerDev &L, int l)
{
    using F = F16T<T>;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, c = blockIdx.x;
    if ((p.mode & M_FFN) && l > 0) {
        // the dynamic producer must have finished reading layer l-1's list
        bool ok = true;
        wait_cta(S.lst_free, (l - 1) & 1, p, fail_word(S), ok);
        if (!cons_sync_ok(fail_word(S))) return false;
    }
    int m, s0, s1;
    if (p.mode & M_PREDICT) {
        const int nw = (L.n + 31) >> 5;
        const int wpt = (nw + kConsumerThreads - 1) / kConsumerThreads; // <= 4 for n <= 65536
        const int wb = min(nw, tid * wpt), we = min(nw, wb + wpt);
        const int hot = hot_rows(L, p), hw = hot >> 5; // words below hw: the hot prefix, never written
        // the mask words, straight from the writers' tagged words (phase B
        // of every SM), polled until all carry this layer's epoch
        unsigned wv[4];
        {
            const unsigned ew = p.epoch + l + (unsigned)p.bar_extra;
            uint64_t raw[4];
            const auto reload = [&]() {
                const uint64_t *stale = nullptr;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    raw[q] = (wb + q < we && wb + q >= hw) ? ld_tagged(p.bmx + wb + q) : ((uint64_t)ew << 32);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (!tag_is(raw[q], ew)) stale = p.bmx + wb + q;
                return stale;
            };
            poll_tags(p, fail_word(S), ew, reload(), reload);
#pragma unroll
            for (int q = 0; q < 4; ++q) wv[q] = (uint32_t)raw[q] | (wb + q < we ? hot_bits(wb + q, hot) : 0u);
        }
        if (!cons_sync_ok(fail_word(S))) return false;
        int cnt = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) cnt += __popc(wv[q]);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        int *wtot = reinterpret_cast<int *>(S.tmp);
        if (lane == 31) wtot[warp] = incl;
        cons_sync();
        if (tid == 0) {
            int run = 0;
            for (int w = 0; w < kConsumerWarps; ++w) {
                const int v = wtot[w];
                wtot[w] = run;
                run += v;
            }
            S.info[INFO_M] = run;
        }
        cons_sync();
        m = S.info[INFO_M];
        s0 = slice_lo(m, c, G);
        s1 = slice_lo(m, c + 1, G);
        // Lane-parallel extraction: every word that overlaps [s0, s1) is
        // broadcast to its warp, lane j ranks bit j by a popcount of the
        // lower bits and writes it if the rank falls in the slice.
        int pos = wtot[warp] + incl - cnt; // global rank of this thread's first set bit
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int pc = __popc(wv[q]);
            const bool mine = pc && pos < s1 && pos + pc > s0;
            unsigned lanes = __ballot_sync(0xffffffffu, mine);
            while (lanes) {
                const int src = __ffs(lanes) - 1;
                lanes &= lanes - 1;
                const unsigned w = __shfl_sync(0xffffffffu, wv[q], src);
                const int base = __shfl_sync(0xffffffffu, pos, src);
                const int widx = __shfl_sync(0xffffffffu, wb + q, src);
                if ((w >> lane) & 1u) {
                    const int rank = base + __popc(w & ((1u << lane) - 1u));
                    if (rank >= s0 && rank < s1) S.slist[rank - s0] = 32 * widx + lane;
                }
            }
            pos += pc;
        }
        cons_sync();
    } else {
        if (p.mode & M_IDX_IN) {
            if (tid == 0) {
                int v = *(volatile const int32_t *)p.count_in;
                if (v < 0 || v > L.n) {
                    raise_error(p, PI_DEV_FLAG);
                    v = 0;
                }
                S.info[INFO_M] = v;
            }
            cons_sync(); // one read, broadcast: the slice bounds must agree across warps
            m = S.info[INFO_M];
        } else {
            m = L.n;
        }
        s0 = slice_lo(m, c, G);
        s1 = slice_lo(m, c + 1, G);
        for (int k = tid; k < s1 - s0; k += kConsumerThreads) {
            int id = s0 + k;
            if (p.mode & M_IDX_IN) {
                id = p.idx_in[s0 + k];
                if (id < 0 || id >= L.n) {
                    raise_error(p, PI_DEV_FLAG);
                    id = -1;
                }
            }
            S.slist[k] = id;
        }
        cons_sync();
    }
    const int ncnt = s1 - s0;
    for (int k = tid; k < ncnt; k += kConsumerThreads) {
        const int id = S.slist[k];
        // with bias tails the bias arrives in the ring stage with the up row
        if (!L.bias_tail) S.sbias[k] = id >= 0 ? F::one(L.b[id]) : 0.f;
        if (p.idx_out) p.idx_out[s0 + k] = id;
        if (p.tr_idx) p.tr_idx[(size_t)l * p.tr_n + s0 + k] = id;
    }
    if (tid == 0) {
        S.info[INFO_NCNT] = ncnt;
        if (c == 0) {
            if (p.count_out) *p.count_out = m;
            if (p.tr_cnt) p.tr_cnt[l] = m;
        }
    }
    cons_sync();
    return true;
}

// ------------------------------------------------------------------ phase C: gather FFN
// The ring delivers stages (npd whole neurons each) in list order.  Stage k
// is owned by a group of P warps (P = 4, 2 or 1 for rings of up to 4, 8 or 16
// stages), group k mod (16 / P); each of them computes its slice of the
// dot products of the stage's neurons over the rows (W_up, W_gate), writes
// the partial sums to shared memory and arrives on the stage's act_full
// barrier (P arrivals); no other warp takes part, so there is no cross-warp
// reduction and no CTA barrier per stage.  Every warp then forms the
// activations from the P partial sums (in part order), adds the stage's
// down-projection rows into the output columns its threads own and releases
// the stage (empty_d counts the 16 warps).  Owners compute ahead, up to
// `ahead` stages past the stage being merged, on stages that have already
// landed.  With few stages of big neurons one warp's pass over a whole row
// was the longest step of a stage's turn (1.8 us for a LLaMA-70B-shaped
// ReGLU neuron), and owners busy with it delayed every stage's release.
// Output columns of thread `tid`: 16-bit rows -> chunks of 8 columns ch = tid
// and tid + 512 (kYSlots = 16 columns); Q4_0 -> half-block hb = tid (16
// columns of block hb/2).
template <typename T>
static __device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8])
{
    using F = F16T<T>;
    const float2 a = F::pair(v.x), b = F::pair(v.y), c = F::pair(v.z), d = F::pair(v.w);
    f[0] = a.x, f[1] = a.y, f[2] = b.x, f[3] = b.y, f[4] = c.x, f[5] = c.y, f[6] = d.x, f[7] = d.y;
}

// 16 nibbles of a Q4_0 half-block (the low nibbles of its 16 bytes, or the
// high ones) as q - 8, exactly, in eight f16 pairs: element e in half (e & 1)
// of pair e / 2.  A byte permute puts bytes e and e + 1 in the two halves;
// masking a nibble into the mantissa under the exponent of 1024 gives the f16
// value 1024 + q (low nibble) or 1024 + 16 q (high nibble), and one f16-pair
// add or fma takes that to q - 8 (every step is exact in f16).
static __device__ __forceinline__ void q4_pairs(const uint4 v, bool high, uint32_t (&h)[8])
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t t = __byte_perm(w[i], 0u, j == 0 ? 0x4140u : 0x4342u); // bytes 4i+2j, 4i+2j+1
            uint32_t m = (t & (high ? 0x00F000F0u : 0x000F000Fu)) | 0x64006400u;
            __half2 x;
            memcpy(&x, &m, 4);
            // the constants by their f16 bits: 1/16 = 0x2C00, -72 = 0xD480, 1032 = 0x6408
            uint32_t c0 = 0x2C002C00u, c1 = 0xD480D480u, c2 = 0x64086408u;
            __half2 k0, k1, k2;
            memcpy(&k0, &c0, 4);
            memcpy(&k1, &c1, 4);
            memcpy(&k2, &c2, 4);
            x = high ? __hfma2(x, k0, k1) // (1024 + 16q)/16 - 72
                     : __hsub2(x, k2);    // 1024 + q - 1032
            memcpy(&h[2 * i + j], &x, 4);
        }
    }
}

// Warps that share the dot products of one stage: one warp's pass over a
// whole row is the longest step of a stage's turn, so the rows are split
// between P warps, each taking a contiguous slice of every row; the stage's
// act_full barrier counts their P arrivals.  P = 4 whenever the partial sums
// of every stage's neurons and parts fit the shared buffer (nsd x neurons per
// stage x P <= 2 x 16 x 8), else 2; the same P for every layer of the launch
// (the barriers are set up once).  Measured at one token, 12-layer stacks, P
// = 4 against 2: Falcon-40B f16 52.1 -> 50.4 us a layer, Q4_0 52.8 -> 52.4,
// OPT-30B 44.8 -> 44.7; P = 8 was slower everywhere (56.4, 48.1, 54.4).
static __device__ __forceinline__ int owner_parts(const StepParams &p)
{
    int npd = 1;
    for (int l = 0; l < p.L; ++l) npd = max(npd, neurons_per_stage(p.layers[l], p));
    return p.nsd * npd * 4 <= 2 * kConsumerWarps * kMaxNeuronsPerStage ? 4 : 2;
}

// One warp: its slice [c0, c1) (16-bit: chunks of 8 elements; Q4_0:
// half-blocks of 16) of the dot products of one neuron's W_up row (at a)
// and, for ReGLU, its W_gate row (at a + upB) with the nt tokens' x_hat in xs
// (16-bit [t][d]); the slice's sums in every lane.
template <typename T, bool Q4, int TGF, bool REGLU>
static __device__ __forceinline__ void row_dots(const LayerDev &L, uint32_t a, uint32_t upB, uint32_t xs, int d,
                                                int nt, int lane, int c0, int c1, float (&au)[TGF], float (&ag)[TGF])
{
#pragma unroll
    for (int t = 0; t < TGF; ++t) au[t] = ag[t] = 0.f;
    if constexpr (!Q4) {
        // two chains per token (alternate chunks) halve the dependent fma run
        float bu[TGF], bg[TGF];
#pragma unroll
        for (int t = 0; t < TGF; ++t) bu[t] = bg[t] = 0.f;
        for (int ch = c0 + lane; ch < c1; ch += 64) {
            const bool two = ch + 32 < c1;
            const uint4 w0 = ld_shared_v4(a + (uint32_t)ch * 16);
            const uint4 w1 = two ? ld_shared_v4(a + (uint32_t)(ch + 32) * 16) : make_uint4(0, 0, 0, 0);
            uint4 g0 = make_uint4(0, 0, 0, 0), g1 = make_uint4(0, 0, 0, 0);
            if (REGLU) {
                g0 = ld_shared_v4(a + upB + (uint32_t)ch * 16);
                if (two) g1 = ld_shared_v4(a + upB + (uint32_t)(ch + 32) * 16);
            }
#pragma unroll
            for (int t = 0; t < TGF; ++t) {
                if (t < nt) {
                    const uint32_t xr = xs + (uint32_t)(t * d) * 2;
                    const uint4 x0 = ld_shared_v4(xr + (uint32_t)ch * 16);
                    const uint4 x1 = two ? ld_shared_v4(xr + (uint32_t)(ch + 32) * 16) : make_uint4(0, 0, 0, 0);
                    au[t] = fma_chunk<T>(w0, x0, au[t]);
                    bu[t] = fma_chunk<T>(w1, x1, bu[t]);
                    if (REGLU) {
                        ag[t] = fma_chunk<T>(g0, x0, ag[t]);
                        bg[t] = fma_chunk<T>(g1, x1, bg[t]);
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TGF; ++t) au[t] += bu[t], ag[t] += bg[t];
    } else {
        // (Q4_0 layers take f16 activations: x_hat pairs and the q - 8 pairs
        // meet in the mixed-precision fma, an exact product rounded once)
        for (int hb = c0 + lane; hb < c1; hb += 32) {
            const int blk = hb >> 1;
            const bool high = (hb & 1) != 0;
            uint32_t qu[8], qg[8];
            q4_pairs(ld_shared_v4(a + L.scB + blk * 16), high, qu);
            const float su = __half2float(__ushort_as_half(ld_shared_u16(a + blk * 2)));
            float sg = 0.f;
            if (REGLU) {
                q4_pairs(ld_shared_v4(a + upB + L.scB + blk * 16), high, qg);
                sg = __half2float(__ushort_as_half(ld_shared_u16(a + upB + blk * 2)));
            }
#pragma unroll
            for (int t = 0; t < TGF; ++t) {
                if (t < nt) {
                    const uint32_t xb = xs + (uint32_t)(t * d + blk * 32 + (hb & 1) * 16) * 2;
                    const uint4 x0 = ld_shared_v4(xb), x1 = ld_shared_v4(xb + 16);
                    const uint32_t xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    float pu = 0.f, pg = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        pu = fma_pair<__half>(qu[e], xv[e], pu);
                        if (REGLU) pg = fma_pair<__half>(qg[e], xv[e], pg);
                    }
                    au[t] = fmaf(su, pu, au[t]);
                    if (REGLU) ag[t] = fmaf(sg, pg, ag[t]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < TGF; ++t) {
        au[t] = butterfly_sum(au[t]);
        if (REGLU) ag[t] = butterfly_sum(ag[t]);
    }
}

template <typename T, bool Q4, int TGF, bool REGLU, bool SQ>
static __device__ bool phase_c_impl(const StepParams &p, const Shm &S, const LayerDev &L, int l, uint32_t &sd,
                                    bool xs_valid)
{
    using F = F16T<T>;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = L.d;
    const int ncnt = S.info[INFO_NCNT];
    const int nb = neuron_bytes(L);
    const int npd = neurons_per_stage(L, p);
    const int nst = (ncnt + npd - 1) / npd;
    const int ngf = (p.B + p.tg - 1) / p.tg;
    const int nch = d >> 3;     // 16-bit: chunks of 8 columns
    const int nhb = d >> 4;     // Q4_0: half-blocks of 16 columns
    const int ahead = max(0, min(p.nsd - 1, p.lookahead)); // lookahead < nsd keeps the ring deadlock-free
    const uint32_t rowB = (uint32_t)L.rowB;
    const uint32_t upB = (uint32_t)L.upB; // offset of the gate row in a neuron
    const uint32_t dnoff = upB + (REGLU ? rowB : 0u); // offset of the W_down^T row
    const uint32_t ring = smem_u32(S.ring);
    const uint32_t xs = smem_u32(S.xs);
    const int P = S.info[INFO_OWNP];    // warps sharing a stage's dot products
    const int G16 = kConsumerWarps / P; // owner groups: group g owns stages g, g + G16, ...
    const int part = warp % P;
    const int units = Q4 ? nhb : nch;  // this warp's slice of every row it computes
    const int c0 = units * part / P, c1 = units * (part + 1) / P;
    // [nsd][npd][P][TGF][2] partial dot sums (up, gate) of the stages in the ring
    float *red = S.red;
    const auto red_at = [&](uint32_t os, int j, int q, int t) {
        return red + ((((int)os * npd + j) * P + q) * TGF + t) * 2;
    };
    bool ok = true;
    for (int g = 0; g < ngf; ++g) {
        const int t0 = g * p.tg, nt = min(p.tg, p.B - t0);
        // phase A left the x_hat of a single token group in xs
        if (!(xs_valid && ngf == 1) && !stage_xhat<T>(p, S, l, t0, nt)) return false;
        float y[TGF][kYSlots];
#pragma unroll
        for (int t = 0; t < TGF; ++t)
#pragma unroll
            for (int e = 0; e < kYSlots; ++e) y[t][e] = 0.f;

        uint32_t slot = sd % p.nsd, par = (sd / p.nsd) & 1; // ring position of stage k
        int own = warp / P;                                  // next stage this warp's group owns
        for (int k = 0; k < nst; ++k) {
            // ---- owned stages up to k + ahead: this warp's part of their dot products
            while (own < nst && own <= k + ahead) {
                const uint32_t sa = sd + (uint32_t)own;
                const uint32_t os = sa % p.nsd, op = (sa / p.nsd) & 1;
                if (own > k && !mbar_test(S.full_d + os, op)) break; // not landed yet: later
                if (wait_cta(S.full_d + os, op, p, fail_word(S), ok)) {
                    if (own == 0 && g == 0) mark(p, 1 + l * kTimelineEvents + 8);
                    const uint32_t base = ring + os * (uint32_t)p.dslotB;
                    const int nn = min(npd, ncnt - own * npd);
                    for (int j = 0; j < nn; ++j) {
                        float au[TGF], ag[TGF];
                        row_dots<T, Q4, TGF, REGLU>(L, base + (uint32_t)(j * nb), upB, xs, d, nt, lane, c0, c1, au, ag);
                        if (lane == 0) {
#pragma unroll
                            for (int t = 0; t < TGF; ++t) {
                                float *r = red_at(os, j, part, t);
                                r[0] = au[t];
                                r[1] = ag[t];
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(S.act_full + os);
                }
                own += G16;
            }
            // ---- stage k: its down-projection rows into this thread's columns
            if (wait_cta(S.full_d + slot, par, p, fail_word(S), ok) && wait_cta(S.act_full + slot, par, p, fail_word(S), ok)) {
                const uint32_t base = ring + slot * (uint32_t)p.dslotB;
                const int nn = min(npd, ncnt - k * npd);
                for (int j = 0; j < nn; ++j) {
                    // the neuron's activation from its P partial sums, added in part order
                    const int pos = k * npd + j;
                    const float bias = L.bias_tail ? F::one(ld_shared_u16(base + (uint32_t)(j * nb) + rowB)) : S.sbias[pos];
                    const bool live = S.slist[pos] >= 0;
                    float a[TGF];
#pragma unroll
                    for (int t = 0; t < TGF; ++t) {
                        float su = 0.f, sg = 0.f;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (q < P) {
                                const float *r = red_at(slot, j, q, t);
                                su += r[0];
                                sg += r[1];
                            }
                        const float rl = fmaxf((REGLU ? sg : su) + bias, 0.f);
                        const float av = REGLU ? rl * su : (SQ ? rl * rl : rl);
                        a[t] = live && t < nt ? av : 0.f;
                    }
                    const uint32_t dn = base + (uint32_t)(j * nb) + dnoff;
                    if (!Q4) {
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            const int ch = tid + q * kConsumerThreads;
                            if (ch < nch) {
                                float wf[8];
                                unpack8<T>(ld_shared_v4(dn + (uint32_t)ch * 16), wf);
#pragma unroll
                                for (int e = 0; e < 8; ++e)
#pragma unroll
                                    for (int t = 0; t < TGF; ++t) y[t][q * 8 + e] = fmaf(a[t], wf[e], y[t][q * 8 + e]);
                            }
                        }
                    } else {
                        const int hb = tid;
                        if (hb < nhb) {
                            const int blk = hb >> 1;
                            uint32_t qh[8];
                            q4_pairs(ld_shared_v4(dn + L.scB + blk * 16), (hb & 1) != 0, qh);
                            const float s = __half2float(__ushort_as_half(ld_shared_u16(dn + blk * 2)));
                            // a * s rounded to f16 (relative error <= 2^-12), then
                            // its exact products with q - 8 in the mixed-precision
                            // fma: no conversion of the nibble pairs to fp32
#pragma unroll
                            for (int t = 0; t < TGF; ++t) {
                                const uint16_t ab = __half_as_ushort(__float2half_rn(a[t] * s));
#pragma unroll
                                for (int e = 0; e < 8; ++e) {
                                    float lo = y[t][2 * e], hi = y[t][2 * e + 1];
                                    asm("{ .reg .b16 ql, qh, ha; mov.b32 {ql, qh}, %2; mov.b16 ha, %3;"
                                        " fma.rn.f32.f16 %0, ql, ha, %0; fma.rn.f32.f16 %1, qh, ha, %1; }"
                                        : "+f"(lo), "+f"(hi)
                                        : "r"(qh[e]), "h"(ab));
                                    y[t][2 * e] = lo, y[t][2 * e + 1] = hi;
                                }
                            }
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(S.empty_d + slot); // this warp is done with stage k
            if (++slot == (uint32_t)p.nsd) slot = 0, par ^= 1;
        }
        sd += (uint32_t)nst;
        // ---- this CTA's fp32 partial of the layer output
        // (tagged with this layer's epoch: the merge polls these words)
        const unsigned ep = p.epoch + l;
        for (int t = 0; t < nt; ++t) {
            uint64_t *dst = p.partx + ((size_t)blockIdx.x * p.B + t0 + t) * d;
            if (!Q4) {
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int ch = tid + q * kConsumerThreads;
                    if (ch < nch) {
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            float a0 = 0.f, a1 = 0.f; // token t's pair (t is not a compile-time index)
#pragma unroll
                            for (int tt = 0; tt < TGF; ++tt)
                                if (tt == t) a0 = y[tt][q * 8 + e], a1 = y[tt][q * 8 + e + 1];
                            st_tagged2(dst + ch * 8 + e, ep, __float_as_uint(a0), __float_as_uint(a1));
                        }
                    }
                }
            } else {
                const int hb = tid;
                if (hb < nhb) {
                    uint64_t *o = dst + (hb >> 1) * 32 + (hb & 1) * 16;
#pragma unroll
                    for (int e = 0; e < 16; e += 2) {
                        float a0 = 0.f, a1 = 0.f;
#pragma unroll
                        for (int tt = 0; tt < TGF; ++tt)
                            if (tt == t) a0 = y[tt][e], a1 = y[tt][e + 1];
                        st_tagged2(o + e, ep, __float_as_uint(a0), __float_as_uint(a1));
                    }
                }
            }
        }
        if (!cons_sync_ok(fail_word(S))) return false; // xs is rewritten by the next group
    }
    return true;
}

template <typename T, bool Q4, int TGF>
static __device__ bool phase_c(const StepParams &p, const Shm &S, const LayerDev &L, int l, uint32_t &sd,
                               bool xs_valid)
{
    if (L.gate) return phase_c_impl<T, Q4, TGF, true, false>(p, S, L, l, sd, xs_valid);
    if (L.act == ACT_SQRELU) return phase_c_impl<T, Q4, TGF, false, true>(p, S, L, l, sd, xs_valid);
    return phase_c_impl<T, Q4, TGF, false, false>(p, S, L, l, sd, xs_valid);
}

// ------------------------------------------------------------------ phase D: merge
// Units of 4 columns; a warp per unit, its lanes over the partials in a fixed
// order, then a butterfly.  x and b_down are loaded alongside the partials.
// The partials are read straight from the writers' tagged words: the first
// read usually finds them all, stale words are polled until phase C of every
// SM has written them, so no grid barrier stands between C and D.  The new
// residual goes to x and, tagged, to xx, which the next layer polls.
template <typename T>
static __device__ void phase_d(const StepParams &p, const Shm &S, const LayerDev &L, int l)
{
    using F = F16T<T>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, d = L.d;
    const int U = p.B * d / 4;
    const int u0 = slice_lo(U, blockIdx.x, G), u1 = slice_lo(U, blockIdx.x + 1, G);
    const size_t stride = (size_t)p.B * d; // words between two SMs' partials
    const unsigned ep = p.epoch + l, ew = ep + (unsigned)p.bar_extra;
    volatile int *fail = fail_word(S);
    for (int u = u0 + warp; u < u1; u += kConsumerWarps) {
        const int j = (4 * u) % d;
        float4 xv = make_float4(0.f, 0.f, 0.f, 0.f);
        uint2 bd = make_uint2(0, 0);
        if (lane == 0) {
            bd = *reinterpret_cast<const uint2 *>(L.bdown + j);
            if (p.mode & M_RESID) xv = __ldcg(reinterpret_cast<const float4 *>(p.x) + u);
        }
        // Request the first 32 * kPre partials of the unit before the first
        // add, so that they cost one L2 round trip instead of one per 32 SMs;
        // the sum keeps the order cc = lane, lane + 32, ...
        constexpr int kPre = 5;
        uint64_t w[kPre][4];
        const auto reload = [&]() {
            const uint64_t *stale = nullptr;
#pragma unroll
            for (int i = 0; i < kPre; ++i) {
                const int cc = lane + 32 * i;
                if (cc < G) {
                    const uint64_t *a = p.partx + (size_t)cc * stride + 4 * (size_t)u;
                    ld_tagged2(a, w[i][0], w[i][1]);
                    ld_tagged2(a + 2, w[i][2], w[i][3]);
                } else {
                    w[i][0] = w[i][1] = w[i][2] = w[i][3] = (uint64_t)ew << 32; // +0.0
                }
            }
#pragma unroll
            for (int i = 0; i < kPre; ++i) {
                const int cc = lane + 32 * i;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (!tag_is(w[i][e], ew)) stale = p.partx + (size_t)cc * stride + 4 * (size_t)u + e;
            }
            return stale;
        };
        poll_tags(p, fail, ew, reload(), reload);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
            acc.x += __uint_as_float((uint32_t)w[i][0]);
            acc.y += __uint_as_float((uint32_t)w[i][1]);
            acc.z += __uint_as_float((uint32_t)w[i][2]);
            acc.w += __uint_as_float((uint32_t)w[i][3]);
        }
        for (int cc = lane + 32 * kPre; cc < G; cc += 32) {
            // (more than 160 SMs only)
            const uint64_t *a = p.partx + (size_t)cc * stride + 4 * (size_t)u;
            uint64_t v[4];
            const auto reload1 = [&]() {
                const uint64_t *stale = nullptr;
                ld_tagged2(a, v[0], v[1]);
                ld_tagged2(a + 2, v[2], v[3]);
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (!tag_is(v[e], ew)) stale = a + e;
                return stale;
            };
            poll_tags(p, fail, ew, reload1(), reload1);
            acc.x += __uint_as_float((uint32_t)v[0]);
            acc.y += __uint_as_float((uint32_t)v[1]);
            acc.z += __uint_as_float((uint32_t)v[2]);
            acc.w += __uint_as_float((uint32_t)v[3]);
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            acc.x += __shfl_xor_sync(0xffffffffu, acc.x, o);
            acc.y += __shfl_xor_sync(0xffffffffu, acc.y, o);
            acc.z += __shfl_xor_sync(0xffffffffu, acc.z, o);
            acc.w += __shfl_xor_sync(0xffffffffu, acc.w, o);
        }
        if (lane == 0) {
            const float2 b01 = F::pair(bd.x), b23 = F::pair(bd.y);
            acc.x += b01.x;
            acc.y += b01.y;
            acc.z += b23.x;
            acc.w += b23.y;
            if (p.mode & M_RESID) {
                xv.x += acc.x;
                xv.y += acc.y;
                xv.z += acc.z;
                xv.w += acc.w;
                __stcg(reinterpret_cast<float4 *>(p.x) + u, xv);
                if (l + 1 < p.L) {
                    st_tagged2(p.xx + 4 * (size_t)u, ep, __float_as_uint(xv.x), __float_as_uint(xv.y));
                    st_tagged2(p.xx + 4 * (size_t)u + 2, ep, __float_as_uint(xv.z), __float_as_uint(xv.w));
                }
            } else if (p.mode & M_YF32) {
                reinterpret_cast<float4 *>(p.yf_out)[u] = acc;
            } else {
                const uint32_t lo = (uint32_t)F::round(acc.x) | ((uint32_t)F::round(acc.y) << 16);
                const uint32_t hi = (uint32_t)F::round(acc.z) | ((uint32_t)F::round(acc.w) << 16);
                reinterpret_cast<uint2 *>(p.y_out)[u] = make_uint2(lo, hi);
            }
        }
    }
}

// ------------------------------------------------------------------ the kernel
template <typename T, bool Q4, int TGF>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const StepParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const Shm S = carve(smem, p, TGF);
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        for (int i = 0; i < p.nss; ++i) {
            mbar_init(S.full_s + i, 1);
            mbar_init(S.empty_s + i, 1);
        }
        for (int i = 0; i < p.nsd; ++i) {
            mbar_init(S.full_d + i, 1);
            mbar_init(S.empty_d + i, kConsumerWarps);
        }
        mbar_init(S.lst_full, 1);
        mbar_init(S.lst_free, 1);
        mbar_init(S.bias_full, 1);
        const int P = p.nsd > 0 ? owner_parts(p) : 1;
        S.info[INFO_OWNP] = P;
        for (int i = 0; i < p.nsd; ++i) mbar_init(S.act_full + i, P);
        fence_barrier_init();
        S.info[INFO_FAIL] = 0;
        S.info[INFO_REGION] = 0;
        // An earlier launch failed and nobody has cleared the state yet.  Read
        // once and broadcast: every warp of the CTA must take the same path,
        // or the consumer warps that stay would block on a named barrier.
        S.info[INFO_FLAG] = aborted(p) ? 1 : 0;
    }
    __syncthreads();
    if (S.info[INFO_FLAG]) return;
    if (warp == kStaticWarp) {
        if ((tid & 31) == 0) static_producer(p, S);
        return;
    }
    if (warp == kDynamicWarp) {
        if ((tid & 31) == 0) dynamic_producer(p, S);
        return;
    }
    // ---- consumers
    uint32_t ss = 0, sd = 0;
    const bool pred = (p.mode & (M_PREDICT | M_COUNTS)) != 0;
    mark(p, 0);
    for (int l = 0; l < p.L; ++l) {
        const LayerDev L = p.layers[l];
        const int ev = 1 + l * kTimelineEvents;
        if ((p.mode & M_RMSNORM) && !pred && !(p.mode & M_FFN)) {
            // x_hat only (for the tensor-core FFN of large batches): CTA 0
            // writes it through the x_hat trace; with M_DENSE | M_COMPACT
            // the whole list follows
            if (blockIdx.x == 0)
                for (int t0 = 0; t0 < p.B; t0 += p.tg)
                    if (!stage_xhat<T>(p, S, l, t0, min(p.tg, p.B - t0))) return;
            if (!(p.mode & M_COMPACT)) continue;
        }
        if (pred) {
            if (!phase_a<T>(p, S, L, l, ss)) return;
            mark(p, ev + 0);
            mark(p, ev + 1); // (no barrier: phase B polls the tagged h)
            if (!phase_b<T>(p, S, L, l, ss)) return;
            mark(p, ev + 2);
            // without an FFN phase the static producer may now refill the
            // bias slices for the next layer
            if (!(p.mode & M_FFN) && threadIdx.x == 0) atomicAdd(S.info + INFO_REGION, 1);
            if (!(p.mode & (M_FFN | M_COMPACT))) continue;
            mark(p, ev + 3); // (no barrier: the list resolution polls the tagged mask words)
        }
        if (p.mode & (M_FFN | M_COMPACT)) {
            if (!resolve_list<T>(p, S, L, l)) return;
            mark(p, ev + 4);
            if (p.mode & M_FFN) {
                if (threadIdx.x == 0) mbar_arrive(S.lst_full);
                if (!phase_c<T, Q4, TGF>(p, S, L, l, sd, pred)) return;
                // the ring is free again: the static producer may fill it for layer l+1
                if (threadIdx.x == 0) atomicAdd(S.info + INFO_REGION, 1);
                mark(p, ev + 5);
                mark(p, ev + 6); // (no barrier: the merge polls the tagged partials)
                phase_d<T>(p, S, L, l);
                if (!cons_sync_ok(fail_word(S))) return; // (CTA-uniform: every consumer warp leaves or none)
                mark(p, ev + 7);
            }
        }
    }
}

// ------------------------------------------------------------------ launch
// One cooperative launch of step_kernel<T, Q4, tgf> on `grid` CTAs of the
// current device.  The dynamic shared-memory limit is a per-device attribute
// of the kernel, so it is set before every launch (a cached value would be
// wrong for a second device or for a host thread racing with this one; the
// call costs microseconds next to a step of milliseconds).
template <typename T, bool Q4>
cudaError_t launch_step(const StepParams &p, int tgf, int grid, cudaStream_t s)
{
    void (*kern)(const StepParams) =
        tgf == 1 ? step_kernel<T, Q4, 1> : (tgf == 2 ? step_kernel<T, Q4, 2> : step_kernel<T, Q4, 4>);
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

} // namespace pi
