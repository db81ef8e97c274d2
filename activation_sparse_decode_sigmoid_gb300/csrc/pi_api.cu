// Host side of libpi: contexts, layer loading, launch planning and the C ABI
// declared in include/pi.h.  All compute happens in the kernels of
// pi_step_*.cu and pi_load.cu; this file validates arguments, owns device
// memory and plans the shared-memory layout of each launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "pi.h"
#include "pi_kernels.h"

using pi::LayerDev;
using pi::StepParams;

namespace {

struct LayerSlot {
    bool loaded = false;
    int shard = 0, nshards = 1; // neurons shard, shard + nshards, ... of the layer (pi_load_layer_shard)
    pi_layer_desc desc{};
    LayerDev dev{};
    std::vector<void *> bufs;
    // TMA maps of the 16-bit FFN rows for the tensor-core path (one-row boxes for gather4)
    bool maps = false;
    CUtensorMap tm_up{}, tm_gate{}, tm_dn{};
};

int round_up(int v, int a) { return (v + a - 1) / a * a; }

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

} // namespace

struct pi_ctx {
    int device = 0;
    cudaStream_t stream = nullptr;
    int max_layers = 0, max_batch = 0;
    int G = 0;          // SMs = CTAs of the persistent kernels
    int smem_optin = 0; // dynamic shared memory limit per CTA
    std::vector<LayerSlot> layers;
    LayerDev *d_layers = nullptr;
    // workspace
    uint64_t *hx = nullptr;  // tagged predictor hidden layer [max_batch][kMaxRank]
    uint64_t *bmx = nullptr; // tagged mask words [kMaxN / 32]
    unsigned epoch = 1;      // epoch of the next launch's first layer (0 = never written)
    uint64_t *partx = nullptr; // tagged split-K partials [G][max_batch][kMaxD]
    uint64_t *xx = nullptr;    // tagged residual between layers [max_batch][kMaxD]
    float *xstage = nullptr; // [max_batch][kMaxD] residual staging of pi_decode_step_host
    // tensor-core FFN of large batches: activations, x_hat and the list of one layer
    uint16_t *actT = nullptr;    // [2][max_batch][kMaxN]: hi, then lo parts of the activations
    uint16_t *xhat_ws = nullptr; // [max_batch][kMaxD]
    int32_t *lidx = nullptr;     // [kMaxN] list, then [1] its count
    float *mpart = nullptr;      // [8][max_batch][kMaxD] partials of the tensor-core down-projection
    float *hbuf = nullptr;       // [max_batch][kMaxRank] predictor hidden layer of large batches
    uint32_t *mbits = nullptr;   // [kMaxN / 32] union mask words of large batches
    bool h_batched = false;      // the last predictor pass was the batched one (h in hbuf)
    // Batches of at least this many tokens run layer by layer: batched predictor launches and the
    // tensor-core FFN (0: never; -1: by layer kind, see layerwise_min_b).
    int mma_min_b = -1;
    int *ctl = nullptr; // [0..1] grid-barrier counter (u64), [2] status, [3] abort
    // trace
    float *tr_x = nullptr;
    void *tr_xhat = nullptr;
    int32_t *tr_idx = nullptr;
    int32_t *tr_cnt = nullptr;
    unsigned long long wait_ns = 2000000000ull;
    int bar_extra = 0;
    unsigned long long *timeline = nullptr;
    int tl_stride = 0;
    // tuning, see StepParams; prefetch -1: by the weights (paced, mode 2, for
    // Q4_0 stacks, whose FFN phase leaves HBM time to spare; none for 16-bit
    // ones, where it slows the latency-bound reads)
    int prefetch = -1, prefetch_ns = 800, lookahead = 16, rows_ahead = 0;
    std::string err;
};

namespace {

pi_status fail(pi_ctx *c, pi_status code, const char *fmt, ...)
{
    if (c) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        c->err = buf;
    }
    return code;
}

#define CU(call)                                                                                        \
    do {                                                                                                \
        cudaError_t e_ = (call);                                                                        \
        if (e_ != cudaSuccess)                                                                          \
            return fail(c, e_ == cudaErrorMemoryAllocation ? PI_ERR_OOM : PI_ERR_CUDA, "%s: %s (%s:%d)", \
                        #call, cudaGetErrorString(e_), __FILE__, __LINE__);                            \
    } while (0)

void free_layer(LayerSlot &s)
{
    for (void *p : s.bufs) cudaFree(p);
    s.bufs.clear();
    s.loaded = false;
    s.dev = LayerDev{};
}

bool valid_dtype16(int dt) { return dt == PI_F16 || dt == PI_BF16; }

pi_status check_desc(pi_ctx *c, const pi_layer_desc *d)
{
    if (!d) return fail(c, PI_ERR_ARG, "desc is NULL");
    if (d->act != PI_RELU && d->act != PI_REGLU && d->act != PI_SQRELU) return fail(c, PI_ERR_ARG, "act %d invalid", d->act);
    if (!valid_dtype16(d->act_dtype)) return fail(c, PI_ERR_ARG, "act_dtype %d invalid", d->act_dtype);
    if (d->w_dtype != d->act_dtype && !(d->w_dtype == PI_Q4_0 && d->act_dtype == PI_F16))
        return fail(c, PI_ERR_ARG, "w_dtype %d with act_dtype %d unsupported", d->w_dtype, d->act_dtype);
    if (d->d_model < 8 || d->d_model > pi::kMaxD || d->d_model % 8)
        return fail(c, PI_ERR_SHAPE, "d_model %d outside [8, %d] or not a multiple of 8", d->d_model, pi::kMaxD);
    if (d->w_dtype == PI_Q4_0 && d->d_model % 32)
        return fail(c, PI_ERR_SHAPE, "Q4_0 needs d_model %% 32 == 0 (got %d)", d->d_model);
    if (d->d_ffn < 1 || d->d_ffn > pi::kMaxN) return fail(c, PI_ERR_SHAPE, "d_ffn %d outside [1, %d]", d->d_ffn, pi::kMaxN);
    if (d->rank < 8 || d->rank > pi::kMaxRank || d->rank % 8)
        return fail(c, PI_ERR_SHAPE, "rank %d outside [8, %d] or not a multiple of 8", d->rank, pi::kMaxRank);
    return PI_OK;
}

pi_status dev_alloc(pi_ctx *c, LayerSlot &s, void **out, size_t bytes)
{
    void *p = nullptr;
    CU(cudaMalloc(&p, bytes < 16 ? 16 : bytes));
    s.bufs.push_back(p);
    *out = p;
    return PI_OK;
}

// The stack = slots 0..L-1, all loaded, same d_model / act_dtype / weight kind.
pi_status stack_layers(pi_ctx *c, int *L_out)
{
    int L = 0;
    while (L < c->max_layers && c->layers[L].loaded) ++L;
    if (L == 0) return fail(c, PI_ERR_NOT_LOADED, "no layer loaded in slot 0");
    for (int l = L; l < c->max_layers; ++l)
        if (c->layers[l].loaded) return fail(c, PI_ERR_NOT_LOADED, "slot %d empty but slot %d loaded", L, l);
    const pi_layer_desc &d0 = c->layers[0].desc;
    for (int l = 1; l < L; ++l) {
        const pi_layer_desc &d = c->layers[l].desc;
        if (d.d_model != d0.d_model || d.act_dtype != d0.act_dtype || (d.w_dtype == PI_Q4_0) != (d0.w_dtype == PI_Q4_0))
            return fail(c, PI_ERR_UNSUPPORTED, "layer %d differs from layer 0 in d_model, act_dtype or weight kind", l);
    }
    *L_out = L;
    return PI_OK;
}

// Shared-memory plan of one launch of the step kernel: the ring region is
// time-shared between the static view (16 KB slots for predictor rows) and
// the dynamic view (stages holding whole neurons for the FFN phase).
pi_status plan(pi_ctx *c, StepParams &p, int l0, int L, int B, int mode, int *tgf_out)
{
    const pi_layer_desc &d0 = c->layers[l0].desc;
    const int d = d0.d_model, G = c->G;
    int rmax = 0, nmax = 0, nbmax = 0;
    for (int l = l0; l < l0 + L; ++l) {
        const LayerSlot &s = c->layers[l];
        rmax = std::max(rmax, s.desc.rank);
        nmax = std::max(nmax, s.desc.d_ffn);
        nbmax = std::max(nbmax, s.dev.upB + (s.desc.act == PI_REGLU ? 2 : 1) * s.dev.rowB);
    }
    const bool pred = (mode & (pi::M_PREDICT | pi::M_COUNTS)) != 0;
    const bool ffn = (mode & pi::M_FFN) != 0;
    // token-group width of the FFN phase: 1, 2 or 4 tokens (the y accumulators
    // of a wider group do not fit the registers of 576 threads and spill)
    const int tgf = B == 1 ? 1 : (B == 2 ? 2 : 4);
    p.d = d;
    p.B = B;
    p.tg = std::min(B, tgf);
    p.tgB = pred ? std::min(B, 4) : 1;
    const int xsB = round_up(p.tg * d * 2, 128);
    const int hB = pred ? round_up(p.tgB * rmax * 4, 128) : 0;
    p.lcap = (nmax + G - 1) / G + 2;
    const int words = (nmax + 31) / 32;
    p.wcap = (words + G - 1) / G + 1;
    p.rcap = std::max((rmax + G - 1) / G + 1, p.wcap * 32);
    const int misc_bound = pi::misc_layout(pi::kConsumerWarps, 16, p.lcap, p.wcap, p.rcap, tgf).total;
    const int ringB = (c->smem_optin - misc_bound - xsB - hB) / 128 * 128;
    p.slotB = 16384;
    p.nss = pred ? std::min(pi::kConsumerWarps, ringB / p.slotB) : 0; // one consumer warp per slot
    if (pred && p.nss < 2) return fail(c, PI_ERR_UNSUPPORTED, "predictor ring does not fit shared memory");
    // FFN stages: as many as the ring holds, up to 16, each of up to three
    // whole neurons within about 28 KB: a 16-bit neuron of 24 KB or more takes
    // a stage of its own, three Q4_0 neurons share one.  Measured at one token
    // (Falcon-40B-shaped Q4_0, 12-layer stack, us a layer): one neuron a stage
    // 53.5, two 50.3, three 49.6, four 52.0
    const int per_stage = std::min(3, std::max(1, 28672 / std::max(1, nbmax)));
    p.dslotB = ffn ? round_up(per_stage * nbmax, 128) : 0;
    p.nsd = ffn ? std::min(16, ringB / p.dslotB) : 0;
    if (ffn && p.nsd < 2)
        return fail(c, PI_ERR_UNSUPPORTED, "a neuron (%d bytes) does not fit two pipeline stages", nbmax);
    p.ringB = ringB;
    p.off_h = ringB;
    p.hB = hB;
    p.off_xs = p.off_h + hB;
    p.off_misc = p.off_xs + xsB;
    p.smem_bytes = p.off_misc + pi::misc_layout(p.nss, p.nsd, p.lcap, p.wcap, p.rcap, tgf).total;
    if (p.smem_bytes > c->smem_optin) return fail(c, PI_ERR_UNSUPPORTED, "plan needs %d bytes of shared memory", p.smem_bytes);
    *tgf_out = tgf;
    return PI_OK;
}

pi_status launch(pi_ctx *c, int l0, int L, int B, int mode, StepParams &p)
{
    int tgf = 1;
    pi_status st = plan(c, p, l0, L, B, mode, &tgf);
    if (st) return st;
    p.layers = c->d_layers + l0;
    p.L = L;
    p.mode = mode;
    if (mode & (pi::M_PREDICT | pi::M_COUNTS)) c->h_batched = false;
    if (c->epoch > 0xF0000000u - (unsigned)L) {
        // epochs would wrap: clear every tag so that no stale word can match
        const size_t bd = (size_t)c->max_batch * pi::kMaxD;
        cudaError_t e = cudaMemsetAsync(c->hx, 0, sizeof(uint64_t) * (size_t)c->max_batch * pi::kMaxRank, c->stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(c->bmx, 0, sizeof(uint64_t) * (size_t)(pi::kMaxN / 32), c->stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(c->partx, 0, sizeof(uint64_t) * (size_t)c->G * bd, c->stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(c->xx, 0, sizeof(uint64_t) * bd, c->stream);
        if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "tag reset: %s", cudaGetErrorString(e));
        c->epoch = 1;
    }
    p.hx = c->hx;
    p.bmx = c->bmx;
    p.epoch = c->epoch;
    p.partx = c->partx;
    p.xx = c->xx;
    p.status = c->ctl + 2;
    p.abort_flag = c->ctl + 3;
    p.wait_ns = c->wait_ns;
    p.bar_extra = c->bar_extra;
    p.timeline = c->timeline;
    p.tl_stride = c->tl_stride;
    const pi_layer_desc &d0 = c->layers[l0].desc;
    // (Falcon-40B-shaped stacks at one token, tokens/s without / with the paced
    // prefetch: Q4_0 339.3 / 344.6, f16 333.1 / 308.5)
    p.prefetch = c->prefetch >= 0 ? c->prefetch : (d0.w_dtype == PI_Q4_0 ? 2 : 0);
    p.prefetch_ns = c->prefetch_ns;
    p.lookahead = c->lookahead;
    p.rows_ahead = c->rows_ahead;
    cudaError_t e;
    if (d0.w_dtype == PI_Q4_0) e = pi::launch_step_q4(p, tgf, c->G, c->stream);
    else if (d0.act_dtype == PI_BF16) e = pi::launch_step_bf16(p, tgf, c->G, c->stream);
    else e = pi::launch_step_f16(p, tgf, c->G, c->stream);
    if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "step kernel launch: %s", cudaGetErrorString(e));
    c->epoch += (unsigned)L; // the next launch's words can never match this one's
    return PI_OK;
}

pi_status check_layer(pi_ctx *c, int layer)
{
    if (layer < 0 || layer >= c->max_layers) return fail(c, PI_ERR_ARG, "layer %d outside [0, %d)", layer, c->max_layers);
    if (!c->layers[layer].loaded) return fail(c, PI_ERR_NOT_LOADED, "layer %d not loaded", layer);
    return PI_OK;
}

pi_status check_batch(pi_ctx *c, int B)
{
    if (B < 1 || B > c->max_batch) return fail(c, PI_ERR_ARG, "batch %d outside [1, %d]", B, c->max_batch);
    return PI_OK;
}

} // namespace

extern "C" {

pi_status pi_create(pi_ctx **out, int32_t device, void *stream, int32_t max_layers, int32_t max_batch)
{
    if (!out) return PI_ERR_ARG;
    *out = nullptr;
    if (max_layers < 1 || max_layers > 4096 || max_batch < 1 || max_batch > pi::kMaxBatch) return PI_ERR_ARG;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return PI_ERR_CUDA;
    DeviceGuard g(device);
    pi_ctx *c = new pi_ctx();
    c->device = device;
    c->stream = (cudaStream_t)stream;
    c->max_layers = max_layers;
    c->max_batch = max_batch;
    c->layers.resize(max_layers);
    // tuning knobs (defaults are the measured best on GB300)
    if (const char *v = getenv("PI_PREFETCH")) c->prefetch = atoi(v);
    if (const char *v = getenv("PI_PREFETCH_NS")) c->prefetch_ns = atoi(v);
    if (const char *v = getenv("PI_LOOKAHEAD")) c->lookahead = atoi(v) >= 0 ? atoi(v) : 0;
    if (const char *v = getenv("PI_ROWS_AHEAD")) c->rows_ahead = atoi(v) > 0 ? atoi(v) : 0;
    int coop = 0;
    cudaError_t e = cudaDeviceGetAttribute(&c->G, cudaDevAttrMultiProcessorCount, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
    if (e != cudaSuccess || !coop) {
        delete c;
        return PI_ERR_CUDA;
    }
    size_t need[] = {sizeof(LayerDev) * (size_t)max_layers,
                     sizeof(uint64_t) * (size_t)max_batch * pi::kMaxRank,
                     sizeof(uint64_t) * (size_t)(pi::kMaxN / 32),
                     sizeof(float) * (size_t)max_batch * pi::kMaxD,
                     sizeof(uint64_t) * (size_t)c->G * max_batch * pi::kMaxD,
                     sizeof(uint64_t) * (size_t)max_batch * pi::kMaxD,
                     sizeof(int) * 64,
                     2 * sizeof(uint16_t) * (size_t)max_batch * pi::kMaxN,
                     sizeof(uint16_t) * (size_t)max_batch * pi::kMaxD,
                     sizeof(int32_t) * ((size_t)pi::kMaxN + 64),
                     sizeof(float) * 8 * (size_t)max_batch * pi::kMaxD,
                     sizeof(float) * (size_t)max_batch * pi::kMaxRank,
                     sizeof(uint32_t) * (size_t)(pi::kMaxN / 32)};
    constexpr int kBufs = (int)(sizeof need / sizeof need[0]);
    void *ptrs[kBufs] = {};
    for (int i = 0; i < kBufs && e == cudaSuccess; ++i) e = cudaMalloc(&ptrs[i], need[i]);
    // zero everything: epoch 0 is never a valid tag
    for (int i = 0; i < kBufs && e == cudaSuccess; ++i)
        if (i != 3) e = cudaMemset(ptrs[i], 0, need[i]);
    if (e != cudaSuccess) {
        for (void *p : ptrs) cudaFree(p);
        delete c;
        return e == cudaErrorMemoryAllocation ? PI_ERR_OOM : PI_ERR_CUDA;
    }
    c->d_layers = (LayerDev *)ptrs[0];
    c->hx = (uint64_t *)ptrs[1];
    c->bmx = (uint64_t *)ptrs[2];
    c->xstage = (float *)ptrs[3];
    c->partx = (uint64_t *)ptrs[4];
    c->xx = (uint64_t *)ptrs[5];
    c->ctl = (int *)ptrs[6];
    c->actT = (uint16_t *)ptrs[7];
    c->xhat_ws = (uint16_t *)ptrs[8];
    c->lidx = (int32_t *)ptrs[9];
    c->mpart = (float *)ptrs[10];
    c->hbuf = (float *)ptrs[11];
    c->mbits = (uint32_t *)ptrs[12];
    *out = c;
    return PI_OK;
}

pi_status pi_destroy(pi_ctx *c)
{
    if (!c) return PI_ERR_ARG;
    {
        DeviceGuard g(c->device);
        cudaStreamSynchronize(c->stream);
        for (LayerSlot &s : c->layers) free_layer(s);
        cudaFree(c->d_layers);
        cudaFree(c->hx);
        cudaFree(c->bmx);
        cudaFree(c->partx);
        cudaFree(c->xx);
        cudaFree(c->xstage);
        cudaFree(c->ctl);
        cudaFree(c->actT);
        cudaFree(c->xhat_ws);
        cudaFree(c->lidx);
        cudaFree(c->mpart);
        cudaFree(c->hbuf);
        cudaFree(c->mbits);
    }
    delete c;
    return PI_OK;
}

pi_status pi_set_stream(pi_ctx *c, void *stream)
{
    if (!c) return PI_ERR_ARG;
    c->stream = (cudaStream_t)stream;
    return PI_OK;
}

// Load the neurons sel[0..nl) (host, original ids in [0, desc->d_ffn); NULL =
// all of them in order, nl = d_ffn) into slot `layer`: physical neuron i of
// the slot is original neuron sel[i].  The predictor's hidden layer (W1, b1)
// is copied whole; W2 rows, b2, the FFN rows and their biases only for the
// selected neurons; b_down when with_bdown, else zeros.
static pi_status load_rows(pi_ctx *c, int32_t layer, const pi_layer_desc *desc, const pi_layer_weights *w,
                           const int32_t *sel, int nl, bool with_bdown);

pi_status pi_load_layer(pi_ctx *c, int32_t layer, const pi_layer_desc *desc, const pi_layer_weights *w,
                        const int32_t *perm)
{
    if (!c) return PI_ERR_ARG;
    if (layer < 0 || layer >= c->max_layers) return fail(c, PI_ERR_ARG, "layer %d outside [0, %d)", layer, c->max_layers);
    pi_status st = check_desc(c, desc);
    if (st) return st;
    const int n = desc->d_ffn;
    if (perm) {
        std::vector<char> seen(n, 0);
        for (int i = 0; i < n; ++i) {
            if (perm[i] < 0 || perm[i] >= n || seen[perm[i]]) return fail(c, PI_ERR_ARG, "perm is not a permutation of 0..%d", n - 1);
            seen[perm[i]] = 1;
        }
    }
    st = load_rows(c, layer, desc, w, perm, n, true);
    if (!st) c->layers[layer].shard = 0, c->layers[layer].nshards = 1;
    return st;
}

pi_status pi_load_layer_shard(pi_ctx *c, int32_t layer, const pi_layer_desc *desc, const pi_layer_weights *w,
                              const int32_t *perm, int32_t shard, int32_t nshards)
{
    if (!c) return PI_ERR_ARG;
    if (layer < 0 || layer >= c->max_layers) return fail(c, PI_ERR_ARG, "layer %d outside [0, %d)", layer, c->max_layers);
    pi_status st = check_desc(c, desc);
    if (st) return st;
    const int n = desc->d_ffn;
    if (nshards < 1 || shard < 0 || shard >= nshards || nshards > n)
        return fail(c, PI_ERR_ARG, "shard %d of %d invalid for %d neurons", shard, nshards, n);
    std::vector<int32_t> sel;
    for (int i = shard; i < n; i += nshards) sel.push_back(perm ? perm[i] : i);
    if (perm) {
        std::vector<char> seen(n, 0);
        for (int i = 0; i < n; ++i) {
            if (perm[i] < 0 || perm[i] >= n || seen[perm[i]]) return fail(c, PI_ERR_ARG, "perm is not a permutation of 0..%d", n - 1);
            seen[perm[i]] = 1;
        }
    }
    st = load_rows(c, layer, desc, w, sel.data(), (int)sel.size(), shard == 0);
    if (!st) c->layers[layer].shard = shard, c->layers[layer].nshards = nshards;
    return st;
}

static pi_status load_rows(pi_ctx *c, int32_t layer, const pi_layer_desc *desc, const pi_layer_weights *w,
                           const int32_t *perm, int nl, bool with_bdown)
{
    if (!w || !w->w_up || !w->w_down || !w->p_w1 || !w->p_w2) return fail(c, PI_ERR_ARG, "missing weight pointer");
    if (desc->act == PI_REGLU && !w->w_gate) return fail(c, PI_ERR_ARG, "ReGLU needs w_gate");
    const int d = desc->d_model, nsrc = desc->d_ffn, r = desc->rank;
    const int n = nl; // neurons held by the slot
    DeviceGuard g(c->device);
    CU(cudaStreamSynchronize(c->stream));
    LayerSlot &s = c->layers[layer];
    free_layer(s);
    const bool q4 = desc->w_dtype == PI_Q4_0;
    const bool reglu = desc->act == PI_REGLU;
    const int scB = q4 ? round_up((d / 32) * 2, 16) : 0;
    const int rowB = q4 ? scB + d / 2 : 2 * d;
    const size_t srcRow = q4 ? (size_t)(d / 32) * 18 : (size_t)2 * d; // bytes of a source FFN row
    LayerDev &L = s.dev;
    L.d = d;
    L.n = n;
    L.r = r;
    L.act = desc->act;
    L.q4 = q4;
    L.rowB = rowB;
    L.scB = scB;
    L.upB = rowB + 16; // W_up rows carry the neuron's bias in a 16-byte tail
    L.bias_tail = 1;
    void *pw1 = nullptr, *pb1 = nullptr, *pw2 = nullptr, *pb2 = nullptr, *pup = nullptr, *pgate = nullptr,
         *pdn = nullptr, *pb = nullptr, *pbd = nullptr;
#define ALLOC(ptr, bytes)                                 \
    do {                                                  \
        pi_status s_ = dev_alloc(c, s, &(ptr), (bytes)); \
        if (s_) {                                         \
            free_layer(s);                                \
            return s_;                                    \
        }                                                 \
    } while (0)
    ALLOC(pw1, (size_t)r * d * 2);
    ALLOC(pb1, (size_t)r * 2 + 32); // + 32: the kernel copies 16-byte-rounded slices
    ALLOC(pw2, (size_t)n * r * 2);
    ALLOC(pb2, (size_t)n * 2 + 32);
    ALLOC(pup, (size_t)n * (rowB + 16));
    if (reglu) ALLOC(pgate, (size_t)n * rowB);
    ALLOC(pdn, (size_t)n * rowB);
    ALLOC(pb, (size_t)n * 2);
    ALLOC(pbd, (size_t)d * 2);
#undef ALLOC
    // staging of host sources and of the permutation
    std::vector<void *> tmp;
    auto cleanup = [&]() {
        for (void *p : tmp) cudaFree(p);
    };
    auto src = [&](const void *p, size_t bytes, const void **out) -> pi_status {
        if (!p) {
            *out = nullptr;
            return PI_OK;
        }
        if (w->on_device) {
            *out = p;
            return PI_OK;
        }
        void *dptr = nullptr;
        cudaError_t e = cudaMalloc(&dptr, bytes);
        if (e != cudaSuccess) return fail(c, PI_ERR_OOM, "staging %zu bytes: %s", bytes, cudaGetErrorString(e));
        tmp.push_back(dptr);
        e = cudaMemcpy(dptr, p, bytes, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "staging copy: %s", cudaGetErrorString(e));
        *out = dptr;
        return PI_OK;
    };
    const void *s_up, *s_gate, *s_b, *s_dn, *s_bd, *s_w1, *s_b1, *s_w2, *s_b2;
    int32_t *dperm = nullptr;
    pi_status rc = PI_OK;
    if (!rc) rc = src(w->w_up, nsrc * srcRow, &s_up);
    if (!rc) rc = src(w->w_gate, nsrc * srcRow, &s_gate);
    if (!rc) rc = src(w->b, (size_t)nsrc * 2, &s_b);
    if (!rc) rc = src(w->w_down, q4 ? nsrc * srcRow : (size_t)d * nsrc * 2, &s_dn);
    if (!rc) rc = src(with_bdown ? w->b_down : nullptr, (size_t)d * 2, &s_bd);
    if (!rc) rc = src(w->p_w1, (size_t)r * d * 2, &s_w1);
    if (!rc) rc = src(w->p_b1, (size_t)r * 2, &s_b1);
    if (!rc) rc = src(w->p_w2, (size_t)nsrc * r * 2, &s_w2);
    if (!rc) rc = src(w->p_b2, (size_t)nsrc * 2, &s_b2);
    if (!rc && perm) {
        cudaError_t e = cudaMalloc((void **)&dperm, (size_t)n * 4);
        if (e == cudaSuccess) {
            tmp.push_back(dperm);
            e = cudaMemcpy(dperm, perm, (size_t)n * 4, cudaMemcpyHostToDevice);
        }
        if (e != cudaSuccess) rc = fail(c, PI_ERR_CUDA, "perm staging: %s", cudaGetErrorString(e));
    }
    cudaStream_t st0 = c->stream;
    cudaError_t e = cudaSuccess;
    auto chk = [&](cudaError_t x) {
        if (e == cudaSuccess) e = x;
    };
    if (!rc) {
        if (q4) {
            chk(pi::launch_q4_split((const uint8_t *)s_up, (uint8_t *)pup, dperm, n, d, scB, st0, (size_t)rowB + 16));
            if (reglu) chk(pi::launch_q4_split((const uint8_t *)s_gate, (uint8_t *)pgate, dperm, n, d, scB, st0));
            chk(pi::launch_q4_split((const uint8_t *)s_dn, (uint8_t *)pdn, dperm, n, d, scB, st0));
        } else {
            chk(pi::launch_permute_rows(s_up, pup, dperm, n, (size_t)rowB, st0, (size_t)rowB + 16));
            if (reglu) chk(pi::launch_permute_rows(s_gate, pgate, dperm, n, (size_t)rowB, st0));
            chk(pi::launch_transpose_permute16((const uint16_t *)s_dn, (uint16_t *)pdn, dperm, d, n, nsrc, st0));
        }
        if (s_b) chk(pi::launch_permute16((const uint16_t *)s_b, (uint16_t *)pb, dperm, n, st0));
        else chk(cudaMemsetAsync(pb, 0, (size_t)n * 2, st0));
        chk(pi::launch_bias_tail((const uint16_t *)pb, (uint8_t *)pup, n, (size_t)rowB, (size_t)rowB + 16, st0));
        chk(cudaMemcpyAsync(pw1, s_w1, (size_t)r * d * 2, cudaMemcpyDeviceToDevice, st0));
        if (s_b1) chk(cudaMemcpyAsync(pb1, s_b1, (size_t)r * 2, cudaMemcpyDeviceToDevice, st0));
        else chk(cudaMemsetAsync(pb1, 0, (size_t)r * 2, st0));
        chk(pi::launch_permute_rows(s_w2, pw2, dperm, n, (size_t)r * 2, st0));
        if (s_b2) chk(pi::launch_permute16((const uint16_t *)s_b2, (uint16_t *)pb2, dperm, n, st0));
        else chk(cudaMemsetAsync(pb2, 0, (size_t)n * 2, st0));
        if (s_bd) chk(cudaMemcpyAsync(pbd, s_bd, (size_t)d * 2, cudaMemcpyDeviceToDevice, st0));
        else chk(cudaMemsetAsync(pbd, 0, (size_t)d * 2, st0));
        chk(cudaStreamSynchronize(st0));
        if (e != cudaSuccess) rc = fail(c, PI_ERR_CUDA, "layer load: %s", cudaGetErrorString(e));
    }
    cleanup();
    if (rc) {
        free_layer(s);
        return rc;
    }
    L.w1 = (const uint16_t *)pw1;
    L.b1 = (const uint16_t *)pb1;
    L.w2 = (const uint16_t *)pw2;
    L.b2 = (const uint16_t *)pb2;
    L.up = (const uint8_t *)pup;
    L.gate = (const uint8_t *)pgate;
    L.dn = (const uint8_t *)pdn;
    L.b = (const uint16_t *)pb;
    L.bdown = (const uint16_t *)pbd;
    e = cudaMemcpy(c->d_layers + layer, &L, sizeof(LayerDev), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        free_layer(s);
        return fail(c, PI_ERR_CUDA, "layer table: %s", cudaGetErrorString(e));
    }
    s.desc = *desc;
    s.desc.d_ffn = n; // the neurons this slot holds
    s.loaded = true;
    s.maps = false;
    if (q4) {
        s.maps = true; // batches dequantise the rows in the tensor-core kernels' shared memory
    } else {
        cudaError_t me = pi::encode_map(&s.tm_up, pup, (uint64_t)d, (uint64_t)n, (uint64_t)rowB + 16, 1);
        if (me == cudaSuccess && reglu) me = pi::encode_map(&s.tm_gate, pgate, (uint64_t)d, (uint64_t)n, (uint64_t)rowB, 1);
        if (me == cudaSuccess) me = pi::encode_map(&s.tm_dn, pdn, (uint64_t)d, (uint64_t)n, (uint64_t)rowB, 1);
        s.maps = me == cudaSuccess; // without maps the layer keeps the CUDA-core path
    }
    return PI_OK;
}

pi_status pi_perm_from_counts(const int32_t *counts, int32_t n, int32_t *perm)
{
    if (!counts || !perm || n < 1) return PI_ERR_ARG;
    for (int i = 0; i < n; ++i) perm[i] = i;
    std::stable_sort(perm, perm + n, [&](int32_t a, int32_t b) { return counts[a] > counts[b]; });
    return PI_OK;
}

pi_status pi_hot_prefix_crossover(const int32_t *counts, int32_t n, int32_t T, int32_t B, double pred_bytes,
                                  double ffn_bytes, int32_t *hot)
{
    if (!counts || !hot || n < 1 || T < 1 || B < 1 || !(pred_bytes > 0.0) || !(ffn_bytes > 0.0)) return PI_ERR_ARG;
    for (int i = 0; i < n; ++i)
        if (counts[i] < 0 || counts[i] > T) return PI_ERR_ARG;
    // computing neuron i unconditionally saves its predictor bytes P and costs
    // F (1 - q_i) more FFN bytes, q_i = 1 - (1 - c_i / T)^B the chance that the
    // union over B tokens selects it: the prefix runs while (1 - q_i) F < P
    const double keep = pred_bytes / ffn_bytes;
    int h = 0;
    while (h < n && std::pow((double)(T - counts[h]) / (double)T, (double)B) < keep) ++h;
    *hot = h;
    return PI_OK;
}

static void neuron_cost(const pi_layer_desc &d, double &pred, double &ffn)
{
    const double w = d.w_dtype == PI_Q4_0 ? 18.0 / 32.0 : 2.0;
    pred = 2.0 * d.rank + 2.0;                                              // W2 row + b2
    ffn = (d.act == PI_REGLU ? 2.0 : 1.0) * d.d_model * w + 2.0 + d.d_model * w; // up (+ gate) + bias + down
}

pi_status pi_choose_hot_prefix(pi_ctx *c, int32_t layer, const int32_t *counts, int32_t T, int32_t B, int32_t *hot)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_layer(c, layer);
    if (st) return st;
    double pred, ffn;
    neuron_cost(c->layers[layer].desc, pred, ffn);
    st = pi_hot_prefix_crossover(counts, c->layers[layer].desc.d_ffn, T, B, pred, ffn, hot);
    return st ? fail(c, st, "counts/hot NULL, T or B < 1, or a count outside [0, T]") : PI_OK;
}

pi_status pi_set_hot_prefix(pi_ctx *c, int32_t layer, int32_t hot)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_layer(c, layer);
    if (st) return st;
    LayerSlot &s = c->layers[layer];
    if (hot < 0 || hot > s.desc.d_ffn) return fail(c, PI_ERR_ARG, "hot prefix %d outside [0, %d]", hot, s.desc.d_ffn);
    DeviceGuard g(c->device);
    // steps in flight read the layer's descriptor
    CU(cudaStreamSynchronize(c->stream));
    s.dev.hot = hot;
    CU(cudaMemcpy(c->d_layers + layer, &s.dev, sizeof(LayerDev), cudaMemcpyHostToDevice));
    return PI_OK;
}

pi_status pi_layer_counts(pi_ctx *c, int32_t layer, const void *x_hat, int32_t T, int32_t *counts)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_layer(c, layer);
    if (st) return st;
    if (!x_hat || !counts || T < 1) return fail(c, PI_ERR_ARG, "x_hat/counts NULL or T < 1");
    DeviceGuard g(c->device);
    const pi_layer_desc &d = c->layers[layer].desc;
    CU(cudaMemsetAsync(counts, 0, (size_t)d.d_ffn * 4, c->stream));
    for (int t0 = 0; t0 < T; t0 += c->max_batch) {
        StepParams p{};
        p.xhat_in = (const uint16_t *)x_hat + (size_t)t0 * d.d_model;
        p.counts_out = counts;
        st = launch(c, layer, 1, std::min(c->max_batch, T - t0), pi::M_COUNTS, p);
        if (st) return st;
    }
    return PI_OK;
}

// Batches of at least mma_min_b tokens take the tensor-core gather-GEMM
// (pi_mma.cu; Q4_0 layers pi_mma_q4.cu); smaller ones the step kernel.
// A layer without tensor maps (none could be made) stays on the step kernel.
// The smallest batch that runs layer by layer.  Unless set, 2 tokens for
// 16-bit layers and 3 for Q4_0 ones: at 2 tokens the persistent kernel's
// two-token groups beat the short launches only where those first
// dequantise the listed rows.
static int layerwise_min_b(const pi_ctx *c, int layer)
{
    if (c->mma_min_b >= 0) return c->mma_min_b;
    return c->layers[layer].desc.w_dtype == PI_Q4_0 ? 3 : 2;
}

static bool use_mma(const pi_ctx *c, int layer, int B)
{
    const int mb = layerwise_min_b(c, layer);
    return mb > 0 && B >= mb && c->layers[layer].maps;
}

// The FFN of one layer on the tensor cores: into y (16-bit), or added into
// the fp32 residual x.  idx/count NULL = every neuron.
static pi_status mma_ffn(pi_ctx *c, int layer, const uint16_t *xhat, int B, const int32_t *idx, const int32_t *count,
                         uint16_t *y, float *x)
{
    const LayerSlot &ls = c->layers[layer];
    const pi_layer_desc &dsc = ls.desc;
    pi::MmaParams q{};
    q.tm_up = ls.tm_up;
    q.tm_gate = ls.tm_gate;
    q.tm_dn = ls.tm_dn;
    const int np = (B + 15) / 16 * 16;
    if (reinterpret_cast<uintptr_t>(xhat) & 15u) return fail(c, PI_ERR_ARG, "x_hat must be 16-byte aligned");
    cudaError_t me = pi::encode_map(&q.tm_x, xhat, (uint64_t)dsc.d_model, (uint64_t)B, (uint64_t)dsc.d_model * 2, np);
    uint16_t *actL = c->actT + (size_t)c->max_batch * pi::kMaxN;
    if (me == cudaSuccess)
        me = pi::encode_map(&q.tm_act, c->actT, (uint64_t)pi::kMaxN, (uint64_t)B, (uint64_t)pi::kMaxN * 2, np);
    if (me == cudaSuccess)
        me = pi::encode_map(&q.tm_act_lo, actL, (uint64_t)pi::kMaxN, (uint64_t)B, (uint64_t)pi::kMaxN * 2, np);
    if (me != cudaSuccess) return fail(c, PI_ERR_CUDA, "tensor map: %s", cudaGetErrorString(me));
    q.layer = c->d_layers + layer;
    q.xhat = xhat;
    q.B = B;
    q.Npad = (B + 15) / 16 * 16;
    q.d = dsc.d_model;
    q.idx = idx;
    q.count = count;
    q.actT = c->actT;
    q.actL = actL;
    q.mstride = pi::kMaxN;
    q.y = y;
    q.x = x;
    q.part = c->mpart;
    q.status = c->ctl + 2;
    q.abort_flag = c->ctl + 3;
    q.wait_ns = c->wait_ns;
    const cudaError_t e = dsc.w_dtype == PI_Q4_0
                              ? pi::launch_ffn_mma_q4(q, dsc.act == PI_REGLU, c->G, c->stream)
                              : pi::launch_ffn_mma(q, dsc.act_dtype == PI_BF16, dsc.act == PI_REGLU, c->G, c->stream);
    if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "tensor-core FFN launch: %s", cudaGetErrorString(e));
    return PI_OK;
}

// Batches of at least mma_min_b tokens run the predictor as short launches
// of register-tiled dot products (pi_pred.cu) instead of the step kernel.
static bool use_pred_batch(const pi_ctx *c, int layer, int B)
{
    const int mb = layerwise_min_b(c, layer);
    return mb > 0 && B >= mb;
}

static pi::PredParams pred_params(pi_ctx *c, int layer, int B)
{
    pi::PredParams q{};
    q.L = c->layers[layer].dev;
    q.B = B;
    q.h = c->hbuf;
    q.mask = c->mbits;
    q.status = c->ctl + 2;
    q.abort_flag = c->ctl + 3;
    q.wait_ns = c->wait_ns;
    return q;
}

static pi_status pred_batch(pi_ctx *c, const pi::PredParams &q, int layer)
{
    const cudaError_t e =
        pi::launch_predict_batch(q, c->layers[layer].desc.act_dtype == PI_BF16, c->G, c->stream);
    if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "predictor launch: %s", cudaGetErrorString(e));
    c->h_batched = true;
    return PI_OK;
}

pi_status pi_predict(pi_ctx *c, int32_t layer, const void *x_hat, int32_t B, int32_t *idx, int32_t *count)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_layer(c, layer);
    if (!st) st = check_batch(c, B);
    if (st) return st;
    if (!x_hat || !idx || !count) return fail(c, PI_ERR_ARG, "x_hat/idx/count NULL");
    DeviceGuard g(c->device);
    if (use_pred_batch(c, layer, B)) {
        if (reinterpret_cast<uintptr_t>(x_hat) & 15u) return fail(c, PI_ERR_ARG, "x_hat must be 16-byte aligned");
        pi::PredParams q = pred_params(c, layer, B);
        q.xhat = (uint16_t *)x_hat;
        q.idx = idx;
        q.count = count;
        return pred_batch(c, q, layer);
    }
    StepParams p{};
    p.xhat_in = (const uint16_t *)x_hat;
    p.idx_out = idx;
    p.count_out = count;
    return launch(c, layer, 1, B, pi::M_PREDICT | pi::M_COMPACT, p);
}

pi_status pi_sparse_ffn(pi_ctx *c, int32_t layer, const void *x_hat, int32_t B, const int32_t *idx,
                        const int32_t *count, void *y)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_layer(c, layer);
    if (!st) st = check_batch(c, B);
    if (st) return st;
    if (!x_hat || !idx || !count || !y) return fail(c, PI_ERR_ARG, "x_hat/idx/count/y NULL");
    DeviceGuard g(c->device);
    if (use_mma(c, layer, B)) return mma_ffn(c, layer, (const uint16_t *)x_hat, B, idx, count, (uint16_t *)y, nullptr);
    StepParams p{};
    p.xhat_in = (const uint16_t *)x_hat;
    p.idx_in = idx;
    p.count_in = count;
    p.y_out = (uint16_t *)y;
    return launch(c, layer, 1, B, pi::M_IDX_IN | pi::M_FFN, p);
}

pi_status pi_dense_ffn(pi_ctx *c, int32_t layer, const void *x_hat, int32_t B, void *y)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_layer(c, layer);
    if (!st) st = check_batch(c, B);
    if (st) return st;
    if (!x_hat || !y) return fail(c, PI_ERR_ARG, "x_hat/y NULL");
    DeviceGuard g(c->device);
    if (use_mma(c, layer, B)) return mma_ffn(c, layer, (const uint16_t *)x_hat, B, nullptr, nullptr, (uint16_t *)y, nullptr);
    StepParams p{};
    p.xhat_in = (const uint16_t *)x_hat;
    p.y_out = (uint16_t *)y;
    return launch(c, layer, 1, B, pi::M_DENSE | pi::M_FFN, p);
}

static pi_status step_common(pi_ctx *c, float *x, int32_t B, int mode)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_batch(c, B);
    if (st) return st;
    if (!x) return fail(c, PI_ERR_ARG, "x NULL");
    int L = 0;
    st = stack_layers(c, &L);
    if (st) return st;
    DeviceGuard g(c->device);
    StepParams p{};
    p.x = x;
    p.tr_x = c->tr_x;
    p.tr_xhat = (uint16_t *)c->tr_xhat;
    p.tr_idx = c->tr_idx;
    p.tr_cnt = c->tr_cnt;
    int nmax = 0;
    for (int l = 0; l < L; ++l) nmax = std::max(nmax, c->layers[l].desc.d_ffn);
    p.tr_n = nmax;
    const int d = c->layers[0].desc.d_model;
    const bool dense = (mode & pi::M_DENSE) != 0;
    const bool bf16 = c->layers[0].desc.act_dtype == PI_BF16;
    if (!use_mma(c, 0, B)) {
        if (dense || !use_pred_batch(c, 0, B)) return launch(c, 0, L, B, mode, p);
        // Q4_0 batches, per layer: x_hat = RMSNorm(x), the batched predictor,
        // then the step kernel's FFN on that list adds the layer into x
        for (int l = 0; l < L; ++l) {
            pi::PredParams q = pred_params(c, l, B);
            q.x = x;
            q.tr_x = c->tr_x ? c->tr_x + (size_t)l * B * d : nullptr;
            q.xhat = c->xhat_ws;
            q.idx = c->lidx;
            q.count = c->lidx + pi::kMaxN;
            q.tr_idx = c->tr_idx ? c->tr_idx + (size_t)l * nmax : nullptr;
            q.tr_cnt = c->tr_cnt ? c->tr_cnt + l : nullptr;
            const cudaError_t e = pi::launch_rmsnorm_rows(q, bf16, c->stream);
            if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "RMSNorm launch: %s", cudaGetErrorString(e));
            st = pred_batch(c, q, l);
            if (st) return st;
            if (c->tr_xhat) {
                const cudaError_t e2 = cudaMemcpyAsync((uint16_t *)c->tr_xhat + (size_t)l * B * d, c->xhat_ws,
                                                       (size_t)B * d * 2, cudaMemcpyDeviceToDevice, c->stream);
                if (e2 != cudaSuccess) return fail(c, PI_ERR_CUDA, "x_hat trace: %s", cudaGetErrorString(e2));
            }
            StepParams f{};
            f.x = x;
            f.xhat_in = c->xhat_ws;
            f.idx_in = c->lidx;
            f.count_in = c->lidx + pi::kMaxN;
            st = launch(c, l, 1, B, pi::M_IDX_IN | pi::M_FFN | pi::M_RESID, f);
            if (st) return st;
        }
        return PI_OK;
    }
    // Large batch, per layer: x_hat = RMSNorm(x) into the workspace, the
    // predicted list (or the whole list), then the tensor-core FFN adds the
    // layer's output into x.
    for (int l = 0; l < L; ++l) {
        pi::PredParams q = pred_params(c, l, B);
        q.x = x;
        q.tr_x = c->tr_x ? c->tr_x + (size_t)l * B * d : nullptr;
        q.xhat = c->xhat_ws;
        q.idx = c->lidx;
        q.count = c->lidx + pi::kMaxN;
        q.tr_idx = c->tr_idx ? c->tr_idx + (size_t)l * nmax : nullptr;
        q.tr_cnt = c->tr_cnt ? c->tr_cnt + l : nullptr;
        cudaError_t e = pi::launch_rmsnorm_rows(q, bf16, c->stream);
        if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "RMSNorm launch: %s", cudaGetErrorString(e));
        if (dense) {
            if (q.tr_idx || q.tr_cnt) {
                e = pi::launch_list_all(q, c->stream);
                if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "list launch: %s", cudaGetErrorString(e));
            }
        } else {
            st = pred_batch(c, q, l);
            if (st) return st;
        }
        if (c->tr_xhat) {
            const cudaError_t e = cudaMemcpyAsync((uint16_t *)c->tr_xhat + (size_t)l * B * d, c->xhat_ws,
                                                  (size_t)B * d * 2, cudaMemcpyDeviceToDevice, c->stream);
            if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "x_hat trace: %s", cudaGetErrorString(e));
        }
        st = mma_ffn(c, l, c->xhat_ws, B, dense ? nullptr : c->lidx, dense ? nullptr : c->lidx + pi::kMaxN, nullptr,
                     x);
        if (st) return st;
    }
    return PI_OK;
}

pi_status pi_decode_step(pi_ctx *c, float *x, int32_t B)
{
    return step_common(c, x, B, pi::M_RMSNORM | pi::M_PREDICT | pi::M_FFN | pi::M_RESID);
}

pi_status pi_decode_step_host(pi_ctx *c, const float *x_in, float *x_out, int32_t B)
{
    if (!c) return PI_ERR_ARG;
    if (!x_in || !x_out) return fail(c, PI_ERR_ARG, "host buffer NULL");
    pi_status st = check_batch(c, B);
    if (st) return st;
    int L = 0;
    st = stack_layers(c, &L);
    if (st) return st;
    DeviceGuard g(c->device);
    const size_t bytes = (size_t)B * c->layers[0].desc.d_model * sizeof(float);
    cudaError_t e = cudaMemcpyAsync(c->xstage, x_in, bytes, cudaMemcpyHostToDevice, c->stream);
    if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "x to device: %s", cudaGetErrorString(e));
    st = pi_decode_step(c, c->xstage, B);
    if (st) return st;
    e = cudaMemcpyAsync(x_out, c->xstage, bytes, cudaMemcpyDeviceToHost, c->stream);
    if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "x to host: %s", cudaGetErrorString(e));
    return pi_sync_status(c);
}

pi_status pi_dense_step(pi_ctx *c, float *x, int32_t B)
{
    return step_common(c, x, B, pi::M_RMSNORM | pi::M_DENSE | pi::M_FFN | pi::M_RESID);
}

pi_status pi_layer_partial(pi_ctx *c, int32_t layer, const float *x, int32_t B, float *u)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_layer(c, layer);
    if (!st) st = check_batch(c, B);
    if (st) return st;
    if (!x || !u) return fail(c, PI_ERR_ARG, "x/u NULL");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(u)) & 15u)
        return fail(c, PI_ERR_ARG, "x and u must be 16-byte aligned");
    DeviceGuard g(c->device);
    const pi_layer_desc &dsc = c->layers[layer].desc;
    const int d = dsc.d_model;
    const bool bf16 = dsc.act_dtype == PI_BF16;
    if (!use_pred_batch(c, layer, B)) {
        // one persistent launch: RMSNorm, predictor, list, FFN, merge into u
        StepParams p{};
        p.x = const_cast<float *>(x); // (read only: M_RESID is not set)
        p.yf_out = u;
        p.tr_x = c->tr_x;
        p.tr_xhat = (uint16_t *)c->tr_xhat;
        p.tr_idx = c->tr_idx;
        p.tr_cnt = c->tr_cnt;
        p.tr_n = dsc.d_ffn;
        return launch(c, layer, 1, B, pi::M_RMSNORM | pi::M_PREDICT | pi::M_FFN | pi::M_YF32, p);
    }
    // layer by layer: RMSNorm, the batched predictor, then the FFN adds into u = 0
    pi::PredParams q = pred_params(c, layer, B);
    q.x = x;
    q.tr_x = c->tr_x;
    q.xhat = c->xhat_ws;
    q.idx = c->lidx;
    q.count = c->lidx + pi::kMaxN;
    q.tr_idx = c->tr_idx;
    q.tr_cnt = c->tr_cnt;
    cudaError_t e = pi::launch_rmsnorm_rows(q, bf16, c->stream);
    if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "RMSNorm launch: %s", cudaGetErrorString(e));
    st = pred_batch(c, q, layer);
    if (st) return st;
    if (c->tr_xhat) {
        e = cudaMemcpyAsync(c->tr_xhat, c->xhat_ws, (size_t)B * d * 2, cudaMemcpyDeviceToDevice, c->stream);
        if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "x_hat trace: %s", cudaGetErrorString(e));
    }
    e = cudaMemsetAsync(u, 0, sizeof(float) * (size_t)B * d, c->stream);
    if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "update clear: %s", cudaGetErrorString(e));
    if (use_mma(c, layer, B)) return mma_ffn(c, layer, c->xhat_ws, B, c->lidx, c->lidx + pi::kMaxN, nullptr, u);
    StepParams f{};
    f.x = u;
    f.xhat_in = c->xhat_ws;
    f.idx_in = c->lidx;
    f.count_in = c->lidx + pi::kMaxN;
    return launch(c, layer, 1, B, pi::M_IDX_IN | pi::M_FFN | pi::M_RESID, f);
}

pi_status pi_residual_add(pi_ctx *c, float *x, const float *u, int32_t B)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_batch(c, B);
    if (st) return st;
    if (!x || !u) return fail(c, PI_ERR_ARG, "x/u NULL");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(u)) & 15u)
        return fail(c, PI_ERR_ARG, "x and u must be 16-byte aligned");
    int L = 0;
    st = stack_layers(c, &L);
    if (st) return st;
    DeviceGuard g(c->device);
    const cudaError_t e = pi::launch_residual_add(x, u, (size_t)B * c->layers[0].desc.d_model, c->stream);
    return e == cudaSuccess ? PI_OK : fail(c, PI_ERR_CUDA, "residual add: %s", cudaGetErrorString(e));
}

pi_status pi_layer_shard(pi_ctx *c, int32_t layer, int32_t *shard, int32_t *nshards)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_layer(c, layer);
    if (st) return st;
    if (!shard || !nshards) return fail(c, PI_ERR_ARG, "shard/nshards NULL");
    *shard = c->layers[layer].shard;
    *nshards = c->layers[layer].nshards;
    return PI_OK;
}

pi_status pi_set_trace(pi_ctx *c, float *x_trace, void *xhat_trace, int32_t *idx_trace, int32_t *count_trace)
{
    if (!c) return PI_ERR_ARG;
    c->tr_x = x_trace;
    c->tr_xhat = xhat_trace;
    c->tr_idx = idx_trace;
    c->tr_cnt = count_trace;
    return PI_OK;
}

pi_status pi_sync_status(pi_ctx *c)
{
    if (!c) return PI_ERR_ARG;
    DeviceGuard g(c->device);
    cudaError_t e = cudaStreamSynchronize(c->stream);
    if (e != cudaSuccess) return fail(c, PI_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
    int ctl[4];
    CU(cudaMemcpy(ctl, c->ctl, sizeof ctl, cudaMemcpyDeviceToHost));
    if (ctl[2] != 0 || ctl[3] != 0) {
        // a failed launch leaves the barrier counter wherever its CTAs stopped
        CU(cudaMemset(c->ctl, 0, sizeof(int) * 4));
        const int code = ctl[2] ? ctl[2] : PI_ERR_TIMEOUT;
        return fail(c, code, code == PI_ERR_TIMEOUT ? "a device-side wait timed out" : "a kernel flagged invalid device data");
    }
    return PI_OK;
}

const char *pi_last_error(pi_ctx *c)
{
    if (!c) return "null context";
    return c->err.c_str();
}

int32_t pi_grid_size(pi_ctx *c) { return c ? c->G : 0; }

pi_status pi_debug_set_wait_limit(pi_ctx *c, uint64_t ns)
{
    if (!c || ns == 0) return PI_ERR_ARG;
    c->wait_ns = ns;
    return PI_OK;
}

pi_status pi_debug_set_timeline(pi_ctx *c, uint64_t *stamps, int32_t per_cta)
{
    if (!c || (stamps && per_cta < 1)) return PI_ERR_ARG;
    c->timeline = (unsigned long long *)stamps;
    c->tl_stride = stamps ? per_cta : 0;
    return PI_OK;
}

pi_status pi_debug_set_tuning(pi_ctx *c, int32_t prefetch, int32_t prefetch_ns, int32_t lookahead,
                              int32_t rows_ahead)
{
    if (!c || prefetch < 0 || prefetch > 3 || prefetch_ns < 0 || lookahead < 0 || rows_ahead < 0)
        return PI_ERR_ARG;
    c->prefetch = prefetch;
    c->prefetch_ns = prefetch_ns;
    c->lookahead = lookahead;
    c->rows_ahead = rows_ahead;
    return PI_OK;
}

pi_status pi_debug_copy_hidden(pi_ctx *c, float *dst, int32_t count)
{
    if (!c || !dst || count < 0 || (size_t)count > (size_t)c->max_batch * pi::kMaxRank) return PI_ERR_ARG;
    DeviceGuard g(c->device);
    // batched pass: plain fp32 [B][rank]; step kernel: the low halves of the tagged words
    const cudaError_t e =
        c->h_batched ? cudaMemcpyAsync(dst, c->hbuf, sizeof(float) * (size_t)count, cudaMemcpyDefault, c->stream)
                     : cudaMemcpy2DAsync(dst, sizeof(float), c->hx, sizeof(uint64_t), sizeof(float), (size_t)count,
                                         cudaMemcpyDefault, c->stream);
    return e == cudaSuccess ? PI_OK : fail(c, PI_ERR_CUDA, "copy of h: %s", cudaGetErrorString(e));
}

pi_status pi_debug_set_mma_min_batch(pi_ctx *c, int32_t min_batch)
{
    if (!c || min_batch < -1) return PI_ERR_ARG;
    c->mma_min_b = min_batch;
    return PI_OK;
}

pi_status pi_layerwise_min_batch(pi_ctx *c, int32_t layer, int32_t *min_batch)
{
    if (!c) return PI_ERR_ARG;
    pi_status st = check_layer(c, layer);
    if (st) return st;
    if (!min_batch) return fail(c, PI_ERR_ARG, "min_batch NULL");
    const int mb = layerwise_min_b(c, layer);
    *min_batch = mb > 0 && c->layers[layer].maps ? mb : 0;
    return PI_OK;
}

pi_status pi_debug_barrier_extra(pi_ctx *c, int32_t extra)
{
    if (!c || extra < 0) return PI_ERR_ARG;
    c->bar_extra = extra;
    return PI_OK;
}

} // extern "C"
