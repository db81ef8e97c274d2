// pi_sparse_ffn_noalloc: the sparse FFN of the step kernel for callers that
// cannot allocate device memory.
//
// Some embedders run this library where cudaMalloc is not theirs to call: an
// inference server whose memory is carved up by its own pool and must not
// see a foreign allocation appear mid-run, a process that runs under a fixed
// device-memory budget, or code that is only handed pre-allocated buffers.
// For them pi_create (which allocates the workspace) is not an option.  This
// entry point needs no context: the caller passes the layer's rows, the
// inputs and the output buffers, and the scratch the kernel needs (split-K
// partials, the grid-barrier counter, the status words, a one-layer
// descriptor table and a zero run standing in for absent biases) lives in the
// file-scope array below, which exists once per GPU that loads the library,
// from load until process exit.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "pi.h"
#include "pi_kernels.h"

namespace {

// Byte layout of the static scratch array.
constexpr size_t kCtlOff = 0;              // (unused u64), int status, int abort
constexpr size_t kLayerOff = 256;          // one pi::LayerDev
constexpr size_t kZeroOff = 4096;          // zeros for absent biases (65536 x 16-bit)
constexpr size_t kZeroBytes = 65536 * 2;
constexpr size_t kPartialOff = kZeroOff + kZeroBytes;
constexpr size_t kScratchBytes = 16u << 20; // 16 MiB in total
constexpr size_t kPartialWords = (kScratchBytes - kPartialOff) / 8; // epoch-tagged fp32 partials

static_assert(sizeof(pi::LayerDev) <= kZeroOff - kLayerOff, "layer table does not fit its slot");

constexpr int kMaxDevices = 64;

} // namespace

// The scratch.  Host code must not use this name as a device address (in host
// code it names a host-side stand-in); noalloc_scratch() returns the real one.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

std::mutex g_mu;
unsigned char *g_ptr[kMaxDevices] = {};
unsigned g_epoch[kMaxDevices] = {}; // epoch of the last call on each device (the array starts zeroed)

// Device address of the scratch array on the current device.  The first call
// on a device resolves it (cudaGetSymbolAddress may load the module; the
// array starts zeroed, as every device variable without an initialiser);
// later calls only read the cache.
cudaError_t noalloc_scratch(int dev, cudaStream_t s, unsigned char **out, unsigned *epoch)
{
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ptr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_ptr[dev] = static_cast<unsigned char *>(ptr);
    }
    *out = g_ptr[dev];
    // every call writes its partials under a new epoch, so what earlier
    // calls left in the array can never be taken for this call's; before
    // the 32-bit epoch could wrap, the tags are cleared on the caller's
    // stream (ordered before this call's kernel)
    if (++g_epoch[dev] == 0xF0000000u) {
        const cudaError_t e = cudaMemsetAsync(g_ptr[dev] + kPartialOff, 0, kPartialWords * 8, s);
        if (e != cudaSuccess) return e;
        g_epoch[dev] = 1;
    }
    *epoch = g_epoch[dev];
    return cudaSuccess;
}

int round_up(int v, int a) { return (v + a - 1) / a * a; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

} // namespace

extern "C" pi_status pi_sparse_ffn_noalloc(const pi_ffn_rows *w, const void *x_hat, int32_t B, const int32_t *idx,
                                           const int32_t *count, void *y, int32_t *dev_status, void *stream)
{
    if (!w || !x_hat || !idx || !count || !y || !w->up || !w->down_rows) return PI_ERR_ARG;
    if (w->act != PI_RELU && w->act != PI_REGLU && w->act != PI_SQRELU) return PI_ERR_ARG;
    if (w->act == PI_REGLU && !w->gate) return PI_ERR_ARG;
    if (w->act_dtype != PI_F16 && w->act_dtype != PI_BF16) return PI_ERR_ARG;
    const int d = w->d_model, n = w->d_ffn;
    if (d < 8 || d > pi::kMaxD || d % 8 || n < 1 || n > pi::kMaxN) return PI_ERR_SHAPE;
    if (B < 1 || B > pi::kMaxBatch) return PI_ERR_ARG;
    // rows are streamed with bulk copies: every row must start on 16 bytes
    if (!aligned16(w->up) || !aligned16(w->down_rows) || (w->gate && !aligned16(w->gate)) || !aligned16(x_hat) ||
        !aligned16(y) || (w->b_down && (reinterpret_cast<uintptr_t>(w->b_down) & 7u)))
        return PI_ERR_ARG;

    int dev = 0, G = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PI_ERR_CUDA;
    if (cudaDeviceGetAttribute(&G, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PI_ERR_CUDA;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return PI_ERR_CUDA;
    // the fp32 split-K partials of every SM must fit the fixed scratch
    if ((size_t)G * B * d > kPartialWords) return PI_ERR_SHAPE;
    unsigned char *scratch = nullptr;
    unsigned epoch = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (noalloc_scratch(dev, s, &scratch, &epoch) != cudaSuccess) return PI_ERR_CUDA;

    // shared-memory plan of the FFN-only launch (no predictor phases)
    pi::StepParams p{};
    const int rowB = 2 * d;
    const int nb = (w->act == PI_REGLU ? 3 : 2) * rowB;
    const int tgf = B == 1 ? 1 : 4;
    p.d = d;
    p.B = B;
    p.L = 1;
    p.mode = pi::M_IDX_IN | pi::M_FFN;
    p.tg = std::min(B, tgf);
    p.tgB = 1;
    p.lcap = (n + G - 1) / G + 2;
    p.wcap = ((n + 31) / 32 + G - 1) / G + 1;
    p.rcap = std::max(2, p.wcap * 32);
    const int xsB = round_up(p.tg * d * 2, 128);
    const int misc_bound = pi::misc_layout(0, 16, p.lcap, p.wcap, p.rcap, tgf).total;
    p.ringB = (optin - misc_bound - xsB) / 128 * 128;
    p.slotB = 16384;
    p.nss = 0;
    p.dslotB = round_up(std::max(nb, 24576), 128);
    p.nsd = std::min(16, p.ringB / p.dslotB);
    if (p.nsd < 2) return PI_ERR_UNSUPPORTED;
    p.off_h = p.ringB;
    p.hB = 0;
    p.off_xs = p.off_h;
    p.off_misc = p.off_xs + xsB;
    p.smem_bytes = p.off_misc + pi::misc_layout(0, p.nsd, p.lcap, p.wcap, p.rcap, tgf).total;
    if (p.smem_bytes > optin) return PI_ERR_UNSUPPORTED;

    // the one-layer descriptor, pointing at the caller's rows
    pi::LayerDev L{};
    L.d = d;
    L.n = n;
    L.r = 8;
    L.act = w->act;
    L.rowB = rowB;
    L.upB = rowB;      // the caller's rows have no bias tail: biases are read from b[]
    L.bias_tail = 0;
    L.up = static_cast<const uint8_t *>(w->up);
    L.gate = w->act == PI_REGLU ? static_cast<const uint8_t *>(w->gate) : nullptr;
    L.dn = static_cast<const uint8_t *>(w->down_rows);
    L.b = w->b ? static_cast<const uint16_t *>(w->b) : reinterpret_cast<const uint16_t *>(scratch + kZeroOff);
    L.bdown = w->b_down ? static_cast<const uint16_t *>(w->b_down)
                        : reinterpret_cast<const uint16_t *>(scratch + kZeroOff);

    // the array keeps the previous call's contents: clear the status words,
    // then publish this call's layer descriptor
    if (cudaMemsetAsync(scratch + kCtlOff, 0, 16, s) != cudaSuccess) return PI_ERR_CUDA;
    if (dev_status && cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s) != cudaSuccess) return PI_ERR_CUDA;
    if (cudaMemcpyAsync(scratch + kLayerOff, &L, sizeof L, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return PI_ERR_CUDA;

    p.layers = reinterpret_cast<const pi::LayerDev *>(scratch + kLayerOff);
    p.xhat_in = static_cast<const uint16_t *>(x_hat);
    p.idx_in = idx;
    p.count_in = count;
    p.y_out = static_cast<uint16_t *>(y);
    p.partx = reinterpret_cast<uint64_t *>(scratch + kPartialOff);
    p.epoch = epoch;
    p.status = dev_status ? dev_status : reinterpret_cast<int *>(scratch + kCtlOff + 8);
    p.abort_flag = reinterpret_cast<int *>(scratch + kCtlOff + 12);
    p.wait_ns = 2000000000ull;
    p.prefetch = 0;
    p.lookahead = 16;
    const cudaError_t e = w->act_dtype == PI_BF16 ? pi::launch_step_bf16(p, tgf, G, s) : pi::launch_step_f16(p, tgf, G, s);
    return e == cudaSuccess ? PI_OK : PI_ERR_CUDA;
}
