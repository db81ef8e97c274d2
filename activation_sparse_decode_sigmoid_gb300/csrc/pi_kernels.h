// Structures shared by the host side of libpi and its kernels.
#pragma once

#include <cuda.h> // CUtensorMap (types only; the encoder is fetched from the driver at run time)
#include <cuda_runtime.h>
#include <stdint.h>

namespace pi {

// Thread layout of the persistent step kernel: 16 consumer warps, then one
// producer warp for the static weight stream (predictor W1/W2 slices) and
// one for the dynamic stream (rows of the predicted neurons).
constexpr int kConsumerWarps = 16;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 64;
constexpr int kStaticWarp = kConsumerWarps;
constexpr int kDynamicWarp = kConsumerWarps + 1;

constexpr int kMaxD = 8192;          // d_model limit (x_hat row fits a 16 KB slot)
constexpr int kMaxRank = 2048;       // predictor width limit
constexpr int kMaxN = 65536;         // neurons per layer
constexpr int kMaxBatch = 64;        // tokens per call
constexpr int kYSlots = 16;          // output columns a consumer thread owns (d <= 8192)
constexpr int kMaxNeuronsPerStage = 8;
constexpr int kPhaseBTokens = 4;     // tokens per inner pass of the W2 dot products
constexpr int kTimelineEvents = 9;   // stamps per layer in the debug timeline

// activation families (mirror pi.h's pi_act)
constexpr int ACT_RELU = 0, ACT_REGLU = 1, ACT_SQRELU = 2;

// device status codes (mirror pi.h)
constexpr int PI_DEV_TIMEOUT = -6;
constexpr int PI_DEV_FLAG = -7;

// mode bits of one launch of the step kernel
enum : int {
    M_RMSNORM = 1,   // x_hat = RMSNorm(x) per layer (else x_hat given)
    M_PREDICT = 2,   // run the predictor; the FFN list is its union
    M_IDX_IN = 4,    // FFN list given (idx_in / count_in)
    M_DENSE = 8,     // FFN list = every neuron
    M_FFN = 16,      // run the sparse FFN and the merge
    M_RESID = 32,    // merge into the fp32 residual x (else write y)
    M_COUNTS = 64,   // predictor: per-neuron selection counts over the tokens
    M_COMPACT = 128, // predictor: write the ascending idx list + count
    M_YF32 = 256,    // merge: write the fp32 update to yf_out (x is only read, by the RMSNorm)
};

struct LayerDev {
    int d, n, r, act, q4;
    int rowB;               // bytes of one FFN row (16-bit: 2d; Q4_0: scB + d/2)
    int scB;                // Q4_0: bytes of the scale part of a row (16-byte padded)
    int upB;                // bytes of one W_up row in `up`: rowB, or rowB + 16 with the bias tail
    int bias_tail;          // 1: neuron i's bias (16-bit) sits at up row i + rowB, so it arrives
                            //    with the row; 0: read from b[]
    int hot;                // neurons [0, hot) are always active: their predictor rows are not
                            // evaluated (0 = every neuron predicted)
    const uint16_t *w1;     // [r][d]
    const uint16_t *b1;     // [r]
    const uint16_t *w2;     // [n][r]   rows in physical order
    const uint16_t *b2;     // [n]
    const uint8_t *up;      // [n] rows of rowB bytes
    const uint8_t *gate;    // [n] rows (ReGLU) or null
    const uint8_t *dn;      // [n] rows of W_down transposed
    const uint16_t *b;      // [n] up bias (ReLU) / gate bias (ReGLU)
    const uint16_t *bdown;  // [d]
};

struct StepParams {
    const LayerDev *layers; // device array [L]
    int L, B, mode, d;
    float *x;               // [B][d] fp32 residual
    const uint16_t *xhat_in;// [B][d]
    const int32_t *idx_in;
    const int32_t *count_in;
    int32_t *idx_out;
    int32_t *count_out;
    uint16_t *y_out;        // [B][d]
    int32_t *counts_out;    // [n]
    float *yf_out;          // [B][d] fp32 layer update (mode M_YF32: written instead of added into x)
    // workspace
    // Cross-SM exchanges that need no grid barrier: every 64-bit word holds
    // a value (low half) and the epoch of the layer that wrote it (high
    // half); a reader polls the words themselves until they carry the
    // epoch it expects, so the data read is also the synchronisation.
    uint64_t *hx;           // [B][r_max] predictor hidden activations (fp32 bits)
    uint64_t *bmx;          // [ceil(n_max/32)] predicted-mask words (union over tokens)
    unsigned epoch;         // epoch of layer 0 of this launch; layer l writes epoch + l
    uint64_t *partx;        // [G][B][d] split-K partials of the FFN output (fp32 bits)
    uint64_t *xx;           // [B][d] the residual after each layer (fp32 bits), read by the next
    int *status;            // first device error
    int *abort_flag;
    // trace
    float *tr_x;            // [L][B][d]
    uint16_t *tr_xhat;      // [L][B][d]
    int32_t *tr_idx;        // [L][tr_n]
    int32_t *tr_cnt;        // [L]
    int tr_n;
    int bar_extra;          // test hook: readers expect epoch + bar_extra, which never comes
    unsigned long long wait_ns;
    unsigned long long *timeline; // [G][tl_stride] globaltimer stamps (debug)
    int tl_stride;
    // tuning: L2 prefetch of the predictor slices (0 off; the next layer's
    // during phase C: 1 all at once, 2 paced at one 16 KB chunk per
    // prefetch_ns; 3 this layer's W2 slice as one burst once phase C of the
    // previous layer is over), how many stages past the one being merged an
    // owner warp may compute activations for (phase C), and how many neurons of the
    // CTA's list the dynamic producer prefetches into L2 ahead of its ring
    // loads (0 off)
    int prefetch;
    int prefetch_ns;
    int lookahead;
    int rows_ahead;
    // shared-memory plan.  The ring region [0, ringB) is time-shared: during
    // the predictor phases it is nss static slots of slotB bytes, during the
    // FFN phase nsd dynamic stages of dslotB bytes.
    int ringB;
    int slotB, nss;
    int dslotB, nsd;
    int off_h, hB;          // predictor hidden staging (tgB tokens)
    int off_xs;             // x_hat of tg tokens
    int off_misc;
    int tg;                 // tokens per x_hat pass (phase A and FFN)
    int tgB;                // tokens per h pass (phase B)
    int lcap;               // capacity of the per-CTA neuron list
    int wcap;               // capacity of the per-CTA mask words
    int rcap;               // capacity of the per-CTA predictor-bias cache
    int smem_bytes;
};


// Byte offsets of the small shared-memory objects of the step kernel (the
// "misc" region).  Computed identically by the host planner and the kernel.
struct MiscLayout {
    int bars, info, tmp, slist, sbias, swords, pbias, red, total;
};

__host__ __device__ inline MiscLayout misc_layout(int nss, int nsd, int lcap, int wcap, int rcap, int tgf)
{
    MiscLayout m;
    int o = 0;
    m.bars = o;
    o += (2 * nss + 3 * nsd + 3) * 8;
    o = (o + 15) & ~15;
    m.info = o;
    o += 16 * 4;
    m.tmp = o;
    o += 256 * 4;
    m.slist = o;
    o += lcap * 4;
    m.sbias = o;
    o += lcap * 4;
    m.swords = o;
    o += wcap * 4;
    o = (o + 15) & ~15;
    m.pbias = o; // two 16-bit bias slices (b1, b2), each a 16-byte-rounded copy
    o += 2 * ((rcap * 2 + 32 + 15) & ~15);
    o = (o + 15) & ~15;
    m.red = o;
    o += 2 * kConsumerWarps * kMaxNeuronsPerStage * tgf * 2 * 4;
    m.total = (o + 127) & ~127;
    return m;
}

// Parameters of the tensor-core FFN kernels (pi_mma.cu), batches of 2..64.
struct MmaParams {
    // TMA maps (16-bit elements, 64-column boxes, 128-byte swizzle): the
    // layer's W_up / W_gate / W_down^T rows (one-row boxes, for gather4),
    // x_hat and the two 16-bit parts of A^T (tile boxes of Npad rows; rows
    // past B read as zeros)
    CUtensorMap tm_up, tm_gate, tm_dn, tm_x, tm_act, tm_act_lo;
    const LayerDev *layer;   // device pointer to the layer's descriptor
    const uint16_t *xhat;    // [B][d] 16-bit
    int B, Npad, d;          // tokens, tokens rounded up to 16, d_model
    const int32_t *idx;      // [m] physical neuron ids, ascending; NULL = all n neurons (dense)
    const int32_t *count;    // device m; NULL = n
    // The activations A^T as two 16-bit parts in the weights' type: hi =
    // round(a), lo = round(a - hi).  The down-projection multiplies both with
    // the same W_down^T tile into one fp32 accumulator, so a reaches it with
    // about twice the 16-bit precision (a 16-bit tensor-core product takes
    // both operands in one type).
    uint16_t *actT;          // [B][mstride] hi parts
    uint16_t *actL;          // [B][mstride] lo parts
    size_t mstride;          // row stride of actT / actL (multiple of 64, >= m rounded up to 64)
    uint16_t *y;             // [B][d] 16-bit output, or NULL when x is set
    float *x;                // [B][d] fp32 residual to add into, or NULL
    float *part;             // [8][B][d] fp32 partials of column blocks split over list shares
    int *status;
    int *abort_flag;
    unsigned long long wait_ns;
};

// Launchers (host side of the kernels), in the step/load translation units.
// tgf: tokens per FFN pass of the step kernel: 1, 2 or 4
cudaError_t launch_step_f16(const StepParams &p, int tgf, int grid, cudaStream_t s);
cudaError_t launch_step_bf16(const StepParams &p, int tgf, int grid, cudaStream_t s);
cudaError_t launch_step_q4(const StepParams &p, int tgf, int grid, cudaStream_t s);
// the union-mask FFN on tcgen05: up/gate kernel on `grid` SMs, then the down kernel
cudaError_t launch_ffn_mma(const MmaParams &p, bool bf16, bool reglu, int grid, cudaStream_t s);
// the same for a Q4_0 layer (f16 activations): the rows are dequantised in shared memory
cudaError_t launch_ffn_mma_q4(const MmaParams &p, bool reglu, int grid, cudaStream_t s);
// y (or x +=) = the down kernel's nks share partials added in share order, + b_down
cudaError_t launch_ffn_merge(const MmaParams &p, bool bf16, int nks, int grid, cudaStream_t s);

// Programmatic dependent launch for the layer-by-layer path: each kernel is
// launched so that it may be scheduled while its predecessor in the stream
// finishes.  It first waits for the predecessor's results (a no-op when it
// was launched without the attribute), then lets its own successor be
// scheduled; a successor can only start once every CTA of this grid is
// resident, so the two never wait on each other's resources.
// The bits of mask word w (neurons [32 w, 32 w + 32)) that a hot prefix of
// h neurons sets.
#ifdef __CUDACC__
__host__ __device__
#endif
inline unsigned hot_bits(int w, int h)
{
    const int k = h - 32 * w;
    return k >= 32 ? ~0u : (k <= 0 ? 0u : (1u << k) - 1u);
}

#ifdef __CUDACC__
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif
template <typename... P, typename... A>
cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, A... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The predictor of one layer for a batch of several tokens (pi_pred.cu).
struct PredParams {
    LayerDev L;               // the layer (device pointers)
    int B;                    // tokens
    const float *x;           // [B][d] fp32 residual: input of the RMSNorm launch
    float *tr_x;              // [B][d] copy of x (trace), or NULL
    uint16_t *xhat;           // [B][d] x_hat: written by the RMSNorm launch, read by the predictor
    float *h;                 // [B][r] fp32 hidden activations
    uint32_t *mask;           // [ceil(n/32)] union mask words
    int32_t *idx, *count;     // the ascending list of predicted neurons and its length
    int32_t *tr_idx, *tr_cnt; // copies of the list and its length (trace), or NULL
    int dense;                // list launch only: the list of every neuron
    int *status;
    int *abort_flag;
    unsigned long long wait_ns;
};
// x_hat = RMSNorm(x) of B tokens, in the step kernel's reduction order
cudaError_t launch_rmsnorm_rows(const PredParams &p, bool bf16, cudaStream_t s);
// h, the union mask, then the list (three launches on `sms` SMs)
cudaError_t launch_predict_batch(const PredParams &p, bool bf16, int sms, cudaStream_t s);
// the list of every neuron 0..n-1 (dense steps), with its trace copies
cudaError_t launch_list_all(const PredParams &p, cudaStream_t s);
// a 2D TMA map over a row-major 16-bit matrix: box = 64 columns x box_rows rows, 128-byte swizzle
cudaError_t encode_map(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t row_bytes,
                       uint32_t box_rows);

cudaError_t launch_permute_rows(const void *src, void *dst, const int32_t *perm, int rows, size_t rowBytes,
                                cudaStream_t s, size_t dstStride = 0);
cudaError_t launch_bias_tail(const uint16_t *b, uint8_t *up, int n, size_t rowB, size_t upB, cudaStream_t s);
cudaError_t launch_transpose_permute16(const uint16_t *src, uint16_t *dst, const int32_t *perm, int d, int n,
                                       int nsrc, cudaStream_t s);
cudaError_t launch_residual_add(float *x, const float *u, size_t n, cudaStream_t s);
cudaError_t launch_q4_split(const uint8_t *src, uint8_t *dst, const int32_t *perm, int n, int d, int scB,
                            cudaStream_t s, size_t dstStride = 0);
cudaError_t launch_permute16(const uint16_t *src, uint16_t *dst, const int32_t *perm, int n, cudaStream_t s);
} // namespace pi
