/*
 * pi.h -- C ABI of libpi, a GB300 (sm_103a) implementation of the PowerInfer
 * decode hot path: a per-layer activation predictor followed by a
 * neuron-aware sparse FFN.
 *
 * What the calls compute (PowerInfer: Fast LLM Serving with a Consumer-grade
 * GPU):
 *   - blog.csdn.net QbitAI/IPADS article, section "充分利用模型和硬件特点":
 *     before a layer's FFN runs, a small per-layer routing predictor decides
 *     which neurons the input activates; only those neurons are computed
 *     (about 10% of an OPT FFN's neurons suffice).
 *   - chatpaper.ai abstract: adaptive predictors and neuron-aware sparse
 *     operators; hot neurons (power-law activation) are kept close to compute.
 *   - same article, section "CPU/GPU混合推理设计": neurons are placed by an
 *     offline hot/cold profile, executors compute their share of the
 *     predicted neurons, and the partial results are merged.  On one GB300 the
 *     whole model is resident in HBM; the hot/cold split becomes an offline
 *     neuron permutation (hot neurons first) and the merge is a split-K
 *     reduction in fp32.
 *   - de.news.hada.io summary: ReLU / ReGLU / squared-ReLU activations,
 *     Q4_0 INT4 weights.
 * The pages print no formulas; the readings used (z > 0 for "sigmoid > 0.5",
 * the canonical fp32 predictor order, Q4_0 block layout, weightless RMSNorm
 * between layers, union of per-token sets for a batch) are documented with
 * the calls below.
 *
 * Conventions for every call
 *   - Returns PI_OK (0) or a negative pi_status.  Argument and shape errors
 *     are detected on the host before anything is launched.  Errors raised
 *     inside a kernel (a bounded wait that ran out) are written to a device
 *     status word that pi_sync_status() returns; nothing traps or aborts.
 *   - Compute calls are asynchronous on the context's current stream
 *     (pi_set_stream); device buffers passed in must stay valid until the
 *     stream has reached the call.
 *   - "dev" pointers are CUDA device pointers, "host" pointers are ordinary
 *     host memory.  16-bit activations are IEEE binary16 (PI_F16) or bfloat16
 *     (PI_BF16) bit patterns.
 *   - Neuron indices are physical: after the layer's neuron permutation.
 *     perm[i] (as passed to pi_load_layer) is the original id of physical
 *     neuron i.
 *   - A context is single-threaded: do not call it from two host threads at
 *     once.
 */
#ifndef PI_H
#define PI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t pi_status;
#define PI_OK 0
#define PI_ERR_ARG (-1)          /* null pointer or invalid enum / count */
#define PI_ERR_SHAPE (-2)        /* dimension outside the supported range */
#define PI_ERR_CUDA (-3)         /* a CUDA runtime call failed */
#define PI_ERR_OOM (-4)          /* device allocation failed */
#define PI_ERR_NOT_LOADED (-5)   /* layer slot empty, or stack not contiguous */
#define PI_ERR_TIMEOUT (-6)      /* a bounded device-side wait ran out */
#define PI_ERR_DEVICE_FLAG (-7)  /* a kernel flagged invalid device data */
#define PI_ERR_UNSUPPORTED (-8)  /* valid request this build does not serve */

/* Activation families (de.news.hada.io summary, "Einschränkungen und FAQ":
 * ReLU, ReGLU and squared ReLU models):
 *   PI_RELU    a_i = max(W_up[i].x_hat + b_i, 0)
 *   PI_REGLU   a_i = max(W_gate[i].x_hat + b_i, 0) * (W_up[i].x_hat)
 *   PI_SQRELU  a_i = max(W_up[i].x_hat + b_i, 0)^2
 * A neuron is active (its activation nonzero) exactly when its ReLU is. */
typedef enum { PI_RELU = 0, PI_REGLU = 1, PI_SQRELU = 2 } pi_act;
typedef enum { PI_F16 = 0, PI_BF16 = 1, PI_Q4_0 = 2 } pi_dtype;

/* Shape and types of one FFN layer and its predictor.
 *   d_model in [8, 8192], multiple of 8 (of 32 for Q4_0 weights)
 *   d_ffn   in [1, 65536]      (neurons n)
 *   rank    in [8, 2048], multiple of 8 (predictor hidden width r)
 *   act_dtype: PI_F16 or PI_BF16 -- x_hat, predictor weights, biases, y
 *   w_dtype:   act_dtype, or PI_Q4_0 (only with act_dtype PI_F16) for
 *              W_up / W_gate / W_down. */
typedef struct {
    int32_t d_model, d_ffn, rank;
    int32_t act;       /* pi_act */
    int32_t w_dtype;   /* pi_dtype */
    int32_t act_dtype; /* pi_dtype */
} pi_layer_desc;

/* Weights of one layer in the model's own layout (original neuron order).
 *   w_up   [n][d]  row i = neuron i (ReLU: u_i = w_up[i].x + b[i])
 *   w_gate [n][d]  ReGLU only, else NULL (a_i = max(w_gate[i].x + b[i], 0) * (w_up[i].x))
 *   b      [n]     bias of the up projection (ReLU) or of the gate (ReGLU); NULL = 0
 *   w_down [d][n]  column i = neuron i's output vector
 *   b_down [d]     NULL = 0
 *   p_w1   [r][d], p_b1 [r] (NULL = 0), p_w2 [n][r], p_b2 [n] (NULL = 0)
 * Q4_0 weights: w_up / w_gate are [n] rows of d/32 Q4_0 blocks, and w_down is
 * given TRANSPOSED, as [n] rows of d/32 blocks along d.  A Q4_0 block is 18
 * bytes: little-endian fp16 scale s, then 16 bytes whose low nibble j is
 * element j and high nibble j is element j+16; weight = (nibble - 8) * s.
 * on_device = 1: all pointers are device pointers; 0: host pointers. */
typedef struct {
    const void *w_up, *w_gate, *b, *w_down, *b_down;
    const void *p_w1, *p_b1, *p_w2, *p_b2;
    int32_t on_device;
} pi_layer_weights;

typedef struct pi_ctx pi_ctx;

/* Create a context on CUDA device `device`.  `stream` is a cudaStream_t (NULL
 * = the legacy default stream).  max_layers bounds the layer slots of the
 * stack, max_batch the tokens per call (1..64).  Allocates the workspace;
 * layers are allocated by pi_load_layer.  *out receives the context. */
pi_status pi_create(pi_ctx **out, int32_t device, void *stream, int32_t max_layers, int32_t max_batch);

/* Free every device buffer of the context (synchronises its stream first). */
pi_status pi_destroy(pi_ctx *ctx);

/* Make `stream` (a cudaStream_t) the stream of subsequent calls. */
pi_status pi_set_stream(pi_ctx *ctx, void *stream);

/* Load (or replace) layer slot `layer` (0 <= layer < max_layers).  Copies the
 * weights into buffers the library owns, applying the neuron permutation
 * `perm` (host [n], perm[i] = original id of physical neuron i; NULL =
 * identity; must be a permutation of 0..n-1), transposing W_down into rows of
 * WdT (one contiguous row per neuron) and splitting Q4_0 rows into separate
 * scale and nibble arrays.  This is the offline placement step of the
 * "CPU/GPU混合推理设计" section, mapped to one device: hot neurons first.
 * Synchronous: returns when the copy is done; the caller keeps its buffers. */
pi_status pi_load_layer(pi_ctx *ctx, int32_t layer, const pi_layer_desc *desc,
                        const pi_layer_weights *w, const int32_t *perm);

/* Neuron-sharded layer, for splitting one layer's neurons over several GPUs
 * (multi-GPU support is listed as future work on the de.news.hada.io
 * summary, "Jüngste Updates und Pläne").  Like pi_load_layer, but slot
 * `layer` keeps only the neurons of shard `shard` of `nshards`, round-robin
 * over the physical order: physical neuron i (after `perm`) belongs to shard
 * i mod nshards, so every shard gets the same mix of hot and cold neurons.
 * The slot holds the whole predictor hidden layer (W1, b1: every shard
 * computes h), the W2 rows and b2 of its neurons, their FFN rows and biases,
 * and b_down on shard 0 only (zeros elsewhere), so that the shards' updates
 * add up to the unsplit layer's.  Local neuron j of the slot is physical
 * neuron shard + j * nshards; lists of the slot (pi_predict, traces) hold
 * local ids, and its d_ffn is the number of neurons it holds.  The other
 * rules (arguments, ownership, errors) are pi_load_layer's; PI_ERR_ARG for
 * nshards < 1, shard outside [0, nshards) or nshards > d_ffn. */
pi_status pi_load_layer_shard(pi_ctx *ctx, int32_t layer, const pi_layer_desc *desc, const pi_layer_weights *w,
                              const int32_t *perm, int32_t shard, int32_t nshards);

/* *shard, *nshards of slot `layer` (0 and 1 for a layer loaded whole). */
pi_status pi_layer_shard(pi_ctx *ctx, int32_t layer, int32_t *shard, int32_t *nshards);

/* One layer's update of the residual stream, written instead of added
 * (the merge step of the "CPU/GPU混合推理设计" section, left to the caller
 * when the layer is split over devices): for x (dev fp32 [B][d], read only)
 *   x_hat = act_dtype(x / sqrt(mean(x^2) + 1e-5)),
 *   list  = the predicted union over the B tokens (as pi_predict),
 *   u     = sparse FFN of x_hat on the list, in fp32 (as pi_sparse_ffn)
 * into u (dev fp32 [B][d]).  For a shard layer, u is the shard's part: the
 * sum of u over the shards equals the unsplit layer's update, so a caller
 * that reduces u over its devices (one all-reduce of B * d floats per layer)
 * and adds it with pi_residual_add takes the same step as pi_decode_step.
 * x and u 16-byte aligned.  The trace set by pi_set_trace, if any, gets this
 * layer's x, x_hat, list and count in its slot 0. */
pi_status pi_layer_partial(pi_ctx *ctx, int32_t layer, const float *x, int32_t B, float *u);

/* x += u, element by element in fp32, for B tokens of the stack's d_model
 * (x, u dev fp32 [B][d], 16-byte aligned): adds a reduced layer update from
 * pi_layer_partial into the residual stream. */
pi_status pi_residual_add(pi_ctx *ctx, float *x, const float *u, int32_t B);

/* Offline activation profile ("稀疏激活带来的推理局部性": count how often
 * each neuron is activated over general inputs).  For T calibration inputs
 * x_hat (dev [T][d], act_dtype), counts[i] (dev int32 [n]) is set to the
 * number of tokens for which the predictor selects physical neuron i. */
pi_status pi_layer_counts(pi_ctx *ctx, int32_t layer, const void *x_hat, int32_t T, int32_t *counts);

/* Host helper: perm (host [n]) = neurons in descending count order, ties to
 * the lower id -- the permutation that makes hot neurons contiguous. */
pi_status pi_perm_from_counts(const int32_t *counts, int32_t n, int32_t *perm);

/* Hot prefix: the one-device analog of the hot/cold split of the
 * "CPU/GPU混合推理设计" section (CSDN page "2080 Ti就能跑70B大模型..."): after
 * the calibrated permutation the hottest neurons are the first physical ones,
 * and neurons [0, hot) of `layer` are then always active -- their predictor
 * rows are not evaluated, and every list (pi_predict, the decode steps)
 * holds them, followed by the predicted neurons >= hot.  hot = 0 (the
 * default after pi_load_layer) predicts every neuron; hot = n is the dense
 * FFN.  pi_layer_counts still evaluates every row.  Synchronises the
 * context's stream before it changes the layer; a CUDA graph captured before
 * the change keeps the old prefix.  PI_ERR_ARG if hot is outside [0, n]. */
pi_status pi_set_hot_prefix(pi_ctx *ctx, int32_t layer, int32_t hot);

/* Host helper: the hot-prefix length at which always computing a neuron
 * costs no more HBM bytes than predicting it.  Predicting neuron i costs
 * pred_bytes (its W2 row and b2); when the union over B tokens misses it,
 * which happens with probability (1 - counts[i] / T)^B, that saves its
 * ffn_bytes (its FFN rows and bias).  *hot = the length of the longest prefix
 * of counts (host int32 [n], physical order; counts[i] = tokens out of T for
 * which the predictor selected neuron i) whose every neuron has
 * (1 - counts[i]/T)^B < pred_bytes / ffn_bytes.  PI_ERR_ARG for NULL
 * pointers, n, T or B < 1, bytes <= 0, or a count outside [0, T]. */
pi_status pi_hot_prefix_crossover(const int32_t *counts, int32_t n, int32_t T, int32_t B, double pred_bytes,
                                  double ffn_bytes, int32_t *hot);

/* pi_hot_prefix_crossover with the bytes of the loaded layer: pred_bytes =
 * 2 r + 2; ffn_bytes = (2 with ReGLU, else 1) d w + 2 + d w, w = 2 bytes per
 * 16-bit weight or 18/32 for Q4_0.  counts: host int32 [n], as above. */
pi_status pi_choose_hot_prefix(pi_ctx *ctx, int32_t layer, const int32_t *counts, int32_t T, int32_t B,
                               int32_t *hot);

/* Predictor ("充分利用模型和硬件特点": a small per-layer routing module
 * predicts the neurons each input activates).  For B tokens x_hat (dev
 * [B][d], act_dtype):
 *   h_t = max(CDOT(W1, x_t) + b1, 0)   (fp32, r values, not rounded)
 *   z_t = CDOT(W2, h_t) + b2           (fp32, n values)
 *   neuron i is selected for token t iff sigmoid(z) > 0.5, i.e. z > 0
 *   (so +0, -0 and NaN are not selected).
 * CDOT is a fixed fp32 order: 32 lanes, lane l accumulates fma over the
 * 8-element chunks l, l+32, ... in order, then a butterfly add over lane
 * distances 16, 8, 4, 2, 1; it makes the index list a deterministic function
 * of the input bytes.
 * Output: idx (dev int32, capacity n) = ascending physical ids of the union
 * over the B tokens, together with the layer's hot prefix (pi_set_hot_prefix);
 * *count (dev int32) = its length. */
pi_status pi_predict(pi_ctx *ctx, int32_t layer, const void *x_hat, int32_t B, int32_t *idx, int32_t *count);

/* Neuron-aware sparse FFN on the listed neurons only.  x_hat dev [B][d];
 * idx dev int32 [*count] physical ids (any order, no duplicates, each in
 * [0, n)); count dev int32.  Every token uses the whole list.
 *   a_{t,i} = ReLU:  max(W_up[i].x_t + b_i, 0)
 *             ReGLU: max(W_gate[i].x_t + b_i, 0) * (W_up[i].x_t)
 *             squared ReLU: max(W_up[i].x_t + b_i, 0)^2
 *   y_t = sum_i a_{t,i} W_down[:, i] + b_down        (fp32 accumulate)
 * y: dev [B][d] act_dtype.  An id outside [0, n) or a count outside [0, n]
 * sets PI_ERR_DEVICE_FLAG (returned by pi_sync_status) and that entry or the
 * whole call is skipped. */
pi_status pi_sparse_ffn(pi_ctx *ctx, int32_t layer, const void *x_hat, int32_t B, const int32_t *idx,
                        const int32_t *count, void *y);

/* No counterpart on the PowerInfer pages: an addition for callers that may
 * not allocate device memory.
 *
 * pi_sparse_ffn_noalloc computes what pi_sparse_ffn computes, for one layer,
 * without a context and without allocating anything.  It is meant for code
 * that only receives pre-allocated buffers, runs under a fixed device-memory
 * budget, or sits inside a server whose memory pool must not see foreign
 * allocations -- callers for which pi_create (which allocates its workspace)
 * is not an option.  The caller passes the layer's rows, the inputs and the
 * output; the kernel's scratch (epoch-tagged fp32 split-K partials, status
 * words, a one-layer descriptor, zeros for absent biases) lives in one
 * 16 MiB array that the library keeps on every GPU that loads it, until the
 * process exits.
 *
 * w: the layer in the library's row layout, all device pointers, original
 *    neuron order (no permutation):
 *      up        [n][d]  W_up rows (16-byte aligned)
 *      gate      [n][d]  W_gate rows, ReGLU only (else NULL)
 *      down_rows [n][d]  W_down TRANSPOSED: row i = neuron i's output vector
 *      b [n], b_down [d] may be NULL (= 0)
 *    act_dtype PI_F16 or PI_BF16 for every tensor (no Q4_0 here);
 *    d_model in [8, 8192] and a multiple of 8, d_ffn in [1, 65536].
 * x_hat dev [B][d], idx/count dev int32 as for pi_sparse_ffn, y dev [B][d];
 * B in [1, 64] and SMs * B * d_model <= 2,080,256 (the fp32 partials of
 * every SM, 8 bytes each with their tag, must fit the array beside its
 * 135,168 bytes of control words, descriptor and zeros: on a 152-SM GB300,
 * B * d_model <= 13,685), else PI_ERR_SHAPE.  Misaligned pointers give
 * PI_ERR_ARG.
 * dev_status: optional dev int32, set to 0, then to the first device-side
 * error (PI_ERR_DEVICE_FLAG for an index or count out of range,
 * PI_ERR_TIMEOUT); when NULL that word stays inside the array.
 * stream: cudaStream_t; the call runs on the current device.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, which may load the module): make it before any
 * stream capture.  Every call shares the array and leaves its contents
 * behind: each call clears what must start at zero (its status words, on
 * `stream`) and tags its partials with a new epoch; once in about four
 * billion calls the tags are cleared on `stream` first.  Calls whose kernels
 * can overlap on the GPU (other streams, other host threads) race on the
 * array, so serialise them. */
typedef struct {
    int32_t d_model, d_ffn;
    int32_t act;       /* pi_act */
    int32_t act_dtype; /* PI_F16 or PI_BF16 */
    const void *up, *gate, *down_rows, *b, *b_down;
} pi_ffn_rows;

pi_status pi_sparse_ffn_noalloc(const pi_ffn_rows *w, const void *x_hat, int32_t B, const int32_t *idx,
                                const int32_t *count, void *y, int32_t *dev_status, void *stream);

/* The same FFN over every neuron (the dense baseline, no predictor). */
pi_status pi_dense_ffn(pi_ctx *ctx, int32_t layer, const void *x_hat, int32_t B, void *y);

/* One decode step over the loaded stack (slots 0..L-1, all with the same
 * d_model and act_dtype), in place on the fp32 residual stream x (dev
 * [B][d]):  for each layer l:
 *   x_hat = act_dtype(x / sqrt(mean(x^2) + 1e-5))   (weightless RMSNorm)
 *   idx = predicted union over the B tokens (as pi_predict)
 *   x += sparse FFN of x_hat on idx (as pi_sparse_ffn, kept in fp32)
 * One persistent kernel runs the whole stack. */
pi_status pi_decode_step(pi_ctx *ctx, float *x, int32_t B);

/* pi_decode_step on host buffers, for callers whose residual stream lives in
 * host memory: x_in host fp32 [B][d] is copied to a device staging buffer of
 * the context, the step runs, the result is copied to x_out (host fp32
 * [B][d]; may equal x_in) and the stream is synchronised.  Page-locked host
 * buffers give asynchronous copies; pageable ones work but are staged by the
 * driver.  Returns the step's status as pi_sync_status would (device-side
 * errors included), so x_out is valid only on PI_OK. */
pi_status pi_decode_step_host(pi_ctx *ctx, const float *x_in, float *x_out, int32_t B);

/* The same step with every neuron computed (dense baseline). */
pi_status pi_dense_step(pi_ctx *ctx, float *x, int32_t B);

/* Optional per-layer trace of pi_decode_step / pi_dense_step, for checking a
 * stack against a reference layer by layer: x_trace dev fp32 [L][B][d] (the
 * residual entering each layer), xhat_trace dev [L][B][d] act_dtype,
 * idx_trace dev int32 [L][n_max] (n_max = largest d_ffn of the stack),
 * count_trace dev int32 [L].  NULL pointers disable that part. */
pi_status pi_set_trace(pi_ctx *ctx, float *x_trace, void *xhat_trace, int32_t *idx_trace, int32_t *count_trace);

/* Synchronise the context's stream and return the first device-side error
 * since the previous call (PI_ERR_TIMEOUT, PI_ERR_DEVICE_FLAG), or a CUDA
 * error, and clear it. */
pi_status pi_sync_status(pi_ctx *ctx);

/* Text of the last error on this context (never NULL; owned by the context). */
const char *pi_last_error(pi_ctx *ctx);

/* Number of SMs the persistent kernels use (one CTA per SM). */
int32_t pi_grid_size(pi_ctx *ctx);

/* Test and profiling hooks.  pi_debug_set_wait_limit: nanoseconds a device-side wait may
 * spin before it gives up with PI_ERR_TIMEOUT (default 2e9).
 * pi_debug_barrier_extra: make every cross-SM exchange of the following
 * launches wait for an epoch `extra` steps ahead of the one its writers tag
 * (SMs pass h, mask words, partials and the residual to one another as
 * epoch-tagged words instead of meeting at grid barriers), so the first
 * exchange can never complete and must time out (0 restores normal
 * operation). */
pi_status pi_debug_set_wait_limit(pi_ctx *ctx, uint64_t ns);
pi_status pi_debug_barrier_extra(pi_ctx *ctx, int32_t extra);

/* Debug timeline: when `stamps` (dev uint64 [grid][per_cta]) is set, thread 0
 * of every CTA of the step kernel writes %globaltimer (ns) at phase ends:
 * index 0 = start, then per layer l at 1 + 9*l + k, k = 0 predictor hidden
 * layer done, 1 (same moment: no barrier follows), 2 predictor output done,
 * 3 (same), 4 list resolved, 5 FFN done, 6 (same), 7 merge done, 8 first FFN
 * rows landed.  Stamps past per_cta are dropped.  NULL disables. */
pi_status pi_debug_set_timeline(pi_ctx *ctx, uint64_t *stamps, int32_t per_cta);

/* Tuning knobs of the step kernel (also read from PI_PREFETCH, PI_PREFETCH_NS,
 * PI_LOOKAHEAD and PI_ROWS_AHEAD at pi_create): prefetch = L2 prefetch of the
 * predictor weights: 0 none (the default for 16-bit stacks); the next layer's
 * slice during the FFN phase, 1 all at once or 2 paced at one 16 KB chunk per
 * prefetch_ns per SM (the default for Q4_0 stacks, prefetch_ns 800);
 * 3 each layer's W2 slice in one burst as soon as the previous layer's FFN
 * phase is over.  lookahead = how many ring stages past the one being merged
 * an owner warp may compute activations for in the FFN phase (capped at the
 * ring size minus one; default 16).  rows_ahead = neurons of an SM's list
 * whose rows are prefetched into L2 ahead of the shared-memory ring (0 none).
 * Results do not depend on them. */
pi_status pi_debug_set_tuning(pi_ctx *ctx, int32_t prefetch, int32_t prefetch_ns, int32_t lookahead,
                              int32_t rows_ahead);

/* Copy the first `count` floats of the predictor's hidden layer as the last
 * predictor pass left it, batched or in the step kernel (fp32 [B][rank],
 * h = max(W1 x_hat + b1, 0)) to dst
 * (device or host memory), asynchronously on the context's stream, so a test
 * can compare h itself, not only the index list it leads to.  count is at
 * most max_batch * 2048. */
pi_status pi_debug_copy_hidden(pi_ctx *ctx, float *dst, int32_t count);

/* Smallest batch (tokens) that runs layer by layer: the predictor as
 * batched launches and the FFN as a gather-GEMM (up to 4 tokens the 16-bit
 * up/gate rows stream whole through the CUDA cores, else tcgen05; the down
 * projection on tcgen05; Q4_0 rows dequantised to f16 in the tensor-core
 * kernels' shared memory).  Smaller
 * batches run in the persistent step kernel (CUDA cores).  -1 (the default)
 * chooses by weight type: 2 tokens for 16-bit layers, 3 for Q4_0 layers.  0
 * keeps every batch on the step kernel.  For comparing the two paths.
 * PI_ERR_ARG below -1. */
pi_status pi_debug_set_mma_min_batch(pi_ctx *ctx, int32_t min_batch);

/* *min_batch = the smallest batch for which `layer`'s FFN runs layer by
 * layer, as set by pi_debug_set_mma_min_batch (0: never, e.g. when the
 * layer's rows could not be mapped for the tensor cores).  A decode step
 * takes the path of layer 0 for the whole stack. */
pi_status pi_layerwise_min_batch(pi_ctx *ctx, int32_t layer, int32_t *min_batch);

#ifdef __cplusplus
}
#endif
#endif /* PI_H */
