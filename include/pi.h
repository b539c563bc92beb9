/*
 * pi.h - C ABI of libpi, the predictor-gated, neuron-aware sparse FFN for
 * one NVIDIA GB300 (sm_103a).
 *
 * The method is PowerInfer's decode-time FFN block ("PowerInfer: Fast Large
 * Language Model Serving with a Consumer-grade GPU", egguo-blog reading
 * report): per layer an adaptive predictor (section 2.3, core module 3)
 * selects the neurons expected to fire, and neuron-aware operators (section
 * 2.3, core module 4) compute only those neurons, directly on the rows of the
 * weight matrices, with no sparse-format conversion.  The offline profile
 * (section 2.3, core module 1) becomes a hot-first neuron order of the
 * resident weight layout.
 *
 * Conventions shared by every call:
 *  - fp16 data is passed as IEEE binary16 bit patterns (uint16_t).
 *  - "device" pointers are CUDA device (or managed) memory of the current
 *    device; "host" pointers are ordinary CPU memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Every call except create/destroy/perm/hot_first_perm/device_status is
 *    asynchronous on that stream, allocates nothing and copies nothing to
 *    the host, so a sequence of calls can be captured in a CUDA graph.
 *  - Active-set sizes never leave the device: `count` is a device int32.
 *  - Arguments are validated on the host before any launch; a rejected call
 *    launches nothing.  Device-side checks (an index or count out of range)
 *    never trap: the offending element is skipped and a status word in the
 *    layer is set, which pi_device_status() reports.
 *  - pi_last_error() returns a thread-local message for the last failure.
 */
#ifndef PI_H_
#define PI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PI_OK = 0,
  PI_ERR_INVALID_ARG = 1,   /* bad pointer, size or shape; nothing launched      */
  PI_ERR_UNSUPPORTED = 2,   /* shape outside the library's supported range       */
  PI_ERR_OOM = 3,           /* pi_layer_create could not allocate device memory  */
  PI_ERR_CUDA = 4,          /* a CUDA runtime call failed (see pi_last_error)    */
  PI_ERR_DEVICE_CHECK = 5   /* a kernel found an out-of-range index or count     */
} pi_status;

typedef enum {
  PI_ACT_RELU = 0,   /* a_i = max(0, W_up_i.x + b_i)                           */
  PI_ACT_REGLU = 1,  /* a_i = max(0, W_gate_i.x + b_i) * (W_up_i.x)            */
  PI_ACT_SWIGLU = 2  /* a_i = SiLU(W_gate_i.x + b_i) * (W_up_i.x), SiLU(z) = z / (1 + e^-z):
                        section 2.3 variable table and section 4.4 limitation 1 (SwiGLU
                        models: neurons pruned with a small effect, about half kept); the
                        sum runs over the predicted set, which skips the pruned neurons */
} pi_act;

/* Storage of the up / gate / down rows that the sparse operators gather.
 * The report's results include quantised weights (section 3.1, Finding 2:
 * INT4 runs); this library's quantised format is its own choice: FP8 E4M3
 * codes with one fp32 scale per stored row, which halves the bytes a gathered
 * row costs while the predictor stays fp16.
 *   PI_ROWS_FP8_E4M3: for each row w of W_up, W_gate and W_down^T (d values):
 *     s = max_j |w_j| / 448 in binary32 (s = 1 when the row is all zero),
 *     q_j = the E4M3 code of w_j / s (binary32 division, round to nearest
 *           even, saturating to +-448),
 *   and the row stands for s * q_j.  The FFN is the FFN of these weights. */
typedef enum {
  PI_ROWS_FP16 = 0,
  PI_ROWS_FP8_E4M3 = 1
} pi_row_format;

/* Shape limits (PI_ERR_UNSUPPORTED outside them). */
#define PI_MAX_D      16384   /* d % 8 == 0 */
#define PI_MAX_RANK   2048    /* rank % 8 == 0 */
#define PI_MAX_FFN    (1 << 20)
#define PI_MAX_BATCH  128
/* pi_stack_forward runs one persistent kernel per this many layers (1-2 tokens). */
#define PI_STACK_LAYERS_PER_LAUNCH 32

typedef struct pi_layer pi_layer;

/* One FFN layer in model space, PyTorch nn.Linear weight layouts, all device
 * pointers.  Read only during pi_layer_create / pi_profile_activations.
 *   W_up   [ffn, d]   fp16  up projection
 *   W_gate [ffn, d]   fp16  gate projection (PI_ACT_REGLU / PI_ACT_SWIGLU, else NULL)
 *   b      [ffn]      fp32  bias of the gated projection (up for ReLU, gate otherwise)
 *   W_down [d, ffn]   fp16  down projection
 *   W_p1   [rank, d]  fp16  predictor first layer (no bias)
 *   W_p2   [ffn, rank] fp16 predictor second layer
 *   c_p    [ffn]      fp32  predictor output bias, or NULL for zero
 *   row_format        pi_row_format of the stored up / gate / down rows
 *                     (0, PI_ROWS_FP16, keeps them as given) */
typedef struct {
  int32_t d, ffn, rank;
  int32_t act;               /* pi_act */
  const uint16_t *W_up;
  const uint16_t *W_gate;
  const float *b;
  const uint16_t *W_down;
  const uint16_t *W_p1;
  const uint16_t *W_p2;
  const float *c_p;
  int32_t row_format;        /* pi_row_format */
} pi_layer_desc;

/* Build a layer object that owns a permuted, neuron-major copy of the weights
 * (section 2.3, core module 1 and variable table: neurons ordered by profiled
 * activation frequency v_i = f_i, hot first).
 *   perm  host int32 [ffn] or NULL (identity): the caller's neuron order, for
 *         example hot-first from pi_hot_first_perm; must be a permutation of
 *         0..ffn-1.  The layer deals this order round-robin over G slices,
 *         G = the device's SM count: the k-th neuron of `perm` is stored in
 *         slice k % G at place k / G, slices (sizes differing by at most one)
 *         laid out one after another.  Every slice then holds the same mix of
 *         hot and cold neurons, which balances the persistent step's per-SM
 *         work.  pi_layer_perm returns the resulting storage order.
 * The library copies W_p1 as is, permutes the rows of W_up, W_gate, b, W_p2,
 * c_p, and stores W_down transposed and permuted as W_down^T [ffn, d] so that
 * each neuron's down weights are one contiguous row.  Peak device memory is
 * the caller's weights plus one layer copy.  Synchronous: returns after the
 * copy finished on `stream`.  The caller may free its buffers afterwards.
 * With row_format PI_ROWS_FP8_E4M3 the permuted up / gate / down^T rows are
 * quantised on the device as described at pi_row_format and only the codes
 * and scales are kept (d + 4 bytes per row).  Such a layer runs in every
 * entry point but pi_sparse_ffn_noalloc (PI_ERR_UNSUPPORTED): the decode step
 * of pi_layer_forward / pi_stack_forward (1 or 2 tokens) reads the codes in
 * its persistent kernel; pi_sparse_ffn, pi_ffn_dense_ref and the batches of
 * 3 or more tokens read them in the generic CUDA-core kernels (the
 * tensor-core path takes fp16 rows only).
 * Errors: PI_ERR_INVALID_ARG (NULL pointer, bad perm, unknown row_format),
 * PI_ERR_UNSUPPORTED (shape), PI_ERR_OOM, PI_ERR_CUDA. *out is NULL on
 * failure. */
pi_status pi_layer_create(pi_layer **out, const pi_layer_desc *desc,
                          const int32_t *perm, void *stream);

/* Free the layer and its device memory (synchronizes the device first).
 * NULL is accepted. */
pi_status pi_layer_destroy(pi_layer *layer);

/* Shape of a layer (any output pointer may be NULL). */
pi_status pi_layer_info(const pi_layer *layer, int32_t *d, int32_t *ffn,
                        int32_t *rank, int32_t *act);

/* Copy the stored FP8 rows of a PI_ROWS_FP8_E4M3 layer, in storage order:
 *   matrix  0 W_up, 1 W_gate (ReGLU only), 2 W_down^T
 *   codes   device uint8 [ffn, d] (E4M3 bit patterns)
 *   scales  device fp32 [ffn]
 * Asynchronous on `stream`.  PI_ERR_UNSUPPORTED for an fp16 layer. */
pi_status pi_layer_rows_fp8(const pi_layer *layer, int32_t matrix, uint8_t *codes,
                            float *scales, void *stream);

/* Copy the layer's storage order (host int32 [ffn]): position k holds model
 * neuron perm[k].  Active-set indices returned by this library are positions
 * k, i.e. in permuted space. */
pi_status pi_layer_perm(const pi_layer *layer, int32_t *perm);

/* Bytes of device workspace that pi_predict, pi_sparse_ffn, pi_ffn_dense_ref
 * and pi_layer_forward need for batches of up to B_max tokens (0 on bad
 * arguments).  The workspace is caller-owned scratch; calls that run
 * concurrently need separate workspaces. */
size_t pi_workspace_bytes(const pi_layer *layer, int32_t B_max);

/* Adaptive predictor (section 2.3, core module 3): for each token b < B,
 *   h = max(0, W_p1 x_b)            binary32 accumulation, h kept in binary32
 *   l = W_p2 h + c_p                binary32
 *   mask[b, i] = (l_i > 0)          i.e. sigmoid(l_i) > 0.5; l_i == 0 is inactive
 *   x       device fp16 [B, d] (model space; rows contiguous)
 *   mask    device uint8 [B, ffn] (permuted space), values 0/1, or NULL
 *   logits  device fp32 [B, ffn] (permuted space), or NULL
 *   ws      device workspace of at least pi_workspace_bytes(layer, B) bytes
 * 1 <= B <= PI_MAX_BATCH.  At least one of mask/logits must be non-NULL. */
pi_status pi_predict(pi_layer *layer, const uint16_t *x, int32_t B,
                     uint8_t *mask, float *logits, void *ws, size_t ws_bytes,
                     void *stream);

/* Active-index compaction (section 2.3, core module 4 computes on the
 * predicted neurons directly; section 4.4 limitation 3: with a batch, the set
 * is the union over the batch):
 *   idx[0..count) = ascending positions i with mask[b, i] != 0 for some b.
 *   mask   device uint8 [B, ffn]
 *   idx    device int32 [ffn]   (entries past count are left untouched)
 *   count  device int32 [1] */
pi_status pi_compact_active(const pi_layer *layer, const uint8_t *mask,
                            int32_t B, int32_t *idx, int32_t *count,
                            void *stream);

/* Neuron-aware sparse FFN (section 2.3, core module 4; variable table,
 * "sparsity": neurons outside the set contribute exactly nothing):
 *   for k < *count, i = idx[k]:  a_i(b) per the layer's activation
 *   y[b, :] = sum_k a_{idx[k]}(b) * W_down^T[idx[k], :]
 * Only the rows idx[0..count) of W_up (and W_gate), and of W_down^T, are read.
 * binary32 accumulation; the reduction over neurons is split over CTAs and
 * combined in a fixed order, so results are bitwise reproducible run to run.
 *   x      device fp16 [B, d]
 *   idx    device int32 [>= *count], positions in [0, ffn), any order
 *   count  device int32 [1], 0 <= *count <= ffn
 *   y      device fp32 [B, d], overwritten
 * Out-of-range idx entries are skipped and *count is clamped to [0, ffn];
 * either sets the layer's device status. */
pi_status pi_sparse_ffn(pi_layer *layer, const uint16_t *x, int32_t B,
                        const int32_t *idx, const int32_t *count, float *y,
                        void *ws, size_t ws_bytes, void *stream);

/* Dense comparator: the same kernels as pi_sparse_ffn over every neuron
 * (idx = 0..ffn-1), without the predictor. */
pi_status pi_ffn_dense_ref(pi_layer *layer, const uint16_t *x, int32_t B,
                           float *y, void *ws, size_t ws_bytes, void *stream);

/* The whole layer for one batch: the results of pi_predict, then
 * pi_compact_active, then pi_sparse_ffn.  For B <= 2 this is one persistent
 * cooperative kernel (see pi_stack_forward).  For 3 <= B <= 32 (rank a
 * multiple of 64, d of 32) the predictor, the union over the batch and the
 * ascending list are one cooperative launch with one CTA per SM and three
 * grid-wide barriers (bounded waits, as in pi_stack_forward); above, or for
 * other shapes, separate kernels.  The FFN then runs on the tensor cores
 * (d a multiple of 64, d >= 128) or on the generic kernels.
 *   idx, count  device outputs as in pi_compact_active
 *   y           device fp32 [B, d] */
pi_status pi_layer_forward(pi_layer *layer, const uint16_t *x, int32_t B,
                           int32_t *idx, int32_t *count, float *y,
                           void *ws, size_t ws_bytes, void *stream);

/* A decode step through a stack of layers in order (layer l reads x[l] and
 * writes y[l]; each layer's result is complete before the next layer
 * starts, as when the next input depends on it).  All layers must share d,
 * ffn, rank, activation and device.
 *   layers  host array of n_layers layer objects
 *   x       device fp16 [n_layers, B, d]
 *   idx     device int32 [n_layers, ffn] active lists, or NULL (B <= 2 only)
 *   count   device int32 [n_layers] active counts, or NULL (B <= 2 only)
 *   y       device fp32 [n_layers, B, d]
 *   ws      workspace of pi_workspace_bytes(layers[0], B) bytes
 * For B <= 2 each group of up to PI_STACK_LAYERS_PER_LAUNCH layers is one
 * cooperative launch with one CTA per SM and three grid-wide barriers per
 * layer (predictor hidden layer; split partial sums; output).  The partial
 * sums of y are added in a fixed order, so y is bitwise reproducible.  Barrier
 * waits are bounded: a wait that runs out sets a status bit
 * (PI_ERR_DEVICE_CHECK from pi_device_status on layers[0]) and the kernel
 * returns. */
pi_status pi_stack_forward(pi_layer *const *layers, int32_t n_layers,
                           const uint16_t *x, int32_t B, int32_t *idx,
                           int32_t *count, float *y, void *ws,
                           size_t ws_bytes, void *stream);

/* The same decode step with each layer's input formed from the previous
 * layer's output on the device (a decoder's data dependence; the attention
 * blocks between FFN blocks are outside this library):
 *   x[l] = fp16(y[l-1] / RMS(y[l-1])) for l >= 1, per token,
 *   RMS(v) = sqrt(mean(v^2) + 1e-12) in binary32.
 *   x  device fp16 [n_layers, B, d]: x[0] is the input; x[1..n_layers) are
 *      overwritten with the inputs the layers used.
 * Other arguments, results and errors as pi_stack_forward.  No input of
 * layer l >= 1 is read before layer l - 1's y is complete. */
pi_status pi_stack_forward_chained(pi_layer *const *layers, int32_t n_layers,
                                   uint16_t *x, int32_t B, int32_t *idx,
                                   int32_t *count, float *y, void *ws,
                                   size_t ws_bytes, void *stream);

/* T decode steps from host memory in one call: copies x_host into x_dev,
 * runs pi_stack_forward (or, with chained != 0, pi_stack_forward_chained) for
 * each token t on x_dev[t] -> y_dev[t], and copies y_dev into y_host, all
 * asynchronously on `stream` (the copies are part of the call, so a caller
 * that times it from host buffers to host buffers times the copies too).
 *   x_host  host fp16 [T, n_layers, B, d]; y_host host fp32 [T, n_layers, B, d]
 *           (page-locked memory lets the copies run asynchronously at full
 *           rate; pageable memory works, the copies then block the host)
 *   x_dev   device fp16 [T, n_layers, B, d], y_dev device fp32 [T, n_layers, B, d]
 *           (caller-owned staging; in chained mode x_dev[t][1..] is overwritten)
 *   idx     device int32 [n_layers, ffn] (the last token's lists) or NULL (B <= 2)
 *   count   device int32 [T, n_layers] or NULL (B <= 2)
 * Errors as pi_stack_forward; nothing is launched after the first failure. */
pi_status pi_stack_forward_host(pi_layer *const *layers, int32_t n_layers, int32_t T,
                                const uint16_t *x_host, int32_t B, float *y_host,
                                uint16_t *x_dev, float *y_dev, int32_t *idx,
                                int32_t *count, int32_t chained, void *ws,
                                size_t ws_bytes, void *stream);

/* pi_sparse_ffn without a workspace, for callers that cannot allocate device
 * memory when they call in (for example a serving framework that has already
 * handed all GPU memory to its own pool, or a plug-in that receives only input
 * and output pointers).  The pages have no counterpart: this is a calling
 * convention of this library, not part of the method.
 * Same arguments and results as pi_sparse_ffn (x, idx, count, y device
 * pointers), batches of 1 or 2 tokens only.  The split partial sums live in a
 * fixed 16 MiB device array inside the library, reserved on a GPU when that
 * GPU loads the array (with CUDA's default lazy module loading: this entry
 * point's first call on it; with CUDA_MODULE_LOADING=EAGER: when the library
 * is loaded) and kept until the process exits.  A call whose d and B need
 * more than that (4 * splits * B * d bytes, splits = the CTAs of the fused
 * kernel: the SM count times 4 for d <= 1024, 3 for d <= 1280, 2 for
 * d <= 2048 and 1 above) returns PI_ERR_UNSUPPORTED without launching.
 * Nothing is allocated and nothing in the array has to start at zero.
 * The array's device address is looked up (cudaGetSymbolAddress) on the first
 * call in each device context and cached for that context; a new context (for
 * example after cudaDeviceReset) looks it up again.  Make the first call in a
 * context outside any stream capture.  All calls share the one array: calls
 * whose kernels can overlap on the GPU (other streams, other host threads)
 * race on it and must be serialised by the caller. */
pi_status pi_sparse_ffn_noalloc(pi_layer *layer, const uint16_t *x, int32_t B,
                                const int32_t *idx, const int32_t *count, float *y,
                                void *stream);

/* Offline activation profile (section 2.3, core module 1 "LLM profiler";
 * section 2.2, profiling data): for T tokens x_t, in model space,
 *   counts[i] += #{t : z_i(x_t) > 0}, z = W_up x + b (ReLU) or W_gate x + b (ReGLU)
 *   x       device fp16 [T, d]
 *   counts  device int32 [ffn], accumulated into (the caller zeroes it)
 * Reads the desc's model-space weights; needs no layer object. */
pi_status pi_profile_activations(const pi_layer_desc *desc, const uint16_t *x,
                                 int32_t T, int32_t *counts, void *stream);

/* Hot-first order from a profile (section 2.3, variable table: impact
 * v_i = f_i; hot neurons are the frequently activated ones): perm lists the
 * neurons by count descending, ties by ascending index.  Host arrays. */
pi_status pi_hot_first_perm(const int32_t *counts, int32_t ffn, int32_t *perm);

/* Profiling hook.  While ev_before / ev_after (cudaEvent_t passed as void*)
 * are set, each call on this layer records ev_before on its stream
 * immediately before its main kernel and ev_after immediately after it (as
 * external event-record nodes when the stream is being captured into a CUDA
 * graph), so the caller can time that kernel alone with cudaEventElapsedTime.
 * The main kernel is the up/down kernel of pi_sparse_ffn / pi_ffn_dense_ref
 * (and of pi_layer_forward for B > 2), and the persistent step kernel of
 * pi_layer_forward / pi_stack_forward for B <= 2 (hook of layers[0]).  Both
 * NULL switches it off.  The setting is per layer and read at call time. */
pi_status pi_layer_set_timing_events(pi_layer *layer, void *ev_before, void *ev_after);

/* Hot-neuron hint for the persistent step (section 2.3, variable table: hot
 * neurons are the few that are activated most often; section 3.1 Finding 1).
 * n_hot = how many leading neurons of the order given to pi_layer_create are
 * hot (e.g. those a profile shows active on more than half of the tokens).
 * pi_layer_forward / pi_stack_forward (B <= 2) then load the rows of each
 * SM slice's leading hot places (at most a few per slice, as many as its
 * registers hold) while the previous layer finishes and the predictor runs,
 * before the predictor has decided, so that HBM is busy during the predictor
 * phases.  Results do not change; a hot neuron the predictor leaves out only
 * costs bandwidth.
 * 0 (the default) disables it.  0 <= n_hot <= ffn. */
pi_status pi_layer_set_hot_count(pi_layer *layer, int32_t n_hot);

/* Number of kernel launches one pi_layer_forward call makes for a batch of B
 * tokens (0 on bad arguments). */
int32_t pi_forward_launches(const pi_layer *layer, int32_t B);

/* Synchronize `stream`, then return PI_ERR_DEVICE_CHECK if any kernel on this
 * layer flagged an out-of-range index or count since the last query (and
 * clear the flag), else PI_OK. */
pi_status pi_device_status(pi_layer *layer, void *stream);

/* Thread-local text of the last error ("" if none). */
const char *pi_last_error(void);

/* Name of a status code. */
const char *pi_status_string(pi_status status);

#ifdef __cplusplus
}
#endif

#endif /* PI_H_ */
