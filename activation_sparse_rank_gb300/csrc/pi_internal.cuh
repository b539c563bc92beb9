// Internal declarations shared by the translation units of libpi.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "pi.h"

// Device status bits (set with atomicOr, read and cleared by pi_device_status).
#define PI_STATUS_BAD_INDEX 1u
#define PI_STATUS_BAD_COUNT 2u
#define PI_STATUS_BARRIER_TIMEOUT 4u

struct pi_layer {
  int d = 0, ffn = 0, rank = 0, act = 0;
  int device = 0, num_sms = 0;
  char *base = nullptr;          // one device allocation holding everything below
  size_t bytes = 0;
  __half *W_p1 = nullptr;        // [rank, d]
  __half *W_p2 = nullptr;        // [ffn, p2_ld]  permuted rows (rank values, then padding)
  int p2_ld = 0;                 // elements between stored W_p2 rows
  __half *W_up = nullptr;        // [ffn, d]      permuted rows
  __half *W_gate = nullptr;      // [ffn, d]      permuted rows (ReGLU)
  __half *W_dT = nullptr;        // [ffn, d]      W_down^T, permuted rows
  // PI_ROWS_FP8_E4M3 layers keep the rows as E4M3 codes with a per-row scale
  // instead (the fp16 row pointers above are then NULL)
  int row_format = PI_ROWS_FP16;
  uint8_t *Q_up = nullptr, *Q_gate = nullptr, *Q_dT = nullptr;   // [ffn, d]
  float *s_up = nullptr, *s_gate = nullptr, *s_dT = nullptr;     // [ffn]
  float *b = nullptr;            // [ffn]         permuted
  float *c_p = nullptr;          // [ffn]         permuted (zeros when absent)
  unsigned int *status = nullptr;
  std::vector<int32_t> perm;     // host copy of the permutation
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;   // profiling hook
  int n_hot = 0;                 // leading neurons of the caller's order treated as hot
};

namespace pi {

// ---- errors ---------------------------------------------------------------
pi_status fail(pi_status s, const char *fmt, ...);
void clear_error();                 // empty this thread's pi_last_error text
pi_status cuda_fail(cudaError_t e, const char *what);

#define PI_TRY_CUDA(call)                                     \
  do {                                                        \
    cudaError_t e_ = (call);                                  \
    if (e_ != cudaSuccess) return pi::cuda_fail(e_, #call);   \
  } while (0)

// ---- workspace --------------------------------------------------------------
// Layout of the caller's workspace for batches of up to B tokens.
struct WsLayout {
  size_t h = 0;        // float [B, rank]
  size_t a = 0;        // float [B, ffn]        activations by list position
  size_t partial = 0;  // float [nsplit, B, d]  split-K partial sums
  size_t mask = 0;     // uint8 [max(B, kMaxStack), ffn]
  size_t idx = 0;      // int32 [ffn]           (pi_layer_forward when idx not given)
  size_t count = 0;    // int32 [4]
  size_t cnt = 0;      // int32 [G]             per-CTA active counts (persistent step)
  size_t bar = 0;      // uint32                grid-barrier counter
  size_t abuf = 0;     // fp16 [2*Bp, ffn_pad]  activations (hi; lo) of the tensor-core path
  size_t hbuf = 0;     // fp16 [2*Bp, rank_pad] predictor hidden layer (hi; lo), tensor-core path
  size_t tcpart = 0;   // float [2 G, 2 Bp, 128] tensor-core tiles split between CTAs
  size_t tcnt = 0;     // int32 [ffn_pad / 128] active rows per logits tile
  size_t total = 0;
};

// Layers per persistent launch (longer stacks are split into several launches).
constexpr int kMaxStack = PI_STACK_LAYERS_PER_LAUNCH;


// Device pointers of one layer, as the persistent kernel sees them.
struct LayerDev {
  const __half *W_p1, *W_p2;         // W_p2 rows p2_ld elements apart (StackParams::p2_stride bytes)
  const void *R_up, *R_gate, *R_dT;   // rows: fp16, or E4M3 codes (FP8 layers)
  const float *s_up, *s_gate, *s_dT;  // per-row scales (FP8 layers)
  const float *b, *c_p;
  int hot_per_slice;     // leading slice positions whose rows are fetched speculatively
};

// Kernel parameters of the persistent step (passed by value, < 4 KB).
struct StackParams {
  int n_layers, d, ffn, rank;
  int G, staged, lanes_l, pf_rows;
  int chained;                   // x of layer l > 0 formed from y of layer l - 1
  int lgt_s;                     // log2 threads per staged W_p2 row (logits)
  int mma_logits, p2_stride;     // staged logits on tensor cores; bytes between staged W_p2 rows
  int off_flag, off_list, off_lb, off_a, off_stage, stage_bytes, slice_pad;   // shared memory layout
  int soff_c, soff_b, soff_p1, soff_p2;                     // offsets inside a stage buffer
  int soff_su, soff_sg, soff_sd;                            // row-scale slices (FP8 layers)
  int gate_silu;                                            // gated layers: SiLU gate (SwiGLU)
  const __half *x;       // [n_layers, B, d] (chained: only layer 0 is read)
  __half *x_out;         // chained: [n_layers, B, d], the inputs formed (layer 0 untouched); else nullptr
  __half *x_next;        // chained: [B, d], the input of the layer after this launch, or nullptr
  float *y;              // [n_layers, B, d]
  int32_t *count;        // [n_layers] or nullptr
  uint8_t *mask_out;     // [n_layers, ffn] union masks (for the idx output) or nullptr
  float *h;              // scratch [B, rank]
  int32_t *cnt;          // scratch [G]
  float *partial;        // scratch [G, B, d]
  unsigned *bar;         // scratch barrier counter (zeroed before launch)
  unsigned *status;
  LayerDev layers[kMaxStack];
};
// Stored W_p2 row length in elements: a rank that is a multiple of 64 gets 32
// elements (64 bytes) of padding per row, so that the decode step's
// tensor-core logits, which read 16 bytes of 8 consecutive rows at once from
// a staged copy of the rows, hit distinct shared-memory banks.
inline int p2_ld_for(int rank) { return rank % 64 == 0 ? rank + 32 : rank; }
int step_grid(const pi_layer *L);
int step_slice(const pi_layer *L);
bool step_staged(const pi_layer *L, int B);
size_t step_smem(const pi_layer *L, int B);
// Ascending active lists of n layers from their union masks [n, ffn] (one CTA per layer).
cudaError_t run_compact_layers(const pi_layer *L, const uint8_t *masks, int n, int32_t *idx,
                               int32_t *count, cudaStream_t s);
// chained: x of layer l > 0 is fp16(y_{l-1} / RMS(y_{l-1})), written to x_out
// [n, B, d]; x_next (or nullptr) receives the input of the layer after layer n - 1.
cudaError_t run_stack(pi_layer *const *layers, int n, const __half *x, int B, int32_t *idx,
                      int32_t *count, float *y, const WsLayout &w, char *ws, cudaStream_t s,
                      bool chained = false, __half *x_out = nullptr, __half *x_next = nullptr);
WsLayout ws_layout(const pi_layer *L, int B);
int fused_splits(const pi_layer *L);        // CTAs of the batch-1 fused kernel
int down_splits(const pi_layer *L, int B);  // split count of the generic down kernel
int down_colblocks(const pi_layer *L);      // column blocks of the generic down kernel

// ---- launch helpers ---------------------------------------------------------
// Launch with programmatic dependent launch (the kernel must execute
// griddepcontrol.wait before touching anything a predecessor writes).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Record the layer's profiling event (if set) on s; external record when capturing.
cudaError_t record_hook(cudaEvent_t ev, cudaStream_t s);

// Stage launchers (pi_predict.cu / pi_sparse.cu).  All asynchronous.
// union_mask: mask is [ffn], 1 where any token of the batch is active
cudaError_t run_predict(const pi_layer *L, const __half *x, int B, uint8_t *mask,
                        float *logits, float *h_ws, cudaStream_t s, bool union_mask = false);
cudaError_t run_compact(const pi_layer *L, const uint8_t *mask, int B, int32_t *idx,
                        int32_t *count, cudaStream_t s);
// idx == nullptr means the identity list 0..count_const-1 (count ignored).
cudaError_t run_sparse_ffn(const pi_layer *L, const __half *x, int B, const int32_t *idx,
                           const int32_t *count, int count_const, float *y,
                           const WsLayout &w, char *ws, cudaStream_t s);
// Tensor-core (tcgen05) batched path for 3 <= B <= PI_MAX_BATCH (pi_tc.cu).
bool tc_supported(const pi_layer *L, int B);
int tc_bpad(int B);
int tc_ffn_pad(const pi_layer *L);
bool tc_predict_supported(const pi_layer *L, int B);
int tc_rank_pad(const pi_layer *L);
// h (fp16 pair, in hbuf [2Bp, rank_pad]), the batch-union mask [ffn] and its
// ascending list idx / count on the tensor cores; piece: fp32 scratch of
// tc_piece_bytes for tiles split between CTAs; tile_cnt: int [ffn_pad / 128].
cudaError_t run_predict_tc(const pi_layer *L, const __half *x, int B, uint8_t *mask_union, __half *hbuf,
                           float *piece, int32_t *tile_cnt, int32_t *idx, int32_t *count, cudaStream_t s);
size_t tc_piece_bytes(const pi_layer *L, int B);
// The same predictor (hbuf as [2B, rank], the union mask, idx / count) in one
// cooperative launch for 3 <= B <= 32 (pi_pbatch.cu); partial: fp32 scratch
// of tc_piece_bytes; cnt: int [num_sms]; bar: a grid-barrier counter.
bool pbatch_supported(const pi_layer *L, int B);
cudaError_t run_predict_batch(const pi_layer *L, const __half *x, int B, uint8_t *mask_union, __half *hbuf,
                              float *partial, int32_t *cnt, unsigned *bar, int32_t *idx, int32_t *count,
                              cudaStream_t s);
cudaError_t run_sparse_ffn_tc(const pi_layer *L, const __half *x, int B, const int32_t *idx,
                              const int32_t *count, int count_const, float *y, const WsLayout &w,
                              char *ws, cudaStream_t s);
cudaError_t run_reduce(const float *partial, int nsplit, int n, float *y, cudaStream_t s);
cudaError_t run_profile(const pi_layer_desc *desc, const __half *x, int T, int32_t *counts,
                        cudaStream_t s);

}  // namespace pi

// ---- device helpers ---------------------------------------------------------
namespace pidev {

__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Streaming 16-byte load of weights (read once per use; do not keep in L1).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Ask L2 to fetch `bytes` (multiple of 16, 16-byte aligned) starting at p.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// acc += sum of the 8 products w[e] * x[e]; fp16 products are exact in fp32.
__device__ __forceinline__ float dot8(float acc, const uint4 &w, const uint4 &x) {
  const __half2 *wh = reinterpret_cast<const __half2 *>(&w);
  const __half2 *xh = reinterpret_cast<const __half2 *>(&x);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float2 wf = __half22float2(wh[e]);
    float2 xf = __half22float2(xh[e]);
    acc = fmaf(wf.x, xf.x, acc);
    acc = fmaf(wf.y, xf.y, acc);
  }
  return acc;
}

// acc[e] += s * w[e] for the 8 halves of w.
__device__ __forceinline__ void axpy8(float *acc, float s, const uint4 &w) {
  const __half2 *wh = reinterpret_cast<const __half2 *>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float2 wf = __half22float2(wh[e]);
    acc[2 * e] = fmaf(s, wf.x, acc[2 * e]);
    acc[2 * e + 1] = fmaf(s, wf.y, acc[2 * e + 1]);
  }
}

// The same for 8 E4M3 codes (w) against 8 halves (x); E4M3 values are exact
// in fp16 and the products exact in fp32.
__device__ __forceinline__ float dot8_e4m3(float acc, const uint2 &w, const uint4 &x) {
  const __nv_fp8x2_storage_t *wq = reinterpret_cast<const __nv_fp8x2_storage_t *>(&w);
  const __half2 *xh = reinterpret_cast<const __half2 *>(&x);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(wq[e], __NV_E4M3);
    float2 wf = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
    float2 xf = __half22float2(xh[e]);
    acc = fmaf(wf.x, xf.x, acc);
    acc = fmaf(wf.y, xf.y, acc);
  }
  return acc;
}

__device__ __forceinline__ void axpy8_e4m3(float *acc, float s, const uint2 &w) {
  const __nv_fp8x2_storage_t *wq = reinterpret_cast<const __nv_fp8x2_storage_t *>(&w);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(wq[e], __NV_E4M3);
    float2 wf = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
    acc[2 * e] = fmaf(s, wf.x, acc[2 * e]);
    acc[2 * e + 1] = fmaf(s, wf.y, acc[2 * e + 1]);
  }
}

__device__ __forceinline__ uint2 ld_stream2(const uint2 *p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// Gate of a gated neuron: ReLU (ReGLU) or SiLU (SwiGLU).
__device__ __forceinline__ float gate_act(float z, bool silu) {
  return silu ? z / (1.0f + expf(-z)) : (z > 0.f ? z : 0.f);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Read *count once, clamp it to [0, limit] and flag values out of range.
__device__ __forceinline__ int load_count(const int32_t *count, int count_const, int limit,
                                          unsigned int *status) {
  if (count == nullptr) return count_const;
  int c = *count;
  if (c < 0 || c > limit) {
    if (threadIdx.x == 0) atomicOr(status, PI_STATUS_BAD_COUNT);
    c = c < 0 ? 0 : limit;
  }
  return c;
}

}  // namespace pidev
