// pi_sparse_ffn_noalloc: the sparse FFN of pi_sparse_ffn for callers that
// cannot hand the library a workspace.
//
// Some hosts cannot allocate device memory when they call in: a serving
// framework that has already carved the whole GPU into its own memory pool, or
// a plug-in that only receives input and output pointers through a fixed
// interface and has no allocator to ask.  For them this entry point keeps its
// scratch (the per-CTA partial sums of the split reduction) in a file-scope
// device array, so the call needs nothing beyond its inputs and outputs.
//
// The array is reserved on a GPU when that GPU loads this file's module (with
// CUDA's default lazy module loading: at this entry point's first call on the
// GPU) and stays until the process exits, so it is kept modest: kScratchBytes
// below.  All calls share it: calls whose kernels overlap on the GPU
// (different streams, or different host threads) race on it and must be
// serialised by the caller.
#include <cuda.h>

#include <mutex>

#include "pi_internal.cuh"

namespace {

constexpr size_t kScratchBytes = 16u << 20;   // 16 MiB per device
constexpr int kMaxDevices = 64;

// Holds the partial sums [splits, B, d] fp32 of the sparse FFN.  Every CTA
// writes its whole slice before the reduction reads it, so no call depends on
// what an earlier call left here and nothing needs clearing.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mutex;
struct Cached {
  CUcontext ctx = nullptr;   // the context the address belongs to
  void *ptr = nullptr;
};
Cached g_cache[kMaxDevices];

// The driver's cuCtxGetCurrent, looked up through the runtime (the library
// does not link libcuda).
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

// Device address of the scratch array in the current context of device dev.
// Host code must not use the symbol itself as a device pointer.  The address
// is looked up once per context: a new context (after cudaDeviceReset, or
// after the primary context was released and created again) looks it up anew.
pi_status scratch_for_device(int dev, void **out) {
  if (dev < 0 || dev >= kMaxDevices) return pi::fail(PI_ERR_UNSUPPORTED, "device %d out of range", dev);
  const CtxGetCurrentFn get = ctx_get_current();
  if (!get) return pi::fail(PI_ERR_CUDA, "cuCtxGetCurrent is not available from the driver");
  std::lock_guard<std::mutex> lock(g_mutex);
  CUcontext ctx = nullptr;
  if (get(&ctx) != CUDA_SUCCESS) return pi::fail(PI_ERR_CUDA, "cuCtxGetCurrent failed");
  Cached &c = g_cache[dev];
  if (!c.ptr || !ctx || ctx != c.ctx) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);   // makes the context current
    if (e != cudaSuccess) return pi::cuda_fail(e, "cudaGetSymbolAddress(g_noalloc_scratch)");
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return pi::fail(PI_ERR_CUDA, "no current context on device %d", dev);
    c.ctx = ctx;
    c.ptr = p;
  }
  *out = c.ptr;
  return PI_OK;
}

}  // namespace

extern "C" pi_status pi_sparse_ffn_noalloc(pi_layer *L, const uint16_t *x, int32_t B,
                                           const int32_t *idx, const int32_t *count, float *y,
                                           void *stream) {
  pi::clear_error();
  if (!L) return pi::fail(PI_ERR_INVALID_ARG, "layer is NULL");
  if (L->row_format != PI_ROWS_FP16)
    return pi::fail(PI_ERR_UNSUPPORTED, "pi_sparse_ffn_noalloc needs a layer with fp16 rows");
  if (B < 1 || B > 2)
    return pi::fail(PI_ERR_UNSUPPORTED, "pi_sparse_ffn_noalloc handles batches of 1 or 2 tokens, got %d", B);
  if (!x || (reinterpret_cast<uintptr_t>(x) & 15u))
    return pi::fail(PI_ERR_INVALID_ARG, "x must be non-NULL and 16-byte aligned");
  if (!idx || !count || (reinterpret_cast<uintptr_t>(idx) & 3u) || (reinterpret_cast<uintptr_t>(count) & 3u))
    return pi::fail(PI_ERR_INVALID_ARG, "idx and count must be non-NULL and 4-byte aligned");
  if (!y || (reinterpret_cast<uintptr_t>(y) & 15u))
    return pi::fail(PI_ERR_INVALID_ARG, "y must be non-NULL and 16-byte aligned");
  const size_t need = sizeof(float) * (size_t)pi::fused_splits(L) * (size_t)B * (size_t)L->d;
  if (need > kScratchBytes)
    return pi::fail(PI_ERR_UNSUPPORTED,
                    "pi_sparse_ffn_noalloc needs %zu bytes of scratch for d=%d, B=%d; its fixed "
                    "scratch holds %zu (use pi_sparse_ffn with a workspace)",
                    need, L->d, B, kScratchBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pi::cuda_fail(e, "cudaGetDevice");
  if (dev != L->device)
    return pi::fail(PI_ERR_INVALID_ARG, "current device %d is not the layer's device %d", dev, L->device);
  void *scratch = nullptr;
  const pi_status st = scratch_for_device(dev, &scratch);
  if (st != PI_OK) return st;
  pi::WsLayout w;          // only the partial sums live in the scratch (batches of <= 2)
  w.partial = 0;
  w.total = need;
  e = pi::run_sparse_ffn(L, reinterpret_cast<const __half *>(x), B, idx, count, 0, y, w,
                         static_cast<char *>(scratch), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return pi::cuda_fail(e, "pi_sparse_ffn_noalloc launch");
  return PI_OK;
}
