// C ABI of libpi: layer objects, argument checking, workspace layout, the
// offline activation profiler and the hot-first order.
//
// "PowerInfer: Fast Large Language Model Serving with a Consumer-grade GPU"
// (egguo-blog reading report), section 2.3: core module 1 (LLM profiler,
// per-neuron activation counts), the variable table (neuron impact
// v_i = f_i, hot neurons = the frequently activated ones), core modules 3-4
// (predictor and neuron-aware operators, launched from here).
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <numeric>
#include <new>

#include "pi_internal.cuh"

namespace {

thread_local char g_err[512] = "";

// the persistent step takes its whole layer table by value
static_assert(sizeof(pi::StackParams) <= 4096, "StackParams must fit the classic 4 KB parameter space");

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// dst[k, 0:cols] = src[perm[k], :] for rows of `cols` halves (cols % 8 == 0),
// dst rows dst_ld halves apart; the dst_ld - cols halves after each row are zeroed.
__global__ void k_permute_rows(const __half *__restrict__ src, __half *__restrict__ dst,
                               const int32_t *__restrict__ perm, int rows, int cols, int dst_ld) {
  const int nv = cols >> 3, nvd = dst_ld >> 3;
  for (int k = blockIdx.x; k < rows; k += gridDim.x) {
    const uint4 *s = reinterpret_cast<const uint4 *>(src + (size_t)perm[k] * cols);
    uint4 *o = reinterpret_cast<uint4 *>(dst + (size_t)k * dst_ld);
    for (int v = threadIdx.x; v < nvd; v += blockDim.x) o[v] = v < nv ? s[v] : make_uint4(0, 0, 0, 0);
  }
}

// dst[k] = src ? src[perm[k]] : 0
// Per-row E4M3 quantisation of W [rows, d] fp16 (the format of
// PI_ROWS_FP8_E4M3): s = max |w| / 448 (1 for an all-zero row), codes of
// w / s rounded to nearest even and saturated, both in binary32.
__global__ void __launch_bounds__(256) k_quantize_rows(const __half *__restrict__ W, uint8_t *__restrict__ Q,
                                                       float *__restrict__ scale, int rows, int d) {
  __shared__ float red[8];
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const __half *w = W + (size_t)r * d;
    float m = 0.f;
    for (int j = threadIdx.x; j < d; j += blockDim.x) m = fmaxf(m, fabsf(__half2float(w[j])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    m = red[0];
    for (int k = 1; k < (int)(blockDim.x >> 5); ++k) m = fmaxf(m, red[k]);
    const float s = m > 0.f ? m / 448.0f : 1.0f;
    for (int j = threadIdx.x; j < d; j += blockDim.x)
      Q[(size_t)r * d + j] = __nv_cvt_float_to_fp8(__half2float(w[j]) / s, __NV_SATFINITE, __NV_E4M3);
    if (threadIdx.x == 0) scale[r] = s;
    __syncthreads();                  // red[] is reused by the next row
  }
}

__global__ void k_permute_vec(const float *__restrict__ src, float *__restrict__ dst,
                              const int32_t *__restrict__ perm, int n) {
  for (int k = blockIdx.x * blockDim.x + threadIdx.x; k < n; k += gridDim.x * blockDim.x)
    dst[k] = src ? src[perm[k]] : 0.f;
}

// W_dT[k, j] = W_down[j, perm[k]]: 32x32 tiles through shared memory.
__global__ void k_transpose_perm(const __half *__restrict__ W_down, __half *__restrict__ W_dT,
                                 const int32_t *__restrict__ perm, int d, int ffn) {
  __shared__ __half tile[32][33];
  const int k0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;   // 32 x 8
  const int k = k0 + tx;
  const int col = k < ffn ? perm[k] : 0;
  for (int jj = ty; jj < 32; jj += 8) {
    const int j = j0 + jj;
    if (j < d && k < ffn) tile[jj][tx] = W_down[(size_t)j * ffn + col];
  }
  __syncthreads();
  for (int kk = ty; kk < 32; kk += 8) {
    const int kr = k0 + kk, j = j0 + tx;
    if (kr < ffn && j < d) W_dT[(size_t)kr * d + j] = tile[tx][kk];
  }
}

// counts[i] += #{t : W[i,:].X[t,:] + bias[i] > 0}.  64 neurons x 64 tokens per
// CTA, 4x4 outputs per thread, K tiles of 32 staged (as fp32) in shared memory.
__global__ void __launch_bounds__(256) k_profile(const __half *__restrict__ W,
                                                 const float *__restrict__ bias,
                                                 const __half *__restrict__ X, int ffn, int d,
                                                 int T, int32_t *__restrict__ counts) {
  __shared__ float As[32][64 + 4];
  __shared__ float Bs[32][64 + 4];
  __shared__ int cnt_s[64];
  const int n0 = blockIdx.x * 64, t0 = blockIdx.y * 64;
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  if (tid < 64) cnt_s[tid] = 0;
  float acc[4][4] = {};
  const int lr = tid >> 2, lk = (tid & 3) * 8;   // loader: row, first k of its vector
  for (int k0 = 0; k0 < d; k0 += 32) {
    const int kk = k0 + lk;
    uint4 av = make_uint4(0, 0, 0, 0), bv = make_uint4(0, 0, 0, 0);
    if (kk < d && n0 + lr < ffn) av = *reinterpret_cast<const uint4 *>(W + (size_t)(n0 + lr) * d + kk);
    if (kk < d && t0 + lr < T) bv = *reinterpret_cast<const uint4 *>(X + (size_t)(t0 + lr) * d + kk);
    const __half *ah = reinterpret_cast<const __half *>(&av);
    const __half *bh = reinterpret_cast<const __half *>(&bv);
    __syncthreads();
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      As[lk + e][lr] = __half2float(ah[e]);
      Bs[lk + e][lr] = __half2float(bh[e]);
    }
    __syncthreads();
#pragma unroll 8
    for (int q = 0; q < 32; ++q) {
      const float4 a = *reinterpret_cast<const float4 *>(&As[q][ty * 4]);
      const float4 b = *reinterpret_cast<const float4 *>(&Bs[q][tx * 4]);
      const float ar[4] = {a.x, a.y, a.z, a.w}, br[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = n0 + ty * 4 + i;
    if (n >= ffn) continue;
    int c = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (t0 + tx * 4 + j < T && acc[i][j] + bias[n] > 0.f) ++c;
    if (c) atomicAdd(&cnt_s[ty * 4 + i], c);
  }
  __syncthreads();
  if (tid < 64 && n0 + tid < ffn && cnt_s[tid]) atomicAdd(&counts[n0 + tid], cnt_s[tid]);
}

pi_status check_desc(const pi_layer_desc *D) {
  if (!D) return pi::fail(PI_ERR_INVALID_ARG, "desc is NULL");
  if (D->act != PI_ACT_RELU && D->act != PI_ACT_REGLU && D->act != PI_ACT_SWIGLU)
    return pi::fail(PI_ERR_INVALID_ARG, "act %d is not PI_ACT_RELU, PI_ACT_REGLU or PI_ACT_SWIGLU", D->act);
  if (D->d < 8 || D->d > PI_MAX_D || D->d % 8)
    return pi::fail(PI_ERR_UNSUPPORTED, "d=%d: need 8 <= d <= %d and d %% 8 == 0", D->d, PI_MAX_D);
  if (D->rank < 8 || D->rank > PI_MAX_RANK || D->rank % 8)
    return pi::fail(PI_ERR_UNSUPPORTED, "rank=%d: need 8 <= rank <= %d and rank %% 8 == 0",
                    D->rank, PI_MAX_RANK);
  if (D->ffn < 1 || D->ffn > PI_MAX_FFN)
    return pi::fail(PI_ERR_UNSUPPORTED, "ffn=%d: need 1 <= ffn <= %d", D->ffn, PI_MAX_FFN);
  if (!D->W_up || !D->b || !D->W_down || !D->W_p1 || !D->W_p2)
    return pi::fail(PI_ERR_INVALID_ARG, "a required weight pointer is NULL");
  if ((D->act != PI_ACT_RELU) != (D->W_gate != nullptr))
    return pi::fail(PI_ERR_INVALID_ARG, "W_gate must be given exactly for a gated act (ReGLU, SwiGLU)");
  if (D->row_format != PI_ROWS_FP16 && D->row_format != PI_ROWS_FP8_E4M3)
    return pi::fail(PI_ERR_INVALID_ARG, "row_format %d is neither PI_ROWS_FP16 nor PI_ROWS_FP8_E4M3",
                    D->row_format);
  const void *h16[] = {D->W_up, D->W_gate, D->W_down, D->W_p1, D->W_p2};
  for (const void *p : h16)
    if (p && !aligned16(p)) return pi::fail(PI_ERR_INVALID_ARG, "fp16 weights must be 16-byte aligned");
  if (!aligned4(D->b) || (D->c_p && !aligned4(D->c_p)))
    return pi::fail(PI_ERR_INVALID_ARG, "fp32 vectors must be 4-byte aligned");
  const void *all[] = {D->W_up, D->W_gate, D->W_down, D->W_p1, D->W_p2, D->b, D->c_p};
  for (const void *p : all) {
    if (!p) continue;
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
      cudaGetLastError();
      return pi::fail(PI_ERR_INVALID_ARG, "pointer %p is not known to CUDA", p);
    }
    if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
      return pi::fail(PI_ERR_INVALID_ARG, "pointer %p is not device or managed memory", p);
  }
  return PI_OK;
}

}  // namespace

namespace pi {

void clear_error() { g_err[0] = 0; }

pi_status fail(pi_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

pi_status cuda_fail(cudaError_t e, const char *what) {
  const pi_status s = (e == cudaErrorMemoryAllocation) ? PI_ERR_OOM : PI_ERR_CUDA;
  snprintf(g_err, sizeof(g_err), "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
  return s;
}

WsLayout ws_layout(const pi_layer *L, int B) {
  WsLayout w;
  size_t off = 0;
  const int nsplit = std::max(fused_splits(L), down_splits(L, B));
  w.h = off;       off += align_up(sizeof(float) * (size_t)B * L->rank);
  w.a = off;       off += align_up(sizeof(float) * (size_t)B * L->ffn);
  w.partial = off; off += align_up(sizeof(float) * (size_t)nsplit * B * L->d);
  w.mask = off;    off += align_up((size_t)std::max(B, kMaxStack) * L->ffn);
  w.idx = off;     off += align_up(sizeof(int32_t) * (size_t)L->ffn);
  w.count = off;   off += align_up(sizeof(int32_t) * 4);
  w.cnt = off;     off += align_up(sizeof(int32_t) * (size_t)step_grid(L));
  w.bar = off;     off += align_up(sizeof(unsigned));
  w.abuf = off;    off += align_up(2 * sizeof(__half) * (size_t)tc_bpad(B) * tc_ffn_pad(L));
  w.hbuf = off;    off += align_up(2 * sizeof(__half) * (size_t)tc_bpad(B) * tc_rank_pad(L));
  w.tcpart = off;  off += B >= 3 ? align_up(tc_piece_bytes(L, B)) : 0;
  w.tcnt = off;    off += B >= 3 ? align_up(sizeof(int32_t) * (size_t)(tc_ffn_pad(L) / 128)) : 0;
  w.total = off;
  return w;
}

cudaError_t record_hook(cudaEvent_t ev, cudaStream_t s) {
  if (!ev) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cudaEventRecordWithFlags(ev, s, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                            : cudaEventRecordDefault);
}

cudaError_t run_profile(const pi_layer_desc *D, const __half *x, int T, int32_t *counts,
                        cudaStream_t s) {
  const __half *W = reinterpret_cast<const __half *>(D->act != PI_ACT_RELU ? D->W_gate : D->W_up);
  const int tiles_t = (T + 63) / 64;
  const int max_y = 65535;
  for (int ty0 = 0; ty0 < tiles_t; ty0 += max_y) {
    const int ny = std::min(max_y, tiles_t - ty0);
    dim3 grid((D->ffn + 63) / 64, ny);
    k_profile<<<grid, 256, 0, s>>>(W, D->b, x + (size_t)ty0 * 64 * D->d, D->ffn, D->d,
                                   T - ty0 * 64, counts);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pi

// ===========================================================================
extern "C" {

const char *pi_last_error(void) { return g_err; }

const char *pi_status_string(pi_status s) {
  switch (s) {
    case PI_OK: return "PI_OK";
    case PI_ERR_INVALID_ARG: return "PI_ERR_INVALID_ARG";
    case PI_ERR_UNSUPPORTED: return "PI_ERR_UNSUPPORTED";
    case PI_ERR_OOM: return "PI_ERR_OOM";
    case PI_ERR_CUDA: return "PI_ERR_CUDA";
    case PI_ERR_DEVICE_CHECK: return "PI_ERR_DEVICE_CHECK";
  }
  return "PI_ERR_UNKNOWN";
}

pi_status pi_layer_create(pi_layer **out, const pi_layer_desc *D, const int32_t *perm,
                          void *stream) {
  g_err[0] = 0;
  if (!out) return pi::fail(PI_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  pi_status st = check_desc(D);
  if (st != PI_OK) return st;
  const int d = D->d, ffn = D->ffn, r = D->rank;
  std::vector<int32_t> p(ffn);
  if (perm) {
    std::vector<char> seen(ffn, 0);
    for (int k = 0; k < ffn; ++k) {
      const int32_t v = perm[k];
      if (v < 0 || v >= ffn || seen[v])
        return pi::fail(PI_ERR_INVALID_ARG, "perm is not a permutation of 0..ffn-1 (entry %d = %d)", k, v);
      seen[v] = 1;
      p[k] = v;
    }
  } else {
    std::iota(p.begin(), p.end(), 0);
  }

  pi_layer *L = new (std::nothrow) pi_layer();
  if (!L) return pi::fail(PI_ERR_OOM, "host allocation failed");
  L->d = d; L->ffn = ffn; L->rank = r; L->act = D->act;
  L->row_format = D->row_format;
  const bool q8 = D->row_format == PI_ROWS_FP8_E4M3;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto bail = [&](pi_status code) {
    if (L->base) cudaFree(L->base);
    delete L;
    return code;
  };
  if (cudaGetDevice(&L->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->device) != cudaSuccess)
    return bail(pi::fail(PI_ERR_CUDA, "no usable CUDA device"));
  // Deal the caller's order round-robin over the G SM slices of the persistent
  // step: the k-th neuron of `p` goes to slice k % G, place k / G within it.
  // Each slice then holds every G-th neuron of a hot-first order, the same mix
  // of hot and cold neurons.
  {
    const int G = pi::step_grid(L), q = ffn / G, rr = ffn % G;
    L->perm.resize(ffn);
    for (int k = 0; k < ffn; ++k) {
      const int c = k % G, j = k / G;
      L->perm[(size_t)c * q + std::min(c, rr) + j] = p[k];
    }
  }

  const size_t wrow = (size_t)ffn * d * sizeof(__half);
  size_t off = 0;
  const size_t o_p1 = off; off += align_up((size_t)r * d * sizeof(__half));
  L->p2_ld = pi::p2_ld_for(r);
  const size_t o_p2 = off; off += align_up((size_t)ffn * L->p2_ld * sizeof(__half));
  // the gathered rows: fp16, or E4M3 codes (1 byte) plus one scale per row
  const size_t rowmat = q8 ? (size_t)ffn * d : wrow;
  const size_t o_up = off; off += align_up(rowmat);
  const bool gated = D->act != PI_ACT_RELU;
  const size_t o_gate = off; if (gated) off += align_up(rowmat);
  const size_t o_dT = off; off += align_up(rowmat);
  const size_t vsc = q8 ? align_up((size_t)ffn * sizeof(float)) : 0;
  const size_t o_sup = off; off += vsc;
  const size_t o_sgate = off; if (gated) off += vsc;
  const size_t o_sdT = off; off += vsc;
  const size_t o_b = off; off += align_up((size_t)ffn * sizeof(float));
  const size_t o_c = off; off += align_up((size_t)ffn * sizeof(float));
  const size_t o_perm = off; off += align_up((size_t)ffn * sizeof(int32_t));
  const size_t o_st = off; off += align_up(sizeof(unsigned int));
  L->bytes = off;

  size_t free_b = 0, total_b = 0;
  if (cudaMemGetInfo(&free_b, &total_b) == cudaSuccess && L->bytes > free_b)
    return bail(pi::fail(PI_ERR_OOM, "layer needs %zu bytes, %zu free", L->bytes, free_b));
  cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&L->base), L->bytes);
  if (e != cudaSuccess) {
    L->base = nullptr;
    cudaGetLastError();
    return bail(pi::cuda_fail(e, "cudaMalloc(layer)"));
  }
  char *b = L->base;
  L->W_p1 = reinterpret_cast<__half *>(b + o_p1);
  L->W_p2 = reinterpret_cast<__half *>(b + o_p2);
  if (!q8) {
    L->W_up = reinterpret_cast<__half *>(b + o_up);
    L->W_gate = gated ? reinterpret_cast<__half *>(b + o_gate) : nullptr;
    L->W_dT = reinterpret_cast<__half *>(b + o_dT);
  } else {
    L->Q_up = reinterpret_cast<uint8_t *>(b + o_up);
    L->Q_gate = gated ? reinterpret_cast<uint8_t *>(b + o_gate) : nullptr;
    L->Q_dT = reinterpret_cast<uint8_t *>(b + o_dT);
    L->s_up = reinterpret_cast<float *>(b + o_sup);
    L->s_gate = gated ? reinterpret_cast<float *>(b + o_sgate) : nullptr;
    L->s_dT = reinterpret_cast<float *>(b + o_sdT);
  }
  L->b = reinterpret_cast<float *>(b + o_b);
  L->c_p = reinterpret_cast<float *>(b + o_c);
  int32_t *perm_dev = reinterpret_cast<int32_t *>(b + o_perm);
  L->status = reinterpret_cast<unsigned int *>(b + o_st);

#define PI_CREATE_CUDA(call)                                  \
  do {                                                        \
    cudaError_t e_ = (call);                                  \
    if (e_ != cudaSuccess) return bail(pi::cuda_fail(e_, #call)); \
  } while (0)

  PI_CREATE_CUDA(cudaMemcpyAsync(perm_dev, L->perm.data(), sizeof(int32_t) * ffn,
                                 cudaMemcpyHostToDevice, s));
  PI_CREATE_CUDA(cudaMemsetAsync(L->status, 0, sizeof(unsigned int), s));
  PI_CREATE_CUDA(cudaMemcpyAsync(L->W_p1, D->W_p1, (size_t)r * d * sizeof(__half),
                                 cudaMemcpyDeviceToDevice, s));
  const int grid_rows = std::min(ffn, 65535);
  k_permute_rows<<<grid_rows, 256, 0, s>>>(reinterpret_cast<const __half *>(D->W_p2), L->W_p2,
                                           perm_dev, ffn, r, L->p2_ld);
  // FP8 layers: each permuted fp16 matrix goes through one temporary buffer
  // and is quantised row by row into the layer
  __half *tmp = nullptr;
  if (q8) {
    e = cudaMalloc(reinterpret_cast<void **>(&tmp), wrow);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return bail(pi::cuda_fail(e, "cudaMalloc(quantisation buffer)"));
    }
  }
  auto fail_tmp = [&](cudaError_t e_, const char *what) {
    if (tmp) {
      cudaStreamSynchronize(s);
      cudaFree(tmp);
    }
    return bail(pi::cuda_fail(e_, what));
  };
  const int grid_q = std::min(ffn, 4 * L->num_sms * 8);
  k_permute_rows<<<grid_rows, 256, 0, s>>>(reinterpret_cast<const __half *>(D->W_up), q8 ? tmp : L->W_up,
                                           perm_dev, ffn, d, d);
  if (q8) k_quantize_rows<<<grid_q, 256, 0, s>>>(tmp, L->Q_up, L->s_up, ffn, d);
  if (gated) {
    k_permute_rows<<<grid_rows, 256, 0, s>>>(reinterpret_cast<const __half *>(D->W_gate), q8 ? tmp : L->W_gate,
                                             perm_dev, ffn, d, d);
    if (q8) k_quantize_rows<<<grid_q, 256, 0, s>>>(tmp, L->Q_gate, L->s_gate, ffn, d);
  }
  k_permute_vec<<<(ffn + 255) / 256, 256, 0, s>>>(D->b, L->b, perm_dev, ffn);
  k_permute_vec<<<(ffn + 255) / 256, 256, 0, s>>>(D->c_p, L->c_p, perm_dev, ffn);
  k_transpose_perm<<<dim3((ffn + 31) / 32, (d + 31) / 32), dim3(32, 8), 0, s>>>(
      reinterpret_cast<const __half *>(D->W_down), q8 ? tmp : L->W_dT, perm_dev, d, ffn);
  if (q8) k_quantize_rows<<<grid_q, 256, 0, s>>>(tmp, L->Q_dT, L->s_dT, ffn, d);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail_tmp(e, "layer copy kernels");
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail_tmp(e, "cudaStreamSynchronize(create)");
  if (tmp) cudaFree(tmp);
#undef PI_CREATE_CUDA
  *out = L;
  return PI_OK;
}

pi_status pi_layer_destroy(pi_layer *L) {
  g_err[0] = 0;
  if (!L) return PI_OK;
  cudaError_t e = cudaDeviceSynchronize();
  cudaError_t f = L->base ? cudaFree(L->base) : cudaSuccess;
  delete L;
  if (e != cudaSuccess) return pi::cuda_fail(e, "cudaDeviceSynchronize");
  if (f != cudaSuccess) return pi::cuda_fail(f, "cudaFree");
  return PI_OK;
}

pi_status pi_layer_info(const pi_layer *L, int32_t *d, int32_t *ffn, int32_t *rank, int32_t *act) {
  if (!L) return pi::fail(PI_ERR_INVALID_ARG, "layer is NULL");
  if (d) *d = L->d;
  if (ffn) *ffn = L->ffn;
  if (rank) *rank = L->rank;
  if (act) *act = L->act;
  return PI_OK;
}

pi_status pi_layer_rows_fp8(const pi_layer *L, int32_t matrix, uint8_t *codes, float *scales,
                            void *stream) {
  g_err[0] = 0;
  if (!L) return pi::fail(PI_ERR_INVALID_ARG, "layer is NULL");
  if (L->row_format != PI_ROWS_FP8_E4M3) return pi::fail(PI_ERR_UNSUPPORTED, "the layer stores fp16 rows");
  if (!codes || !scales) return pi::fail(PI_ERR_INVALID_ARG, "codes and scales must be non-NULL");
  const uint8_t *q = matrix == 0 ? L->Q_up : matrix == 1 ? L->Q_gate : matrix == 2 ? L->Q_dT : nullptr;
  const float *sc = matrix == 0 ? L->s_up : matrix == 1 ? L->s_gate : matrix == 2 ? L->s_dT : nullptr;
  if (!q || !sc) return pi::fail(PI_ERR_INVALID_ARG, "matrix %d: need 0 (up), 1 (gate, ReGLU) or 2 (down)", matrix);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PI_TRY_CUDA(cudaMemcpyAsync(codes, q, (size_t)L->ffn * L->d, cudaMemcpyDeviceToDevice, s));
  PI_TRY_CUDA(cudaMemcpyAsync(scales, sc, sizeof(float) * (size_t)L->ffn, cudaMemcpyDeviceToDevice, s));
  return PI_OK;
}

pi_status pi_layer_perm(const pi_layer *L, int32_t *perm) {
  if (!L || !perm) return pi::fail(PI_ERR_INVALID_ARG, "layer or perm is NULL");
  std::memcpy(perm, L->perm.data(), sizeof(int32_t) * L->ffn);
  return PI_OK;
}

size_t pi_workspace_bytes(const pi_layer *L, int32_t B_max) {
  if (!L || B_max < 1 || B_max > PI_MAX_BATCH) return 0;
  return pi::ws_layout(L, B_max).total;
}

static pi_status check_common(const pi_layer *L, const uint16_t *x, int32_t B, const void *ws,
                              size_t ws_bytes, pi::WsLayout *w) {
  if (!L) return pi::fail(PI_ERR_INVALID_ARG, "layer is NULL");
  if (B < 1 || B > PI_MAX_BATCH)
    return pi::fail(PI_ERR_INVALID_ARG, "B=%d: need 1 <= B <= %d", B, PI_MAX_BATCH);
  if (!x || !aligned16(x)) return pi::fail(PI_ERR_INVALID_ARG, "x must be non-NULL and 16-byte aligned");
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)))
    return pi::fail(PI_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
  *w = pi::ws_layout(L, B);
  if (ws_bytes < w->total)
    return pi::fail(PI_ERR_INVALID_ARG, "workspace of %zu bytes, need %zu for B=%d", ws_bytes,
                    w->total, B);
  return PI_OK;
}

pi_status pi_predict(pi_layer *L, const uint16_t *x, int32_t B, uint8_t *mask, float *logits,
                     void *ws, size_t ws_bytes, void *stream) {
  g_err[0] = 0;
  pi::WsLayout w;
  pi_status st = check_common(L, x, B, ws, ws_bytes, &w);
  if (st != PI_OK) return st;
  if (!mask && !logits) return pi::fail(PI_ERR_INVALID_ARG, "mask and logits are both NULL");
  if (logits && !aligned4(logits)) return pi::fail(PI_ERR_INVALID_ARG, "logits must be 4-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  PI_TRY_CUDA(pi::run_predict(L, reinterpret_cast<const __half *>(x), B, mask, logits,
                              reinterpret_cast<float *>(static_cast<char *>(ws) + w.h), s));
  return PI_OK;
}

pi_status pi_compact_active(const pi_layer *L, const uint8_t *mask, int32_t B, int32_t *idx,
                            int32_t *count, void *stream) {
  g_err[0] = 0;
  if (!L) return pi::fail(PI_ERR_INVALID_ARG, "layer is NULL");
  if (B < 1 || B > PI_MAX_BATCH)
    return pi::fail(PI_ERR_INVALID_ARG, "B=%d: need 1 <= B <= %d", B, PI_MAX_BATCH);
  if (!mask || !idx || !count || !aligned4(idx) || !aligned4(count))
    return pi::fail(PI_ERR_INVALID_ARG, "mask, idx and count must be non-NULL (idx, count 4-byte aligned)");
  PI_TRY_CUDA(pi::run_compact(L, mask, B, idx, count, static_cast<cudaStream_t>(stream)));
  return PI_OK;
}

pi_status pi_sparse_ffn(pi_layer *L, const uint16_t *x, int32_t B, const int32_t *idx,
                        const int32_t *count, float *y, void *ws, size_t ws_bytes, void *stream) {
  g_err[0] = 0;
  pi::WsLayout w;
  pi_status st = check_common(L, x, B, ws, ws_bytes, &w);
  if (st != PI_OK) return st;
  if (!idx || !count || !aligned4(idx) || !aligned4(count))
    return pi::fail(PI_ERR_INVALID_ARG, "idx and count must be non-NULL and 4-byte aligned");
  if (!y || !aligned16(y)) return pi::fail(PI_ERR_INVALID_ARG, "y must be non-NULL and 16-byte aligned");
  PI_TRY_CUDA(pi::run_sparse_ffn(L, reinterpret_cast<const __half *>(x), B, idx, count, 0, y, w,
                                 static_cast<char *>(ws), static_cast<cudaStream_t>(stream)));
  return PI_OK;
}

pi_status pi_ffn_dense_ref(pi_layer *L, const uint16_t *x, int32_t B, float *y, void *ws,
                           size_t ws_bytes, void *stream) {
  g_err[0] = 0;
  pi::WsLayout w;
  pi_status st = check_common(L, x, B, ws, ws_bytes, &w);
  if (st != PI_OK) return st;
  if (!y || !aligned16(y)) return pi::fail(PI_ERR_INVALID_ARG, "y must be non-NULL and 16-byte aligned");
  PI_TRY_CUDA(pi::run_sparse_ffn(L, reinterpret_cast<const __half *>(x), B, nullptr, nullptr,
                                 L->ffn, y, w, static_cast<char *>(ws),
                                 static_cast<cudaStream_t>(stream)));
  return PI_OK;
}

pi_status pi_layer_forward(pi_layer *L, const uint16_t *x, int32_t B, int32_t *idx,
                           int32_t *count, float *y, void *ws, size_t ws_bytes, void *stream) {
  g_err[0] = 0;
  pi::WsLayout w;
  pi_status st = check_common(L, x, B, ws, ws_bytes, &w);
  if (st != PI_OK) return st;
  if (!idx || !count || !aligned4(idx) || !aligned4(count))
    return pi::fail(PI_ERR_INVALID_ARG, "idx and count must be non-NULL and 4-byte aligned");
  if (!y || !aligned16(y)) return pi::fail(PI_ERR_INVALID_ARG, "y must be non-NULL and 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *wsb = static_cast<char *>(ws);
  const __half *xh = reinterpret_cast<const __half *>(x);
  if (B <= 2) {
    PI_TRY_CUDA(pi::run_stack(&L, 1, xh, B, idx, count, y, w, wsb, s));
    return PI_OK;
  }
  uint8_t *mask = reinterpret_cast<uint8_t *>(wsb + w.mask);
  if (pi::pbatch_supported(L, B)) {
    PI_TRY_CUDA(pi::run_predict_batch(L, xh, B, mask, reinterpret_cast<__half *>(wsb + w.hbuf),
                                       reinterpret_cast<float *>(wsb + w.tcpart),
                                       reinterpret_cast<int32_t *>(wsb + w.cnt),
                                       reinterpret_cast<unsigned *>(wsb + w.bar), idx, count, s));
  } else if (pi::tc_predict_supported(L, B)) {
    PI_TRY_CUDA(pi::run_predict_tc(L, xh, B, mask, reinterpret_cast<__half *>(wsb + w.hbuf),
                                    reinterpret_cast<float *>(wsb + w.tcpart),
                                    reinterpret_cast<int32_t *>(wsb + w.tcnt), idx, count, s));
  } else {
    PI_TRY_CUDA(pi::run_predict(L, xh, B, mask, nullptr, reinterpret_cast<float *>(wsb + w.h), s, true));
    PI_TRY_CUDA(pi::run_compact(L, mask, 1, idx, count, s));
  }
  PI_TRY_CUDA(pi::run_sparse_ffn(L, xh, B, idx, count, 0, y, w, wsb, s));
  return PI_OK;
}

}  // extern "C"

namespace {

// Chained input of the next layer: x[t] = fp16(y[t] / RMS(y[t])) with
// RMS(v) = sqrt(mean(v^2) + 1e-12), binary32, one CTA per token.
__global__ void __launch_bounds__(256) k_chain_x(const float *__restrict__ y, __half *__restrict__ x, int d) {
  __shared__ float red[8];
  const float *yt = y + (size_t)blockIdx.x * d;
  float s = 0.f;
  for (int j = threadIdx.x; j < d; j += 256) s = fmaf(yt[j], yt[j], s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < 8; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / (float)d + 1e-12f);
  for (int j = threadIdx.x; j < d; j += 256) x[(size_t)blockIdx.x * d + j] = __float2half_rn(yt[j] * inv);
}

pi_status stack_forward_impl(pi_layer *const *layers, int32_t n_layers, uint16_t *x_mut,
                             const uint16_t *x, int32_t B, int32_t *idx, int32_t *count, float *y,
                             void *ws, size_t ws_bytes, void *stream, bool chained) {
  if (!layers || n_layers < 1) return pi::fail(PI_ERR_INVALID_ARG, "layers is NULL or n_layers < 1");
  for (int l = 0; l < n_layers; ++l) {
    const pi_layer *Ll = layers[l];
    if (!Ll) return pi::fail(PI_ERR_INVALID_ARG, "layers[%d] is NULL", l);
    if (Ll->d != layers[0]->d || Ll->ffn != layers[0]->ffn || Ll->rank != layers[0]->rank ||
        Ll->act != layers[0]->act || Ll->device != layers[0]->device ||
        Ll->row_format != layers[0]->row_format)
      return pi::fail(PI_ERR_INVALID_ARG, "layers[%d] differs in shape, activation, row format or device", l);
  }
  pi_layer *L = layers[0];
  pi::WsLayout w;
  pi_status st = check_common(L, x, B, ws, ws_bytes, &w);
  if (st != PI_OK) return st;
  if (!y || !aligned16(y)) return pi::fail(PI_ERR_INVALID_ARG, "y must be non-NULL and 16-byte aligned");
  if ((idx && !aligned4(idx)) || (count && !aligned4(count)))
    return pi::fail(PI_ERR_INVALID_ARG, "idx and count must be 4-byte aligned");
  if (idx && !count) return pi::fail(PI_ERR_INVALID_ARG, "an idx output needs a count output");
  if (B > 2 && (!idx || !count))
    return pi::fail(PI_ERR_INVALID_ARG, "B > 2 needs idx and count buffers");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char *wsb = static_cast<char *>(ws);
  const __half *xh = reinterpret_cast<const __half *>(x);
  __half *xm = reinterpret_cast<__half *>(x_mut);
  const size_t xs = (size_t)B * L->d;
  if (B <= 2) {
    for (int l0 = 0; l0 < n_layers; l0 += pi::kMaxStack) {
      const int n = std::min(pi::kMaxStack, n_layers - l0);
      __half *x_next = chained && l0 + n < n_layers ? xm + (l0 + n) * xs : nullptr;
      PI_TRY_CUDA(pi::run_stack(layers + l0, n, xh + l0 * xs, B, idx ? idx + (size_t)l0 * L->ffn : nullptr,
                                count ? count + l0 : nullptr, y + l0 * xs, w, wsb, s, chained,
                                chained ? xm + l0 * xs : nullptr, x_next));
    }
    return PI_OK;
  }

  for (int l = 0; l < n_layers; ++l) {
    pi_layer *Ll = layers[l];
    uint8_t *mask = reinterpret_cast<uint8_t *>(wsb + w.mask);
    if (pi::pbatch_supported(Ll, B)) {
      PI_TRY_CUDA(pi::run_predict_batch(Ll, xh + l * xs, B, mask, reinterpret_cast<__half *>(wsb + w.hbuf),
                                         reinterpret_cast<float *>(wsb + w.tcpart),
                                         reinterpret_cast<int32_t *>(wsb + w.cnt),
                                         reinterpret_cast<unsigned *>(wsb + w.bar), idx + (size_t)l * L->ffn,
                                         count + l, s));
    } else if (pi::tc_predict_supported(Ll, B)) {
      PI_TRY_CUDA(pi::run_predict_tc(Ll, xh + l * xs, B, mask, reinterpret_cast<__half *>(wsb + w.hbuf),
                                      reinterpret_cast<float *>(wsb + w.tcpart),
                                      reinterpret_cast<int32_t *>(wsb + w.tcnt), idx + (size_t)l * L->ffn,
                                      count + l, s));
    } else {
      PI_TRY_CUDA(pi::run_predict(Ll, xh + l * xs, B, mask, nullptr, reinterpret_cast<float *>(wsb + w.h), s, true));
      PI_TRY_CUDA(pi::run_compact(Ll, mask, 1, idx + (size_t)l * L->ffn, count + l, s));
    }
    PI_TRY_CUDA(pi::run_sparse_ffn(Ll, xh + l * xs, B, idx + (size_t)l * L->ffn, count + l, 0,
                                   y + l * xs, w, wsb, s));
    if (chained && l + 1 < n_layers) {
      k_chain_x<<<B, 256, 0, s>>>(y + l * xs, xm + (l + 1) * xs, L->d);
      PI_TRY_CUDA(cudaGetLastError());
    }
  }
  return PI_OK;
}

}  // namespace

extern "C" {

pi_status pi_stack_forward(pi_layer *const *layers, int32_t n_layers, const uint16_t *x,
                           int32_t B, int32_t *idx, int32_t *count, float *y, void *ws,
                           size_t ws_bytes, void *stream) {
  g_err[0] = 0;
  return stack_forward_impl(layers, n_layers, nullptr, x, B, idx, count, y, ws, ws_bytes, stream,
                            false);
}

pi_status pi_stack_forward_chained(pi_layer *const *layers, int32_t n_layers, uint16_t *x,
                                   int32_t B, int32_t *idx, int32_t *count, float *y, void *ws,
                                   size_t ws_bytes, void *stream) {
  g_err[0] = 0;
  return stack_forward_impl(layers, n_layers, x, x, B, idx, count, y, ws, ws_bytes, stream, true);
}

pi_status pi_stack_forward_host(pi_layer *const *layers, int32_t n_layers, int32_t T,
                                const uint16_t *x_host, int32_t B, float *y_host, uint16_t *x_dev,
                                float *y_dev, int32_t *idx, int32_t *count, int32_t chained,
                                void *ws, size_t ws_bytes, void *stream) {
  g_err[0] = 0;
  if (T < 1) return pi::fail(PI_ERR_INVALID_ARG, "T=%d: need at least one token", T);
  if (!x_host || !y_host) return pi::fail(PI_ERR_INVALID_ARG, "x_host and y_host must be non-NULL");
  if (!layers || n_layers < 1 || !layers[0]) return pi::fail(PI_ERR_INVALID_ARG, "layers is NULL or n_layers < 1");
  if (B < 1 || B > PI_MAX_BATCH) return pi::fail(PI_ERR_INVALID_ARG, "B=%d: need 1 <= B <= %d", B, PI_MAX_BATCH);
  if (!x_dev || !aligned16(x_dev) || !y_dev || !aligned16(y_dev))
    return pi::fail(PI_ERR_INVALID_ARG, "x_dev and y_dev must be non-NULL and 16-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t per_tok = (size_t)n_layers * B * layers[0]->d;     // elements of one token's x or y
  PI_TRY_CUDA(cudaMemcpyAsync(x_dev, x_host, sizeof(uint16_t) * per_tok * T, cudaMemcpyHostToDevice, s));
  for (int t = 0; t < T; ++t) {
    uint16_t *xt = x_dev + per_tok * t;
    const pi_status st = stack_forward_impl(layers, n_layers, xt, xt, B, idx, count ? count + (size_t)t * n_layers : nullptr,
                                            y_dev + per_tok * t, ws, ws_bytes, stream, chained != 0);
    if (st != PI_OK) return st;
  }
  PI_TRY_CUDA(cudaMemcpyAsync(y_host, y_dev, sizeof(float) * per_tok * T, cudaMemcpyDeviceToHost, s));
  return PI_OK;
}

pi_status pi_profile_activations(const pi_layer_desc *D, const uint16_t *x, int32_t T,
                                 int32_t *counts, void *stream) {
  g_err[0] = 0;
  pi_status st = check_desc(D);
  if (st != PI_OK) return st;
  if (T < 0) return pi::fail(PI_ERR_INVALID_ARG, "T=%d is negative", T);
  if (T == 0) return PI_OK;
  if (!x || !aligned16(x) || !counts || !aligned4(counts))
    return pi::fail(PI_ERR_INVALID_ARG, "x (16-byte aligned) and counts must be non-NULL");
  PI_TRY_CUDA(pi::run_profile(D, reinterpret_cast<const __half *>(x), T, counts,
                              static_cast<cudaStream_t>(stream)));
  return PI_OK;
}

pi_status pi_hot_first_perm(const int32_t *counts, int32_t ffn, int32_t *perm) {
  g_err[0] = 0;
  if (!counts || !perm || ffn < 1) return pi::fail(PI_ERR_INVALID_ARG, "bad counts/perm/ffn");
  std::vector<int32_t> p(ffn);
  std::iota(p.begin(), p.end(), 0);
  std::stable_sort(p.begin(), p.end(), [&](int32_t a, int32_t b) { return counts[a] > counts[b]; });
  std::memcpy(perm, p.data(), sizeof(int32_t) * ffn);
  return PI_OK;
}

pi_status pi_layer_set_timing_events(pi_layer *L, void *ev_before, void *ev_after) {
  g_err[0] = 0;
  if (!L) return pi::fail(PI_ERR_INVALID_ARG, "layer is NULL");
  if ((ev_before == nullptr) != (ev_after == nullptr))
    return pi::fail(PI_ERR_INVALID_ARG, "set both events or neither");
  L->ev_before = static_cast<cudaEvent_t>(ev_before);
  L->ev_after = static_cast<cudaEvent_t>(ev_after);
  return PI_OK;
}

pi_status pi_layer_set_hot_count(pi_layer *L, int32_t n_hot) {
  g_err[0] = 0;
  if (!L) return pi::fail(PI_ERR_INVALID_ARG, "layer is NULL");
  if (n_hot < 0 || n_hot > L->ffn) return pi::fail(PI_ERR_INVALID_ARG, "n_hot=%d outside [0, ffn]", n_hot);
  L->n_hot = n_hot;
  return PI_OK;
}

int32_t pi_forward_launches(const pi_layer *L, int32_t B) {
  if (!L || B < 1 || B > PI_MAX_BATCH) return 0;
  // B <= 2: the persistent step and the ordered compaction of its masks
  // (memsets not counted).  Otherwise the predictor, then the FFN.  The
  // predictor: one cooperative launch (B <= 32, pi_pbatch.cu); else on the
  // tensor cores hidden layer and logits (each with its split-tile fix-up)
  // and tile compaction; else predict_h, predict_l, compact.  The FFN on the
  // tensor cores: up (+ fix-up), down, column reduce; else up, down, reduce.
  if (B <= 2) return 2;
  const int pred = pi::pbatch_supported(L, B) ? 1 : (pi::tc_predict_supported(L, B) ? 5 : 3);
  return pred + (pi::tc_supported(L, B) ? 4 : 3);
}

pi_status pi_device_status(pi_layer *L, void *stream) {
  g_err[0] = 0;
  if (!L) return pi::fail(PI_ERR_INVALID_ARG, "layer is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  PI_TRY_CUDA(cudaStreamSynchronize(s));
  PI_TRY_CUDA(cudaMemcpy(&v, L->status, sizeof(v), cudaMemcpyDeviceToHost));
  if (v) {
    PI_TRY_CUDA(cudaMemset(L->status, 0, sizeof(v)));
    return pi::fail(PI_ERR_DEVICE_CHECK, "device check failed:%s%s%s",
                    (v & PI_STATUS_BAD_INDEX) ? " index out of range" : "",
                    (v & PI_STATUS_BAD_COUNT) ? " count out of range" : "",
                    (v & PI_STATUS_BARRIER_TIMEOUT) ? " grid barrier timed out" : "");
  }
  return PI_OK;
}

}  // extern "C"
