// Neuron-aware sparse FFN over a list of active neurons.
//
// "PowerInfer: Fast Large Language Model Serving with a Consumer-grade GPU"
// (egguo-blog reading report), section 2.3, core module 4: the operators
// work directly on individual neurons, reading only the weight rows of the
// neurons the predictor selected, with no conversion to a sparse format.
// For each listed neuron i:  ReLU  a_i = max(0, W_up_i.x + b_i)
//                            ReGLU a_i = max(0, W_gate_i.x + b_i) * (W_up_i.x)
// and y = sum_i a_i W_down^T_i.
//
// Work split: the active list is cut into one contiguous chunk per CTA, each
// CTA forms a partial y over its chunk, and k_reduce adds the partials in a
// fixed order (deterministic, no floating-point atomics).  Every weight row
// is 2d contiguous bytes, read once with 16-byte loads; the fused kernel first
// asks L2 to stream in the rows of the next window of neurons with bulk
// prefetches so that the HBM stream never waits on the arithmetic.
#include "pi_internal.cuh"

namespace {

constexpr int kBT = 8;

// ---------------------------------------------------------------------------
// Fused up+down for batches of 1 or 2 tokens.  Thread t owns 16-byte column
// vectors v = t + c*blockDim (c < CPT) of every row: for the up rows it forms
// partial dot products, for the down rows partial outputs.  The CTA walks its
// chunk in windows of `sub` neurons (<= kWinMax); the rows of the next window
// are bulk-prefetched into L2 while the current one is consumed, and inside a
// window rows are loaded in groups of G so every load of a group is in flight
// before any arithmetic uses it.
// ---------------------------------------------------------------------------
constexpr int kWinMax = 32;

template <int CPT, bool REGLU>
struct FusedShape {
  static constexpr int loads = CPT == 1 ? 16 : 8;              // 16-byte loads in flight per thread
  static constexpr int G = loads / (CPT * (REGLU ? 2 : 1)) > 0 ? loads / (CPT * (REGLU ? 2 : 1)) : 1;
};

template <int CPT, int NB, bool REGLU>
__global__ void __launch_bounds__(512) k_fused_small(
    const __half *__restrict__ W_up, const __half *__restrict__ W_gate,
    const float *__restrict__ bias, const __half *__restrict__ W_dT,
    const __half *__restrict__ x, int d, int ffn, const int32_t *__restrict__ idx,
    const int32_t *__restrict__ count_p, int count_const, int sub,
    float *__restrict__ partial, unsigned int *status, int silu) {
  constexpr int G = FusedShape<CPT, REGLU>::G;
  constexpr int NR = REGLU ? 2 : 1;
  __shared__ float red_s[16][NB][NR][kWinMax];
  __shared__ float a_s[NB][kWinMax];
  __shared__ int i_s[2][kWinMax];

  pidev::griddep_wait();
  pidev::griddep_launch();

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int nthr = blockDim.x, nwarps = nthr >> 5;
  const int nv = d >> 3;
  const int count = pidev::load_count(count_p, count_const, ffn, status);
  const int nsplit = gridDim.x;
  const int chunk = (count + nsplit - 1) / nsplit;
  const int k0 = min(count, blockIdx.x * chunk);
  const int k1 = min(count, k0 + chunk);
  const uint32_t row_bytes = (uint32_t)d * 2u;

  // token vectors this thread needs, kept in registers
  uint4 xr[NB][CPT];
#pragma unroll
  for (int t = 0; t < NB; ++t)
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int v = tid + c * nthr;
      xr[t][c] = v < nv ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)t * d) + v)
                        : make_uint4(0, 0, 0, 0);
    }

  float acc[NB][CPT][8];
#pragma unroll
  for (int t = 0; t < NB; ++t)
#pragma unroll
    for (int c = 0; c < CPT; ++c)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[t][c][e] = 0.f;

  auto prefetch_window = [&](int s0, int buf) {
    const int s1 = min(k1, s0 + sub);
    for (int k = s0 + tid; k < s1; k += nthr) {
      int i = idx ? idx[k] : k;
      if (i < 0 || i >= ffn) {
        atomicOr(status, PI_STATUS_BAD_INDEX);
        i = -1;
      }
      i_s[buf][k - s0] = i;
      if (i >= 0) {
        pidev::prefetch_l2_bulk(W_up + (size_t)i * d, row_bytes);
        if (REGLU) pidev::prefetch_l2_bulk(W_gate + (size_t)i * d, row_bytes);
        pidev::prefetch_l2_bulk(W_dT + (size_t)i * d, row_bytes);
      }
    }
  };

  if (k0 < k1) prefetch_window(k0, 0);
  __syncthreads();

  int buf = 0;
  for (int s0 = k0; s0 < k1; s0 += sub, buf ^= 1) {
    const int n_here = min(sub, k1 - s0);
    if (s0 + sub < k1) prefetch_window(s0 + sub, buf ^ 1);

    // phase 1: dot products of the window's up (and gate) rows with x
    for (int g0 = 0; g0 < n_here; g0 += G) {
      uint4 w[G][NR][CPT];
#pragma unroll
      for (int n = 0; n < G; ++n) {
        const int i = g0 + n < n_here ? i_s[buf][g0 + n] : -1;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          const int v = tid + c * nthr;
          const bool ok = i >= 0 && v < nv;
          w[n][0][c] = ok ? pidev::ld_stream(reinterpret_cast<const uint4 *>(W_up + (size_t)i * d) + v)
                          : make_uint4(0, 0, 0, 0);
          if (REGLU)
            w[n][NR - 1][c] = ok ? pidev::ld_stream(reinterpret_cast<const uint4 *>(W_gate + (size_t)i * d) + v)
                                 : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int n = 0; n < G; ++n)
#pragma unroll
        for (int q = 0; q < NR; ++q)
#pragma unroll
          for (int t = 0; t < NB; ++t) {
            float p = 0.f;
#pragma unroll
            for (int c = 0; c < CPT; ++c) p = pidev::dot8(p, w[n][q][c], xr[t][c]);
            p = pidev::warp_sum(p);
            if (lane == 0 && g0 + n < n_here) red_s[wid][t][q][g0 + n] = p;
          }
    }
    __syncthreads();
    for (int e = tid; e < NB * n_here; e += nthr) {
      const int t = e / n_here, n = e % n_here;
      const int i = i_s[buf][n];
      float a = 0.f;
      if (i >= 0) {
        float su = 0.f, sg = 0.f;
        for (int q = 0; q < nwarps; ++q) {   // fixed order over warps
          su += red_s[q][t][0][n];
          if (REGLU) sg += red_s[q][t][NR - 1][n];
        }
        if (REGLU) {
          const float gz = sg + bias[i];
          a = pidev::gate_act(gz, silu != 0) * su;
        } else {
          const float z = su + bias[i];
          a = z > 0.f ? z : 0.f;
        }
      }
      a_s[t][n] = a;
    }
    __syncthreads();

    // phase 2: accumulate the window's down rows, scaled by a
    constexpr int G2 = FusedShape<CPT, false>::G;
    for (int g0 = 0; g0 < n_here; g0 += G2) {
      uint4 w[G2][CPT];
#pragma unroll
      for (int n = 0; n < G2; ++n) {
        const int i = g0 + n < n_here ? i_s[buf][g0 + n] : -1;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          const int v = tid + c * nthr;
          w[n][c] = (i >= 0 && v < nv)
                        ? pidev::ld_stream(reinterpret_cast<const uint4 *>(W_dT + (size_t)i * d) + v)
                        : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int n = 0; n < G2; ++n) {
        if (g0 + n < n_here) {
#pragma unroll
          for (int t = 0; t < NB; ++t) {
            const float an = a_s[t][g0 + n];
#pragma unroll
            for (int c = 0; c < CPT; ++c) pidev::axpy8(acc[t][c], an, w[n][c]);
          }
        }
      }
    }
    __syncthreads();   // i_s / a_s / red_s of this window are reused later
  }

  // partial[split, t, :]
#pragma unroll
  for (int t = 0; t < NB; ++t)
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int v = tid + c * nthr;
      if (v < nv) {
        float4 *dst = reinterpret_cast<float4 *>(partial + ((size_t)blockIdx.x * NB + t) * d) + 2 * v;
        dst[0] = make_float4(acc[t][c][0], acc[t][c][1], acc[t][c][2], acc[t][c][3]);
        dst[1] = make_float4(acc[t][c][4], acc[t][c][5], acc[t][c][6], acc[t][c][7]);
      }
    }
}

// ---------------------------------------------------------------------------
// Generic batch: up kernel writes a[b, k] (by list position), down kernel
// forms split partials over (chunk of the list) x (2048-column block).
// ---------------------------------------------------------------------------
// FP8: the rows are E4M3 codes (d bytes each, 8 codes per 8-byte load) and
// a dot product is multiplied by its row's scale before the bias.
template <bool REGLU, bool FP8>
__global__ void __launch_bounds__(256) k_sparse_up(
    const void *__restrict__ R_up, const void *__restrict__ R_gate, const float *__restrict__ sc_up,
    const float *__restrict__ sc_gate, const float *__restrict__ bias, const __half *__restrict__ x, int B,
    int d, int ffn, const int32_t *__restrict__ idx, const int32_t *__restrict__ count_p, int count_const,
    float *__restrict__ a, unsigned int *status, int silu) {
  pidev::griddep_wait();
  pidev::griddep_launch();
  const int lane = threadIdx.x & 31;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int count = pidev::load_count(count_p, count_const, ffn, status);
  const int nv = d >> 3;
  for (int k = gw; k < count; k += nw) {
    const int i = idx ? idx[k] : k;
    const bool ok = i >= 0 && i < ffn;
    if (!ok && lane == 0) atomicOr(status, PI_STATUS_BAD_INDEX);
    for (int b0 = 0; b0 < B; b0 += kBT) {
      const int nb = min(kBT, B - b0);
      float su[kBT], sg[kBT];
#pragma unroll
      for (int t = 0; t < kBT; ++t) su[t] = sg[t] = 0.f;
      if (ok) {
        const size_t rb = FP8 ? (size_t)d : (size_t)d * 2;     // bytes per row
        const char *ru = static_cast<const char *>(R_up) + (size_t)i * rb;
        const char *rg = static_cast<const char *>(R_gate) + (size_t)(REGLU ? i : 0) * rb;
#pragma unroll 2
        for (int v = lane; v < nv; v += 32) {
          uint4 wu = make_uint4(0, 0, 0, 0), wg = make_uint4(0, 0, 0, 0);
          uint2 qu = make_uint2(0, 0), qg = make_uint2(0, 0);
          if (FP8) {
            qu = pidev::ld_stream2(reinterpret_cast<const uint2 *>(ru) + v);
            if (REGLU) qg = pidev::ld_stream2(reinterpret_cast<const uint2 *>(rg) + v);
          } else {
            wu = pidev::ld_stream(reinterpret_cast<const uint4 *>(ru) + v);
            if (REGLU) wg = pidev::ld_stream(reinterpret_cast<const uint4 *>(rg) + v);
          }
#pragma unroll
          for (int t = 0; t < kBT; ++t) {
            if (t < nb) {
              const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(b0 + t) * d) + v);
              if (FP8) {
                su[t] = pidev::dot8_e4m3(su[t], qu, xv);
                if (REGLU) sg[t] = pidev::dot8_e4m3(sg[t], qg, xv);
              } else {
                su[t] = pidev::dot8(su[t], wu, xv);
                if (REGLU) sg[t] = pidev::dot8(sg[t], wg, xv);
              }
            }
          }
        }
      }
      const float scu = (FP8 && ok) ? sc_up[i] : 1.f;
      const float scg = (FP8 && REGLU && ok) ? sc_gate[i] : 1.f;
#pragma unroll
      for (int t = 0; t < kBT; ++t) {
        const float u = pidev::warp_sum(su[t]) * scu;
        const float g = REGLU ? pidev::warp_sum(sg[t]) * scg : 0.f;
        if (lane == 0 && t < nb) {
          float av = 0.f;
          if (ok) {
            if (REGLU) {
              const float gz = g + bias[i];
              av = pidev::gate_act(gz, silu != 0) * u;
            } else {
              const float z = u + bias[i];
              av = z > 0.f ? z : 0.f;
            }
          }
          a[(size_t)(b0 + t) * ffn + k] = av;
        }
      }
    }
  }
}

template <bool FP8>
__global__ void __launch_bounds__(256) k_sparse_down(
    const void *__restrict__ R_dT, const float *__restrict__ sc_dT, const float *__restrict__ a, int B, int d,
    int ffn, const int32_t *__restrict__ idx, const int32_t *__restrict__ count_p, int count_const,
    float *__restrict__ partial, unsigned int *status) {
  pidev::griddep_wait();
  pidev::griddep_launch();
  const int count = pidev::load_count(count_p, count_const, ffn, status);
  const int nsplit = gridDim.x;
  const int chunk = (count + nsplit - 1) / nsplit;
  const int k0 = min(count, blockIdx.x * chunk);
  const int k1 = min(count, k0 + chunk);
  const int v = blockIdx.y * blockDim.x + threadIdx.x;   // 16-byte column vector
  const bool active = v < (d >> 3);
  for (int b0 = 0; b0 < B; b0 += kBT) {
    const int nb = min(kBT, B - b0);
    float acc[kBT][8];
#pragma unroll
    for (int t = 0; t < kBT; ++t)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[t][e] = 0.f;
    if (active) {
#pragma unroll 2
      for (int k = k0; k < k1; ++k) {
        const int i = idx ? idx[k] : k;
        if (i < 0 || i >= ffn) continue;   // flagged by the up kernel
        if (FP8) {
          const uint2 q = pidev::ld_stream2(
              reinterpret_cast<const uint2 *>(static_cast<const uint8_t *>(R_dT) + (size_t)i * d) + v);
          const float sc = sc_dT[i];
#pragma unroll
          for (int t = 0; t < kBT; ++t)
            if (t < nb) pidev::axpy8_e4m3(acc[t], a[(size_t)(b0 + t) * ffn + k] * sc, q);
        } else {
          const uint4 w = pidev::ld_stream(
              reinterpret_cast<const uint4 *>(static_cast<const __half *>(R_dT) + (size_t)i * d) + v);
#pragma unroll
          for (int t = 0; t < kBT; ++t)
            if (t < nb) pidev::axpy8(acc[t], a[(size_t)(b0 + t) * ffn + k], w);
        }
      }
      for (int t = 0; t < nb; ++t) {
        float4 *dst = reinterpret_cast<float4 *>(partial + ((size_t)blockIdx.x * B + b0 + t) * d) + 2 * v;
        dst[0] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
        dst[1] = make_float4(acc[t][4], acc[t][5], acc[t][6], acc[t][7]);
      }
    }
  }
}

// y[e] = sum over splits s = 0..nsplit-1 of partial[s][e], e < n (float4
// granularity).  Thread (g, col): g = 16 split groups, col = 16 float4 columns;
// group g sums splits g, g+16, ... in order, then the 16 group sums are added
// in order g = 0..15.  The order depends only on nsplit: deterministic.
__global__ void __launch_bounds__(256) k_reduce(const float *__restrict__ partial, int nsplit,
                                                int n4, float *__restrict__ y) {
  __shared__ float4 part_s[16][16];
  pidev::griddep_wait();
  pidev::griddep_launch();
  const int col = threadIdx.x & 15, g = threadIdx.x >> 4;
  const int e4 = blockIdx.x * 16 + col;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  if (e4 < n4) {
    const float4 *p = reinterpret_cast<const float4 *>(partial);
#pragma unroll 4
    for (int sp = g; sp < nsplit; sp += 16) {
      const float4 v = p[(size_t)sp * n4 + e4];
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
  }
  part_s[g][col] = s;
  __syncthreads();
  if (g == 0 && e4 < n4) {
    float4 t = part_s[0][col];
    for (int q = 1; q < 16; ++q) {
      const float4 v = part_s[q][col];
      t.x += v.x; t.y += v.y; t.z += v.z; t.w += v.w;
    }
    reinterpret_cast<float4 *>(y)[e4] = t;
  }
}

int fused_threads(int d) {
  int t = d / 8;
  t = (t + 31) / 32 * 32;
  if (t < 128) t = 128;
  if (t > 512) t = 512;
  return t;
}

template <int CPT, int NB, bool REGLU>
cudaError_t launch_fused(const pi_layer *L, const __half *x, const int32_t *idx,
                         const int32_t *count, int count_const, float *partial, cudaStream_t s) {
  const int threads = fused_threads(L->d);
  const int nsplit = pi::fused_splits(L);
  // window: about 192 KB of rows per CTA, at most kWinMax neurons
  const int rows_per_neuron = REGLU ? 3 : 2;
  int sub = (192 * 1024) / (2 * L->d * rows_per_neuron);
  if (sub > kWinMax) sub = kWinMax;
  if (sub < 1) sub = 1;
  return pi::launch_pdl(k_fused_small<CPT, NB, REGLU>, dim3(nsplit), dim3(threads), 0, s,
                        L->W_up, L->W_gate, L->b, L->W_dT, x, L->d, L->ffn, idx, count,
                        count_const, sub, partial, L->status, L->act == PI_ACT_SWIGLU ? 1 : 0);
}

template <int NB, bool REGLU>
cudaError_t dispatch_fused(const pi_layer *L, const __half *x, const int32_t *idx,
                           const int32_t *count, int count_const, float *partial, cudaStream_t s) {
  const int threads = fused_threads(L->d);
  const int cpt = (L->d / 8 + threads - 1) / threads;
  switch (cpt) {
    case 1: return launch_fused<1, NB, REGLU>(L, x, idx, count, count_const, partial, s);
    case 2: return launch_fused<2, NB, REGLU>(L, x, idx, count, count_const, partial, s);
    case 3: return launch_fused<3, NB, REGLU>(L, x, idx, count, count_const, partial, s);
    case 4: return launch_fused<4, NB, REGLU>(L, x, idx, count, count_const, partial, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

namespace pi {

int fused_splits(const pi_layer *L) {
  const int threads = fused_threads(L->d);
  return L->num_sms * (512 / threads > 4 ? 4 : 512 / threads);
}

int down_colblocks(const pi_layer *L) { return (L->d / 8 + 255) / 256; }

int down_splits(const pi_layer *L, int B) {
  (void)B;
  int n = (2 * L->num_sms) / down_colblocks(L);
  return n < 1 ? 1 : n;
}

cudaError_t run_reduce(const float *partial, int nsplit, int n, float *y, cudaStream_t s) {
  const int n4 = n / 4;
  return launch_pdl(k_reduce, dim3((n4 + 15) / 16), dim3(256), 0, s, partial, nsplit, n4, y);
}

cudaError_t run_sparse_ffn(const pi_layer *L, const __half *x, int B, const int32_t *idx,
                           const int32_t *count, int count_const, float *y, const WsLayout &w,
                           char *ws, cudaStream_t s) {
  // E4M3 rows: the tensor-core path converts the codes in shared memory; the
  // generic kernels take them below 3 tokens (the decode step has its own
  // E4M3 path) and for shapes off the tensor cores
  const bool q8 = L->row_format == PI_ROWS_FP8_E4M3;
  if (B > 2 && tc_supported(L, B)) return run_sparse_ffn_tc(L, x, B, idx, count, count_const, y, w, ws, s);
  float *partial = reinterpret_cast<float *>(ws + w.partial);
  const bool reglu = L->act != PI_ACT_RELU;      // gated: ReGLU or SwiGLU
  const int silu = L->act == PI_ACT_SWIGLU ? 1 : 0;
  cudaError_t e;
  int nsplit;
  if (B <= 2 && !q8) {
    nsplit = fused_splits(L);
    e = record_hook(L->ev_before, s);
    if (e != cudaSuccess) return e;
    if (B == 1)
      e = reglu ? dispatch_fused<1, true>(L, x, idx, count, count_const, partial, s)
                : dispatch_fused<1, false>(L, x, idx, count, count_const, partial, s);
    else
      e = reglu ? dispatch_fused<2, true>(L, x, idx, count, count_const, partial, s)
                : dispatch_fused<2, false>(L, x, idx, count, count_const, partial, s);
    if (e != cudaSuccess) return e;
    e = record_hook(L->ev_after, s);
  } else {
    float *a = reinterpret_cast<float *>(ws + w.a);
    const int grid_up = L->num_sms * 4;
    e = record_hook(L->ev_before, s);
    if (e != cudaSuccess) return e;
    const void *ru = q8 ? (const void *)L->Q_up : (const void *)L->W_up;
    const void *rg = q8 ? (const void *)L->Q_gate : (const void *)L->W_gate;
    const void *rd = q8 ? (const void *)L->Q_dT : (const void *)L->W_dT;
    const dim3 gu(grid_up), bu(256);
    if (q8)
      e = reglu ? launch_pdl(k_sparse_up<true, true>, gu, bu, 0, s, ru, rg, L->s_up, L->s_gate, L->b, x, B, L->d,
                             L->ffn, idx, count, count_const, a, L->status, silu)
                : launch_pdl(k_sparse_up<false, true>, gu, bu, 0, s, ru, rg, L->s_up, L->s_gate, L->b, x, B, L->d,
                             L->ffn, idx, count, count_const, a, L->status, silu);
    else
      e = reglu ? launch_pdl(k_sparse_up<true, false>, gu, bu, 0, s, ru, rg, L->s_up, L->s_gate, L->b, x, B, L->d,
                             L->ffn, idx, count, count_const, a, L->status, silu)
                : launch_pdl(k_sparse_up<false, false>, gu, bu, 0, s, ru, rg, L->s_up, L->s_gate, L->b, x, B, L->d,
                             L->ffn, idx, count, count_const, a, L->status, silu);
    if (e != cudaSuccess) return e;
    nsplit = down_splits(L, B);
    const dim3 gd(nsplit, down_colblocks(L)), bd(256);
    e = q8 ? launch_pdl(k_sparse_down<true>, gd, bd, 0, s, rd, (const float *)L->s_dT, (const float *)a, B, L->d,
                        L->ffn, idx, count, count_const, partial, L->status)
           : launch_pdl(k_sparse_down<false>, gd, bd, 0, s, rd, (const float *)L->s_dT, (const float *)a, B, L->d,
                        L->ffn, idx, count, count_const, partial, L->status);
    if (e != cudaSuccess) return e;
    e = record_hook(L->ev_after, s);
  }
  if (e != cudaSuccess) return e;
  const int n4 = B * L->d / 4;
  return launch_pdl(k_reduce, dim3((n4 + 15) / 16), dim3(256), 0, s, (const float *)partial,
                    nsplit, n4, y);
}

}  // namespace pi
