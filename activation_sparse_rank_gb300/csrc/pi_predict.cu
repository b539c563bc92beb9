// Adaptive activation predictor and active-index compaction.
//
// "PowerInfer: Fast Large Language Model Serving with a Consumer-grade GPU"
// (egguo-blog reading report), section 2.3, core module 3: a small MLP per
// layer predicts which FFN neurons fire for the current token; here
// h = ReLU(W_p1 x), l = W_p2 h + c_p, neuron active iff l > 0 (sigmoid > 1/2).
// Section 2.3, core module 4 (neuron-aware operators) then consumes the list
// of active neurons; with a batch the list is the union over tokens
// (section 4.4, limitation 3).
//
// All three kernels are HBM- or latency-bound GEMV / scan work: plain
// coalesced 16-byte loads, fp32 accumulation, warp-shuffle reductions.
#include "pi_internal.cuh"

namespace {

constexpr int kBT = 8;   // tokens handled per pass over a weight row

// h[b, k] = max(0, W_p1[k, :] . x[b, :]).  One warp per row k; each lane
// takes every 32nd 16-byte vector of the row.
__global__ void __launch_bounds__(128) k_predict_h(const __half *__restrict__ W_p1,
                                                   const __half *__restrict__ x, int B, int d,
                                                   int r, float *__restrict__ h) {
  pidev::griddep_wait();
  pidev::griddep_launch();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= r) return;
  const uint4 *w = reinterpret_cast<const uint4 *>(W_p1 + (size_t)warp * d);
  const int nv = d >> 3;
  for (int b0 = 0; b0 < B; b0 += kBT) {
    const int nb = min(kBT, B - b0);
    float acc[kBT];
#pragma unroll
    for (int t = 0; t < kBT; ++t) acc[t] = 0.f;
#pragma unroll 4
    for (int v = lane; v < nv; v += 32) {
      const uint4 wv = pidev::ld_stream(w + v);
#pragma unroll
      for (int t = 0; t < kBT; ++t) {
        if (t < nb) {
          const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)(b0 + t) * d) + v);
          acc[t] = pidev::dot8(acc[t], wv, xv);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kBT; ++t) {
      const float s = pidev::warp_sum(acc[t]);
      if (lane == 0 && t < nb) h[(size_t)(b0 + t) * r + warp] = s > 0.f ? s : 0.f;
    }
  }
}

// l[b, i] = W_p2[i, :] . h[b, :] + c_p[i]; mask = l > 0.  G lanes share a row
// (G = 8, 16 or 32 from the rank), h staged in shared memory per token group.
// W_p2 rows are ld elements apart.
__global__ void __launch_bounds__(256) k_predict_l(const __half *__restrict__ W_p2, int ld,
                                                   const float *__restrict__ c_p,
                                                   const float *__restrict__ h, int B, int r,
                                                   int ffn, int G, uint8_t *__restrict__ mask,
                                                   float *__restrict__ logits, int union_mask) {
  extern __shared__ float h_s[];   // [kBT, r]
  pidev::griddep_wait();
  pidev::griddep_launch();
  const int lane = threadIdx.x & 31;
  const int sub = lane % G;                 // lane within the row group
  const int groups_per_warp = 32 / G;
  const int gid = ((blockIdx.x * blockDim.x + threadIdx.x) >> 5) * groups_per_warp + lane / G;
  const int ngroups = ((gridDim.x * blockDim.x) >> 5) * groups_per_warp;
  const int nv = r >> 3;
  // every lane of a row group iterates the same number of times (shuffles stay converged)
  const int rows_iter = (ffn + ngroups - 1) / ngroups;
  for (int b0 = 0; b0 < B; b0 += kBT) {
    const int nb = min(kBT, B - b0);
    __syncthreads();
    for (int e = threadIdx.x; e < nb * r; e += blockDim.x) h_s[e] = h[(size_t)b0 * r + e];
    __syncthreads();
    for (int it = 0; it < rows_iter; ++it) {
      const int row = gid + it * ngroups;
      const bool valid = row < ffn;
      float acc[kBT];
#pragma unroll
      for (int t = 0; t < kBT; ++t) acc[t] = 0.f;
      if (valid) {
        const uint4 *w = reinterpret_cast<const uint4 *>(W_p2 + (size_t)row * ld);
        for (int v = sub; v < nv; v += G) {
          const uint4 wv = pidev::ld_stream(w + v);
          const __half2 *wh = reinterpret_cast<const __half2 *>(&wv);
#pragma unroll
          for (int t = 0; t < kBT; ++t) {
            if (t < nb) {
              const float4 *hp = reinterpret_cast<const float4 *>(h_s + t * r + v * 8);
              const float4 h0 = hp[0], h1 = hp[1];
              float2 w0 = __half22float2(wh[0]), w1 = __half22float2(wh[1]);
              float2 w2 = __half22float2(wh[2]), w3 = __half22float2(wh[3]);
              float a = acc[t];
              a = fmaf(w0.x, h0.x, a); a = fmaf(w0.y, h0.y, a);
              a = fmaf(w1.x, h0.z, a); a = fmaf(w1.y, h0.w, a);
              a = fmaf(w2.x, h1.x, a); a = fmaf(w2.y, h1.y, a);
              a = fmaf(w3.x, h1.z, a); a = fmaf(w3.y, h1.w, a);
              acc[t] = a;
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < kBT; ++t) {
        float s = acc[t];
        for (int o = G >> 1; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (valid && sub == 0 && t < nb) {
          const float l = s + c_p[row];
          const size_t o = (size_t)(b0 + t) * ffn + row;
          if (mask) {
            if (!union_mask) mask[o] = l > 0.f ? 1 : 0;
            else if (l > 0.f) mask[row] = 1;      // OR over the batch (zeroed before the launch)
          }
          if (logits) logits[o] = l;
        }
      }
    }
  }
}

// Ordered compaction of the union of mask rows: one CTA of 1024 threads, each
// thread owns 16 consecutive neurons per pass; warp and block prefix sums give
// every thread its output offset, so idx comes out ascending.
__global__ void __launch_bounds__(1024) k_compact(const uint8_t *__restrict__ mask, int B,
                                                  int ffn, int vec, int32_t *__restrict__ idx,
                                                  int32_t *__restrict__ count) {
  __shared__ int warp_tot[32];
  pidev::griddep_wait();
  pidev::griddep_launch();
  // one CTA per problem: blockIdx.x selects a [B, ffn] mask, an idx row and a count
  mask += (size_t)blockIdx.x * B * ffn;
  idx += (size_t)blockIdx.x * ffn;
  count += blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  int base = 0;
  for (int i0 = 0; i0 < ffn; i0 += 1024 * 16) {
    const int i = i0 + tid * 16;
    uint32_t bits = 0;
    if (i < ffn) {
      if (vec && i + 16 <= ffn) {
        for (int b = 0; b < B; ++b) {
          const uint4 m = *reinterpret_cast<const uint4 *>(mask + (size_t)b * ffn + i);
          const uint32_t wds[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if ((wds[q] >> (8 * e)) & 0xffu) bits |= 1u << (4 * q + e);
        }
      } else {
        for (int j = 0; j < 16 && i + j < ffn; ++j)
          for (int b = 0; b < B; ++b)
            if (mask[(size_t)b * ffn + i + j]) bits |= 1u << j;
      }
    }
    const int c = __popc(bits);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
      const int v = warp_tot[lane];
      int s = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, s, o);
        if (lane >= o) s += n;
      }
      warp_tot[lane] = s - v;   // exclusive prefix of warp totals
    }
    __syncthreads();
    int off = base + warp_tot[wid] + incl - c;
    while (bits) {
      const int j = __ffs(bits) - 1;
      idx[off++] = i + j;
      bits &= bits - 1;
    }
    // block total = exclusive prefix of the last warp + its inclusive total
    const int last_incl = __shfl_sync(0xffffffffu, incl, 31);
    __syncthreads();
    if (wid == 31 && lane == 0) warp_tot[0] = warp_tot[31] + last_incl;
    __syncthreads();
    base += warp_tot[0];
    __syncthreads();
  }
  if (tid == 0) *count = base;
}

}  // namespace

namespace pi {

cudaError_t run_predict(const pi_layer *L, const __half *x, int B, uint8_t *mask, float *logits,
                        float *h_ws, cudaStream_t s, bool union_mask) {
  const int warps_h = 4;
  const int grid_h = (L->rank + warps_h - 1) / warps_h;
  cudaError_t e = launch_pdl(k_predict_h, dim3(grid_h), dim3(32 * warps_h), 0, s, L->W_p1, x, B,
                             L->d, L->rank, h_ws);
  if (e != cudaSuccess) return e;
  int G = 32;
  while (G > 8 && G * 8 > L->rank) G >>= 1;
  const int rows_per_cta = (256 / 32) * (32 / G);
  int grid_l = (L->ffn + rows_per_cta - 1) / rows_per_cta;
  const int cap = L->num_sms * 8;
  if (grid_l > cap) grid_l = cap;
  const size_t smem = sizeof(float) * kBT * L->rank;
  if (smem > 48 * 1024) {
    e = cudaFuncSetAttribute(k_predict_l, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  if (union_mask) {
    e = cudaMemsetAsync(mask, 0, (size_t)L->ffn, s);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(k_predict_l, dim3(grid_l), dim3(256), smem, s, L->W_p2, L->p2_ld, L->c_p, h_ws, B,
                    L->rank, L->ffn, G, mask, logits, union_mask ? 1 : 0);
}

cudaError_t run_compact(const pi_layer *L, const uint8_t *mask, int B, int32_t *idx,
                        int32_t *count, cudaStream_t s) {
  const int vec = ((reinterpret_cast<uintptr_t>(mask) & 15) == 0) && (L->ffn % 16 == 0);
  return launch_pdl(k_compact, dim3(1), dim3(1024), 0, s, mask, B, L->ffn, vec, idx, count);
}

cudaError_t run_compact_layers(const pi_layer *L, const uint8_t *masks, int n, int32_t *idx,
                               int32_t *count, cudaStream_t s) {
  const int vec = ((reinterpret_cast<uintptr_t>(masks) & 15) == 0) && (L->ffn % 16 == 0);
  return launch_pdl(k_compact, dim3(n), dim3(1024), 0, s, masks, 1, L->ffn, vec, idx, count);
}

}  // namespace pi
