// Persistent decode step: a stack of sparse-FFN layers in one cooperative
// launch.
//
// "PowerInfer: Fast Large Language Model Serving with a Consumer-grade GPU"
// (egguo-blog reading report), section 2.3, core modules 3 (predictor) and 4
// (neuron-aware operators), run layer after layer for one decode batch.
//
// One CTA per SM.  Per layer, four grid-wide phases separated by barriers:
//   A  h = ReLU(W_p1 x): predictor rows k = cta, cta+G, ... (whole CTA per row)
//   C  l = W_p2 h + c_p over the CTA's contiguous neuron slice, threshold,
//      ordered local active list; the CTA immediately asks L2 to stream in the
//      up/gate/down rows of its own active neurons, so HBM traffic for the
//      sparse FFN starts before the global list exists
//   E  global list = concatenation of the local lists (prefix of their
//      counts); CTA j takes the j-th equal chunk of it, forms a and its
//      partial y (rows stream through L2 in windows), and meanwhile prefetches
//      the next layer's predictor weights into L2
//   F  y = sum of the partials in fixed split order (deterministic)
// A barrier follows F so the next layer may depend on y, as in real decode.
//
// Grid barriers spin on a global counter with an iteration cap; on timeout a
// status bit is set and every CTA returns (no trap, no unbounded wait).  Data
// written inside the kernel (h, counts, lists, partials) is read with
// ld.global.cg (L2, coherent); only weights and x use the read-only path.
#include "pi_internal.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kWin = 32;               // max neurons per phase-E window
constexpr unsigned kSpinLimit = 1u << 22;   // ~seconds of polling, then give up

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

template <typename T>
__device__ __forceinline__ T ldcg(const T *p) { return __ldcg(p); }

// Grid barrier number `epoch` (1, 2, ...).  Returns false (after setting the
// timeout bit) if the other CTAs did not arrive within the spin cap or an
// error was already flagged.
__device__ bool grid_barrier(unsigned *bar, unsigned epoch, unsigned *status) {
  __shared__ int ok_s;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned target = epoch * gridDim.x;
    __threadfence();
    atomicAdd(bar, 1u);
    int ok = 1;
    unsigned it = 0;
    while (true) {
      const unsigned v = ld_acquire(bar);
      if ((int)(v - target) >= 0) break;
      if (++it > kSpinLimit) {
        atomicOr(status, PI_STATUS_BARRIER_TIMEOUT);
        ok = 0;
        break;
      }
    }
    __threadfence();
    ok_s = ok;
  }
  __syncthreads();
  return ok_s != 0;
}

#ifdef PI_PHASE_TIMING
// Diagnostic build only: globaltimer stamps at phase boundaries of CTA 0 and
// CTA G-1 for the first 16 layers of the most recent launch.
__device__ unsigned long long g_phase_ts[3][16][16];
#define PHASE_STAMP(l, ph)                                                        \
  do {                                                                            \
    const int w_ = blockIdx.x == 0 ? 0 : blockIdx.x == gridDim.x / 2 ? 1 : blockIdx.x == gridDim.x - 1 ? 2 : -1; \
    if (threadIdx.x == 0 && w_ >= 0 && (l) < 16) {                               \
      unsigned long long t_;                                                      \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                      \
      g_phase_ts[w_][l][ph] = t_;                                                 \
    }                                                                             \
  } while (0)
#else
#define PHASE_STAMP(l, ph) do {} while (0)
#endif

template <int CPT, int NB, bool REGLU>
__global__ void __launch_bounds__(kThreads, 1) k_stack_step(const __grid_constant__ pi::StackParams p) {
  constexpr int G1 = CPT == 1 ? 16 : 8 / CPT > 0 ? 8 / CPT : 1;     // phase-E loads per group
  constexpr int GU = (REGLU ? G1 / 2 : G1) > 0 ? (REGLU ? G1 / 2 : G1) : 1;
  constexpr int NR = REGLU ? 2 : 1;
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ float red_s[kWarps][NB][NR][kWin];
  __shared__ float a_s[NB][kWin];
  __shared__ int win_s[2][kWin];
  __shared__ float4 fred_s[16][32];

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int G = gridDim.x, cta = blockIdx.x;
  const int d = p.d, ffn = p.ffn, r = p.rank, nv = d >> 3;
  const int slice = p.slice;
  const uint32_t row_bytes = (uint32_t)d * 2u;
  unsigned *status = p.status;
  unsigned epoch = 0;

  // dynamic shared memory carve-up
  float *h_s = reinterpret_cast<float *>(smem);                         // [NB, r]
  int *pre_s = reinterpret_cast<int *>(h_s + NB * r);                   // [G + 1]
  int *list_s = pre_s + ((G + 1 + 3) & ~3);                             // [slice]
  int *chunk_s = list_s + slice;                                        // [slice]
  unsigned char *flag_s = reinterpret_cast<unsigned char *>(chunk_s + slice);   // [slice]

  const int s0 = min(ffn, cta * slice), s1 = min(ffn, s0 + slice);     // my predictor slice

  for (int l = 0; l < p.n_layers; ++l) {
    const pi::LayerDev &Ld = p.layers[l];
    const __half *x = p.x + (size_t)l * NB * d;

    uint4 xr[NB][CPT];
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        const int v = tid + c * kThreads;
        xr[t][c] = v < nv ? __ldg(reinterpret_cast<const uint4 *>(x + (size_t)t * d) + v)
                          : make_uint4(0, 0, 0, 0);
      }

    PHASE_STAMP(l, 0);
    // ---------------- A: h = ReLU(W_p1 x), rows cta, cta + G, ...
    for (int k0 = cta; k0 < r; k0 += 2 * G) {
      uint4 w[2][CPT];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int k = k0 + q * G;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          const int v = tid + c * kThreads;
          w[q][c] = (k < r && v < nv)
                        ? pidev::ld_stream(reinterpret_cast<const uint4 *>(Ld.W_p1 + (size_t)k * d) + v)
                        : make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int t = 0; t < NB; ++t) {
          float s = 0.f;
#pragma unroll
          for (int c = 0; c < CPT; ++c) s = pidev::dot8(s, w[q][c], xr[t][c]);
          s = pidev::warp_sum(s);
          if (lane == 0) red_s[wid][t][0][q] = s;
        }
      __syncthreads();
      if (tid < 2 * NB) {
        const int q = tid / NB, t = tid % NB;
        const int k = k0 + q * G;
        if (k < r) {
          float s = 0.f;
          for (int w2 = 0; w2 < kWarps; ++w2) s += red_s[w2][t][0][q];
          p.h[(size_t)t * r + k] = s > 0.f ? s : 0.f;
        }
      }
      __syncthreads();
    }
    PHASE_STAMP(l, 1);
    if (!grid_barrier(p.bar, ++epoch, status)) return;
    PHASE_STAMP(l, 2);

    // ---------------- C: logits over my slice, local ordered active list
    for (int e = tid; e < NB * r; e += kThreads) h_s[e] = ldcg(p.h + e);
    __syncthreads();
    PHASE_STAMP(l, 3);
    {
      const int GL = p.lanes_l;                 // lanes per predictor row (8, 16, 32)
      const int rows_per_warp = 32 / GL;
      const int sub = lane % GL;
      const int nvr = r >> 3;
      const int n_rows = s1 - s0;
      const int iters = (n_rows + kWarps * rows_per_warp - 1) / (kWarps * rows_per_warp);
      constexpr int RU = 8;                     // rows in flight per lane
      for (int it0 = 0; it0 < iters; it0 += RU) {
        float acc[RU][NB];
#pragma unroll
        for (int u = 0; u < RU; ++u)
#pragma unroll
          for (int t = 0; t < NB; ++t) acc[u][t] = 0.f;
        for (int v = sub; v < nvr; v += GL) {
          uint4 wv[RU];
#pragma unroll
          for (int u = 0; u < RU; ++u) {
            const int rl = ((it0 + u) * kWarps + wid) * rows_per_warp + lane / GL;
            wv[u] = (it0 + u < iters && rl < n_rows)
                        ? pidev::ld_stream(reinterpret_cast<const uint4 *>(Ld.W_p2 + (size_t)(s0 + rl) * r) + v)
                        : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int t = 0; t < NB; ++t) {
            const float4 *hp = reinterpret_cast<const float4 *>(h_s + t * r + v * 8);
            const float4 h0 = hp[0], h1 = hp[1];
#pragma unroll
            for (int u = 0; u < RU; ++u) {
              const __half2 *wh = reinterpret_cast<const __half2 *>(&wv[u]);
              const float2 w0 = __half22float2(wh[0]), w1 = __half22float2(wh[1]);
              const float2 w2 = __half22float2(wh[2]), w3 = __half22float2(wh[3]);
              float a = acc[u][t];
              a = fmaf(w0.x, h0.x, a); a = fmaf(w0.y, h0.y, a);
              a = fmaf(w1.x, h0.z, a); a = fmaf(w1.y, h0.w, a);
              a = fmaf(w2.x, h1.x, a); a = fmaf(w2.y, h1.y, a);
              a = fmaf(w3.x, h1.z, a); a = fmaf(w3.y, h1.w, a);
              acc[u][t] = a;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < RU; ++u) {
          const int rl = ((it0 + u) * kWarps + wid) * rows_per_warp + lane / GL;
          const bool valid = it0 + u < iters && rl < n_rows;
          bool on = false;
#pragma unroll
          for (int t = 0; t < NB; ++t) {
            float s = acc[u][t];
            for (int o = GL >> 1; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            if (valid) on |= (s + Ld.c_p[s0 + rl]) > 0.f;
          }
          if (valid && sub == 0) flag_s[rl] = on ? 1 : 0;
        }
      }
    }
    __syncthreads();
    PHASE_STAMP(l, 4);
    // ordered compaction of flag_s[0 .. s1-s0)
    {
      const int n_rows = s1 - s0;
      int base = 0;
      for (int c0 = 0; c0 < n_rows; c0 += kThreads) {
        const int i = c0 + tid;
        const bool on = i < n_rows && flag_s[i];
        const unsigned bal = __ballot_sync(0xffffffffu, on);
        __shared__ int wtot_s[kWarps];
        if (lane == 0) wtot_s[wid] = __popc(bal);
        __syncthreads();
        int wpre = 0, tot = 0;
        for (int q = 0; q < kWarps; ++q) {
          const int v = wtot_s[q];
          if (q < wid) wpre += v;
          tot += v;
        }
        if (on) {
          const int pos = base + wpre + __popc(bal & ((1u << lane) - 1u));
          list_s[pos] = s0 + i;
        }
        base += tot;
        __syncthreads();
      }
      const int lcount = base;
      for (int j = tid; j < lcount; j += kThreads) p.lists[(size_t)cta * slice + j] = list_s[j];
      if (tid == 0) p.cnt[cta] = lcount;
      // stream my own active rows towards L2 now (bounded by the prefetch budget)
      const int npf = min(lcount, p.pf_rows);
      for (int j = tid; j < npf; j += kThreads) {
        const int i = list_s[j];
        pidev::prefetch_l2_bulk(Ld.W_up + (size_t)i * d, row_bytes);
        if (REGLU) pidev::prefetch_l2_bulk(Ld.W_gate + (size_t)i * d, row_bytes);
        pidev::prefetch_l2_bulk(Ld.W_dT + (size_t)i * d, row_bytes);
      }
    }
    PHASE_STAMP(l, 5);
    if (!grid_barrier(p.bar, ++epoch, status)) return;
    PHASE_STAMP(l, 6);

    // ---------------- E: my chunk of the global list, up + down
    if (tid < 32) {
      // exclusive prefix of the G local counts (one warp; all loads issued first)
      constexpr int kCntRegs = 8;
      int cv[kCntRegs];
#pragma unroll
      for (int q = 0; q < kCntRegs; ++q) {
        const int c = q * 32 + lane;
        cv[q] = c < G ? ldcg(p.cnt + c) : 0;
      }
      int carry = 0;
      for (int c0 = 0; c0 < G; c0 += 32) {
        const int q = c0 / 32;
        int v = 0;
#pragma unroll
        for (int qq = 0; qq < kCntRegs; ++qq)
          if (qq == q) v = cv[qq];
        if (q >= kCntRegs) v = c0 + lane < G ? ldcg(p.cnt + c0 + lane) : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += n;
        }
        if (c0 + lane < G) pre_s[c0 + lane] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) pre_s[G] = carry;
    }
    __syncthreads();
    const int total = pre_s[G];
    if (cta == 0 && tid == 0 && p.count) p.count[l] = total;
    if (p.idx) {
      const int my0 = pre_s[cta], myn = pre_s[cta + 1] - my0;
      for (int j = tid; j < myn; j += kThreads) p.idx[(size_t)l * ffn + my0 + j] = list_s[j];
    }
    const int chunk = (total + G - 1) / G;
    const int k0 = min(total, cta * chunk), k1 = min(total, k0 + chunk);
    for (int j = tid; j < k1 - k0; j += kThreads) {
      const int k = k0 + j;
      int lo = 0, hi = G - 1;                 // largest o with pre_s[o] <= k
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre_s[mid] <= k) lo = mid; else hi = mid - 1;
      }
      chunk_s[j] = ldcg(p.lists + (size_t)lo * slice + (k - pre_s[lo]));
    }
    __syncthreads();
    PHASE_STAMP(l, 7);
    // next layer's predictor weights: start them towards L2 now
    if (p.pf_next && l + 1 < p.n_layers) {
      const pi::LayerDev &Ln = p.layers[l + 1];
      if (tid == 0)
        for (int k = cta; k < r; k += G) pidev::prefetch_l2_bulk(Ln.W_p1 + (size_t)k * d, row_bytes);
      const uint32_t p2_bytes = (uint32_t)(s1 - s0) * (uint32_t)r * 2u;
      if (tid == 1 && s1 > s0) {
        // bulk prefetch sizes are limited; split into 64 KB pieces
        const char *base = reinterpret_cast<const char *>(Ln.W_p2 + (size_t)s0 * r);
        for (uint32_t o = 0; o < p2_bytes; o += 65536u)
          pidev::prefetch_l2_bulk(base + o, min(65536u, p2_bytes - o));
      }
    }

    float acc[NB][CPT][8];
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
      for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[t][c][e] = 0.f;

    const int n_chunk = k1 - k0;
    const int win = p.sub;
    auto prefetch_window = [&](int w0, int buf) {
      const int w1 = min(n_chunk, w0 + win);
      for (int j = w0 + tid; j < w1; j += kThreads) {
        const int i = chunk_s[j];
        win_s[buf][j - w0] = i;
        pidev::prefetch_l2_bulk(Ld.W_up + (size_t)i * d, row_bytes);
        if (REGLU) pidev::prefetch_l2_bulk(Ld.W_gate + (size_t)i * d, row_bytes);
        pidev::prefetch_l2_bulk(Ld.W_dT + (size_t)i * d, row_bytes);
      }
    };
    if (n_chunk > 0) prefetch_window(0, 0);
    __syncthreads();
    int buf = 0;
    for (int w0 = 0; w0 < n_chunk; w0 += win, buf ^= 1) {
      const int n_here = min(win, n_chunk - w0);
      if (w0 + win < n_chunk) prefetch_window(w0 + win, buf ^ 1);
      for (int g0 = 0; g0 < n_here; g0 += GU) {
        uint4 w[GU][NR][CPT];
#pragma unroll
        for (int n = 0; n < GU; ++n) {
          const int i = g0 + n < n_here ? win_s[buf][g0 + n] : -1;
#pragma unroll
          for (int c = 0; c < CPT; ++c) {
            const int v = tid + c * kThreads;
            const bool ok = i >= 0 && v < nv;
            w[n][0][c] = ok ? pidev::ld_stream(reinterpret_cast<const uint4 *>(Ld.W_up + (size_t)i * d) + v)
                            : make_uint4(0, 0, 0, 0);
            if (REGLU)
              w[n][NR - 1][c] = ok ? pidev::ld_stream(reinterpret_cast<const uint4 *>(Ld.W_gate + (size_t)i * d) + v)
                                   : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int n = 0; n < GU; ++n)
#pragma unroll
          for (int q = 0; q < NR; ++q)
#pragma unroll
            for (int t = 0; t < NB; ++t) {
              float s = 0.f;
#pragma unroll
              for (int c = 0; c < CPT; ++c) s = pidev::dot8(s, w[n][q][c], xr[t][c]);
              s = pidev::warp_sum(s);
              if (lane == 0 && g0 + n < n_here) red_s[wid][t][q][g0 + n] = s;
            }
      }
      __syncthreads();
      for (int e = tid; e < NB * n_here; e += kThreads) {
        const int t = e / n_here, n = e % n_here;
        const int i = win_s[buf][n];
        float su = 0.f, sg = 0.f;
        for (int q = 0; q < kWarps; ++q) {
          su += red_s[q][t][0][n];
          if (REGLU) sg += red_s[q][t][NR - 1][n];
        }
        float a;
        if (REGLU) {
          const float gz = sg + Ld.b[i];
          a = (gz > 0.f ? gz : 0.f) * su;
        } else {
          const float z = su + Ld.b[i];
          a = z > 0.f ? z : 0.f;
        }
        a_s[t][n] = a;
      }
      __syncthreads();
      for (int g0 = 0; g0 < n_here; g0 += G1) {
        uint4 w[G1][CPT];
#pragma unroll
        for (int n = 0; n < G1; ++n) {
          const int i = g0 + n < n_here ? win_s[buf][g0 + n] : -1;
#pragma unroll
          for (int c = 0; c < CPT; ++c) {
            const int v = tid + c * kThreads;
            w[n][c] = (i >= 0 && v < nv)
                          ? pidev::ld_stream(reinterpret_cast<const uint4 *>(Ld.W_dT + (size_t)i * d) + v)
                          : make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int n = 0; n < G1; ++n) {
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
      __syncthreads();
    }
    PHASE_STAMP(l, 8);
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        const int v = tid + c * kThreads;
        if (v < nv) {
          float4 *dst = reinterpret_cast<float4 *>(p.partial + ((size_t)cta * NB + t) * d) + 2 * v;
          dst[0] = make_float4(acc[t][c][0], acc[t][c][1], acc[t][c][2], acc[t][c][3]);
          dst[1] = make_float4(acc[t][c][4], acc[t][c][5], acc[t][c][6], acc[t][c][7]);
        }
      }
    PHASE_STAMP(l, 9);
    if (!grid_barrier(p.bar, ++epoch, status)) return;
    PHASE_STAMP(l, 10);

    // ---------------- F: y = sum of partials, columns c = cta, cta + G, ... (float4)
    {
      const int n4 = NB * d / 4;
      const int col_l = tid & 31, g = tid >> 5;     // 32 columns x 16 split groups per pass
      float *y = p.y + (size_t)l * NB * d;
      for (int c0 = cta * 32; c0 < n4; c0 += G * 32) {
        const int c = c0 + col_l;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < n4) {
          const float4 *pp = reinterpret_cast<const float4 *>(p.partial);
          constexpr int kPR = 16;                  // split loads in flight per thread
          for (int sp0 = g; sp0 < G; sp0 += kWarps * kPR) {
            float4 v[kPR];
#pragma unroll
            for (int q = 0; q < kPR; ++q) {
              const int sp = sp0 + q * kWarps;
              v[q] = sp < G ? ldcg(pp + (size_t)sp * n4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < kPR; ++q) {
              s.x += v[q].x; s.y += v[q].y; s.z += v[q].z; s.w += v[q].w;
            }
          }
        }
        fred_s[g][col_l] = s;
        __syncthreads();
        if (g == 0 && c < n4) {
          float4 t4 = fred_s[0][col_l];
          for (int q = 1; q < kWarps; ++q) {
            const float4 v = fred_s[q][col_l];
            t4.x += v.x; t4.y += v.y; t4.z += v.z; t4.w += v.w;
          }
          reinterpret_cast<float4 *>(y)[c] = t4;
        }
        __syncthreads();
      }
    }
    PHASE_STAMP(l, 11);
    if (!grid_barrier(p.bar, ++epoch, status)) return;
    PHASE_STAMP(l, 12);
  }
}

#ifdef PI_PHASE_TIMING
}  // namespace
extern "C" int pi_debug_phase_times(unsigned long long *out) {
  return (int)cudaMemcpyFromSymbol(out, g_phase_ts, sizeof(g_phase_ts));
}
namespace {
#endif

template <int CPT, int NB, bool REGLU>
cudaError_t launch_step(const pi::StackParams &p, size_t smem, cudaStream_t s) {
  auto kern = k_stack_step<CPT, NB, REGLU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int occ = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
  if (e != cudaSuccess) return e;
  if (occ < 1) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int NB, bool REGLU>
cudaError_t dispatch_step(const pi::StackParams &p, size_t smem, cudaStream_t s) {
  const int cpt = (p.d / 8 + kThreads - 1) / kThreads;
  switch (cpt) {
    case 1: return launch_step<1, NB, REGLU>(p, smem, s);
    case 2: return launch_step<2, NB, REGLU>(p, smem, s);
    case 3: return launch_step<3, NB, REGLU>(p, smem, s);
    case 4: return launch_step<4, NB, REGLU>(p, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

namespace pi {

int step_grid(const pi_layer *L) { return L->num_sms; }

int step_slice(const pi_layer *L) { return (L->ffn + step_grid(L) - 1) / step_grid(L); }

size_t step_smem(const pi_layer *L, int B) {
  const int G = step_grid(L), slice = step_slice(L);
  size_t b = sizeof(float) * (size_t)B * L->rank;
  b += sizeof(int) * (size_t)((G + 1 + 3) & ~3);
  b += sizeof(int) * 2 * (size_t)slice + (size_t)slice;
  return (b + 15) & ~(size_t)15;
}

cudaError_t run_stack(pi_layer *const *layers, int n, const __half *x, int B, int32_t *idx,
                      int32_t *count, float *y, const WsLayout &w, char *ws, cudaStream_t s) {
  const pi_layer *L0 = layers[0];
  StackParams p = {};
  p.n_layers = n;
  p.d = L0->d;
  p.ffn = L0->ffn;
  p.rank = L0->rank;
  p.G = step_grid(L0);
  p.slice = step_slice(L0);
  int GL = 32;
  while (GL > 8 && GL * 8 > L0->rank) GL >>= 1;
  p.lanes_l = GL;
  const int rows_per_neuron = L0->act == PI_ACT_REGLU ? 3 : 2;
  int sub = (192 * 1024) / (2 * L0->d * rows_per_neuron);
  p.sub = sub < 1 ? 1 : (sub > kWin ? kWin : sub);
  // early prefetch of the local active rows: up to ~384 KB of rows per CTA
  int pf = (384 * 1024) / (2 * L0->d * rows_per_neuron);
  p.pf_rows = pf < 1 ? 1 : pf;
  // next layer's predictor weights into L2 only when they are small
  const size_t pred_bytes = 2ull * L0->rank * L0->d + 2ull * L0->ffn * L0->rank;
  p.pf_next = pred_bytes <= (32ull << 20);
  p.x = x;
  p.y = y;
  p.idx = idx;
  p.count = count;
  p.h = reinterpret_cast<float *>(ws + w.h);
  p.cnt = reinterpret_cast<int32_t *>(ws + w.cnt);
  p.lists = reinterpret_cast<int32_t *>(ws + w.lists);
  p.partial = reinterpret_cast<float *>(ws + w.partial);
  p.bar = reinterpret_cast<unsigned *>(ws + w.bar);
  p.status = L0->status;
  for (int l = 0; l < n; ++l) {
    const pi_layer *Ll = layers[l];
    p.layers[l] = LayerDev{Ll->W_p1, Ll->W_p2, Ll->W_up, Ll->W_gate, Ll->W_dT, Ll->b, Ll->c_p};
  }
  cudaError_t e = cudaMemsetAsync(p.bar, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const size_t smem = step_smem(L0, B);
  const bool reglu = L0->act == PI_ACT_REGLU;
  e = record_hook(L0->ev_before, s);
  if (e != cudaSuccess) return e;
  if (B == 1)
    e = reglu ? dispatch_step<1, true>(p, smem, s) : dispatch_step<1, false>(p, smem, s);
  else
    e = reglu ? dispatch_step<2, true>(p, smem, s) : dispatch_step<2, false>(p, smem, s);
  if (e != cudaSuccess) return e;
  return record_hook(L0->ev_after, s);
}

}  // namespace pi
