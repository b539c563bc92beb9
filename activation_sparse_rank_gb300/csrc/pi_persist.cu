// Persistent decode step: a stack of sparse-FFN layers in one cooperative
// launch.
//
// "PowerInfer: Fast Large Language Model Serving with a Consumer-grade GPU"
// (egguo-blog reading report), section 2.3, core modules 3 (predictor) and 4
// (neuron-aware operators), run layer after layer for one decode batch.
//
// One CTA per SM.  The layer's neurons are stored hot-first and dealt
// round-robin over the G SM slices (see pi_layer_create), so every CTA's
// contiguous slice holds the same mix of hot and cold neurons and a similar
// expected number of active ones.  Per layer, three grid-wide barriers:
//   A  h = ReLU(W_p1 x): predictor rows k = cta, cta+G, ... (whole CTA per row)
//   -- barrier 1 (h complete)
//   C  l = W_p2 h + c_p over the CTA's slice, threshold, ordered local list
//   E  the CTA streams the up/gate/down rows of its own active neurons (bulk
//      L2 prefetch of all of them first, then 16-byte loads in windows), forms
//      a and its partial y; meanwhile the next layer's predictor weights land
//      in shared memory by TMA (or are prefetched into L2 when too big)
//   -- barrier 2 (partials complete)
//   F  y = sum of the G partials in a fixed order (deterministic)
//   -- barrier 3 (y complete: the next layer may depend on it, as in decode)
// In chained mode the next layer's input is formed from y on the device,
// x_{l+1} = fp16(y_l / RMS(y_l)), after barrier 3 (nothing of x_{l+1} is
// read earlier).
//
// Grid barriers are a release-add on a global counter and an acquire poll
// with an iteration cap; mbarrier waits are capped too.  On a cap the kernel
// sets a status bit and returns (no trap, no unbounded wait).  Data written
// inside the kernel (h, counts, partials) is read with ld.global.cg (L2,
// coherent); only weights and x use the read-only path.
#include <type_traits>

#include "pi_internal.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
// The last warp issues the asynchronous copies and prefetches (TMA staging,
// L2 prefetch): those instructions can stall their issuing thread, so they
// go to a warp that has no other work on the critical path.
constexpr int kIssuer = kThreads - 32;
constexpr unsigned kSpinLimit = 1u << 22;   // polls before a wait gives up (seconds)

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

template <typename T>
__device__ __forceinline__ T ldcg(const T *p) { return __ldcg(p); }

// Grid barrier number `epoch` (1, 2, ...).  False if the wait ran out (status set).
__device__ bool grid_barrier(unsigned *bar, unsigned epoch, unsigned *status) {
  __shared__ int ok_s;
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned target = epoch * gridDim.x;
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
    int ok = 1;
    unsigned it = 0;
    while ((int)(ld_acquire(bar) - target) < 0) {
      if (++it > kSpinLimit) {
        atomicOr(status, PI_STATUS_BARRIER_TIMEOUT);
        ok = 0;
        break;
      }
    }
    ok_s = ok;
  }
  __syncthreads();
  return ok_s != 0;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Bounded wait for mbarrier phase `parity`.  False if it ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t mbar, uint32_t parity) {
  for (unsigned it = 0; it < kSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(mbar), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void tma_load_1d(void *dst_smem, const void *src, uint32_t bytes,
                                            uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(mbar)
      : "memory");
}

#ifdef PI_PHASE_TIMING
// Diagnostic build only: globaltimer stamps at phase boundaries of three CTAs
// for the first 16 layers of the most recent launch.
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
// per CTA and layer: up/down phase duration (ns) and local active count
__device__ unsigned long long g_cta_e[160][16][2];
#define CTA_E_BEGIN(l) unsigned long long te0_ = 0; if (threadIdx.x == 0) asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(te0_));
#define CTA_E_END(l, cnt)                                                            \
  do {                                                                               \
    if (threadIdx.x == 0 && blockIdx.x < 160 && (l) < 16) {                          \
      unsigned long long t_;                                                         \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                         \
      g_cta_e[blockIdx.x][l][0] = t_ - te0_;                                         \
      g_cta_e[blockIdx.x][l][1] = (unsigned long long)(cnt);                         \
    }                                                                                \
  } while (0)
#else
#define PHASE_STAMP(l, ph) do {} while (0)
#define CTA_E_BEGIN(l) do {} while (0)
#define CTA_E_END(l, cnt) do {} while (0)
#endif

// Stage the inputs of one layer for this CTA into shared memory (one thread,
// TMA bulk copies completing on `mbar`): the token rows x [NB, d] (unless
// with_x is false), the CTA's
// slices of c_p and b (from the 16-byte boundary at or below s0; the layer
// allocation pads both vectors to 256 bytes, so the rounded-up end stays
// inside it) and, when `with_pred`, its W_p1 rows k = cta, cta+G, ... and
// its W_p2 slice.
// Called by lane 0 of one warp.  W_p2 rows are p2_stride bytes apart, in the
// layer and in the copy alike (the slice is one contiguous bulk copy).
__device__ __forceinline__ void stage_layer(const pi::LayerDev &Ld, const __half *x, int nb, bool with_x,
                                            int cta, int G, int d, int r, int s0, int s1, bool with_pred,
                                            int p2_stride, __half *x_s, float *c_s, float *b_s,
                                            __half *p1_s, unsigned char *p2_s, float *su_s, float *sg_s,
                                            float *sd_s, uint32_t mbar, int part = 0) {
  // su_s / sg_s / sd_s: the row-scale slices of an FP8 layer (up, gate for
  // ReGLU, down^T), or nullptr
  const int s0a = s0 & ~3;
  const uint32_t cb_bytes = (uint32_t)(((s1 - s0a) + 3) & ~3) * 4u;
  const uint32_t x_bytes = with_x ? (uint32_t)nb * (uint32_t)d * 2u : 0u;
  const uint32_t row_bytes = (uint32_t)d * 2u;
  const uint32_t p2_bytes = with_pred ? (uint32_t)(s1 - s0) * (uint32_t)p2_stride : 0u;
  int na = 0;
  if (with_pred)
    for (int k = cta; k < r; k += G) ++na;
  const uint32_t nsc = su_s ? (sg_s ? 3u : 2u) : 0u;
  const uint32_t total = x_bytes + (cb_bytes ? (2u + nsc) * cb_bytes : 0u) + (uint32_t)na * row_bytes + p2_bytes;
  if (part == 2) {                     // the W_p2 slice only (the expectation is already set)
    if (p2_bytes)
      tma_load_1d(p2_s, reinterpret_cast<const unsigned char *>(Ld.W_p2) + (size_t)s0 * p2_stride, p2_bytes, mbar);
    return;
  }
  if (part != 1)                        // part 1: the caller set the expectation already
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(total) : "memory");
  if (x_bytes) tma_load_1d(x_s, x, x_bytes, mbar);
  if (cb_bytes) {
    tma_load_1d(c_s, Ld.c_p + s0a, cb_bytes, mbar);
    tma_load_1d(b_s, Ld.b + s0a, cb_bytes, mbar);
    if (su_s) {
      tma_load_1d(su_s, Ld.s_up + s0a, cb_bytes, mbar);
      if (sg_s) tma_load_1d(sg_s, Ld.s_gate + s0a, cb_bytes, mbar);
      tma_load_1d(sd_s, Ld.s_dT + s0a, cb_bytes, mbar);
    }
  }
  int q = 0;
  for (int k = cta; q < na; k += G, ++q)
    tma_load_1d(p1_s + (size_t)q * d, Ld.W_p1 + (size_t)k * d, row_bytes, mbar);
  if (p2_bytes && part == 0)
    tma_load_1d(p2_s, reinterpret_cast<const unsigned char *>(Ld.W_p2) + (size_t)s0 * p2_stride, p2_bytes, mbar);
}

// Tensor-core fragment helpers (mma.sync m16n8k16, fp16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// (hi, lo) fp16 pair of a binary32 value: hi = fp16(v), lo = fp16(v - hi)
__device__ __forceinline__ void f32_to_pair(float v, __half &hi, __half &lo) {
  hi = __float2half_rn(v);
  lo = __float2half_rn(v - __half2float(hi));
}
__device__ __forceinline__ uint32_t pack_h2(__half a, __half b) {
  return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

template <int CPT, int NB, bool REGLU, bool FP8>
__global__ void __launch_bounds__(kThreads, 1) k_stack_step(const __grid_constant__ pi::StackParams p) {
  // FP8: the up / gate / down rows are E4M3 codes (8 bytes per 8 elements,
  // loaded as uint2) with a per-row scale applied to each dot product and
  // activation; otherwise fp16 (uint4 per 8 elements)
  using RowVec = typename std::conditional<FP8, uint2, uint4>::type;
  constexpr int NR = REGLU ? 2 : 1;                          // gated rows per neuron
  constexpr int LOADS = CPT == 1 ? 24 : 16;                  // 16-byte loads in flight per thread
  constexpr int GU0 = LOADS / (CPT * NR), GD0 = LOADS / CPT;
  constexpr int GU = GU0 > 0 ? GU0 : 1;                      // neurons per up-pass window
  constexpr int GD = GD0 > 0 ? GD0 : 1;                      // neurons per down-pass window
  // one-pass windows: each neuron's up (+gate) and down rows loaded together,
  // 96 registers of rows in flight per thread (56 with two tokens, whose
  // inputs and accumulators take twice the registers)
  constexpr int RV = FP8 ? 2 : 4;                            // 32-bit registers per row vector
  constexpr int GW0 = (NB == 1 ? 96 : 56) / ((NR + 1) * CPT * RV);
  constexpr int GW = GW0 > 0 ? GW0 : 1;                      // neurons per window
  constexpr int GR = GU > GW ? GU : GW;
  // Measured on GB300: the one-pass windows win with E4M3 rows (a window of
  // 24 neurons covers nearly every CTA's list), with two tokens and with
  // ReGLU (three rows per neuron); with one token of fp16 ReLU rows the two
  // passes are as fast or slightly faster.
  constexpr bool kOnePass = FP8 || NB == 2 || REGLU;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float red_s[kWarps][NB][NR][GR];
  __shared__ float ared_s[kWarps][NB][8];
  __shared__ float4 fred_s[2][8];
  __shared__ int wtot_s[kWarps];
  __shared__ __align__(8) unsigned long long mbar_s[2];

  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int G = gridDim.x, cta = blockIdx.x;
  const int d = p.d, ffn = p.ffn, r = p.rank, nv = d >> 3;
  const int p2_ld = p.p2_stride >> 1;                          // elements between W_p2 rows
  const uint32_t row_bytes = (uint32_t)d * 2u;                 // an fp16 row (predictor)
  const uint32_t rrow = FP8 ? (uint32_t)d : row_bytes;          // a gathered up / gate / down row
  unsigned *status = p.status;
  const bool chained = p.chained != 0;
  __shared__ float ss_s[kWarps][NB];
  // 8-element vector v of gathered row i of R (fp16 or E4M3 codes)
  auto ldrow = [&](const void *R, int i, int v) -> RowVec {
    const char *row = static_cast<const char *>(R) + (size_t)i * rrow;
    if constexpr (FP8) return pidev::ld_stream2(reinterpret_cast<const uint2 *>(row) + v);
    else return pidev::ld_stream(reinterpret_cast<const uint4 *>(row) + v);
  };
  auto rowdot = [](float acc, const RowVec &w, const uint4 &x) {
    if constexpr (FP8) return pidev::dot8_e4m3(acc, w, x);
    else return pidev::dot8(acc, w, x);
  };
  auto rowaxpy = [](float *acc, float a, const RowVec &w) {
    if constexpr (FP8) pidev::axpy8_e4m3(acc, a, w);
    else pidev::axpy8(acc, a, w);
  };
  auto rowpf = [&](const void *R, int i) {
    pidev::prefetch_l2_bulk(static_cast<const char *>(R) + (size_t)i * rrow, rrow);
  };
  unsigned epoch = 0;
  const uint32_t mbar0 = smem_u32(&mbar_s[0]);

  // this CTA's neuron slice [s0, s1): sizes differ by at most one
  const int q_sl = ffn / G, r_sl = ffn % G;
  const int s0 = cta * q_sl + min(cta, r_sl);
  const int s1 = s0 + q_sl + (cta < r_sl ? 1 : 0);
  const int n_rows = s1 - s0;

  // dynamic shared memory carve-up (sizes from pi::step_smem)
  float *h_s = reinterpret_cast<float *>(smem);                                     // [NB, r]
  unsigned char *flag_s = reinterpret_cast<unsigned char *>(smem) + p.off_flag;    // [slice]
  int *list_s = reinterpret_cast<int *>(smem + p.off_list);                        // [slice]
  float *lb_s = reinterpret_cast<float *>(smem + p.off_lb);                        // [slice] b of list
  float *a_all = reinterpret_cast<float *>(smem + p.off_a);                         // [NB, slice] a of list
  // two stage buffers (layer l uses buffer l & 1), each [x | c_p slice | b slice | W_p1 rows | W_p2 slice]
  auto stage_buf = [&](int k) { return smem + p.off_stage + (size_t)k * p.stage_bytes; };
  const int s0a = s0 & ~3;                       // c / b slices start at this neuron
  auto stage_total = [&](int layer) -> uint32_t {   // bytes stage(layer) copies (staged layers)
    const int s0a_ = s0 & ~3;
    const uint32_t cb = (uint32_t)(((s1 - s0a_) + 3) & ~3) * 4u;
    const uint32_t xb = (!chained || layer == 0) ? (uint32_t)NB * (uint32_t)d * 2u : 0u;
    int na = 0;
    for (int k = cta; k < r; k += G) ++na;
    const uint32_t nsc = FP8 ? (REGLU ? 3u : 2u) : 0u;
    return xb + (cb ? (2u + nsc) * cb : 0u) + (uint32_t)na * (uint32_t)d * 2u + (uint32_t)(s1 - s0) * (uint32_t)p.p2_stride;
  };
  auto stage = [&](int layer, int part = 0) {    // one thread: issue layer's inputs into its buffer
    unsigned char *bsm = stage_buf(layer & 1);
    stage_layer(p.layers[layer], p.x + (size_t)layer * NB * d, NB, !chained || layer == 0, cta, G, d, r,
                s0, s1, p.staged != 0, p.p2_stride, reinterpret_cast<__half *>(bsm),
                reinterpret_cast<float *>(bsm + p.soff_c), reinterpret_cast<float *>(bsm + p.soff_b),
                reinterpret_cast<__half *>(bsm + p.soff_p1), bsm + p.soff_p2,
                FP8 ? reinterpret_cast<float *>(bsm + p.soff_su) : nullptr,
                FP8 && REGLU ? reinterpret_cast<float *>(bsm + p.soff_sg) : nullptr,
                FP8 ? reinterpret_cast<float *>(bsm + p.soff_sd) : nullptr, mbar0 + 8u * (uint32_t)(layer & 1), part);
  };

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar0));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(mbar0 + 8u));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // layer l's inputs go to buffer l & 1: layer 0's now, layer l + 1's during
  // layer l's logits (buffer (l + 1) & 1 is free once layer l has begun)
  if (tid == kIssuer) stage(0);
  // on a failed wait: let the stage copies this CTA may have in flight land
  auto drain = [&](int first, int last) {
    for (int k = first; k <= last && k < p.n_layers; ++k)
      mbar_wait(mbar0 + 8u * (uint32_t)(k & 1), (uint32_t)((k >> 1) & 1));
  };

  for (int l = 0; l < p.n_layers; ++l) {
    const pi::LayerDev &Ld = p.layers[l];
    PHASE_STAMP(l, 0);

    const uint32_t mbar = mbar0 + 8u * (uint32_t)(l & 1);
    const int n_hot = min(Ld.hot_per_slice, n_rows);
    if (!mbar_wait(mbar, (uint32_t)((l >> 1) & 1))) {
      if (tid == 0) atomicOr(status, PI_STATUS_BARRIER_TIMEOUT);
      drain(l, l);
      return;
    }
    unsigned char *bsm = stage_buf(l & 1);
    const __half *x_s = reinterpret_cast<const __half *>(bsm);
    const float *c_s = reinterpret_cast<const float *>(bsm + p.soff_c);
    const float *b_s = reinterpret_cast<const float *>(bsm + p.soff_b);
    // FP8 layers: row scales of the slice (up, gate for ReGLU, down^T)
    const float *sc_up = reinterpret_cast<const float *>(bsm + p.soff_su);
    const float *sc_gate = reinterpret_cast<const float *>(bsm + p.soff_sg);
    const float *sc_dn = reinterpret_cast<const float *>(bsm + p.soff_sd);
    const __half *p1_s = reinterpret_cast<const __half *>(bsm + p.soff_p1);
    const __half *p2_s = reinterpret_cast<const __half *>(bsm + p.soff_p2);
    uint4 xr[NB][CPT];
    if (chained && l > 0) {
      // x = fp16(y / RMS(y)) of the previous layer's y, complete since
      // barrier 3 (every CTA forms the whole vector in the same order, so all
      // agree bit for bit)
      const float *yp = p.y + (size_t)(l - 1) * NB * d;
      float yv[NB][CPT][8];
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        float ss = 0.f;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          const int v = tid + c * kThreads;
          float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
          if (v < nv) {
            a0 = ldcg(reinterpret_cast<const float4 *>(yp + (size_t)t * d) + 2 * v);
            a1 = ldcg(reinterpret_cast<const float4 *>(yp + (size_t)t * d) + 2 * v + 1);
          }
          yv[t][c][0] = a0.x; yv[t][c][1] = a0.y; yv[t][c][2] = a0.z; yv[t][c][3] = a0.w;
          yv[t][c][4] = a1.x; yv[t][c][5] = a1.y; yv[t][c][6] = a1.z; yv[t][c][7] = a1.w;
#pragma unroll
          for (int k = 0; k < 8; ++k) ss = fmaf(yv[t][c][k], yv[t][c][k], ss);
        }
        ss = pidev::warp_sum(ss);
        if (lane == 0) ss_s[wid][t] = ss;
      }
      __syncthreads();
#pragma unroll
      for (int t = 0; t < NB; ++t) {
        float sum = 0.f;
        for (int w2 = 0; w2 < kWarps; ++w2) sum += ss_s[w2][t];
        const float inv = 1.0f / sqrtf(sum / (float)d + 1e-12f);
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          __half2 hv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            hv[k] = __floats2half2_rn(yv[t][c][2 * k] * inv, yv[t][c][2 * k + 1] * inv);
          xr[t][c] = *reinterpret_cast<const uint4 *>(hv);
          const int v = tid + c * kThreads;
          if (cta == 0 && v < nv)           // the input this layer used, for the caller
            reinterpret_cast<uint4 *>(p.x_out + ((size_t)l * NB + t) * d)[v] = xr[t][c];
        }
      }
    } else {
#pragma unroll
      for (int t = 0; t < NB; ++t)
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          const int v = tid + c * kThreads;
          xr[t][c] = v < nv ? reinterpret_cast<const uint4 *>(x_s + (size_t)t * d)[v]
                            : make_uint4(0, 0, 0, 0);
        }
    }

    // ---------------- A: h = ReLU(W_p1 x), rows cta, cta + G, ... (2 rows per pass)
    for (int q0 = 0; cta + q0 * G < r; q0 += 2) {
      const bool two = cta + (q0 + 1) * G < r;   // uniform over the CTA
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (q == 1 && !two) break;
        const int k = cta + (q0 + q) * G;
        uint4 w[CPT];
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          const int v = tid + c * kThreads;
          if (v < nv)
            w[c] = p.staged ? reinterpret_cast<const uint4 *>(p1_s + (size_t)(q0 + q) * d)[v]
                            : pidev::ld_stream(reinterpret_cast<const uint4 *>(Ld.W_p1 + (size_t)k * d) + v);
          else
            w[c] = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int t = 0; t < NB; ++t) {
          float sum = 0.f;
#pragma unroll
          for (int c = 0; c < CPT; ++c) sum = pidev::dot8(sum, w[c], xr[t][c]);
          sum = pidev::warp_sum(sum);
          if (lane == 0) ared_s[wid][t][q] = sum;
        }
      }
      __syncthreads();
      if (tid < 2 * NB) {
        const int q = tid / NB, t = tid % NB;
        const int k = cta + (q0 + q) * G;
        if (k < r) {
          float sum = 0.f;
          for (int w2 = 0; w2 < kWarps; ++w2) sum += ared_s[w2][t][q];
          p.h[(size_t)t * r + k] = sum > 0.f ? sum : 0.f;
        }
      }
      __syncthreads();
    }
    PHASE_STAMP(l, 1);
    if (!grid_barrier(p.bar, ++epoch, status)) return;   // no copy in flight yet
    PHASE_STAMP(l, 2);

    // ---------------- C: logits over my slice, ordered local active list
    // Hot neurons (the leading places of the slice, from the offline profile)
    // fire on most tokens: start their rows towards L2 now, while HBM would
    // otherwise idle through the logits.  (Issued after barrier 1: a burst
    // before it slowed the barrier itself.)
    if (tid >= kIssuer && tid < kIssuer + n_hot) {
      const int i = s0 + tid - kIssuer;
      rowpf(Ld.R_up, i);
      if (REGLU) rowpf(Ld.R_gate, i);
      rowpf(Ld.R_dT, i);
    }
    // h into shared memory as [NB][2][r / 8] float4: elements 0-3 of each
    // 8-element group in the first half, 4-7 in the second, so that lanes
    // reading different groups hit distinct banks
    const int nvr = r >> 3;
    float4 *h4_s = reinterpret_cast<float4 *>(h_s);
    for (int e = tid; e < NB * (r >> 2); e += kThreads) {
      const int t = e / (r >> 2), g4 = e - t * (r >> 2);
      h4_s[t * 2 * nvr + (g4 & 1) * nvr + (g4 >> 1)] = ldcg(reinterpret_cast<const float4 *>(p.h) + e);
    }
    __syncthreads();
    PHASE_STAMP(l, 9);
    // the next layer's inputs go to the other buffer (free since barrier 1):
    // issued here by the last warp, which has no logits rows to compute when
    // the slice needs fewer than 16 warps
    if (p.staged && p.mma_logits && l + 1 < p.n_layers) {
      // two issuing warps (14 and 15 have no logits rows): the last warp sets
      // the stage's byte expectation and copies the small pieces, warp 14
      // the W_p2 slice once the expectation is set (named barrier 1)
      if (wid == kWarps - 1) {
        if (lane == 0) {
          const uint32_t mb = mbar0 + 8u * (uint32_t)((l + 1) & 1);
          const uint32_t tot = stage_total(l + 1);
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(tot) : "memory");
        }
        __syncwarp();
        asm volatile("bar.arrive 1, 64;" ::: "memory");
        if (lane == 0) stage(l + 1, 1);
      } else if (wid == kWarps - 2) {
        asm volatile("bar.sync 1, 64;" ::: "memory");
        if (lane == 0) stage(l + 1, 2);
      }
    } else if (tid == kIssuer && l + 1 < p.n_layers) {
      stage(l + 1);
    }
    if (p.staged && p.mma_logits) {
      // W_p2 slice in shared memory (padded rows) on the tensor cores: warp m
      // takes rows [16m, 16m + 16) as the A tile (m16n8k16, fp16); B holds h
      // as fp16 pairs, column 2t = hi and 2t + 1 = lo of token t, so that the
      // logit is D[row][2t] + D[row][2t + 1] (binary32 accumulation).  The k
      // order is permuted (lane c of a quad reads 8 consecutive elements of a
      // 32-element block, for two k-steps); A and B use the same permutation.
      const int g = lane >> 2, c4 = lane & 3;
      const int ntile = (n_rows + 15) >> 4;
      const unsigned char *p2b = reinterpret_cast<const unsigned char *>(p2_s);
      for (int m = wid; m < ntile; m += kWarps) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const unsigned char *ra = p2b + (size_t)(16 * m + g) * p.p2_stride + c4 * 16;
        const unsigned char *rb = ra + (size_t)8 * p.p2_stride;
        const int tb = g >> 1;                  // token of this lane's B column (valid when g < 2 NB)
        for (int sp = 0; sp < (r >> 5); ++sp) {
          const uint4 wa = *reinterpret_cast<const uint4 *>(ra + sp * 64);
          const uint4 wb = *reinterpret_cast<const uint4 *>(rb + sp * 64);
          uint32_t b[4] = {0u, 0u, 0u, 0u};
          if (g < 2 * NB) {
            // 8 consecutive h values: elements 0-3 of group 4 sp + c4 in the
            // first half of h4_s, 4-7 in the second
            const float4 h0 = h4_s[tb * 2 * nvr + 4 * sp + c4], h1 = h4_s[tb * 2 * nvr + nvr + 4 * sp + c4];
            const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
            __half pk[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              __half hi, lo;
              f32_to_pair(hv[j], hi, lo);
              pk[j] = (g & 1) ? lo : hi;
            }
            b[0] = pack_h2(pk[0], pk[1]); b[1] = pack_h2(pk[2], pk[3]);
            b[2] = pack_h2(pk[4], pk[5]); b[3] = pack_h2(pk[6], pk[7]);
          }
          mma_16816(acc, wa.x, wb.x, wa.y, wb.y, b[0], b[1]);
          mma_16816(acc, wa.z, wb.z, wa.w, wb.w, b[2], b[3]);
        }
        // lane (g, c4) holds D[g][2 c4 + {0,1}] in acc[0..1] and D[g + 8][...]
        // in acc[2..3]: token c4's hi and lo for rows g and g + 8
        bool on_a = false, on_b = false;
        const int row_a = 16 * m + g, row_b = row_a + 8;
        if (c4 < NB) {
          on_a = row_a < n_rows && (acc[0] + acc[1]) + c_s[s0 + row_a - s0a] > 0.f;
          on_b = row_b < n_rows && (acc[2] + acc[3]) + c_s[s0 + row_b - s0a] > 0.f;
        }
        if (NB == 2) {                          // union over the two tokens (lanes c4 = 0, 1)
          on_a |= __shfl_xor_sync(0xffffffffu, on_a ? 1 : 0, 1) != 0;
          on_b |= __shfl_xor_sync(0xffffffffu, on_b ? 1 : 0, 1) != 0;
        }
        if (c4 == 0) {
          if (row_a < n_rows) flag_s[row_a] = on_a ? 1 : 0;
          if (row_b < n_rows) flag_s[row_b] = on_b ? 1 : 0;
        }
      }
    } else if (p.staged) {
      // W_p2 slice in shared memory: 2^lgt_s threads per row, each summing
      // r / 8 / 2^lgt_s of the row's 16-byte vectors; a row's visiting order
      // is rotated by its place within the quarter-warp so that the 16-byte
      // reads of a quarter-warp fall on distinct banks
      const int lgT = p.lgt_s, T = 1 << lgT;
      const int nk = nvr >> lgT;                 // vectors per thread
      const int rpp = kThreads >> lgT;           // rows per pass
      const int rr = tid >> lgT, sub = tid & (T - 1);
      const int rot = (rr & ((8 >> lgT) - 1)) % nk;
      for (int rb = 0; rb < n_rows; rb += rpp) {
        if (rb + ((wid * 32) >> lgT) >= n_rows) break;   // no row of this warp in this pass or later
        const int rl = rb + rr;
        const bool valid = rl < n_rows;
        const uint4 *wrow = reinterpret_cast<const uint4 *>(p2_s + (size_t)(valid ? rl : 0) * p2_ld);
        float a4[NB][4];
#pragma unroll
        for (int t = 0; t < NB; ++t)
#pragma unroll
          for (int q = 0; q < 4; ++q) a4[t][q] = 0.f;
        int kk = rot;
#pragma unroll 4
        for (int k = 0; k < nk; ++k) {
          const int v = sub + (kk << lgT);
          const uint4 wv = wrow[v];
          const __half2 *wh = reinterpret_cast<const __half2 *>(&wv);
          const float2 w0 = __half22float2(wh[0]), w1 = __half22float2(wh[1]);
          const float2 w2 = __half22float2(wh[2]), w3 = __half22float2(wh[3]);
#pragma unroll
          for (int t = 0; t < NB; ++t) {
            const float4 h0 = h4_s[t * 2 * nvr + v], h1 = h4_s[t * 2 * nvr + nvr + v];
            a4[t][0] = fmaf(w0.x, h0.x, fmaf(w0.y, h0.y, a4[t][0]));
            a4[t][1] = fmaf(w1.x, h0.z, fmaf(w1.y, h0.w, a4[t][1]));
            a4[t][2] = fmaf(w2.x, h1.x, fmaf(w2.y, h1.y, a4[t][2]));
            a4[t][3] = fmaf(w3.x, h1.z, fmaf(w3.y, h1.w, a4[t][3]));
          }
          kk = kk + 1 == nk ? 0 : kk + 1;
        }
        bool on = false;
#pragma unroll
        for (int t = 0; t < NB; ++t) {
          float sl = (a4[t][0] + a4[t][1]) + (a4[t][2] + a4[t][3]);
          for (int o = T >> 1; o > 0; o >>= 1) sl += __shfl_xor_sync(0xffffffffu, sl, o);
          on |= valid && sl + c_s[s0 + rl - s0a] > 0.f;
        }
        if (sub == 0 && valid) flag_s[rl] = on ? 1 : 0;
      }
    } else {
      const int GL = p.lanes_l;                 // lanes per predictor row (8, 16, 32)
      const int rows_per_warp = 32 / GL;
      const int sub = lane % GL;
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
            if (it0 + u < iters && rl < n_rows)
              wv[u] = p.staged ? reinterpret_cast<const uint4 *>(p2_s + (size_t)rl * p2_ld)[v]
                               : pidev::ld_stream(reinterpret_cast<const uint4 *>(Ld.W_p2 + (size_t)(s0 + rl) * p2_ld) + v);
            else
              wv[u] = make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int t = 0; t < NB; ++t) {
            const float4 h0 = h4_s[t * 2 * nvr + v], h1 = h4_s[t * 2 * nvr + nvr + v];
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
        // reduce-scatter of the 8 rows' partial sums over the GL lanes of the
        // row group: 3 halving exchanges leave each lane one row (bits o1, o2,
        // o3 of the lane pick it), then a plain reduction over the low bits.
        const int o1 = GL >> 1, o2 = GL >> 2, o3 = GL >> 3;
        const bool b1 = (lane & o1) != 0, b2 = (lane & o2) != 0, b3 = (lane & o3) != 0;
        bool on = false;
#pragma unroll
        for (int t = 0; t < NB; ++t) {
          float k4[4], k2[2];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float mine = b1 ? acc[j + 4][t] : acc[j][t];
            const float oth = b1 ? acc[j][t] : acc[j + 4][t];
            k4[j] = mine + __shfl_xor_sync(0xffffffffu, oth, o1);
          }
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float mine = b2 ? k4[j + 2] : k4[j];
            const float oth = b2 ? k4[j] : k4[j + 2];
            k2[j] = mine + __shfl_xor_sync(0xffffffffu, oth, o2);
          }
          float k1 = (b3 ? k2[1] : k2[0]) + __shfl_xor_sync(0xffffffffu, b3 ? k2[0] : k2[1], o3);
          for (int o = o3 >> 1; o > 0; o >>= 1) k1 += __shfl_xor_sync(0xffffffffu, k1, o);
          const int u = (b1 ? 4 : 0) + (b2 ? 2 : 0) + (b3 ? 1 : 0);
          const int rl = ((it0 + u) * kWarps + wid) * rows_per_warp + lane / GL;
          if (it0 + u < iters && rl < n_rows) on |= (k1 + c_s[s0 + rl - s0a]) > 0.f;
        }
        {
          const int u = (b1 ? 4 : 0) + (b2 ? 2 : 0) + (b3 ? 1 : 0);
          const int rl = ((it0 + u) * kWarps + wid) * rows_per_warp + lane / GL;
          if ((lane & (o3 - 1)) == 0 && it0 + u < iters && rl < n_rows) flag_s[rl] = on ? 1 : 0;
        }
      }
    }
    __syncthreads();
    PHASE_STAMP(l, 10);
    int lcount = 0;
    {
      for (int c0 = 0; c0 < n_rows; c0 += kThreads) {
        const int i = c0 + tid;
        const bool on = i < n_rows && flag_s[i];
        const unsigned bal = __ballot_sync(0xffffffffu, on);
        if (lane == 0) wtot_s[wid] = __popc(bal);
        __syncthreads();
        int wpre = 0, tot = 0;
        for (int q = 0; q < kWarps; ++q) {
          const int v = wtot_s[q];
          if (q < wid) wpre += v;
          tot += v;
        }
        if (on) list_s[lcount + wpre + __popc(bal & ((1u << lane) - 1u))] = s0 + i;
        lcount += tot;
        __syncthreads();
      }
      PHASE_STAMP(l, 11);
      // ask L2 for all my active rows now (within the prefetch budget).  A
      // list past the budget on an unstaged layer instead has only its down
      // rows asked for, by every thread as the row phase starts: the bulk
      // prefetches of a long list would hold the last warp (and the row phase
      // behind it) for microseconds, while the up rows are loaded first
      // thing in the row phase anyway.
      const bool heavy = !p.staged && lcount > p.pf_rows;
      const int npf = heavy ? 0 : min(lcount, p.pf_rows);
      if (tid >= kIssuer)
        for (int j = tid - kIssuer; j < npf; j += 32) {
          const int i = list_s[j];
          if (i - s0 < n_hot) continue;        // requested after the first barrier
          rowpf(Ld.R_up, i);
          if (REGLU) rowpf(Ld.R_gate, i);
          rowpf(Ld.R_dT, i);
        }
      for (int j = tid; j < lcount; j += kThreads) lb_s[j] = b_s[list_s[j] - s0a];
      if (p.mask_out)
        for (int i = tid; i < n_rows; i += kThreads) p.mask_out[(size_t)l * ffn + s0 + i] = flag_s[i];
      if (tid == 0) p.cnt[cta] = lcount;
    }
    __syncthreads();
    PHASE_STAMP(l, 3);
    CTA_E_BEGIN(l);

    // ---------------- E: up (+gate) and down rows of my active neurons, in
    // windows of one pass or in two passes (kOnePass).
    float acc[NB][CPT][8];
#pragma unroll
    for (int t = 0; t < NB; ++t)
#pragma unroll
      for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[t][c][e] = 0.f;
    if (lcount > p.pf_rows) {
      if (!p.staged) {                          // a long list (above): its down rows
        for (int j = tid; j < lcount; j += kThreads) {
          const int i = list_s[j];
          if (i - s0 >= n_hot) rowpf(Ld.R_dT, i);
        }
      } else {                                  // rows past the early-prefetch budget
        for (int j = p.pf_rows + tid; j < lcount; j += kThreads) {
          const int i = list_s[j];
          rowpf(Ld.R_up, i);
          if (REGLU) rowpf(Ld.R_gate, i);
          rowpf(Ld.R_dT, i);
        }
      }
    }
    if constexpr (kOnePass) {
    // One pass of windows: a window's up (+gate) and down rows are requested
    // together, so a window costs one memory round trip.
    for (int w0 = 0; w0 < lcount; w0 += GW) {
      const int n_here = min(GW, lcount - w0);
      RowVec wu[GW][NR][CPT], wd[GW][CPT];
#pragma unroll
      for (int n = 0; n < GW; ++n) {
        const int i = n < n_here ? list_s[w0 + n] : -1;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          const int v = tid + c * kThreads;
          const bool ok = i >= 0 && v < nv;
          wu[n][0][c] = ok ? ldrow(Ld.R_up, i, v) : RowVec{};
          if (REGLU) wu[n][NR - 1][c] = ok ? ldrow(Ld.R_gate, i, v) : RowVec{};
          wd[n][c] = ok ? ldrow(Ld.R_dT, i, v) : RowVec{};
        }
      }
#pragma unroll
      for (int n = 0; n < GW; ++n)
#pragma unroll
        for (int q = 0; q < NR; ++q)
#pragma unroll
          for (int t = 0; t < NB; ++t) {
            float sdot = 0.f;
#pragma unroll
            for (int c = 0; c < CPT; ++c) sdot = rowdot(sdot, wu[n][q][c], xr[t][c]);
            sdot = pidev::warp_sum(sdot);
            if (lane == 0) red_s[wid][t][q][n] = sdot;
          }
      __syncthreads();
      if (tid < NB * GW) {
        const int t = tid / GW, n = tid % GW;
        if (n < n_here) {
          const float bi = lb_s[w0 + n];
          float su = 0.f, sg = 0.f;
          for (int q = 0; q < kWarps; ++q) {   // fixed order over warps
            su += red_s[q][t][0][n];
            if (REGLU) sg += red_s[q][t][NR - 1][n];
          }
          if (FP8) {                           // row scales (staged slices)
            const int k = list_s[w0 + n] - s0a;
            su *= sc_up[k];
            if (REGLU) sg *= sc_gate[k];
          }
          float a;
          if (REGLU) {
            const float gz = sg + bi;
            a = pidev::gate_act(gz, p.gate_silu != 0) * su;
          } else {
            const float z = su + bi;
            a = z > 0.f ? z : 0.f;
          }
          a_all[t * p.slice_pad + w0 + n] = a;
        }
      }
      __syncthreads();   // a of the window visible; red_s free for the next window
#pragma unroll
      for (int n = 0; n < GW; ++n) {
        if (n < n_here) {
#pragma unroll
          for (int t = 0; t < NB; ++t) {
            float an = a_all[t * p.slice_pad + w0 + n];
            if (FP8) an *= sc_dn[list_s[w0 + n] - s0a];
#pragma unroll
            for (int c = 0; c < CPT; ++c) rowaxpy(acc[t][c], an, wd[n][c]);
          }
        }
      }
    }
    } else {
    // Two passes: all up-row dot products (a into shared memory), then all
    // down rows, which were asked of L2 at the end of phase C and arrive
    // while the up pass runs.
    for (int w0 = 0; w0 < lcount; w0 += GU) {
      const int n_here = min(GU, lcount - w0);
      RowVec wu[GU][NR][CPT];
#pragma unroll
      for (int n = 0; n < GU; ++n) {
        const int i = n < n_here ? list_s[w0 + n] : -1;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          const int v = tid + c * kThreads;
          const bool ok = i >= 0 && v < nv;
          wu[n][0][c] = ok ? ldrow(Ld.R_up, i, v) : RowVec{};
          if (REGLU) wu[n][NR - 1][c] = ok ? ldrow(Ld.R_gate, i, v) : RowVec{};
        }
      }
#pragma unroll
      for (int n = 0; n < GU; ++n)
#pragma unroll
        for (int q = 0; q < NR; ++q)
#pragma unroll
          for (int t = 0; t < NB; ++t) {
            float sdot = 0.f;
#pragma unroll
            for (int c = 0; c < CPT; ++c) sdot = rowdot(sdot, wu[n][q][c], xr[t][c]);
            sdot = pidev::warp_sum(sdot);
            if (lane == 0) red_s[wid][t][q][n] = sdot;
          }
      __syncthreads();
      if (tid < NB * GU) {
        const int t = tid / GU, n = tid % GU;
        if (n < n_here) {
          const float bi = lb_s[w0 + n];
          float su = 0.f, sg = 0.f;
          for (int q = 0; q < kWarps; ++q) {   // fixed order over warps
            su += red_s[q][t][0][n];
            if (REGLU) sg += red_s[q][t][NR - 1][n];
          }
          if (FP8) {                           // row scales (staged slices)
            const int k = list_s[w0 + n] - s0a;
            su *= sc_up[k];
            if (REGLU) sg *= sc_gate[k];
          }
          float a;
          if (REGLU) {
            const float gz = sg + bi;
            a = pidev::gate_act(gz, p.gate_silu != 0) * su;
          } else {
            const float z = su + bi;
            a = z > 0.f ? z : 0.f;
          }
          a_all[t * p.slice_pad + w0 + n] = a;
        }
      }
      __syncthreads();   // red_s is rewritten by the next window
    }
    for (int w0 = 0; w0 < lcount; w0 += GD) {
      const int n_here = min(GD, lcount - w0);
      RowVec wd[GD][CPT];
#pragma unroll
      for (int n = 0; n < GD; ++n) {
        const int i = n < n_here ? list_s[w0 + n] : -1;
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
          const int v = tid + c * kThreads;
          wd[n][c] = (i >= 0 && v < nv) ? ldrow(Ld.R_dT, i, v) : RowVec{};
        }
      }
#pragma unroll
      for (int n = 0; n < GD; ++n) {
        if (n < n_here) {
#pragma unroll
          for (int t = 0; t < NB; ++t) {
            float an = a_all[t * p.slice_pad + w0 + n];
            if (FP8) an *= sc_dn[list_s[w0 + n] - s0a];
#pragma unroll
            for (int c = 0; c < CPT; ++c) rowaxpy(acc[t][c], an, wd[n][c]);
          }
        }
      }
    }
    }
    PHASE_STAMP(l, 4);
    CTA_E_END(l, lcount);
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
    PHASE_STAMP(l, 5);
    if (!grid_barrier(p.bar, ++epoch, status)) {
      drain(l + 1, l + 1);
      return;
    }
    PHASE_STAMP(l, 6);

    // ---------------- F: y = sum of partials.  Columns (float4) c = cta*8 + j
    // (+ G*8 per pass); thread (j, g): j = tid / 64 column, g = tid % 64 split
    // group summing splits g, g+64, ... in order; then a fixed shuffle tree
    // over the 32 lanes of each warp, and the two warps of a column in order.
    if (cta == 0 && p.count && wid == 0) {
      int cv[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) cv[q] = q * 32 + lane < G ? ldcg(p.cnt + q * 32 + lane) : 0;
      int s = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) s += cv[q];
      for (int c = 256 + lane; c < G; c += 32) s += ldcg(p.cnt + c);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) p.count[l] = s;
    }
    {
      const int n4 = NB * d / 4;
      const int j = tid >> 6, g = tid & 63;
      float *y = p.y + (size_t)l * NB * d;
      const float4 *pp = reinterpret_cast<const float4 *>(p.partial);
      for (int c0 = cta * 8; c0 < n4; c0 += G * 8) {
        const int c = c0 + j;
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c < n4) {
          constexpr int kPR = 4;
          for (int sp0 = g; sp0 < G; sp0 += 64 * kPR) {
            float4 v[kPR];
#pragma unroll
            for (int q = 0; q < kPR; ++q) {
              const int sp = sp0 + q * 64;
              v[q] = sp < G ? ldcg(pp + (size_t)sp * n4 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int q = 0; q < kPR; ++q) {
              s.x += v[q].x; s.y += v[q].y; s.z += v[q].z; s.w += v[q].w;
            }
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          s.x += __shfl_xor_sync(0xffffffffu, s.x, o);
          s.y += __shfl_xor_sync(0xffffffffu, s.y, o);
          s.z += __shfl_xor_sync(0xffffffffu, s.z, o);
          s.w += __shfl_xor_sync(0xffffffffu, s.w, o);
        }
        if (lane == 0) fred_s[(tid >> 5) & 1][j] = s;
        __syncthreads();
        if (g == 0 && c < n4) {
          const float4 a0 = fred_s[0][j], a1 = fred_s[1][j];
          reinterpret_cast<float4 *>(y)[c] = make_float4(a0.x + a1.x, a0.y + a1.y, a0.z + a1.z, a0.w + a1.w);
        }
        __syncthreads();
      }
    }
    PHASE_STAMP(l, 7);
    if (!grid_barrier(p.bar, ++epoch, status)) {
      drain(l + 1, l + 1);
      return;
    }
    PHASE_STAMP(l, 8);
  }
  // chained across launches: the input of the layer after this launch
  if (chained && p.x_next && cta == 0 && p.n_layers > 0) {
    const float *yp = p.y + (size_t)(p.n_layers - 1) * NB * d;
#pragma unroll
    for (int t = 0; t < NB; ++t) {
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        const int v = tid + c * kThreads;
        if (v < nv)
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float yk = ldcg(yp + (size_t)t * d + 8 * v + k);
            ss = fmaf(yk, yk, ss);
          }
      }
      ss = pidev::warp_sum(ss);
      if (lane == 0) ss_s[wid][t] = ss;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < NB; ++t) {
      float sum = 0.f;
      for (int w2 = 0; w2 < kWarps; ++w2) sum += ss_s[w2][t];
      const float inv = 1.0f / sqrtf(sum / (float)d + 1e-12f);
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        const int v = tid + c * kThreads;
        if (v < nv) {
          __half2 hv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k)
            hv[k] = __floats2half2_rn(ldcg(yp + (size_t)t * d + 8 * v + 2 * k) * inv,
                                      ldcg(yp + (size_t)t * d + 8 * v + 2 * k + 1) * inv);
          reinterpret_cast<uint4 *>(p.x_next + (size_t)t * d)[v] = *reinterpret_cast<const uint4 *>(hv);
        }
      }
    }
  }
}

#ifdef PI_PHASE_TIMING
}  // namespace
extern "C" int pi_debug_phase_times(unsigned long long *out) {
  return (int)cudaMemcpyFromSymbol(out, g_phase_ts, sizeof(g_phase_ts));
}
extern "C" int pi_debug_cta_e(unsigned long long *out) {
  return (int)cudaMemcpyFromSymbol(out, g_cta_e, sizeof(g_cta_e));
}
namespace {
#endif

template <int CPT, int NB, bool REGLU, bool FP8>
cudaError_t launch_step(const pi::StackParams &p, size_t smem, cudaStream_t s) {
  auto kern = k_stack_step<CPT, NB, REGLU, FP8>;
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

template <int NB, bool REGLU, bool FP8>
cudaError_t dispatch_step(const pi::StackParams &p, size_t smem, cudaStream_t s) {
  const int cpt = (p.d / 8 + kThreads - 1) / kThreads;
  switch (cpt) {
    case 1: return launch_step<1, NB, REGLU, FP8>(p, smem, s);
    case 2: return launch_step<2, NB, REGLU, FP8>(p, smem, s);
    case 3: return launch_step<3, NB, REGLU, FP8>(p, smem, s);
    case 4: return launch_step<4, NB, REGLU, FP8>(p, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

constexpr size_t kSmemBudget = 200 * 1024;   // dynamic shared memory the step may use

size_t align128(size_t v) { return (v + 127) & ~(size_t)127; }
size_t align16(size_t v) { return (v + 15) & ~(size_t)15; }

struct SmemPlan {
  size_t off_flag, off_list, off_lb, off_a, off_stage;   // absolute offsets
  size_t soff_c, soff_b, soff_p1, soff_p2;              // offsets inside a stage buffer
  size_t soff_su, soff_sg, soff_sd;                      // FP8 row-scale slices (empty for fp16)
  size_t stage_small, stage_full;                        // buffer size without / with predictor
  size_t base_end;
};

// The staged logits run on the tensor cores when the rank is a multiple of 64
// (the stored W_p2 rows are then padded, see pi::p2_ld_for); the staged slice
// is allocated in whole 16-row tiles (the last tile reads, and ignores, rows
// past the slice).
bool mma_logits(const pi_layer *L) { return L->rank % 64 == 0 && L->p2_ld == L->rank + 32; }
int p2_stride(const pi_layer *L) { return L->p2_ld * 2; }
size_t p2_rows(const pi_layer *L) {
  const size_t slice = (size_t)pi::step_slice(L);
  return mma_logits(L) ? (slice + 15) / 16 * 16 : slice;
}

SmemPlan smem_plan(const pi_layer *L, int B) {
  const int G = pi::step_grid(L);
  const size_t slice = (size_t)pi::step_slice(L);
  const size_t na_max = (size_t)(L->rank + G - 1) / G;
  SmemPlan s;
  size_t off = align128(sizeof(float) * (size_t)B * L->rank);   // h
  s.off_flag = off;  off = align128(off + slice);
  s.off_list = off;  off = align128(off + sizeof(int) * slice);
  s.off_lb = off;    off = align128(off + sizeof(float) * slice);
  s.off_a = off;     off = align128(off + sizeof(float) * (size_t)B * align16(slice));
  s.off_stage = off;
  s.base_end = off;
  size_t so = align128(2 * (size_t)B * L->d);                     // x
  s.soff_c = so;     so = align128(so + sizeof(float) * (slice + 8));
  s.soff_b = so;     so = align128(so + sizeof(float) * (slice + 8));
  const bool q8 = L->row_format == PI_ROWS_FP8_E4M3;
  const size_t sc = q8 ? sizeof(float) * (slice + 8) : 0;
  s.soff_su = so;    so = align128(so + sc);
  s.soff_sg = so;    so = align128(so + (L->act != PI_ACT_RELU ? sc : 0));
  s.soff_sd = so;    so = align128(so + sc);
  s.stage_small = so;
  s.soff_p1 = so;    so = align128(so + na_max * L->d * 2);
  s.soff_p2 = so;    so = align128(so + p2_rows(L) * (size_t)p2_stride(L));
  s.stage_full = so;
  return s;
}

}  // namespace

namespace pi {

int step_grid(const pi_layer *L) { return L->num_sms; }

int step_slice(const pi_layer *L) { return (L->ffn + step_grid(L) - 1) / step_grid(L); }

bool step_staged(const pi_layer *L, int B) {
  const SmemPlan s = smem_plan(L, B);
  return s.base_end + 2 * s.stage_full <= kSmemBudget;
}

size_t step_smem(const pi_layer *L, int B) {
  const SmemPlan s = smem_plan(L, B);
  return s.base_end + 2 * (step_staged(L, B) ? s.stage_full : s.stage_small);
}

cudaError_t run_stack(pi_layer *const *layers, int n, const __half *x, int B, int32_t *idx,
                      int32_t *count, float *y, const WsLayout &w, char *ws, cudaStream_t s,
                      bool chained, __half *x_out, __half *x_next) {
  const pi_layer *L0 = layers[0];
  const SmemPlan sp = smem_plan(L0, B);
  StackParams p = {};
  p.n_layers = n;
  p.d = L0->d;
  p.ffn = L0->ffn;
  p.rank = L0->rank;
  p.G = step_grid(L0);
  p.staged = step_staged(L0, B) ? 1 : 0;
  p.off_flag = (int)sp.off_flag;
  p.off_list = (int)sp.off_list;
  p.off_lb = (int)sp.off_lb;
  p.off_a = (int)sp.off_a;
  p.slice_pad = (int)align16((size_t)step_slice(L0));
  p.off_stage = (int)sp.off_stage;
  p.stage_bytes = (int)(p.staged ? sp.stage_full : sp.stage_small);
  p.soff_c = (int)sp.soff_c;
  p.soff_b = (int)sp.soff_b;
  p.soff_p1 = (int)sp.soff_p1;
  p.soff_p2 = (int)sp.soff_p2;
  p.soff_su = (int)sp.soff_su;
  p.soff_sg = (int)sp.soff_sg;
  p.soff_sd = (int)sp.soff_sd;
  int GL = 32;
  while (GL > 8 && GL * 8 > L0->rank) GL >>= 1;
  p.lanes_l = GL;
  // staged logits: the most threads per W_p2 row (up to 8, dividing r / 8)
  // that still cover the slice in one pass of the CTA
  int lgt = 0;
  while (lgt < 3 && (step_slice(L0) << (lgt + 1)) <= kThreads && ((L0->rank >> 3) % (2 << lgt)) == 0) ++lgt;
  p.lgt_s = lgt;
  p.mma_logits = mma_logits(L0) ? 1 : 0;
  p.p2_stride = p2_stride(L0);
  const int rows_per_neuron = L0->act != PI_ACT_RELU ? 3 : 2;
  // early L2 prefetch of the local active rows: up to ~768 KB of rows per CTA
  const int rb = L0->row_format == PI_ROWS_FP8_E4M3 ? L0->d : 2 * L0->d;   // bytes of a gathered row
  const int pf = (768 * 1024) / (rb * rows_per_neuron);
  p.pf_rows = pf < 1 ? 1 : pf;
  p.chained = chained ? 1 : 0;
  p.x = x;
  p.x_out = chained ? x_out : nullptr;
  p.x_next = chained ? x_next : nullptr;
  p.y = y;
  p.count = count;
  p.mask_out = idx ? reinterpret_cast<uint8_t *>(ws + w.mask) : nullptr;
  p.h = reinterpret_cast<float *>(ws + w.h);
  p.cnt = reinterpret_cast<int32_t *>(ws + w.cnt);
  p.partial = reinterpret_cast<float *>(ws + w.partial);
  p.bar = reinterpret_cast<unsigned *>(ws + w.bar);
  p.status = L0->status;
  for (int l = 0; l < n; ++l) {
    const pi_layer *Ll = layers[l];
    // the k-th neuron of the caller's order sits at slice k % G, place k / G:
    // the first n_hot of them fill places 0 .. ceil(n_hot / G) - 1 of the slices
    const int hot = (Ll->n_hot + p.G - 1) / p.G;
    const bool q8 = Ll->row_format == PI_ROWS_FP8_E4M3;
    p.layers[l] = LayerDev{Ll->W_p1, Ll->W_p2,
                           q8 ? static_cast<const void *>(Ll->Q_up) : Ll->W_up,
                           q8 ? static_cast<const void *>(Ll->Q_gate) : Ll->W_gate,
                           q8 ? static_cast<const void *>(Ll->Q_dT) : Ll->W_dT,
                           Ll->s_up, Ll->s_gate, Ll->s_dT, Ll->b, Ll->c_p, hot};
  }
  cudaError_t e = cudaMemsetAsync(p.bar, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const size_t smem = step_smem(L0, B);
  const bool reglu = L0->act != PI_ACT_RELU;      // gated: ReGLU or SwiGLU
  p.gate_silu = L0->act == PI_ACT_SWIGLU ? 1 : 0;
  const bool q8 = L0->row_format == PI_ROWS_FP8_E4M3;
  e = record_hook(L0->ev_before, s);
  if (e != cudaSuccess) return e;
  if (B == 1)
    e = q8 ? (reglu ? dispatch_step<1, true, true>(p, smem, s) : dispatch_step<1, false, true>(p, smem, s))
           : (reglu ? dispatch_step<1, true, false>(p, smem, s) : dispatch_step<1, false, false>(p, smem, s));
  else
    e = q8 ? (reglu ? dispatch_step<2, true, true>(p, smem, s) : dispatch_step<2, false, true>(p, smem, s))
           : (reglu ? dispatch_step<2, true, false>(p, smem, s) : dispatch_step<2, false, false>(p, smem, s));
  if (e != cudaSuccess) return e;
  e = record_hook(L0->ev_after, s);
  if (e != cudaSuccess) return e;
  if (idx) {
    // ascending active lists (and counts) from the per-layer masks
    e = run_compact_layers(L0, p.mask_out, n, idx, count, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pi
