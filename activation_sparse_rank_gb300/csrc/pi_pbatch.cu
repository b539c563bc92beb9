// Batched activation predictor in one cooperative launch (3 <= B <= 32).
//
// "PowerInfer: Fast Large Language Model Serving with a Consumer-grade GPU"
// (egguo-blog reading report), section 2.3, core module 3 (a small MLP per
// layer predicts which neurons fire) and section 4.4, limitation 3 (with a
// batch the active set is the union over its tokens):
//   h[b, k]  = ReLU(sum_j W_p1[k, j] x[b, j])
//   l[b, i]  = sum_k W_p2[i, k] h[b, k] + c_p[i]      (c_p = 0 when absent)
//   i active = l[b, i] > 0 for some token b;  idx = active i ascending, count.
//
// One CTA per SM, four phases separated by grid barriers:
//   1. partial hidden layer: CTA (row group, K chunk) multiplies its rows of
//      W_p1 by its chunk of x on the tensor cores (mma.sync m16n8k16, fp16
//      operands, binary32 accumulation) and stores the partial sums;
//   2. each CTA adds the partials of its share of h in a fixed order, applies
//      ReLU and stores h as an fp16 pair (hi = fp16(h), lo = fp16(h - hi));
//   3. each CTA copies h into shared memory and forms the logits of its
//      slice of neurons on the tensor cores (B operand column 2b = hi and
//      2b + 1 = lo of token b, so a logit is D[2b] + D[2b + 1] + c_p), takes
//      the union over the batch and lists its active neurons in order;
//   4. each CTA writes its list after the counts of the CTAs before it (the
//      slices are ascending ranges, so the whole list is ascending).
// The slice's W_p2 rows are asked of L2 when the kernel starts, so phase 3
// reads them from L2 while phases 1 and 2 run.  Every sum has a fixed order
// (deterministic); barrier waits are bounded and set a status bit.
//
// The k order of each 32-element block is permuted the same way in both
// operands of every mma: lane c of a quad takes 8 consecutive elements with
// one 16-byte load and uses them for two k-steps (elements 0-3 for the
// first, 4-7 for the second).  Shared-memory rows sit 64 bytes off a
// multiple of 128 bytes, so the 16-byte loads of a quarter-warp (two rows,
// four lanes each) fall on distinct banks.
#include <cmath>

#include "pi_internal.cuh"

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kSpinLimit = 1u << 22;   // polls before a barrier wait gives up
constexpr size_t kSmemBudget = 200 * 1024;

struct PBParams {
  const __half *x;          // [B, d]
  const __half *W_p1;       // [r, d]
  const __half *W_p2;       // [ffn, p2_ld]
  const float *c_p;         // [ffn] or nullptr
  int B, d, r, ffn, p2_ld;
  int NKC, KC, RS, RG;      // K chunks, chunk length, rows per row group, row groups
  int xs_stride, hs_stride; // bytes between the rows of x / h in shared memory
  int off_flag, off_list;   // shared-memory offsets of the slice's flags and list
  float *partial;           // [NKC, B, r]
  __half *hbuf;             // [2B, r]
  uint8_t *mask;            // [ffn] or nullptr
  int32_t *cnt;             // [G]
  int32_t *idx;             // [ffn]
  int32_t *count;
  unsigned *bar;
  unsigned *status;
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// All CTAs of the grid arrive; returns false (status bit set) if the wait ran out.
__device__ bool grid_sync(unsigned *bar, unsigned target, unsigned *status) {
  __shared__ int ok_s;
  __syncthreads();
  if (threadIdx.x == 0) {
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(bar) : "memory");
    int ok = 1;
    unsigned it = 0;
    while ((int)(ld_acquire_gpu(bar) - target) < 0)
      if (++it > kSpinLimit) {
        atomicOr(status, PI_STATUS_BARRIER_TIMEOUT);
        ok = 0;
        break;
      }
    ok_s = ok;
  }
  __syncthreads();
  return ok_s != 0;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// NT: n tiles of the logits (8 columns = the hi / lo pairs of 4 tokens), B <= 4 NT.
template <int NT>
__global__ void __launch_bounds__(kThreads, 1) k_predict_batch(const __grid_constant__ PBParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int NT1 = (NT + 1) / 2;           // n tiles of the hidden layer (8 tokens each)
  __shared__ float red_s[kThreads];
  __shared__ int wtot_s[kWarps];
  __shared__ int pre_s;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int G = gridDim.x, cta = blockIdx.x;
  const int B = p.B, d = p.d, r = p.r;
  // this CTA's neuron slice [s0, s0 + n_rows): ascending, sizes differ by at most one
  const int q_sl = p.ffn / G, r_sl = p.ffn % G;
  const int s0 = cta * q_sl + min(cta, r_sl);
  const int n_rows = q_sl + (cta < r_sl ? 1 : 0);
  if (tid == 0 && n_rows > 0) {               // the slice's W_p2 rows, for phase 3
    const char *base = reinterpret_cast<const char *>(p.W_p2 + (size_t)s0 * p.p2_ld);
    const uint32_t bytes = (uint32_t)n_rows * (uint32_t)p.p2_ld * 2u;
    for (uint32_t o = 0; o < bytes; o += 65536u) pidev::prefetch_l2_bulk(base + o, min(65536u, bytes - o));
  }

  // ---- phase 1: partial hidden layer over K chunk kc of row group rg
  {
    unsigned char *xs = smem;                 // [8 NT1, KC] fp16, xs_stride bytes apart
    const int kc = cta % p.NKC, rg = cta / p.NKC;
    if (rg < p.RG) {
      const int KC = p.KC, k0 = kc * KC, nv = KC >> 3;
      for (int v = tid; v < 8 * NT1 * nv; v += kThreads) {
        const int b = v / nv, q = v - b * nv;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (b < B) val = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)b * d + k0) + q);
        *reinterpret_cast<uint4 *>(xs + (size_t)b * p.xs_stride + q * 16) = val;
      }
      __syncthreads();
      const int row0 = rg * p.RS, row1 = min(r, row0 + p.RS);
      const int nmt = (row1 - row0 + 15) >> 4;
      for (int mt = wid; mt < nmt; mt += kWarps) {
        const int ra = row0 + 16 * mt + g, rb = ra + 8;
        const uint4 *pa = reinterpret_cast<const uint4 *>(p.W_p1 + (size_t)min(ra, r - 1) * d + k0) + t4;
        const uint4 *pb = reinterpret_cast<const uint4 *>(p.W_p1 + (size_t)min(rb, r - 1) * d + k0) + t4;
        float acc[NT1][4];
#pragma unroll
        for (int j = 0; j < NT1; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll 4
        for (int kb = 0; kb < (KC >> 5); ++kb) {
          const uint4 wa = pidev::ld_stream(pa + 4 * kb), wb = pidev::ld_stream(pb + 4 * kb);
#pragma unroll
          for (int j = 0; j < NT1; ++j) {
            const uint4 xv =
                *reinterpret_cast<const uint4 *>(xs + (size_t)(8 * j + g) * p.xs_stride + kb * 64 + t4 * 16);
            mma16816(acc[j], wa.x, wb.x, wa.y, wb.y, xv.x, xv.y);
            mma16816(acc[j], wa.z, wb.z, wa.w, wb.w, xv.z, xv.w);
          }
        }
        // lane (g, t4): D[g][2 t4 + e] in acc[j][e], D[g + 8][2 t4 + e] in
        // acc[j][2 + e]; column 2 t4 + e of n tile j is token 8 j + 2 t4 + e
#pragma unroll
        for (int j = 0; j < NT1; ++j)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int b = 8 * j + 2 * t4 + e;
            if (b < B) {
              float *dst = p.partial + ((size_t)kc * B + b) * r;
              if (ra < row1) dst[ra] = acc[j][e];
              if (rb < row1) dst[rb] = acc[j][2 + e];
            }
          }
      }
    }
  }
  if (!grid_sync(p.bar, (unsigned)G, p.status)) return;

  // ---- phase 2: h = ReLU(sum of the K-chunk partials) for elements [e0, e1)
  {
    const int E = B * r;
    const int e0 = (int)((long long)cta * E / G), e1 = (int)((long long)(cta + 1) * E / G);
    const int ne = e1 - e0;                   // at most kThreads (checked on the host)
    if (ne > 0) {
      const int qn = kThreads / ne, el = tid % ne, q = tid / ne;
      if (q < qn) {
        float s = 0.f;
        for (int k = q; k < p.NKC; k += qn) s += __ldcg(p.partial + (size_t)k * E + e0 + el);
        red_s[q * ne + el] = s;
      }
      __syncthreads();
      if (tid < ne) {
        float h = 0.f;
        for (int k = 0; k < qn; ++k) h += red_s[k * ne + tid];
        h = h > 0.f ? h : 0.f;
        const int e = e0 + tid, b = e / r, k = e - b * r;
        const __half hi = __float2half_rn(h);
        const __half lo = __float2half_rn(h - __half2float(hi));
        p.hbuf[(size_t)(2 * b) * r + k] = hi;
        p.hbuf[(size_t)(2 * b + 1) * r + k] = lo;
      }
    }
  }
  if (!grid_sync(p.bar, 2u * (unsigned)G, p.status)) return;

  // ---- phase 3: logits of the slice, union over the batch, ordered local list
  unsigned char *hs = smem;                   // [8 NT, r] fp16, hs_stride bytes apart
  unsigned char *flag_s = smem + p.off_flag;  // [n_rows]
  int *list_s = reinterpret_cast<int *>(smem + p.off_list);
  {
    const int nv = r >> 3;
    for (int v = tid; v < 8 * NT * nv; v += kThreads) {
      const int n = v / nv, q = v - n * nv;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (n < 2 * B) val = __ldcg(reinterpret_cast<const uint4 *>(p.hbuf + (size_t)n * r) + q);
      *reinterpret_cast<uint4 *>(hs + (size_t)n * p.hs_stride + q * 16) = val;
    }
  }
  __syncthreads();
  const int nmt = (n_rows + 15) >> 4;
  for (int mt = wid; mt < nmt; mt += kWarps) {
    const int la = 16 * mt + g, lb = la + 8;  // rows within the slice
    const int ia = s0 + min(la, n_rows - 1), ib = s0 + min(lb, n_rows - 1);
    const uint4 *pa = reinterpret_cast<const uint4 *>(p.W_p2 + (size_t)ia * p.p2_ld) + t4;
    const uint4 *pb = reinterpret_cast<const uint4 *>(p.W_p2 + (size_t)ib * p.p2_ld) + t4;
    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
#pragma unroll 4
    for (int kb = 0; kb < (r >> 5); ++kb) {
      const uint4 wa = pidev::ld_stream(pa + 4 * kb), wb = pidev::ld_stream(pb + 4 * kb);
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const uint4 hv = *reinterpret_cast<const uint4 *>(hs + (size_t)(8 * j + g) * p.hs_stride + kb * 64 + t4 * 16);
        mma16816(acc[j], wa.x, wb.x, wa.y, wb.y, hv.x, hv.y);
        mma16816(acc[j], wa.z, wb.z, wa.w, wb.w, hv.z, hv.w);
      }
    }
    // lane (g, t4) holds token 4 j + t4 of n tile j: hi in acc[j][0] (row la)
    // and acc[j][2] (row lb), lo in acc[j][1] and acc[j][3]
    const float ca = p.c_p ? __ldg(p.c_p + ia) : 0.f, cb = p.c_p ? __ldg(p.c_p + ib) : 0.f;
    unsigned on_a = 0u, on_b = 0u;
#pragma unroll
    for (int j = 0; j < NT; ++j)
      if (4 * j + t4 < B) {
        on_a |= (acc[j][0] + acc[j][1]) + ca > 0.f ? 1u : 0u;
        on_b |= (acc[j][2] + acc[j][3]) + cb > 0.f ? 1u : 0u;
      }
    on_a |= __shfl_xor_sync(0xffffffffu, on_a, 1);
    on_a |= __shfl_xor_sync(0xffffffffu, on_a, 2);
    on_b |= __shfl_xor_sync(0xffffffffu, on_b, 1);
    on_b |= __shfl_xor_sync(0xffffffffu, on_b, 2);
    if (t4 == 0) {
      if (la < n_rows) flag_s[la] = (unsigned char)on_a;
      if (lb < n_rows) flag_s[lb] = (unsigned char)on_b;
    }
  }
  __syncthreads();
  int lcount = 0;
  for (int c0 = 0; c0 < n_rows; c0 += kThreads) {
    const int i = c0 + tid;
    const bool on = i < n_rows && flag_s[i];
    const unsigned bal = __ballot_sync(0xffffffffu, on);
    if (lane == 0) wtot_s[wid] = __popc(bal);
    __syncthreads();
    int wpre = 0, tot = 0;
    for (int w = 0; w < kWarps; ++w) {
      const int v = wtot_s[w];
      if (w < wid) wpre += v;
      tot += v;
    }
    if (on) list_s[lcount + wpre + __popc(bal & ((1u << lane) - 1u))] = s0 + i;
    lcount += tot;
    __syncthreads();
  }
  if (p.mask)
    for (int i = tid; i < n_rows; i += kThreads) p.mask[s0 + i] = flag_s[i];
  if (tid == 0) p.cnt[cta] = lcount;
  if (!grid_sync(p.bar, 3u * (unsigned)G, p.status)) return;

  // ---- phase 4: the list at its place in the ascending union list
  if (wid == 0) {
    int s = 0;
    for (int c = lane; c < cta; c += 32) s += __ldcg(p.cnt + c);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) pre_s = s;
  }
  __syncthreads();
  const int pre = pre_s;
  for (int j = tid; j < lcount; j += kThreads) p.idx[pre + j] = list_s[j];
  if (cta == G - 1 && tid == 0) *p.count = pre + lcount;
}

struct PBPlan {
  bool ok = false;
  int NT = 0, NKC = 0, KC = 0, RS = 0, RG = 0, xs_stride = 0, hs_stride = 0, off_flag = 0, off_list = 0;
  size_t smem = 0;
};

size_t align128(size_t v) { return (v + 127) & ~(size_t)127; }
int xs_stride_for(int KC) { return (KC * 2) % 128 == 0 ? KC * 2 + 64 : KC * 2; }

PBPlan pb_plan(const pi_layer *L, int B) {
  PBPlan s;
  const int G = L->num_sms, d = L->d, r = L->rank;
  if (B < 3 || B > 32 || G < 1 || r % 64 != 0 || r > 2048 || d % 32 != 0) return s;
  if ((long long)B * r > (long long)kThreads * G) return s;   // phase 2: one element per thread
  s.NT = B <= 8 ? 2 : (B <= 16 ? 4 : 8);
  const int NT1 = (s.NT + 1) / 2;
  // K chunks (the chunk length a multiple of 32 dividing d, the x chunk
  // within shared memory) and row groups: the split with the fewest bytes
  // per CTA (its W_p1 block and x chunk, its partial sums out, its share of
  // the partials in)
  const int nk_all = d / 32;
  const long long ne = ((long long)B * r + G - 1) / G;
  long long best_cost = -1;
  for (int n = 1; n <= std::min(nk_all, G); ++n) {
    if (nk_all % n != 0) continue;
    const int KC = d / n;
    if ((size_t)8 * NT1 * xs_stride_for(KC) > kSmemBudget / 2) continue;
    const int rg0 = std::max(1, std::min(G / n, (r + 15) / 16));
    const int RS = ((r + rg0 - 1) / rg0 + 15) / 16 * 16;
    const long long cost = (long long)(RS + B) * KC * 2 + (long long)RS * B * 4 + (long long)n * ne * 4;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      s.NKC = n;
      s.KC = KC;
      s.RS = RS;
    }
  }
  if (best_cost < 0) return s;
  s.RG = (r + s.RS - 1) / s.RS;
  s.xs_stride = xs_stride_for(s.KC);
  s.hs_stride = r * 2 + 64;
  const size_t slice = (size_t)(L->ffn + G - 1) / G;
  const size_t region = std::max((size_t)8 * NT1 * s.xs_stride, (size_t)8 * s.NT * s.hs_stride);
  s.off_flag = (int)align128(region);
  s.off_list = (int)align128(s.off_flag + slice);
  s.smem = align128(s.off_list + 4 * slice);
  if (s.smem > kSmemBudget) return s;
  if ((size_t)s.NKC * B * r * sizeof(float) > pi::tc_piece_bytes(L, B)) return s;
  s.ok = true;
  return s;
}

template <int NT>
cudaError_t launch_nt(const PBParams &p, int G, size_t smem, cudaStream_t st) {
  auto kern = k_predict_batch<NT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  void *args[] = {const_cast<PBParams *>(&p)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(G), dim3(kThreads), args, smem, st);
}

}  // namespace

namespace pi {

bool pbatch_supported(const pi_layer *L, int B) { return pb_plan(L, B).ok; }

cudaError_t run_predict_batch(const pi_layer *L, const __half *x, int B, uint8_t *mask_union, __half *hbuf,
                              float *partial, int32_t *cnt, unsigned *bar, int32_t *idx, int32_t *count,
                              cudaStream_t s) {
  const PBPlan pl = pb_plan(L, B);
  if (!pl.ok) return cudaErrorInvalidValue;
  PBParams p = {};
  p.x = x;
  p.W_p1 = L->W_p1;
  p.W_p2 = L->W_p2;
  p.c_p = L->c_p;
  p.B = B;
  p.d = L->d;
  p.r = L->rank;
  p.ffn = L->ffn;
  p.p2_ld = L->p2_ld;
  p.NKC = pl.NKC;
  p.KC = pl.KC;
  p.RS = pl.RS;
  p.RG = pl.RG;
  p.xs_stride = pl.xs_stride;
  p.hs_stride = pl.hs_stride;
  p.off_flag = pl.off_flag;
  p.off_list = pl.off_list;
  p.partial = partial;
  p.hbuf = hbuf;
  p.mask = mask_union;
  p.cnt = cnt;
  p.idx = idx;
  p.count = count;
  p.bar = bar;
  p.status = L->status;
  cudaError_t e = cudaMemsetAsync(bar, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const int G = L->num_sms;
  switch (pl.NT) {
    case 2: return launch_nt<2>(p, G, pl.smem, s);
    case 4: return launch_nt<4>(p, G, pl.smem, s);
    default: return launch_nt<8>(p, G, pl.smem, s);
  }
}

}  // namespace pi
