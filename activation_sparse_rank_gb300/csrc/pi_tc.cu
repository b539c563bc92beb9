// Batched sparse FFN on the tensor cores (tcgen05, TMEM accumulators, TMA).
//
// "PowerInfer: Fast Large Language Model Serving with a Consumer-grade GPU"
// (egguo-blog reading report), section 2.3 core module 4 (neuron-aware
// operators) and section 4.4, limitation 3: with a batch of B tokens the
// active set is the union over the batch, and the union's rows form a dense
// contraction with the batch:
//   up    H[u, b]  = W_up[idx[u], :] . x[b, :]           (and the gate rows)
//         a[u, b]  = ReLU(H + bias)  or  ReLU(G + bias) * H
//   down  y[b, j]  = sum_u a[u, b] W_down^T[idx[u], j]
// Both products run as tcgen05.mma kind::f16 (fp16 operands, fp32 TMEM
// accumulators).  The activations enter the second product as an fp16 pair
// a = a_hi + a_lo (stacked as 2*Bp columns), which keeps their rounding error
// near 2^-22 relative instead of fp16's 2^-11.
//
// k_tc_up:   persistent CTAs over 128-neuron tiles of the active list.  Per
//            64-element K slab, all 128 threads gather the 128 rows with
//            16-byte cp.async copies written straight into the 128-byte
//            swizzled operand layout (a gathered row piece is only 128 bytes,
//            too small for TMA to move at full rate), TMA loads the x slab,
//            and thread 0 issues the MMAs of a multi-stage mbarrier pipeline;
//            four warps then read the accumulators from TMEM.
// k_tc_down: CTA (column tile of 128, split of the list).  Per 64-neuron slab,
//            the threads gather 64 rows x 128 columns of W_down^T (MN-major
//            operand) the same way and TMA loads the matching [a_hi; a_lo]
//            slab; partial sums go to the workspace and k_reduce adds them
//            in split order (deterministic).
// All mbarrier waits are bounded; on a timeout the kernel sets a status bit,
// waits (bounded) for its copies in flight, frees its TMEM and returns.
#include <cuda.h>

#include <algorithm>

#include "pi_internal.cuh"

namespace {

constexpr unsigned kSpin = 1u << 22;
constexpr int kTile = 128;      // MMA M
constexpr int kSlab = 64;       // K elements per slab (128 bytes of fp16)

__device__ __forceinline__ uint32_t su32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ bool mb_wait(uint32_t mbar, uint32_t parity) {
  for (unsigned it = 0; it < kSpin; ++it) {
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

__device__ __forceinline__ void mb_init(uint32_t mbar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(count));
}

__device__ __forceinline__ void mb_expect(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tma_tile2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(mbar)
      : "memory");
}

__device__ __forceinline__ void tma_gather4(uint32_t dst, const CUtensorMap *map, int c0, int r0, int r1, int r2,
                                            int r3, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(
          dst),
      "l"(map), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(mbar)
      : "memory");
}

// 16-byte global -> shared copy (L2 only), and an mbarrier arrival once all of
// this thread's earlier copies have landed (counted against the init count).
__device__ __forceinline__ void cp16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_arrive(uint32_t mbar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(mbar) : "memory");
}
// Offset of 16-byte chunk c of row r in a 128-byte-swizzled tile of 128-byte rows
// (the layout TMA writes with 128B swizzle and the MMA reads with layout type 2).
__device__ __forceinline__ uint32_t sw128(int r, int c) { return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4)); }

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 layout type 2).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16 with f16 A/B and f32 D.
__device__ __forceinline__ uint32_t idesc_f16(int n, int m, bool a_mn_major) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar) : "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float *v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ int tmem_cols_for(int n) {
  int c = 32;
  while (c < n) c <<= 1;
  return c;
}

// ---------------------------------------------------------------------------
// Row-tile GEMM D[128 rows, N] = W[rows, 0:K] . Bop[0:N, 0:K]^T with one of
// three epilogues:
//   kAct     a = ReLU(D + bias) (ReGLU: ReLU(D_gate + bias) * D_up), written
//            as the fp16 pair (hi; lo) into out [2Bp, ld] (the sparse FFN up)
//   kLogits  l = D_hi + D_lo + bias over the pair columns of Bop; mask[row] =
//            1 if l > 0 for some token of the batch (predictor layer 2)
//   kHiddenPart  the predictor's layer 1 split over K: CTA (tile, blockIdx.y)
//            contracts K elements [blockIdx.y * klen, +klen) and writes D in
//            fp32 to fout [split, Bp, ld]; k_hidden_finish adds the splits
//            in order.  (The layer has only r / 128 row tiles, too few CTAs
//            to stream W_p1 at speed.)
constexpr int kAct = 0, kHiddenPart = 1, kLogits = 2;

template <int MODE, bool REGLU>
__global__ void __launch_bounds__(128, 1) k_tc_rows(const __half *__restrict__ Wg,   // rows (gated rows for kAct)
                                                    const __half *__restrict__ Wu,   // up rows (ReGLU)
                                                    const __grid_constant__ CUtensorMap tm_x,   // B operand
                                                    const int32_t *__restrict__ idx, const int32_t *__restrict__ count_p,
                                                    int count_const, const float *__restrict__ bias, int d, int klen,
                                                    int ffn, int B, int Bp, int nstage, int kw,
                                                    __half *__restrict__ abuf, float *__restrict__ fout, int abuf_ld,
                                                    uint8_t *__restrict__ mask_out, unsigned int *status) {
  // d: row length of W; this CTA contracts K elements [koff, koff + klen);
  // ffn: number of rows of W.  A pipeline stage holds kw consecutive
  // 64-element K slabs, so every gathered row contributes kw * 128
  // contiguous bytes per stage.
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  constexpr int NA = REGLU ? 2 : 1;
  const int Nmma = MODE == kLogits ? 2 * Bp : Bp;
  const uint32_t slabA = kTile * 128;                   // one gathered operand slab
  const uint32_t slabX = (uint32_t)Nmma * 128;
  const uint32_t subX = (slabX + 1023) & ~1023u;
  const uint32_t stage_bytes = (uint32_t)kw * (NA * slabA + subX);
  __shared__ __align__(8) unsigned long long full_s[8], empty_s[8], done_s;
  __shared__ int rows_s[kTile];
  __shared__ uint32_t taddr_s;
  __shared__ int fail_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ncols = tmem_cols_for(NA * Nmma);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&taddr_s)), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      mb_init(su32(&full_s[s]), 129);   // 128 copy arrivals + the TMA expect_tx arrival
      mb_init(su32(&empty_s[s]), 1);
    }
    mb_init(su32(&done_s), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fail_s = 0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = taddr_s;

  int count = count_p ? *count_p : count_const;
  if (count < 0 || count > ffn) {
    if (tid == 0) atomicOr(status, PI_STATUS_BAD_COUNT);
    count = count < 0 ? 0 : ffn;
  }
  const int ntiles = (count + kTile - 1) / kTile;
  const int koff = (int)blockIdx.y * klen;
  const int KT = klen / (kSlab * kw);
  const uint32_t idesc = idesc_f16(Nmma, kTile, false);
  uint32_t gslab = 0;          // slabs issued by this CTA so far (pipeline position)
  uint32_t done_phase = 0;

  for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int k0 = tile * kTile;
    {
      const int k = k0 + tid;
      int i = k < count ? (idx ? idx[k] : k) : -1;
      if (k < count && (i < 0 || i >= ffn)) {
        atomicOr(status, PI_STATUS_BAD_INDEX);
        i = -2;
      }
      rows_s[tid] = i;
    }
    __syncthreads();
    {
      // Every thread copies 8 of the 1024 16-byte chunks of each gathered
      // slab (8 threads per 128-byte row piece, rows t/8 + 16 i), straight
      // into the swizzled layout; thread 0 also loads the x slab by TMA and
      // issues the MMAs.  Invalid / padding rows read row 0 (their
      // activation is written as 0).
      const int cch = tid & 7;
      const __half *gsrc[8], *usrc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int q = (tid >> 3) + 16 * i;
        const int rid = rows_s[q] >= 0 ? rows_s[q] : 0;
        gsrc[i] = Wg + (size_t)rid * d + koff + cch * 8;
        usrc[i] = REGLU ? Wu + (size_t)rid * d + koff + cch * 8 : nullptr;
      }
      auto issue = [&](int kt, uint32_t g) {
        const int s = (int)(g % (uint32_t)nstage);
        if (g >= (uint32_t)nstage && !mb_wait(su32(&empty_s[s]), ((g / nstage) - 1) & 1)) fail_s = 1;
        unsigned char *st = sm + (size_t)s * stage_bytes;
        const uint32_t bar = su32(&full_s[s]);
        const uint32_t base = su32(st);
        for (int j = 0; j < kw; ++j) {
          const int k0e = (kt * kw + j) * kSlab;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int q = (tid >> 3) + 16 * i;
            cp16(base + j * slabA + sw128(q, cch), gsrc[i] + k0e);
            if (REGLU) cp16(base + (kw + j) * slabA + sw128(q, cch), usrc[i] + k0e);
          }
        }
        cp_arrive(bar);
        if (tid == 0) {
          mb_expect(bar, kw * slabX);
          for (int j = 0; j < kw; ++j)
            tma_tile2d(su32(st + NA * kw * slabA + j * subX), &tm_x, koff + (kt * kw + j) * kSlab, 0, bar);
        }
      };
      const int pre = min(nstage - 1, KT);
      for (int kt = 0; kt < pre; ++kt) issue(kt, gslab + kt);
      for (int kt = 0; kt < KT; ++kt) {
        if (fail_s) break;
        const uint32_t g = gslab + kt;
        if (kt + nstage - 1 < KT) issue(kt + nstage - 1, g + nstage - 1);
        if (tid == 0) {
          const int s = (int)(g % (uint32_t)nstage);
          if (!mb_wait(su32(&full_s[s]), (g / nstage) & 1)) {
            fail_s = 1;
          } else {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            asm volatile("tcgen05.fence::after_thread_sync;");
            unsigned char *st = sm + (size_t)s * stage_bytes;
            for (int j = 0; j < kw; ++j) {
              const uint32_t xa = su32(st + NA * kw * slabA + j * subX);
              const uint32_t aa = su32(st + j * slabA);
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = sdesc(xa + kk * 32, 16, 1024);
                const uint32_t acc = (kt | j | kk) ? 1u : 0u;
                mma_f16(tmem, sdesc(aa + kk * 32, 16, 1024), bd, idesc, acc);
                if (REGLU)
                  mma_f16(tmem + (uint32_t)Nmma, sdesc(aa + kw * slabA + kk * 32, 16, 1024), bd, idesc, acc);
              }
            }
            mma_commit(su32(&empty_s[s]));
          }
        }
      }
      gslab += KT;
      if (tid == 0) mma_commit(su32(&done_s));
    }
    __syncthreads();
    if (fail_s) break;
    if (!mb_wait(su32(&done_s), done_phase)) { fail_s = 1; break; }
    done_phase ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;");
    // epilogue: TMEM lane = tile row = warp*32 + lane
    const int q = warp * 32 + lane;
    const int i = rows_s[q];
    const float bi = (i >= 0 && bias) ? bias[i] : 0.f;
    const int kq = k0 + q;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    if (MODE == kLogits) {
      bool on = false;
      for (int c0 = 0; c0 < Bp; c0 += 8) {
        float hi8[8], lo8[8];
        tmem_ld8(trow + (uint32_t)c0, hi8);
        tmem_ld8(trow + (uint32_t)(Bp + c0), lo8);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (c0 + j < B) on |= (hi8[j] + lo8[j] + bi) > 0.f;
      }
      if (i >= 0) mask_out[i] = on ? 1 : 0;
    } else if (MODE == kHiddenPart) {
      float *dst = fout + (size_t)blockIdx.y * Bp * abuf_ld + kq;
      for (int c0 = 0; c0 < Bp; c0 += 8) {
        float g8[8];
        tmem_ld8(trow + (uint32_t)c0, g8);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[(size_t)(c0 + j) * abuf_ld] = (i >= 0 && c0 + j < B) ? g8[j] : 0.f;
      }
    } else {
      for (int c0 = 0; c0 < Bp; c0 += 8) {
        float g8[8], u8[8];
        tmem_ld8(trow + (uint32_t)c0, g8);
        if (REGLU) tmem_ld8(trow + (uint32_t)(Bp + c0), u8);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int b = c0 + j;
          float a = 0.f;
          if (i >= 0 && b < B) {
            const float z = g8[j] + bi;
            a = REGLU ? (z > 0.f ? z : 0.f) * u8[j] : (z > 0.f ? z : 0.f);
          }
          const __half hi = __float2half_rn(a);
          const __half lo = __float2half_rn(a - __half2float(hi));
          abuf[(size_t)b * abuf_ld + kq] = hi;
          abuf[(size_t)(Bp + b) * abuf_ld + kq] = lo;
        }
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
  }
  if (fail_s && tid == 0) atomicOr(status, PI_STATUS_BARRIER_TIMEOUT);
  // let every copy issued by this CTA land before leaving (bounded)
  if (tid == 0 && fail_s)
    for (int s = 0; s < nstage; ++s) mb_wait(su32(&full_s[s]), 0), mb_wait(su32(&full_s[s]), 1);
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols));
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 1) k_tc_down(const __half *__restrict__ Wd,                  // W_down^T
                                                    const __grid_constant__ CUtensorMap tm_a,   // abuf, box 64 x 2Bp
                                                    const int32_t *__restrict__ idx, const int32_t *__restrict__ count_p,
                                                    int count_const, int d, int ffn, int B, int Bp, int nstage,
                                                    int cw, float *__restrict__ partial, unsigned int *status) {
  // A CTA owns cw column tiles of 128 (cw * 256 contiguous bytes of every
  // gathered W_down^T row per slab), one TMEM accumulator per tile.
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  const int N2 = 2 * Bp;
  const uint32_t half_bytes = kSlab * 128;                // 64 rows x 64 columns
  const uint32_t tileW = 2 * half_bytes;                  // 128 columns
  const uint32_t slabW = (uint32_t)cw * tileW;
  const uint32_t slabA = (uint32_t)N2 * 128;
  const uint32_t stage_bytes = slabW + ((slabA + 1023) & ~1023u);
  __shared__ __align__(8) unsigned long long full_s[8], empty_s[8], done_s;
  __shared__ uint32_t taddr_s;
  __shared__ int fail_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j0 = blockIdx.x * kTile * cw;
  const int ncols = tmem_cols_for(cw * N2);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&taddr_s)), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      mb_init(su32(&full_s[s]), 129);   // 128 copy arrivals + the TMA expect_tx arrival
      mb_init(su32(&empty_s[s]), 1);
    }
    mb_init(su32(&done_s), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fail_s = 0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = taddr_s;

  int count = count_p ? *count_p : count_const;
  if (count < 0 || count > ffn) count = count < 0 ? 0 : ffn;     // flagged by k_tc_up
  const int KS = (count + kSlab - 1) / kSlab;
  const int per = (KS + gridDim.y - 1) / gridDim.y;
  const int ks0 = min(KS, (int)blockIdx.y * per), ks1 = min(KS, ks0 + per);
  const int nk = ks1 - ks0;
  const uint32_t idesc = idesc_f16(N2, kTile, true);

  if (nk > 0) {
    // Every thread copies 16 of the 2048 16-byte chunks of a slab: chunk
    // c = tid % 8 of column half (tid / 8) % 2 of rows tid / 16 + 8 i, into the
    // MN-major swizzled layout (8 rows of 128 bytes per 1024-byte group);
    // thread 0 also loads the [a_hi; a_lo] slab by TMA and issues the MMAs.
    const int cch = tid & 7, hh = (tid >> 3) & 1, r0 = tid >> 4;
    // row indices of the next slab to issue, loaded one issue ahead so their
    // latency hides behind the copies of the current slab
    int nxt[8];
    auto load_rows = [&](int slab) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int k = slab * kSlab + r0 + 8 * i;
        int rid = k < count ? (idx ? idx[k] : k) : 0;
        nxt[i] = (rid >= 0 && rid < ffn) ? rid : 0;  // padding / invalid: row 0 times a zero activation
      }
    };
    load_rows(ks0);
    auto issue = [&](int t) {
      const int s = t % nstage;
      if (t >= nstage && !mb_wait(su32(&empty_s[s]), ((t / nstage) - 1) & 1)) fail_s = 1;
      unsigned char *st = sm + (size_t)s * stage_bytes;
      const uint32_t bar = su32(&full_s[s]);
      const int slab = ks0 + t;
      int cur[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
      if (t + 1 < nk) load_rows(slab + 1);
      for (int c = 0; c < cw; ++c) {
        const uint32_t base = su32(st) + c * tileW + hh * half_bytes;
        const int col = j0 + c * kTile + hh * 64 + cch * 8;
        const int colc = col < d ? col : 0;          // a column past d reads column 0 (output dropped)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int q = r0 + 8 * i;
          cp16(base + sw128(q, cch), Wd + (size_t)cur[i] * d + colc);
        }
      }
      cp_arrive(bar);
      if (tid == 0) {
        mb_expect(bar, slabA);
        tma_tile2d(su32(st + slabW), &tm_a, slab * kSlab, 0, bar);
      }
    };
    const int pre = min(nstage - 1, nk);
    for (int t = 0; t < pre; ++t) issue(t);
    for (int t = 0; t < nk; ++t) {
      if (fail_s) break;
      if (t + nstage - 1 < nk) issue(t + nstage - 1);
      if (tid == 0) {
        const int s = t % nstage;
        if (!mb_wait(su32(&full_s[s]), (t / nstage) & 1)) {
          fail_s = 1;
        } else {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          asm volatile("tcgen05.fence::after_thread_sync;");
          unsigned char *st = sm + (size_t)s * stage_bytes;
          for (int c = 0; c < cw; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              // A: MN-major (K groups of 8 rows at 1024 B, column halves at half_bytes)
              const uint64_t ad = sdesc(su32(st) + c * tileW + kk * 16 * 128, half_bytes, 1024);
              const uint64_t bd = sdesc(su32(st + slabW) + kk * 32, 16, 1024);
              mma_f16(tmem + (uint32_t)(c * N2), ad, bd, idesc, (t | kk) ? 1u : 0u);
            }
          mma_commit(su32(&empty_s[s]));
        }
      }
    }
    if (tid == 0) mma_commit(su32(&done_s));
  }
  __syncthreads();
  if (nk > 0 && !fail_s) {
    if (!mb_wait(su32(&done_s), 0)) fail_s = 1;
  }
  __syncthreads();
  if (!fail_s) {
    asm volatile("tcgen05.fence::after_thread_sync;");
    for (int c = 0; c < cw; ++c) {
      const int j = j0 + c * kTile + warp * 32 + lane;   // TMEM lane = output column
      const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c * N2);
      for (int c0 = 0; c0 < Bp; c0 += 8) {
        float hi[8], lo[8];
        if (nk > 0) {
          tmem_ld8(trow + (uint32_t)c0, hi);
          tmem_ld8(trow + (uint32_t)(Bp + c0), lo);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q) hi[q] = lo[q] = 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int b = c0 + q;
          if (b < B && j < d) partial[((size_t)blockIdx.y * B + b) * d + j] = hi[q] + lo[q];
        }
      }
    }
  } else if (tid == 0) {
    atomicOr(status, PI_STATUS_BARRIER_TIMEOUT);
    for (int s = 0; s < nstage; ++s) mb_wait(su32(&full_s[s]), 0), mb_wait(su32(&full_s[s]), 1);
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols));
}

// ---------------------------------------------------------------------------
// The driver's tensor-map encoder, looked up through the runtime so that the
// library does not link libcuda (it must load on machines without a driver).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

bool encode_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer) {
  const EncodeTiledFn enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// h = ReLU(sum of the K splits, in split order), written as the fp16 pair
// (hi rows 0..Bp-1, lo rows Bp..2Bp-1) of the logits kernel's B operand.
__global__ void k_hidden_finish(const float *__restrict__ part, int nsplit, int B, int Bp, int rank, int rpad,
                                __half *__restrict__ hbuf) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  const int n = Bp * rpad;
  if (e >= n) return;
  const int b = e / rpad, row = e % rpad;
  float acc = 0.f;
  for (int k = 0; k < nsplit; ++k) acc += part[(size_t)k * n + e];
  const float h = (b < B && row < rank && acc > 0.f) ? acc : 0.f;
  const __half hi = __float2half_rn(h);
  hbuf[e] = hi;
  hbuf[(size_t)n + e] = __float2half_rn(h - __half2float(hi));
}

constexpr size_t kTcSmemBudget = 200 * 1024;

template <int MODE, bool REGLU>
cudaError_t launch_rows(const pi_layer *L, const __half *Wg, const __half *Wu, const CUtensorMap &tm_x,
                        const int32_t *idx, const int32_t *count, int count_const, const float *bias, int K,
                        int nrows, int B, int Bp, __half *out, int out_ld, uint8_t *mask, cudaStream_t s,
                        int ksplit = 1, float *fout = nullptr) {
  // K: row length; each of the ksplit CTAs of a row tile contracts K / ksplit
  const int klen = K / ksplit;
  const int NA = REGLU ? 2 : 1;
  const int Nmma = MODE == kLogits ? 2 * Bp : Bp;
  const size_t sub = NA * (size_t)kTile * 128 + (((size_t)Nmma * 128 + 1023) & ~(size_t)1023);
  // widest stage (kw consecutive slabs per row) that divides K and keeps >= 2 stages
  int kw = 4;
  while (kw > 1 && ((klen / kSlab) % kw != 0 || (kTcSmemBudget - 1024) / (kw * sub) < 2)) kw >>= 1;
  const size_t stage = kw * sub;
  int ns = (int)((kTcSmemBudget - 1024) / stage);
  if (ns > 8) ns = 8;
  if (ns < 2) return cudaErrorInvalidValue;
  const size_t smem = 1024 + ns * stage;
  auto kern = k_tc_rows<MODE, REGLU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int grid = (nrows + kTile - 1) / kTile;
  if (grid > L->num_sms) grid = L->num_sms;
  kern<<<dim3(grid, ksplit), 128, smem, s>>>(Wg, Wu, tm_x, idx, count, count_const, bias, K, klen, nrows, B, Bp,
                                             ns, kw, out, fout, out_ld, mask, L->status);
  return cudaGetLastError();
}

}  // namespace

namespace pi {

bool tc_supported(const pi_layer *L, int B) {
  return B >= 3 && B <= PI_MAX_BATCH && L->d % kSlab == 0 && L->d >= kTile;
}

int tc_bpad(int B) { return (B + 15) & ~15; }   // MMA N: a multiple of 16

int tc_ffn_pad(const pi_layer *L) { return (L->ffn + kTile - 1) / kTile * kTile; }

bool tc_predict_supported(const pi_layer *L, int B) {
  return tc_supported(L, B) && L->rank % kSlab == 0;
}

int tc_rank_pad(const pi_layer *L) { return (L->rank + kTile - 1) / kTile * kTile; }

int tc_hidden_splits(const pi_layer *L) {
  const int tiles = tc_rank_pad(L) / kTile, slabs = L->d / kSlab;
  int k = std::min(kMaxHiddenSplits, std::max(1, L->num_sms / tiles));
  while (k > 1 && slabs % k != 0) --k;
  return k;
}

cudaError_t run_predict_tc(const pi_layer *L, const __half *x, int B, uint8_t *mask_union, __half *hbuf,
                           float *hpart, cudaStream_t s) {
  const int Bp = tc_bpad(B);
  const int rpad = tc_rank_pad(L);
  CUtensorMap tm_x, tm_h;
  if (!encode_2d(&tm_x, x, L->d, B, (uint64_t)L->d * 2, kSlab, Bp) ||
      !encode_2d(&tm_h, hbuf, rpad, 2 * Bp, (uint64_t)rpad * 2, kSlab, 2 * Bp))
    return cudaErrorInvalidValue;
  // h = ReLU(W_p1 x) as an fp16 pair (K split over CTAs, splits added in
  // order), then l = W_p2 h + c_p -> union mask
  const int ks = tc_hidden_splits(L);
  cudaError_t e = launch_rows<kHiddenPart, false>(L, L->W_p1, nullptr, tm_x, nullptr, nullptr, L->rank, nullptr,
                                                  L->d, L->rank, B, Bp, nullptr, rpad, nullptr, s, ks, hpart);
  if (e != cudaSuccess) return e;
  const int n = Bp * rpad;
  k_hidden_finish<<<(n + 255) / 256, 256, 0, s>>>(hpart, ks, B, Bp, L->rank, rpad, hbuf);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_rows<kLogits, false>(L, L->W_p2, nullptr, tm_h, nullptr, nullptr, L->ffn, L->c_p, L->rank, L->ffn, B,
                                     Bp, nullptr, 0, mask_union, s);
}



cudaError_t run_sparse_ffn_tc(const pi_layer *L, const __half *x, int B, const int32_t *idx,
                              const int32_t *count, int count_const, float *y, const WsLayout &w,
                              char *ws, cudaStream_t s) {
  const bool reglu = L->act == PI_ACT_REGLU;
  const int Bp = tc_bpad(B);
  const int ffn_pad = tc_ffn_pad(L);
  __half *abuf = reinterpret_cast<__half *>(ws + w.abuf);
  float *partial = reinterpret_cast<float *>(ws + w.partial);
  CUtensorMap tm_x, tm_a;
  const uint64_t row_bytes = (uint64_t)L->d * 2;
  if (!encode_2d(&tm_x, x, L->d, B, row_bytes, kSlab, Bp) ||
      !encode_2d(&tm_a, abuf, ffn_pad, 2 * Bp, (uint64_t)ffn_pad * 2, kSlab, 2 * Bp))
    return cudaErrorInvalidValue;

  cudaError_t e = record_hook(L->ev_before, s);
  if (e != cudaSuccess) return e;
  e = reglu ? launch_rows<kAct, true>(L, reglu ? L->W_gate : L->W_up, L->W_up, tm_x, idx, count, count_const, L->b,
                                      L->d, L->ffn, B, Bp, abuf, ffn_pad, nullptr, s)
            : launch_rows<kAct, false>(L, L->W_up, nullptr, tm_x, idx, count, count_const, L->b, L->d, L->ffn, B,
                                       Bp, abuf, ffn_pad, nullptr, s);
  if (e != cudaSuccess) return e;

  // down: stages of cw x 16 KB gathered W_down^T + the [a_hi; a_lo] slab
  const int cw = (L->d % (2 * kTile) == 0 && 2 * 2 * Bp <= 512) ? 2 : 1;
  const size_t dn_stage = cw * 2 * (size_t)kSlab * 128 + (((size_t)2 * Bp * 128 + 1023) & ~(size_t)1023);
  int dn_ns = (int)((kTcSmemBudget - 1024) / dn_stage);
  if (dn_ns > 8) dn_ns = 8;
  if (dn_ns < 2) return cudaErrorInvalidValue;
  const size_t dn_smem = 1024 + dn_ns * dn_stage;
  e = cudaFuncSetAttribute(k_tc_down, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dn_smem);
  if (e != cudaSuccess) return e;
  const int ctiles = (L->d + cw * kTile - 1) / (cw * kTile);
  int nsplit = L->num_sms / ctiles;
  if (nsplit < 1) nsplit = 1;
  dim3 grid_dn(ctiles, nsplit);
  k_tc_down<<<grid_dn, 128, dn_smem, s>>>(L->W_dT, tm_a, idx, count, count_const, L->d, L->ffn, B, Bp, dn_ns, cw,
                                         partial, L->status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = record_hook(L->ev_after, s);
  if (e != cudaSuccess) return e;
  return run_reduce(partial, nsplit, B * L->d, y, s);
}

}  // namespace pi
