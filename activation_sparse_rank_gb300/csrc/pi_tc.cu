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
// k_tc_rows: the up rows (and the predictor's two layers), 128-row tiles of
//            the list.  Per stage of kw 64-element K slabs, all 128 threads
//            gather the 128 rows with 16-byte cp.async copies written
//            straight into the 128-byte swizzled operand layout (a gathered
//            row piece is only 128-512 bytes, too small for TMA to move at
//            full rate), TMA loads the x slab, and thread 0 issues the MMAs
//            of a multi-stage mbarrier pipeline; four warps then read the
//            accumulators from TMEM.
// k_tc_down: per 64-neuron slab, the threads gather 64 rows x cw * 128
//            columns of W_down^T (MN-major operand) the same way and TMA
//            loads the matching [a_hi; a_lo] slab.
// Both split their (tile, K stage) work stream-K style over all SMs: each CTA
// takes an equal contiguous share, so no SM idles when the tile count is not
// a multiple of the SM count; tiles shared by several CTAs are summed from
// per-CTA pieces in CTA order (deterministic; no float atomics).
// All mbarrier waits are bounded; on a timeout the kernel sets a status bit,
// waits (bounded) for its copies in flight, frees its TMEM and returns.
#include <cuda.h>

#include <algorithm>

#include "pi_internal.cuh"

namespace {

constexpr unsigned kSpin = 1u << 22;
constexpr int kTile = 128;      // MMA M
constexpr int kSlab = 64;       // K elements per slab (128 bytes of fp16)
// Column tiles of 128 per down-kernel work unit: 4 gives every gathered
// W_down^T row 1 KB of contiguous bytes per slab (two stages still fit in
// shared memory); measured 10-12 % faster than 2 at batches 8 and 32.
#ifndef PI_TC_DOWN_CW
#define PI_TC_DOWN_CW 4
#endif
constexpr int kDownCwMax = PI_TC_DOWN_CW;

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
//   kHidden  h = ReLU(D), written as the pair into out (predictor layer 1)
//   kLogits  l = D_hi + D_lo + bias over the pair columns of Bop; mask[row] =
//            1 if l > 0 for some token of the batch (predictor layer 2)
//
// Work is split stream-K style: the (tile, K stage) iterations of all row
// tiles are laid end to end and CTA c takes the contiguous range
// [c*I/G, (c+1)*I/G), so every CTA streams the same number of bytes whatever
// the tile count (a union of 171 tiles on 152 SMs, or the predictor's r/128
// tiles, no longer leaves SMs idle).  A tile covered by one CTA gets its
// epilogue at once; a tile split between CTAs leaves one fp32 piece per CTA
// (slot 2c for a CTA's first piece, 2c+1 for its last) and k_tc_fixup adds
// the pieces in CTA order (deterministic) and applies the epilogue.
constexpr int kAct = 0, kHidden = 1, kLogits = 2;

__device__ __forceinline__ long long range_start(int c, long long I, int G) { return (long long)c * I / G; }

// At most kCtasPerTile CTAs per row tile take part (a small list leaves the
// rest of the grid idle rather than cutting tiles into slivers); a tile then
// meets at most 2 * kCtasPerTile + 2 CTA ranges, within kMaxPieces.
constexpr int kCtasPerTile = 8;
constexpr int kMaxPieces = 32;

__device__ __forceinline__ int active_ctas(int grid, int ntiles) {
  const long long g = (long long)ntiles * kCtasPerTile;
  return (int)(g < grid ? (g > 0 ? g : 1) : grid);
}

// Row of a tile: index into W (or -1 past the end of the list, -2 when the
// list holds an out-of-range index, which is flagged).
__device__ __forceinline__ int tile_row(const int32_t *idx, int k, int count, int ffn, unsigned *status) {
  if (k >= count) return -1;
  const int i = idx ? idx[k] : k;
  if (i < 0 || i >= ffn) {
    atomicOr(status, PI_STATUS_BAD_INDEX);
    return -2;
  }
  return i;
}

// Epilogue of one tile row (the calling thread's row q, W row i, output
// column kq).  fetch8(c, v) yields D columns c .. c+7 of the row; for kAct
// and kHidden only token columns [c_begin, c_end) are produced.
// Row scales of E4M3 layers for the kAct epilogue (all null for fp16 rows):
// g / u multiply the gated / up dot products, d (the row's W_down^T scale)
// multiplies the activation, which is how the down product's rows get it.
struct RowScales {
  const float *g = nullptr, *u = nullptr, *d = nullptr;
};

template <int MODE, bool REGLU, typename F>
__device__ __forceinline__ bool row_epilogue(F fetch8, int c_begin, int c_end, int i, int kq, float bi, int B,
                                             int Bp, int Nmma, __half *abuf, int abuf_ld, uint8_t *mask_out,
                                             bool silu, const RowScales &sc) {
  // silu: the gate of a gated (kAct, REGLU) row is SiLU (SwiGLU) instead of ReLU
  if (MODE == kLogits) {                // kLogits: token columns [c_begin, c_end); returns l > 0 for one of them
    bool on = false;
    for (int c0 = c_begin; c0 < c_end; c0 += 8) {
      float hi8[8], lo8[8];
      fetch8(c0, hi8);
      fetch8(Bp + c0, lo8);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (c0 + j < B) on |= (hi8[j] + lo8[j] + bi) > 0.f;
    }
    if (i >= 0 && mask_out) mask_out[i] = on ? 1 : 0;
    return on;
  } else {
    float sgi = 1.f, sui = 1.f, sdi = 1.f;
    if (i >= 0) {
      if (sc.g) sgi = sc.g[i];
      if (sc.u) sui = sc.u[i];
      if (sc.d) sdi = sc.d[i];
    }
    for (int c0 = c_begin; c0 < c_end; c0 += 8) {
      float g8[8], u8[8];
      fetch8(c0, g8);
      if (REGLU) fetch8(Nmma + c0, u8);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int b = c0 + j;
        float a = 0.f;
        if (i >= 0 && b < B) {
          const float z = g8[j] * sgi + bi;
          a = REGLU ? pidev::gate_act(z, silu) * (u8[j] * sui) : (z > 0.f ? z : 0.f);
          a *= sdi;
        }
        const __half hi = __float2half_rn(a);
        const __half lo = __float2half_rn(a - __half2float(hi));
        abuf[(size_t)b * abuf_ld + kq] = hi;
        abuf[(size_t)(Bp + b) * abuf_ld + kq] = lo;
      }
    }
    return false;
  }
}

template <int MODE, bool REGLU>
__global__ void __launch_bounds__(128, 1) k_tc_rows(const __half *__restrict__ Wg,   // rows (gated rows for kAct)
                                                    const __half *__restrict__ Wu,   // up rows (ReGLU)
                                                    const __grid_constant__ CUtensorMap tm_x,   // B operand
                                                    const int32_t *__restrict__ idx, const int32_t *__restrict__ count_p,
                                                    int count_const, const float *__restrict__ bias, int d, int wld,
                                                    int ffn, int B, int Bp, int nstage, int kw, __half *__restrict__ abuf,
                                                    int abuf_ld, float *__restrict__ piece,
                                                    uint8_t *__restrict__ mask_out, int32_t *__restrict__ tile_cnt,
                                                    unsigned int *status, int silu) {
  // d: row length of W and contraction length K; wld: elements between the
  // rows of W; ffn: number of rows of W.
  // A pipeline stage holds kw consecutive 64-element K slabs, so every
  // gathered row contributes kw * 128 contiguous bytes per stage.
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  constexpr int NA = REGLU ? 2 : 1;
  const int Nmma = MODE == kLogits ? 2 * Bp : Bp;
  const int ncolD = NA * Nmma;                          // accumulator columns
  const uint32_t slabA = kTile * 128;                   // one gathered operand slab
  const uint32_t slabX = (uint32_t)Nmma * 128;
  const uint32_t subX = (slabX + 1023) & ~1023u;
  const uint32_t stage_bytes = (uint32_t)kw * (NA * slabA + subX);
  __shared__ __align__(8) unsigned long long full_s[8], empty_s[8], done_s;
  __shared__ int rows_s[kTile];
  __shared__ uint32_t taddr_s;
  __shared__ int fail_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ncols = tmem_cols_for(ncolD);
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
  // the set-up above overlaps the previous kernel's tail (programmatic
  // dependent launch); nothing it writes or reads is touched before this
  pidev::griddep_wait();
  pidev::griddep_launch();

  int count = count_p ? *count_p : count_const;
  if (count < 0 || count > ffn) {
    if (tid == 0) atomicOr(status, PI_STATUS_BAD_COUNT);
    count = count < 0 ? 0 : ffn;
  }
  const int ntiles = (count + kTile - 1) / kTile;
  const int KT = d / (kSlab * kw);                      // stages per tile
  const long long I = (long long)ntiles * KT;
  const int G = active_ctas(gridDim.x, ntiles), cta = blockIdx.x;
  const long long rs = cta < G ? range_start(cta, I, G) : 0, re = cta < G ? range_start(cta + 1, I, G) : 0;
  const uint32_t idesc = idesc_f16(Nmma, kTile, false);
  uint32_t gslab = 0;          // stages issued by this CTA so far (pipeline position)
  uint32_t done_phase = 0;

  for (long long s0 = rs; s0 < re;) {
    const int tile = (int)(s0 / KT);
    const int kb = (int)(s0 % KT);
    const int n = (int)min((long long)(KT - kb), re - s0);   // stages of this piece
    const bool whole = (n == KT);
    const int slot = 2 * cta + (s0 == rs ? 0 : 1);
    s0 += n;
    const int k0 = tile * kTile;
    rows_s[tid] = tile_row(idx, k0 + tid, count, ffn, status);
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
        gsrc[i] = Wg + (size_t)rid * wld + cch * 8;
        usrc[i] = REGLU ? Wu + (size_t)rid * wld + cch * 8 : nullptr;
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
            tma_tile2d(su32(st + NA * kw * slabA + j * subX), &tm_x, (kt * kw + j) * kSlab, 0, bar);
        }
      };
      const int pre = min(nstage - 1, n);
      for (int it = 0; it < pre; ++it) issue(kb + it, gslab + it);
      for (int it = 0; it < n; ++it) {
        if (fail_s) break;
        const uint32_t g = gslab + it;
        if (it + nstage - 1 < n) issue(kb + it + nstage - 1, g + nstage - 1);
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
                const uint32_t acc = (it | j | kk) ? 1u : 0u;
                mma_f16(tmem, sdesc(aa + kk * 32, 16, 1024), bd, idesc, acc);
                if (REGLU)
                  mma_f16(tmem + (uint32_t)Nmma, sdesc(aa + kw * slabA + kk * 32, 16, 1024), bd, idesc, acc);
              }
            }
            mma_commit(su32(&empty_s[s]));
          }
        }
      }
      gslab += n;
      if (tid == 0) mma_commit(su32(&done_s));
    }
    __syncthreads();
    if (fail_s) break;
    if (!mb_wait(su32(&done_s), done_phase)) { fail_s = 1; break; }
    done_phase ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;");
    // epilogue: TMEM lane = tile row = warp*32 + lane
    const int q = warp * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    if (whole) {
      const int i = rows_s[q];
      const float bi = (i >= 0 && bias) ? bias[i] : 0.f;
      const bool on = row_epilogue<MODE, REGLU>([&](int c, float *v) { tmem_ld8(trow + (uint32_t)c, v); }, 0, Bp,
                                                i, k0 + q, bi, B, Bp, Nmma, abuf, abuf_ld, mask_out, silu != 0,
                                                RowScales{});
      if (MODE == kLogits) {            // active rows of the tile, for the ordered compaction
        const int n_on = __syncthreads_count(on && i >= 0);
        if (tid == 0) tile_cnt[tile] = n_on;
      }
    } else {
      float *dst = piece + (size_t)slot * ncolD * kTile + q;
      for (int c0 = 0; c0 < ncolD; c0 += 8) {
        float v[8];
        tmem_ld8(trow + (uint32_t)c0, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[(size_t)(c0 + j) * kTile] = v[j];
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
// E4M3 rows on the tensor cores.  The MMA takes fp16 operands, so each stage
// goes through shared memory twice: the codes of a stage are copied with
// 16-byte cp.async into a ring of raw stages (each thread copies, and later
// reads, its own stretch: 16 bytes of padding per stretch keep the reads of
// a quarter-warp on distinct banks), and once a thread's copies of the stage
// have landed (cp.async.wait_group) it converts them to fp16 in the
// 128-byte-swizzled operand buffer (E4M3 values are exact in fp16) and
// arrives on the stage's barrier.  With one operand buffer a stage is
// converted when the MMAs of the one before it completed, while kRaw stages
// of codes are in flight; with two (where they fit) the conversion overlaps
// the previous stage's MMAs and two raw stages are in flight.  The row
// scales enter the up epilogue (the W_down^T row scale multiplies the
// activation).
constexpr int kRaw = 3;

__device__ __forceinline__ void e4m3x16_to_half(const uint4 &q, uint4 &h0, uint4 &h1) {
  const __nv_fp8x2_storage_t *p = reinterpret_cast<const __nv_fp8x2_storage_t *>(&q);
  uint32_t o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(p[e], __NV_E4M3);
    o[e] = (uint32_t)r.x | ((uint32_t)r.y << 16);
  }
  h0 = make_uint4(o[0], o[1], o[2], o[3]);
  h1 = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ void mb_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}

// Up rows (kAct) of an E4M3 layer: Qg the gated rows (the up rows for ReLU),
// Qu the up rows of a gated layer.  Thread t owns row t of the tile.  NOP
// operand buffers: with two, the conversion of a stage overlaps the MMAs of
// the one before it (and two raw stages are in flight instead of three).
template <bool REGLU, int NOP>
__global__ void __launch_bounds__(128, 1) k_tc_rows_q8(const uint8_t *__restrict__ Qg, const uint8_t *__restrict__ Qu,
                                                       const __grid_constant__ CUtensorMap tm_x,
                                                       const int32_t *__restrict__ idx,
                                                       const int32_t *__restrict__ count_p, int count_const,
                                                       const float *__restrict__ bias, int d, int ffn, int B, int Bp,
                                                       int kw, __half *__restrict__ abuf, int abuf_ld,
                                                       float *__restrict__ piece, unsigned int *status, int silu,
                                                       RowScales sc) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  constexpr int NA = REGLU ? 2 : 1;
  const int Nmma = Bp;
  const int ncolD = NA * Nmma;
  const uint32_t slabA = kTile * 128;
  const uint32_t slabX = (uint32_t)Nmma * 128;
  const uint32_t subX = (slabX + 1023) & ~1023u;
  const uint32_t a_bytes = (uint32_t)kw * (NA * slabA + subX);   // the operand stage
  const uint32_t rrow = (uint32_t)kw * kSlab + 16;                // a thread's raw stretch per matrix
  const uint32_t raw_bytes = NA * kTile * rrow;                   // one raw stage
  constexpr int KR = NOP == 2 ? 2 : kRaw;                         // raw stages in the ring
  unsigned char *raw = sm + NOP * a_bytes;
  __shared__ __align__(8) unsigned long long full_s[NOP], empty_s[NOP], done_s;
  __shared__ int rows_s[kTile];
  __shared__ uint32_t taddr_s;
  __shared__ int fail_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ncols = tmem_cols_for(ncolD);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&taddr_s)), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int b = 0; b < NOP; ++b) {
      mb_init(su32(&full_s[b]), 129);   // 128 converting threads + the TMA expect_tx arrival
      mb_init(su32(&empty_s[b]), 1);
    }
    mb_init(su32(&done_s), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fail_s = 0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = taddr_s;
  pidev::griddep_wait();
  pidev::griddep_launch();

  int count = count_p ? *count_p : count_const;
  if (count < 0 || count > ffn) {
    if (tid == 0) atomicOr(status, PI_STATUS_BAD_COUNT);
    count = count < 0 ? 0 : ffn;
  }
  const int ntiles = (count + kTile - 1) / kTile;
  const int KT = d / (kSlab * kw);                      // stages per tile
  const long long I = (long long)ntiles * KT;
  const int G = active_ctas(gridDim.x, ntiles), cta = blockIdx.x;
  const long long rs = cta < G ? range_start(cta, I, G) : 0, re = cta < G ? range_start(cta + 1, I, G) : 0;
  const uint32_t idesc = idesc_f16(Nmma, kTile, false);
  const uint32_t my_raw = su32(raw) + (uint32_t)tid * rrow;
  uint32_t gst = 0;            // operand stages used so far (buffer gst % NOP)
  uint32_t done_phase = 0;

  for (long long s0 = rs; s0 < re;) {
    const int tile = (int)(s0 / KT);
    const int kb = (int)(s0 % KT);
    const int n = (int)min((long long)(KT - kb), re - s0);   // stages of this piece
    const bool whole = (n == KT);
    const int slot = 2 * cta + (s0 == rs ? 0 : 1);
    s0 += n;
    const int k0 = tile * kTile;
    rows_s[tid] = tile_row(idx, k0 + tid, count, ffn, status);
    __syncthreads();
    const int rid = rows_s[tid] >= 0 ? rows_s[tid] : 0;   // invalid / padding rows read row 0 (activation 0)
    const uint8_t *gsrc = Qg + (size_t)rid * d;
    const uint8_t *usrc = REGLU ? Qu + (size_t)rid * d : nullptr;
    auto issue_raw = [&](int kt, int rslot) {
      const uint32_t dst = my_raw + (uint32_t)rslot * raw_bytes;
      const int off = kt * kw * kSlab;                  // byte (= code) offset in the row
      for (int c = 0; c < 4 * kw; ++c) {
        cp16(dst + c * 16, gsrc + off + c * 16);
        if (REGLU) cp16(dst + kTile * rrow + c * 16, usrc + off + c * 16);
      }
    };
    for (int p = 0; p < KR; ++p) {
      if (p < n) issue_raw(kb + p, p);
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int it = 0; it < n; ++it) {
      if (fail_s) break;
      const uint32_t g = gst + (uint32_t)it;
      const int b = (int)(g % NOP);
      unsigned char *opA = sm + (size_t)b * a_bytes;
      const uint32_t full = su32(&full_s[b]), empty = su32(&empty_s[b]);
      // this buffer's previous stage: its MMAs are done
      if (g >= NOP && !mb_wait(empty, ((g / NOP) - 1) & 1)) fail_s = 1;
      if (tid == 0) {
        mb_expect(full, kw * slabX);
        for (int j = 0; j < kw; ++j)
          tma_tile2d(su32(opA + NA * kw * slabA + j * subX), &tm_x, ((kb + it) * kw + j) * kSlab, 0, full);
      }
      asm volatile("cp.async.wait_group %0;" ::"n"(KR - 1) : "memory");
      {
        const unsigned char *src = raw + (size_t)(it % KR) * raw_bytes + (size_t)tid * rrow;
#pragma unroll
        for (int m = 0; m < NA; ++m)
          for (int j = 0; j < kw; ++j) {
            unsigned char *dstA = opA + (size_t)(m * kw + j) * slabA;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 q = *reinterpret_cast<const uint4 *>(src + m * kTile * rrow + j * kSlab + c * 16);
              uint4 h0, h1;
              e4m3x16_to_half(q, h0, h1);
              *reinterpret_cast<uint4 *>(dstA + sw128(tid, 2 * c)) = h0;
              *reinterpret_cast<uint4 *>(dstA + sw128(tid, 2 * c + 1)) = h1;
            }
          }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mb_arrive(full);
      if (it + KR < n) issue_raw(kb + it + KR, it % KR);
      asm volatile("cp.async.commit_group;" ::: "memory");
      if (tid == 0) {
        if (!mb_wait(full, (g / NOP) & 1)) {
          fail_s = 1;
        } else {
          asm volatile("tcgen05.fence::after_thread_sync;");
          for (int j = 0; j < kw; ++j) {
            const uint32_t xa = su32(opA + NA * kw * slabA + j * subX);
            const uint32_t aa = su32(opA + j * slabA);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = sdesc(xa + kk * 32, 16, 1024);
              const uint32_t acc = (it | j | kk) ? 1u : 0u;
              mma_f16(tmem, sdesc(aa + kk * 32, 16, 1024), bd, idesc, acc);
              if (REGLU) mma_f16(tmem + (uint32_t)Nmma, sdesc(aa + kw * slabA + kk * 32, 16, 1024), bd, idesc, acc);
            }
          }
          mma_commit(empty);
        }
      }
    }
    gst += (uint32_t)n;
    if (tid == 0) mma_commit(su32(&done_s));
    __syncthreads();
    if (fail_s) break;
    if (!mb_wait(su32(&done_s), done_phase)) { fail_s = 1; break; }
    done_phase ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;");
    const int q = warp * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    if (whole) {
      const int i = rows_s[q];
      const float bi = (i >= 0 && bias) ? bias[i] : 0.f;
      row_epilogue<kAct, REGLU>([&](int c, float *v) { tmem_ld8(trow + (uint32_t)c, v); }, 0, Bp, i, k0 + q, bi, B,
                                Bp, Nmma, abuf, abuf_ld, nullptr, silu != 0, sc);
    } else {
      float *dst = piece + (size_t)slot * ncolD * kTile + q;
      for (int c0 = 0; c0 < ncolD; c0 += 8) {
        float v[8];
        tmem_ld8(trow + (uint32_t)c0, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) dst[(size_t)(c0 + j) * kTile] = v[j];
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
  }
  // every copy this CTA issued lands before it leaves (the waits are bounded)
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (fail_s && tid == 0) {
    atomicOr(status, PI_STATUS_BARRIER_TIMEOUT);
    for (int b = 0; b < NOP; ++b) mb_wait(su32(&full_s[b]), 0), mb_wait(su32(&full_s[b]), 1);
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols));
}

// Tiles that k_tc_rows split between CTAs: block c finishes the tile whose
// last stage lies in CTA c's range when that tile started in an earlier CTA's
// range.  It adds the tile's pieces in CTA order and applies the epilogue;
// the block has 128 threads per group of token columns (thread = tile row),
// so each thread adds only its group's columns of the pieces.
template <int MODE, bool REGLU>
__global__ void __launch_bounds__(1024) k_tc_fixup(const float *__restrict__ piece, const int32_t *__restrict__ idx,
                                                   const int32_t *__restrict__ count_p, int count_const,
                                                   const float *__restrict__ bias, int ffn, int B, int Bp, int KT,
                                                   int grid, __half *__restrict__ abuf, int abuf_ld,
                                                   uint8_t *__restrict__ mask_out, int32_t *__restrict__ tile_cnt,
                                                   unsigned int *status, int silu, RowScales sc) {
  pidev::griddep_wait();
  pidev::griddep_launch();
  constexpr int NA = REGLU ? 2 : 1;
  const int Nmma = MODE == kLogits ? 2 * Bp : Bp;
  const int ncolD = NA * Nmma;
  int count = count_p ? *count_p : count_const;
  if (count < 0 || count > ffn) count = count < 0 ? 0 : ffn;    // flagged by k_tc_rows
  const int ntiles = (count + kTile - 1) / kTile;
  const long long I = (long long)ntiles * KT;
  const int G = active_ctas(grid, ntiles), c = blockIdx.x;
  if (c >= G) return;
  const long long rs = range_start(c, I, G), re = range_start(c + 1, I, G);
  if (rs >= re || rs % KT == 0) return;          // c's range starts a tile: it completes no split tile
  const int tile = (int)(rs / KT);
  const long long t0 = (long long)tile * KT, t1 = t0 + KT;
  if (re < t1) return;                           // the tile goes on in a later CTA
  __shared__ int slots_s[kMaxPieces];
  __shared__ int nslot_s;
  __shared__ unsigned char on_s[8][kTile];
  if (threadIdx.x == 0) {          // the tile's pieces, in CTA order
    int cf = c;
    while (cf > 0 && range_start(cf, I, G) > t0) --cf;
    int np = 0;
    for (int cc = cf; cc <= c; ++cc) {
      const long long a0 = range_start(cc, I, G), a1 = range_start(cc + 1, I, G);
      const long long p0 = a0 > t0 ? a0 : t0, p1 = a1 < t1 ? a1 : t1;
      if (p0 >= p1) continue;
      if (np == kMaxPieces) {          // more pieces than slots: cannot happen (see kCtasPerTile)
        atomicOr(status, PI_STATUS_BAD_COUNT);
        break;
      }
      slots_s[np++] = 2 * cc + (p0 == a0 ? 0 : 1);
    }
    nslot_s = np;
  }
  __syncthreads();
  const int np = nslot_s;
  const int q = threadIdx.x % kTile, grp = threadIdx.x / kTile, ngrp = blockDim.x / kTile;
  const int i = tile_row(idx, tile * kTile + q, count, ffn, status);
  const float bi = (i >= 0 && bias) ? bias[i] : 0.f;
  auto fetch8 = [&](int col, float *v) {
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = 0.f;
    for (int p0 = 0; p0 < np; p0 += 4) {     // four pieces' loads in flight, added in order
      float t[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (p0 + u < np) {
          const float *src = piece + ((size_t)slots_s[p0 + u] * ncolD + col) * kTile + q;
#pragma unroll
          for (int j = 0; j < 8; ++j) t[u][j] = src[(size_t)j * kTile];
        }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (p0 + u < np)
#pragma unroll
          for (int j = 0; j < 8; ++j) v[j] += t[u][j];
    }
  };
  bool on = false;
  for (int c0 = 8 * grp; c0 < Bp; c0 += 8 * ngrp)
    on |= row_epilogue<MODE, REGLU>(fetch8, c0, c0 + 8, i, tile * kTile + q, bi, B, Bp, Nmma, abuf, abuf_ld,
                                    nullptr, silu != 0, sc);
  if (MODE == kLogits) {
    on_s[grp][q] = on ? 1 : 0;
    __syncthreads();
    bool any = false;
    if (grp == 0) {
      for (int g2 = 0; g2 < ngrp; ++g2) any |= on_s[g2][q] != 0;
      if (i >= 0) mask_out[i] = any ? 1 : 0;
    }
    const int n_on = __syncthreads_count(grp == 0 && any && i >= 0);
    if (threadIdx.x == 0) tile_cnt[tile] = n_on;
  }
}

// Ordered compaction from the logits kernels' per-tile counts: block t writes
// the active rows of tile t (ascending) after the sum of the counts of the
// tiles before it; the last block writes the total.
__global__ void __launch_bounds__(kTile) k_compact_tiles(const uint8_t *__restrict__ mask,
                                                         const int32_t *__restrict__ tile_cnt, int ffn,
                                                         int32_t *__restrict__ idx, int32_t *__restrict__ count) {
  __shared__ int red_s[4];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  pidev::griddep_wait();
  pidev::griddep_launch();
  int pre = 0;
  for (int k = tid; k < t; k += kTile) pre += tile_cnt[k];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, o);
  const int row = t * kTile + tid;
  const bool on = row < ffn && mask[row] != 0;
  const unsigned bal = __ballot_sync(0xffffffffu, on);
  if (lane == 0) red_s[w] = pre;
  __syncthreads();
  const int base = red_s[0] + red_s[1] + red_s[2] + red_s[3];
  __syncthreads();
  if (lane == 0) red_s[w] = __popc(bal);
  __syncthreads();
  int wpre = 0;
  for (int k = 0; k < w; ++k) wpre += red_s[k];
  if (on) idx[base + wpre + __popc(bal & ((1u << lane) - 1u))] = row;
  if (t == gridDim.x - 1 && tid == 0) *count = base + red_s[0] + red_s[1] + red_s[2] + red_s[3];
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128, 1) k_tc_down(const __half *__restrict__ Wd,                  // W_down^T
                                                    const __grid_constant__ CUtensorMap tm_a,   // abuf, box 64 x 2Bp
                                                    const int32_t *__restrict__ idx, const int32_t *__restrict__ count_p,
                                                    int count_const, int d, int ffn, int B, int Bp, int nstage,
                                                    int cw, float *__restrict__ piece, unsigned int *status) {
  // Work units are (column tile of cw * 128 outputs, 64-row slab of the
  // list), column-tile major, split stream-K style over the CTAs: each CTA
  // accumulates its consecutive slabs of one column tile in TMEM (cw * 256
  // contiguous bytes of every gathered W_down^T row per slab) and writes the
  // sum as one fp32 piece [B, cw * 128] to slot 2c (its first piece) or
  // 2c + 1 (its last); k_tc_down_reduce adds each column tile's pieces in CTA
  // order.
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  const int N2 = 2 * Bp;
  const uint32_t half_bytes = kSlab * 128;                // 64 rows x 64 columns
  const uint32_t tileW = 2 * half_bytes;                  // 128 columns
  const uint32_t slabW = (uint32_t)cw * tileW;
  const uint32_t slabA = (uint32_t)N2 * 128;
  const uint32_t stage_bytes = slabW + ((slabA + 1023) & ~1023u);
  const int CW = cw * kTile;                              // outputs per column tile
  __shared__ __align__(8) unsigned long long full_s[8], empty_s[8], done_s;
  __shared__ uint32_t taddr_s;
  __shared__ int fail_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
  pidev::griddep_wait();
  pidev::griddep_launch();

  int count = count_p ? *count_p : count_const;
  if (count < 0 || count > ffn) count = count < 0 ? 0 : ffn;     // flagged by the up kernel
  const int KS = (count + kSlab - 1) / kSlab;
  const int ctiles = (d + CW - 1) / CW;
  const long long I = (long long)ctiles * KS;
  const int G = active_ctas(gridDim.x, ctiles), cta = blockIdx.x;
  const long long rs = cta < G ? range_start(cta, I, G) : 0, re = cta < G ? range_start(cta + 1, I, G) : 0;
  const uint32_t idesc = idesc_f16(N2, kTile, true);
  // Every thread copies 16 of the 2048 16-byte chunks of a slab: chunk
  // c = tid % 8 of column half (tid / 8) % 2 of rows tid / 16 + 8 i, into the
  // MN-major swizzled layout (8 rows of 128 bytes per 1024-byte group);
  // thread 0 also loads the [a_hi; a_lo] slab by TMA and issues the MMAs.
  const int cch = tid & 7, hh = (tid >> 3) & 1, r0 = tid >> 4;
  uint32_t gpos = 0, done_phase = 0;

  for (long long s0 = rs; s0 < re;) {
    const int tile = (int)(s0 / KS);
    const int kb = (int)(s0 % KS);
    const int n = (int)min((long long)(KS - kb), re - s0);   // slabs of this piece
    const int slot = 2 * cta + (s0 == rs ? 0 : 1);
    s0 += n;
    const int j0 = tile * CW;
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
    load_rows(kb);
    auto issue = [&](int it) {
      const uint32_t g = gpos + (uint32_t)it;
      const int s = (int)(g % (uint32_t)nstage);
      if (g >= (uint32_t)nstage && !mb_wait(su32(&empty_s[s]), ((g / nstage) - 1) & 1)) fail_s = 1;
      unsigned char *st = sm + (size_t)s * stage_bytes;
      const uint32_t bar = su32(&full_s[s]);
      const int slab = kb + it;
      int cur[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
      if (it + 1 < n) load_rows(slab + 1);
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
    const int pre = min(nstage - 1, n);
    for (int it = 0; it < pre; ++it) issue(it);
    for (int it = 0; it < n; ++it) {
      if (fail_s) break;
      if (it + nstage - 1 < n) issue(it + nstage - 1);
      if (tid == 0) {
        const uint32_t g = gpos + (uint32_t)it;
        const int s = (int)(g % (uint32_t)nstage);
        if (!mb_wait(su32(&full_s[s]), (g / nstage) & 1)) {
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
              mma_f16(tmem + (uint32_t)(c * N2), ad, bd, idesc, (it | kk) ? 1u : 0u);
            }
          mma_commit(su32(&empty_s[s]));
        }
      }
    }
    gpos += (uint32_t)n;
    if (tid == 0) mma_commit(su32(&done_s));
    __syncthreads();
    if (fail_s) break;
    if (!mb_wait(su32(&done_s), done_phase)) { fail_s = 1; break; }
    done_phase ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;");
    for (int c = 0; c < cw; ++c) {
      const int jl = c * kTile + warp * 32 + lane;           // TMEM lane = output column
      const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c * N2);
      float *dst = piece + (size_t)slot * B * CW + jl;
      for (int c0 = 0; c0 < Bp; c0 += 8) {
        float hi[8], lo[8];
        tmem_ld8(trow + (uint32_t)c0, hi);
        tmem_ld8(trow + (uint32_t)(Bp + c0), lo);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (c0 + q < B) dst[(size_t)(c0 + q) * CW] = hi[q] + lo[q];
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
  }
  if (fail_s && tid == 0) {
    atomicOr(status, PI_STATUS_BARRIER_TIMEOUT);
    for (int s = 0; s < nstage; ++s) mb_wait(su32(&full_s[s]), 0), mb_wait(su32(&full_s[s]), 1);
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols));
}

// W_down^T rows of an E4M3 layer (the row scales are in the activations):
// the units, pieces and MMAs of k_tc_down; thread t copies and converts half
// of row t / 2 of the slab's codes for the column tile (cw * 64 codes); NOP
// operand buffers as in k_tc_rows_q8.
template <int NOP>
__global__ void __launch_bounds__(128, 1) k_tc_down_q8(const uint8_t *__restrict__ Qd,
                                                       const __grid_constant__ CUtensorMap tm_a,
                                                       const int32_t *__restrict__ idx,
                                                       const int32_t *__restrict__ count_p, int count_const, int d,
                                                       int ffn, int B, int Bp, int cw, float *__restrict__ piece,
                                                       unsigned int *status) {
  extern __shared__ __align__(1024) unsigned char smraw[];
  unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~(uintptr_t)1023);
  const int N2 = 2 * Bp;
  const uint32_t half_bytes = kSlab * 128;                // 64 rows x 64 columns
  const uint32_t tileW = 2 * half_bytes;                  // 128 columns
  const uint32_t slabW = (uint32_t)cw * tileW;
  const uint32_t slabA = (uint32_t)N2 * 128;
  const uint32_t a_bytes = slabW + ((slabA + 1023) & ~1023u);
  const uint32_t rrow = (uint32_t)cw * 64 + 16;           // a thread's raw stretch (cw * 64 codes + padding)
  const uint32_t raw_bytes = kTile * rrow;
  const int CW = cw * kTile;                              // outputs per column tile
  constexpr int KR = NOP == 2 ? 2 : kRaw;                 // raw stages in the ring
  unsigned char *raw = sm + NOP * a_bytes;
  __shared__ __align__(8) unsigned long long full_s[NOP], empty_s[NOP], done_s;
  __shared__ uint32_t taddr_s;
  __shared__ int fail_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ncols = tmem_cols_for(cw * N2);
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&taddr_s)), "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int b = 0; b < NOP; ++b) {
      mb_init(su32(&full_s[b]), 129);
      mb_init(su32(&empty_s[b]), 1);
    }
    mb_init(su32(&done_s), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fail_s = 0;
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;");
  const uint32_t tmem = taddr_s;
  pidev::griddep_wait();
  pidev::griddep_launch();

  int count = count_p ? *count_p : count_const;
  if (count < 0 || count > ffn) count = count < 0 ? 0 : ffn;     // flagged by the up kernel
  const int KS = (count + kSlab - 1) / kSlab;
  const int ctiles = (d + CW - 1) / CW;
  const long long I = (long long)ctiles * KS;
  const int G = active_ctas(gridDim.x, ctiles), cta = blockIdx.x;
  const long long rs = cta < G ? range_start(cta, I, G) : 0, re = cta < G ? range_start(cta + 1, I, G) : 0;
  const uint32_t idesc = idesc_f16(N2, kTile, true);
  const int q = tid >> 1, hb = tid & 1;                   // row of the slab, half of its codes
  const uint32_t my_raw = su32(raw) + (uint32_t)tid * rrow;
  uint32_t gst = 0, done_phase = 0;

  for (long long s0 = rs; s0 < re;) {
    const int tile = (int)(s0 / KS);
    const int kb = (int)(s0 % KS);
    const int n = (int)min((long long)(KS - kb), re - s0);   // slabs of this piece
    const int slot = 2 * cta + (s0 == rs ? 0 : 1);
    s0 += n;
    const int j0 = tile * CW;
    auto issue_raw = [&](int slab, int rslot) {
      const int k = slab * kSlab + q;
      int rid = k < count ? (idx ? idx[k] : k) : 0;
      if (rid < 0 || rid >= ffn) rid = 0;                   // padding / invalid: row 0 times a zero activation
      const uint32_t dst = my_raw + (uint32_t)rslot * raw_bytes;
      const int col0 = j0 + hb * cw * 64;
      for (int c = 0; c < 4 * cw; ++c) {
        const int col = col0 + 16 * c;
        cp16(dst + c * 16, Qd + (size_t)rid * d + (col < d ? col : 0));   // a column past d: output dropped
      }
    };
    for (int p = 0; p < KR; ++p) {
      if (p < n) issue_raw(kb + p, p);
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    for (int it = 0; it < n; ++it) {
      if (fail_s) break;
      const uint32_t g = gst + (uint32_t)it;
      const int b = (int)(g % NOP);
      unsigned char *opA = sm + (size_t)b * a_bytes;
      const uint32_t full = su32(&full_s[b]), empty = su32(&empty_s[b]);
      if (g >= NOP && !mb_wait(empty, ((g / NOP) - 1) & 1)) fail_s = 1;
      if (tid == 0) {
        mb_expect(full, slabA);
        tma_tile2d(su32(opA + slabW), &tm_a, (kb + it) * kSlab, 0, full);
      }
      asm volatile("cp.async.wait_group %0;" ::"n"(KR - 1) : "memory");
      {
        const unsigned char *src = raw + (size_t)(it % KR) * raw_bytes + (size_t)tid * rrow;
        for (int c = 0; c < 4 * cw; ++c) {
          const uint4 qv = *reinterpret_cast<const uint4 *>(src + c * 16);
          uint4 h[2];
          e4m3x16_to_half(qv, h[0], h[1]);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int colr = hb * cw * 64 + 16 * c + 8 * e;   // column within the unit
            const int ct = colr >> 7, hh = (colr >> 6) & 1, cch = (colr >> 3) & 7;
            *reinterpret_cast<uint4 *>(opA + ct * tileW + hh * half_bytes + sw128(q, cch)) = h[e];
          }
        }
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mb_arrive(full);
      if (it + KR < n) issue_raw(kb + it + KR, it % KR);
      asm volatile("cp.async.commit_group;" ::: "memory");
      if (tid == 0) {
        if (!mb_wait(full, (g / NOP) & 1)) {
          fail_s = 1;
        } else {
          asm volatile("tcgen05.fence::after_thread_sync;");
          for (int c = 0; c < cw; ++c)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = sdesc(su32(opA) + c * tileW + kk * 16 * 128, half_bytes, 1024);
              const uint64_t bd = sdesc(su32(opA + slabW) + kk * 32, 16, 1024);
              mma_f16(tmem + (uint32_t)(c * N2), ad, bd, idesc, (it | kk) ? 1u : 0u);
            }
          mma_commit(empty);
        }
      }
    }
    gst += (uint32_t)n;
    if (tid == 0) mma_commit(su32(&done_s));
    __syncthreads();
    if (fail_s) break;
    if (!mb_wait(su32(&done_s), done_phase)) { fail_s = 1; break; }
    done_phase ^= 1u;
    asm volatile("tcgen05.fence::after_thread_sync;");
    for (int c = 0; c < cw; ++c) {
      const int jl = c * kTile + warp * 32 + lane;           // TMEM lane = output column
      const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c * N2);
      float *dst = piece + (size_t)slot * B * CW + jl;
      for (int c0 = 0; c0 < Bp; c0 += 8) {
        float hi[8], lo[8];
        tmem_ld8(trow + (uint32_t)c0, hi);
        tmem_ld8(trow + (uint32_t)(Bp + c0), lo);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (c0 + e < B) dst[(size_t)(c0 + e) * CW] = hi[e] + lo[e];
      }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (fail_s && tid == 0) {
    atomicOr(status, PI_STATUS_BARRIER_TIMEOUT);
    for (int b = 0; b < NOP; ++b) mb_wait(su32(&full_s[b]), 0), mb_wait(su32(&full_s[b]), 1);
  }
  asm volatile("tcgen05.fence::before_thread_sync;");
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols));
}

// y[b, j] = the pieces of j's column tile added in CTA order (0 for an empty
// list).  Block (tile, b), one thread per column of the tile (up to 512):
// thread 0 lists the tile's pieces once for the block.
__global__ void __launch_bounds__(512) k_tc_down_reduce(const float *__restrict__ piece,
                                                        const int32_t *__restrict__ count_p, int count_const, int d,
                                                        int ffn, int B, int CW, int grid, float *__restrict__ y) {
  __shared__ int slots_s[2 * kCtasPerTile + 4];
  __shared__ int nslot_s;
  const int tile = blockIdx.x, b = blockIdx.y;
  pidev::griddep_wait();
  pidev::griddep_launch();
  int count = count_p ? *count_p : count_const;
  if (count < 0 || count > ffn) count = count < 0 ? 0 : ffn;
  const long long KS = (count + kSlab - 1) / kSlab;
  const int ctiles = (d + CW - 1) / CW;
  const long long I = (long long)ctiles * KS;
  if (threadIdx.x == 0) {
    int np = 0;
    if (KS > 0) {
      const int G = active_ctas(grid, ctiles);
      const long long t0 = tile * KS, t1 = t0 + KS;
      // CTA holding iteration x: the largest c with c * I / G <= x
      const int cf = (int)(((t0 + 1) * G + I - 1) / I) - 1;
      const int cl = (int)((t1 * G + I - 1) / I) - 1;
      for (int cc = cf; cc <= cl && np < 2 * kCtasPerTile + 4; ++cc) {
        const long long a0 = range_start(cc, I, G), a1 = range_start(cc + 1, I, G);
        const long long p0 = a0 > t0 ? a0 : t0, p1 = a1 < t1 ? a1 : t1;
        if (p0 < p1) slots_s[np++] = 2 * cc + (p0 == a0 ? 0 : 1);
      }
    }
    nslot_s = np;
  }
  __syncthreads();
  const int jl = threadIdx.x, j = tile * CW + jl;
  if (jl >= CW || j >= d) return;
  float acc = 0.f;
  for (int p = 0; p < nslot_s; ++p) acc += piece[((size_t)slots_s[p] * B + b) * CW + jl];
  y[(size_t)b * d + j] = acc;
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

constexpr size_t kTcSmemBudget = 200 * 1024;

// Launch k_tc_rows over nrows candidate rows (count_const, or *count on the
// device when count is given) and then k_tc_fixup for the tiles it split.
// rows_known: the row count is known here (the predictor), so the stage
// width can be chosen to give every active CTA at least one stage; otherwise
// the widest stage is taken (most contiguous bytes per gathered row).
template <int MODE, bool REGLU>
cudaError_t launch_rows(const pi_layer *L, const __half *Wg, const __half *Wu, const CUtensorMap &tm_x,
                        const int32_t *idx, const int32_t *count, int count_const, const float *bias, int K,
                        int wld, int nrows, int B, int Bp, __half *out, int out_ld, uint8_t *mask, float *piece,
                        int32_t *tile_cnt, bool rows_known, cudaStream_t s, int silu = 0) {
  const int NA = REGLU ? 2 : 1;
  const int Nmma = MODE == kLogits ? 2 * Bp : Bp;
  const size_t sub = NA * (size_t)kTile * 128 + (((size_t)Nmma * 128 + 1023) & ~(size_t)1023);
  const int slabs = K / kSlab;
  const long long tiles = (nrows + kTile - 1) / kTile;
  const int G = L->num_sms;
  // widest stage (kw consecutive slabs per row) that divides K and keeps >= 2
  // stages; with a known row count, also >= G stages over all tiles
  int kw = 4;
  while (kw > 1 && (slabs % kw != 0 || (kTcSmemBudget - 1024) / (kw * sub) < 2 ||
                    (rows_known && tiles * (slabs / kw) < std::min<long long>(G, tiles * kCtasPerTile))))
    kw >>= 1;
  const size_t stage = kw * sub;
  int ns = (int)((kTcSmemBudget - 1024) / stage);
  if (ns > 8) ns = 8;
  if (ns < 2) return cudaErrorInvalidValue;
  const size_t smem = 1024 + ns * stage;
  auto kern = k_tc_rows<MODE, REGLU>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = pi::launch_pdl(kern, dim3(G), dim3(128), smem, s, Wg, Wu, tm_x, idx, count, count_const, bias, K, wld, nrows,
                     B, Bp, ns, kw, out, out_ld, piece, mask, tile_cnt, L->status, silu);
  if (e != cudaSuccess) return e;
  const int groups = std::min(Bp / 8, 8);       // 128 threads per group of token columns
  return pi::launch_pdl(k_tc_fixup<MODE, REGLU>, dim3(G), dim3(kTile * groups), 0, s, piece, idx, count, count_const,
                        bias, nrows, B, Bp, slabs / kw, G, out, out_ld, mask, tile_cnt, L->status, silu, RowScales{});
}

// The E4M3 up kernel and its fix-up: the widest stage (kw slabs), with two
// operand buffers and two raw stages if they fit in kQ8Smem2 bytes of shared
// memory, else with one operand buffer and kRaw raw stages.
constexpr size_t kQ8Smem2 = 225 * 1024;

template <bool REGLU>
cudaError_t launch_rows_q8(const pi_layer *L, const CUtensorMap &tm_x, const int32_t *idx, const int32_t *count,
                           int count_const, int B, int Bp, __half *out, int out_ld, float *piece, cudaStream_t s,
                           int silu) {
  constexpr int NA = REGLU ? 2 : 1;
  const size_t subX = ((size_t)Bp * 128 + 1023) & ~(size_t)1023;
  const int slabs = L->d / kSlab;
  int kw = 4, nop = 0;
  size_t smem = 0;
  for (; kw >= 1 && nop == 0; kw >>= 1) {
    if (slabs % kw != 0) continue;
    const size_t a = (size_t)kw * (NA * (size_t)kTile * 128 + subX);
    const size_t raw = (size_t)NA * kTile * (kw * kSlab + 16);
    if (1024 + 2 * a + 2 * raw <= kQ8Smem2) {
      nop = 2;
      smem = 1024 + 2 * a + 2 * raw;
    } else if (1024 + a + kRaw * raw <= kTcSmemBudget) {
      nop = 1;
      smem = 1024 + a + kRaw * raw;
    }
    if (nop) break;
  }
  if (nop == 0) return cudaErrorInvalidValue;
  RowScales sc;
  sc.g = REGLU ? L->s_gate : L->s_up;
  sc.u = REGLU ? L->s_up : nullptr;
  sc.d = L->s_dT;
  const uint8_t *Qg = REGLU ? L->Q_gate : L->Q_up;
  const uint8_t *Qu = REGLU ? L->Q_up : nullptr;
  const int G = L->num_sms;
  auto kern = nop == 2 ? k_tc_rows_q8<REGLU, 2> : k_tc_rows_q8<REGLU, 1>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = pi::launch_pdl(kern, dim3(G), dim3(128), smem, s, Qg, Qu, tm_x, idx, count, count_const, (const float *)L->b,
                     L->d, L->ffn, B, Bp, kw, out, out_ld, piece, L->status, silu, sc);
  if (e != cudaSuccess) return e;
  const int groups = std::min(Bp / 8, 8);
  return pi::launch_pdl(k_tc_fixup<kAct, REGLU>, dim3(G), dim3(kTile * groups), 0, s, piece, idx, count, count_const,
                        (const float *)L->b, L->ffn, B, Bp, slabs / kw, G, out, out_ld, (uint8_t *)nullptr,
                        (int32_t *)nullptr, L->status, silu, sc);
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

size_t tc_piece_bytes(const pi_layer *L, int B) {
  // two slots per CTA: 128 rows x (at most 2 Bp) fp32 accumulator columns of
  // the row kernels, or B x (cw * 128) outputs of the down kernel
  const size_t cols = (size_t)kTile * (kDownCwMax > 2 ? kDownCwMax : 2);
  return sizeof(float) * 2 * (size_t)L->num_sms * cols * (size_t)tc_bpad(B);
}

cudaError_t run_predict_tc(const pi_layer *L, const __half *x, int B, uint8_t *mask_union, __half *hbuf,
                           float *piece, int32_t *tile_cnt, int32_t *idx, int32_t *count, cudaStream_t s) {
  const int Bp = tc_bpad(B);
  const int rpad = tc_rank_pad(L);
  CUtensorMap tm_x, tm_h;
  if (!encode_2d(&tm_x, x, L->d, B, (uint64_t)L->d * 2, kSlab, Bp) ||
      !encode_2d(&tm_h, hbuf, rpad, 2 * Bp, (uint64_t)rpad * 2, kSlab, 2 * Bp))
    return cudaErrorInvalidValue;
  // h = ReLU(W_p1 x) as an fp16 pair, then l = W_p2 h + c_p -> union mask
  // and per-tile counts, then the ordered list of active neurons
  cudaError_t e = launch_rows<kHidden, false>(L, L->W_p1, nullptr, tm_x, nullptr, nullptr, L->rank, nullptr, L->d, L->d,
                                              rpad, B, Bp, hbuf, rpad, nullptr, piece, nullptr, true, s);
  if (e != cudaSuccess) return e;
  e = launch_rows<kLogits, false>(L, L->W_p2, nullptr, tm_h, nullptr, nullptr, L->ffn, L->c_p, L->rank, L->p2_ld, L->ffn, B,
                                  Bp, nullptr, 0, mask_union, piece, tile_cnt, true, s);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_compact_tiles, dim3((L->ffn + kTile - 1) / kTile), dim3(kTile), 0, s, mask_union, tile_cnt,
                    L->ffn, idx, count);
}

cudaError_t run_sparse_ffn_tc(const pi_layer *L, const __half *x, int B, const int32_t *idx,
                              const int32_t *count, int count_const, float *y, const WsLayout &w,
                              char *ws, cudaStream_t s) {
  const bool reglu = L->act != PI_ACT_RELU;      // gated: ReGLU or SwiGLU
  const int silu = L->act == PI_ACT_SWIGLU ? 1 : 0;
  const int Bp = tc_bpad(B);
  const int ffn_pad = tc_ffn_pad(L);
  __half *abuf = reinterpret_cast<__half *>(ws + w.abuf);
  float *piece = reinterpret_cast<float *>(ws + w.tcpart);   // split tiles of the up and down kernels
  CUtensorMap tm_x, tm_a;
  const uint64_t row_bytes = (uint64_t)L->d * 2;
  if (!encode_2d(&tm_x, x, L->d, B, row_bytes, kSlab, Bp) ||
      !encode_2d(&tm_a, abuf, ffn_pad, 2 * Bp, (uint64_t)ffn_pad * 2, kSlab, 2 * Bp))
    return cudaErrorInvalidValue;

  const bool q8 = L->row_format == PI_ROWS_FP8_E4M3;
  cudaError_t e = record_hook(L->ev_before, s);
  if (e != cudaSuccess) return e;
  if (q8)
    e = reglu ? launch_rows_q8<true>(L, tm_x, idx, count, count_const, B, Bp, abuf, ffn_pad, piece, s, silu)
              : launch_rows_q8<false>(L, tm_x, idx, count, count_const, B, Bp, abuf, ffn_pad, piece, s, silu);
  else
    e = reglu ? launch_rows<kAct, true>(L, L->W_gate, L->W_up, tm_x, idx, count, count_const, L->b, L->d, L->d, L->ffn,
                                        B, Bp, abuf, ffn_pad, nullptr, piece, nullptr, false, s, silu)
              : launch_rows<kAct, false>(L, L->W_up, nullptr, tm_x, idx, count, count_const, L->b, L->d, L->d, L->ffn,
                                         B, Bp, abuf, ffn_pad, nullptr, piece, nullptr, false, s);
  if (e != cudaSuccess) return e;

  // down: stages of cw x 16 KB gathered W_down^T + the [a_hi; a_lo] slab
  // (E4M3 rows: one or two such operand stages and raw stages of cw x 8 KB)
  int cw = kDownCwMax;
  while (cw > 1 && (L->d % (cw * kTile) != 0 || cw * 2 * Bp > 512)) cw >>= 1;
  const size_t act_slab = ((size_t)2 * Bp * 128 + 1023) & ~(size_t)1023;
  if (q8) {
    size_t dn_smem = 0;
    int nop = 0;
    for (;; cw >>= 1) {
      const size_t a = cw * 2 * (size_t)kSlab * 128 + act_slab;
      const size_t raw = (size_t)kTile * (cw * 64 + 16);
      if (1024 + 2 * a + 2 * raw <= kQ8Smem2) {
        nop = 2;
        dn_smem = 1024 + 2 * a + 2 * raw;
      } else if (1024 + a + kRaw * raw <= kTcSmemBudget) {
        nop = 1;
        dn_smem = 1024 + a + kRaw * raw;
      }
      if (nop || cw == 1) break;
    }
    if (nop == 0) return cudaErrorInvalidValue;
    auto dkern = nop == 2 ? k_tc_down_q8<2> : k_tc_down_q8<1>;
    e = cudaFuncSetAttribute(dkern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dn_smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(dkern, dim3(L->num_sms), dim3(128), dn_smem, s, (const uint8_t *)L->Q_dT, tm_a, idx, count,
                   count_const, L->d, L->ffn, B, Bp, cw, piece, L->status);
  } else {
    const size_t dn_stage = cw * 2 * (size_t)kSlab * 128 + act_slab;
    int dn_ns = (int)((kTcSmemBudget - 1024) / dn_stage);
    if (dn_ns > 8) dn_ns = 8;
    if (dn_ns < 2) return cudaErrorInvalidValue;
    const size_t dn_smem = 1024 + dn_ns * dn_stage;
    e = cudaFuncSetAttribute(k_tc_down, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dn_smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(k_tc_down, dim3(L->num_sms), dim3(128), dn_smem, s, L->W_dT, tm_a, idx, count, count_const, L->d,
                   L->ffn, B, Bp, dn_ns, cw, piece, L->status);
  }
  if (e != cudaSuccess) return e;
  e = record_hook(L->ev_after, s);
  if (e != cudaSuccess) return e;
  const int CW = cw * kTile;
  return launch_pdl(k_tc_down_reduce, dim3((L->d + CW - 1) / CW, B), dim3(CW), 0, s, piece, count, count_const, L->d,
                    L->ffn, B, CW, L->num_sms, y);
}

}  // namespace pi
