// Per-group clipping search on the tensor cores ("AWQ (activation-aware
// weight quantization)", "Simplifications": the method also searches a
// clipping threshold per group, shrinking the max range; "AWQ vs GPTQ ...",
// "AWQ: move the error away from what matters": a second search shrinks
// each group's clipping range when that lowers output error).
//
// For row r, group G (128 columns) and shrink factor c the group's own share
// of the row's output error is
//   e(r, G, c) = sum_n (sum_{j in G} (X / s)[n, j] * D_c[r, j])^2,
//   D_c = Q_c(t) - t,  t = W * s,
// which is the square sum of one row of the product D_c (128 rows x 128 K)
// times (X / s)_G^T (128 K x N tokens): the search's error GEMM restricted to
// one group.  Here both operands come from shared memory in the 128-byte
// swizzled K-major layout: X / s (fp16, scaled by 2^m) by TMA, and D_c
// (fp16, scaled by 2^e) written there by the producers.
//
// Work item = (128-row tile, group); the items are spread evenly over the
// persistent CTAs (a contiguous range each).  Roles (512 threads):
//   warp 0      TMA loads: the item's two W blocks (128 rows x 64 columns)
//               into a two-stage ring, its two X / s blocks (N tokens x 64
//               columns) into a three-stage ring
//   warp 1      the single tcgen05.mma issuer
//   warp 2      tensor memory owner (512 columns: two accumulators of 256)
//   warpgroups 1 and 2 (producers, thread = row): warpgroup 1 takes the
//               group's first 64 columns, warpgroup 2 the second.  Per item
//               each forms t of its half and the whole group's range (the
//               other half's products only for the range), then for every
//               factor writes D_c of its half into a shared-memory slot (two
//               slots, each both halves of one factor).
//   warpgroup 3 (epilogue, thread = row): per factor, the accumulator's
//               row square sum; keeps the first factor with the smallest
//               share (strict <) and writes clip[r][G] (and the shares).
// Every wait is bounded as in the search kernel.
//
// Rounding as in the search kernel's producers: t * (1/scale) rounded with
// one fused multiply-add against 1.5 * 2^23, clamped to the quantizer's code
// range (the clipped range leaves values beyond it on the end codes).  Next
// to an exact half-integer this can round the other way than the correctly
// rounded quotient; either neighbour is half a step away, so only that
// entry's error changes sign, far below the fp16 rounding of the operands.
#include <algorithm>


#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

constexpr int kCThreads = 512;
constexpr int kCRows = 128;
constexpr int kCKB = 64;  // K columns per block
constexpr int kCG = 128;  // group width of this path
constexpr int kCSW = 2;   // W stages (one item)
constexpr int kCSX = 3;   // X stages
constexpr int kCSlots = 2;
constexpr uint32_t kCW_TILE = kCRows * kCKB * 2;  // 16 KB
constexpr uint32_t kCD_SLOT = 2 * kCW_TILE;       // both halves of one factor
constexpr uint32_t kCCtrl = 2048;
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
constexpr uint32_t kCRegsCtl = 48, kCRegsProd = 200, kCRegsEpi = 64;
static_assert(128 * kCRegsCtl + 256 * kCRegsProd + 128 * kCRegsEpi <= kCThreads * 128,
              "register split");

struct ClipCtrl {
  uint64_t w_full[kCSW], w_empty[kCSW];
  uint64_t x_full[kCSX], x_empty[kCSX];
  uint64_t d_full[kCSlots], d_empty[kCSlots];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  float factors[kMaxClip];  // the kernel argument's factors, indexable without local memory
};
static_assert(sizeof(ClipCtrl) <= kCCtrl, "control block too large");

struct ClipMmaArgs {
  int out, in, T, ngroups, n_items, nf;
  float factors[kMaxClip];
  float Lf, maxqf;
  const float* ss;    // [in] s * 2^e
  const float* ctl;   // {1e-8 * 2^e, 2^-2(e + m)}
  float* clip;        // [out][ngroups]
  float* errs;        // [out][ngroups][nf] or null
  int32_t* status;
  uint32_t* diag;
  uint64_t wait_limit_ns;
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <typename WT>
__device__ __forceinline__ void load_w8c(const uint8_t* stage, int row, int cc, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(stage + row * 128 + ((cc ^ (row & 7)) << 4));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (sizeof(WT) == 2 && std::is_same<WT, __half>::value) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    } else {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}

// This CTA's items [i0, i1): an even share of the (row tile, group) pairs.
__device__ __forceinline__ void item_range(int n_items, int& i0, int& i1) {
  i0 = (int)((int64_t)blockIdx.x * n_items / gridDim.x);
  i1 = (int)((int64_t)(blockIdx.x + 1) * n_items / gridDim.x);
}

template <typename WT, bool SYM>
__global__ void __launch_bounds__(kCThreads, 1)
    clip_mma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                    const ClipMmaArgs p) {
  extern __shared__ uint8_t csmem_raw[];
  const uint32_t raw = smem_addr(csmem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = csmem_raw + (base - raw);
  ClipCtrl& c = *reinterpret_cast<ClipCtrl*>(gbase);
  const uint32_t X_STAGE = (uint32_t)p.T * 128u;
  const uint32_t w_ring = base + kCCtrl;
  const uint32_t d_ring = w_ring + kCSW * kCW_TILE;
  const uint32_t x_ring = d_ring + kCSlots * kCD_SLOT;
  const uint8_t* w_ring_ptr = gbase + kCCtrl;
  uint8_t* d_ring_ptr = gbase + kCCtrl + kCSW * kCW_TILE;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kCSW; ++i) {
      mbar_init(smem_addr(&c.w_full[i]), 1);
      mbar_init(smem_addr(&c.w_empty[i]), 8);  // both producer warpgroups read both stages
    }
    for (int i = 0; i < kCSX; ++i) {
      mbar_init(smem_addr(&c.x_full[i]), 1);
      mbar_init(smem_addr(&c.x_empty[i]), 1);
    }
    for (int i = 0; i < kCSlots; ++i) {
      mbar_init(smem_addr(&c.d_full[i]), 8);
      mbar_init(smem_addr(&c.d_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&c.acc_full[i]), 1);
      mbar_init(smem_addr(&c.acc_empty[i]), 4);
    }
    mbar_init(smem_addr(&c.drain), 1);
    c.abort = 0;
#pragma unroll
    for (int i = 0; i < kMaxClip; ++i) c.factors[i] = p.factors[i];
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_addr(&c.tmem_base), 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&tmW);
    tma_prefetch_map(&tmX);
  }
  __syncthreads();
  tc_fence_after();
  pdl_wait();  // s * 2^e, X / s and the scalings come from earlier kernels
  const uint32_t tmem = c.tmem_base;
  volatile int* abort = &c.abort;
  const uint64_t lim = p.wait_limit_ns;
  int i0, i1;
  item_range(p.n_items, i0, i1);
  const int nf = p.nf;

  if (warp < 4) {
    setmaxnreg_dec<kCRegsCtl>();
    if (warp == 0) {
      // ---------------------------------------------------------- loader
      // (the whole warp runs the loop, the elected lane issues the copies)
      uint32_t wq = 0, xq = 0;
      bool ok = true;
      for (int it = i0; ok && it < i1; ++it) {
        const int rt = it / p.ngroups, g = it % p.ngroups;
        for (int kb = 0; ok && kb < 2; ++kb) {
          const uint32_t ws = wq % kCSW, wph = (wq / kCSW) & 1;
          ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.w_empty[ws]), wph ^ 1, abort, lim,
                                                 p.diag, 21, wq));
          if (!ok) break;
          if (elect_one()) {
            mbar_arrive_expect_tx(smem_addr(&c.w_full[ws]), kCW_TILE);
            tma_load_2d(w_ring + ws * kCW_TILE, &tmW, smem_addr(&c.w_full[ws]),
                        g * kCG + kb * kCKB, rt * kCRows);
          }
          __syncwarp();
          ++wq;
          const uint32_t xs = xq % kCSX, xph = (xq / kCSX) & 1;
          ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.x_empty[xs]), xph ^ 1, abort, lim,
                                                 p.diag, 22, xq));
          if (!ok) break;
          if (elect_one()) {
            mbar_arrive_expect_tx(smem_addr(&c.x_full[xs]), X_STAGE);
            tma_load_2d(x_ring + xs * X_STAGE, &tmX, smem_addr(&c.x_full[xs]),
                        g * kCG + kb * kCKB, 0);
          }
          __syncwarp();
          ++xq;
        }
      }
      int never_set = 0;  // drain the copies still in flight
      for (uint32_t m = wq > kCSW ? wq - kCSW : 0; m < wq; ++m)
        mbar_wait(smem_addr(&c.w_full[m % kCSW]), (m / kCSW) & 1, &never_set, lim);
      for (uint32_t m = xq > kCSX ? xq - kCSX : 0; m < xq; ++m)
        mbar_wait(smem_addr(&c.x_full[m % kCSX]), (m / kCSX) & 1, &never_set, lim);
    } else if (warp == 1) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_f16_f32(kCRows, (uint32_t)p.T);
      uint32_t xq = 0, fq = 0;  // X blocks and factors consumed
      bool ok = true;
      for (int it = i0; ok && it < i1; ++it) {
        uint32_t xs[2];
        for (int kb = 0; ok && kb < 2; ++kb) {
          xs[kb] = (xq + kb) % kCSX;
          ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.x_full[xs[kb]]),
                                                 ((xq + kb) / kCSX) & 1, abort, lim, p.diag, 23,
                                                 xq + kb));
        }
        if (!ok) break;
        for (int f = 0; ok && f < nf; ++f) {
          const uint32_t sl = fq % kCSlots, acc = fq & 1;
          ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.d_full[sl]), (fq / kCSlots) & 1,
                                                 abort, lim, p.diag, 24, fq));
          if (ok && fq >= 2)
            ok = __all_sync(0xffffffffu, mbar_wait(smem_addr(&c.acc_empty[acc]),
                                                   ((fq - 2) / 2) & 1, abort, lim, p.diag, 25,
                                                   fq));
          if (!ok) break;
          tc_fence_after();
          const uint32_t d_t = tmem + acc * 256u;
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            const uint64_t adesc = smem_desc_sw128(d_ring + sl * kCD_SLOT + kb * kCW_TILE);
            const uint64_t bdesc = smem_desc_sw128(x_ring + xs[kb] * X_STAGE);
#pragma unroll
            for (int k = 0; k < kCKB / 16; ++k)
              umma_ss_elect(d_t, adesc + (uint64_t)(2 * k), bdesc + (uint64_t)(2 * k), idesc,
                            (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit_elect(smem_addr(&c.d_empty[sl]));
          umma_commit_elect(smem_addr(&c.acc_full[acc]));
          ++fq;
        }
        if (!ok) break;
        umma_commit_elect(smem_addr(&c.x_empty[xs[0]]));
        umma_commit_elect(smem_addr(&c.x_empty[xs[1]]));
        xq += 2;
      }
      umma_commit_elect(smem_addr(&c.drain));
      int never_set = 0;
      mbar_wait(smem_addr(&c.drain), 0, &never_set, lim);
    }
  } else if (warp < 12) {
    // ------------------------------------------------------------ producers
    setmaxnreg_inc<kCRegsProd>();
    const int half = (warp - 4) >> 2;  // K block of the group this warpgroup takes
    const int row = (warp & 3) * 32 + lane;
    const float clampk = __ldg(p.ctl);
    uint32_t wq = 0, fq = 0;
    bool ok = true;
    for (int it = i0; ok && it < i1; ++it) {
      const int g = it % p.ngroups;
      // the item's two W blocks: stages (2 * item) and (2 * item + 1) of the ring
      for (int h = 0; ok && h < 2; ++h) {
        const uint32_t m = wq + h;
        ok = mbar_wait(smem_addr(&c.w_full[m % kCSW]), (m / kCSW) & 1, abort, lim, p.diag, 26, m);
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // pass 1: t = fl32(w * s * 2^e) of this half, and the group's range
      // over both halves (the other half's products only for the range)
      float t[kCKB];
      float r0 = 0.0f, r1 = 0.0f;  // sym: max|t|; asym: min(min t, 0), max(max t, 0)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = half ^ hh;
        const float* ssg = p.ss + (int64_t)g * kCG + h * kCKB;
        const uint8_t* stg = w_ring_ptr + ((wq + h) % kCSW) * kCW_TILE;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          float w8[8];
          load_w8c<WT>(stg, row, cc, w8);
          const float4 sa = __ldg(reinterpret_cast<const float4*>(ssg + cc * 8));
          const float4 sb = __ldg(reinterpret_cast<const float4*>(ssg + cc * 8 + 4));
          const float s8[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 tv =
                __fmul2_rn(make_float2(w8[e], w8[e + 1]), make_float2(s8[e], s8[e + 1]));
            if (hh == 0) {
              t[cc * 8 + e] = tv.x;
              t[cc * 8 + e + 1] = tv.y;
            }
            if (SYM) {
              r0 = fmax3f(r0, fabsf(tv.x), fabsf(tv.y));
            } else {
              r0 = fmin3f(r0, tv.x, tv.y);
              r1 = fmax3f(r1, tv.x, tv.y);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_addr(&c.w_empty[wq % kCSW]));
        mbar_arrive(smem_addr(&c.w_empty[(wq + 1) % kCSW]));
      }
      // pass 2: every factor's D = t - q * scale (fp16) into a slot
      for (int f = 0; ok && f < p.nf; ++f) {
        const float cf = c.factors[f];
        float scale, qlo, qhi;
        if (SYM) {
          scale = fmaxf(__fdiv_rn(__fmul_rn(cf, r0), p.Lf), clampk);
          qlo = kMagic - p.Lf - 1.0f;
          qhi = kMagic + p.Lf;
        } else {
          const float lo = __fmul_rn(cf, r0), hi = __fmul_rn(cf, r1);
          scale = fmaxf(__fdiv_rn(__fsub_rn(hi, lo), p.maxqf), clampk);
          const float zero = rintf(__fdiv_rn(-lo, scale));
          qlo = kMagic - zero;
          qhi = kMagic + p.maxqf - zero;
        }
        const float rcp = __frcp_rn(scale);
        const uint32_t sl = fq % kCSlots;
        ok = mbar_wait(smem_addr(&c.d_empty[sl]), ((fq / kCSlots) & 1) ^ 1, abort, lim, p.diag,
                       27, fq);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        uint8_t* dst = d_ring_ptr + sl * kCD_SLOT + half * kCW_TILE + row * 128;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 tv = make_float2(t[cc * 8 + 2 * e], t[cc * 8 + 2 * e + 1]);
            float2 av = __ffma2_rn(tv, make_float2(rcp, rcp), make_float2(kMagic, kMagic));
            av.x = fminf(fmaxf(av.x, qlo), qhi);
            av.y = fminf(fmaxf(av.y, qlo), qhi);
            const float2 qv = __fadd2_rn(av, make_float2(-kMagic, -kMagic));
            const float2 ev = __ffma2_rn(qv, make_float2(-scale, -scale), tv);  // t - q * scale
            __half2 h = __float22half2_rn(ev);
            pk[e] = *reinterpret_cast<uint32_t*>(&h);
          }
          *reinterpret_cast<uint4*>(dst + ((cc ^ (row & 7)) << 4)) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&c.d_full[sl]));
        ++fq;
      }
      wq += 2;
    }
    if (!ok) *abort = 1;
  } else {
    // ------------------------------------------------------------ epilogue
    setmaxnreg_dec<kCRegsEpi>();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
    const float unscale = __ldg(p.ctl + 1);
    uint32_t fq = 0;
    bool ok = true;
    for (int it = i0; ok && it < i1; ++it) {
      const int rt = it / p.ngroups, g = it % p.ngroups;
      const int64_t grow = (int64_t)rt * kCRows + row;
      const bool live = grow < p.out;
      float* erow = (p.errs != nullptr && live) ? p.errs + (grow * p.ngroups + g) * p.nf : nullptr;
      float best_e = 0.0f;
      int best = 0;
      for (int f = 0; ok && f < p.nf; ++f) {
        const uint32_t acc = fq & 1;
        ok = mbar_wait(smem_addr(&c.acc_full[acc]), (fq / 2) & 1, abort, lim, p.diag, 28, fq);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        float e = 0.0f;
        const uint32_t cb = tmem + lane_addr + acc * 256u;
        for (int cc = 0; cc < p.T; cc += 16) {
          uint32_t v[16];
          tmem_ld16(cb + (uint32_t)cc, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float x = __uint_as_float(v[i]);
            e = fmaf(x, x, e);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&c.acc_empty[acc]));
        e *= unscale;
        if (f == 0 || e < best_e) {
          best_e = e;
          best = f;
        }
        if (erow != nullptr) erow[f] = e;
        ++fq;
      }
      if (ok && live) p.clip[grow * p.ngroups + g] = c.factors[best];
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && c.abort) set_status(p.status, ST_TIMEOUT);
}

// ctl = {1e-8 * 2^e, 2^-2(e + m)}, ss = s * 2^e and xf = 2^m / s, from
// max|W| (bits in absmax[0]), max|X| (absmax[1]) and the extremes of s: the
// clipped rounding errors are at most max|t| <= max|W| * max(s) and
// |X / s| <= max|X| / min(s), each scaled into the fp16 range
// (pow2_exponent_for).  One CTA.
__global__ void __launch_bounds__(1024) clip_prep_kernel(const float* __restrict__ s, int64_t in,
                                                        const uint32_t* __restrict__ absmax,
                                                        float* __restrict__ ss,
                                                        float* __restrict__ xf,
                                                        float* __restrict__ ctl) {
  pdl_wait();
  pdl_trigger();
  float smax = 0.0f, smin = INFINITY;
  for (int64_t j = threadIdx.x; j < in; j += blockDim.x) {
    smax = fmaxf(smax, s[j]);
    smin = fminf(smin, s[j]);
  }
  for (int o = 16; o > 0; o >>= 1) {
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, o));
    smin = fminf(smin, __shfl_xor_sync(0xffffffffu, smin, o));
  }
  __shared__ float red[2][32];
  __shared__ float sc[2];
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = smax;
    red[1][threadIdx.x >> 5] = smin;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
      smax = fmaxf(smax, red[0][w]);
      smin = fminf(smin, red[1][w]);
    }
    const float wmax = __uint_as_float(absmax[0]), xmax = __uint_as_float(absmax[1]);
    const int e = pow2_exponent_for((double)wmax * (double)smax);
    const int m = smin > 0.0f ? pow2_exponent_for((double)xmax / (double)smin) : 0;
    sc[0] = ldexpf(1.0f, e);
    sc[1] = ldexpf(1.0f, m);
    ctl[0] = 1e-8f * sc[0];
    ctl[1] = (float)ldexp(1.0, -2 * (e + m));
  }
  __syncthreads();
  for (int64_t j = threadIdx.x; j < in; j += blockDim.x) {
    ss[j] = s[j] * sc[0];
    xf[j] = __frcp_rn(s[j]) * sc[1];
  }
}

// xs[n][j] = fp16(X[n][j] * xf[j]), eight columns a thread.
template <typename T>
__global__ void __launch_bounds__(256) clip_xcopy_kernel(const T* __restrict__ X, int64_t N,
                                                         int64_t in, const float* __restrict__ xf,
                                                         uint4* __restrict__ xs) {
  pdl_wait();
  pdl_trigger();
  const int64_t n8 = in / 8, total = N * n8;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t j8 = i % n8;
    float v[8], f[8];
    load8_f32<T>(X + (i / n8) * in + j8 * 8, v);
    load8_f32<float>(xf + j8 * 8, f);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 h = __floats2half2_rn(v[2 * k] * f[2 * k], v[2 * k + 1] * f[2 * k + 1]);
      w[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    xs[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

// With fewer than 32 tokens a share is a sum of few squared dot products,
// and the fp16 rounding of the operands no longer averages out: such layers
// (cheap anyway) take the fp32 path.
bool clip_mma_eligible(int dt, int64_t in, int64_t N, int group) {
  return (dt == kDtF16 || dt == kDtBF16) && group == kCG && in % kCG == 0 && N >= 32 &&
         N <= 256 && in <= (1 << 24);
}

size_t clip_mma_workspace_bytes(int64_t in, int64_t N) {
  return align_up((size_t)in * 4, 256) * 2 + 256 + align_up((size_t)N * in * 2, 256);
}

cudaError_t launch_clip_search_mma(const void* W, const void* X, int dt, int64_t out, int64_t in,
                                   int64_t N, const float* s, int bits, int sym, int nf,
                                   const ClipFactors& cf, void* workspace, float* clip, float* errs,
                                   int32_t* dev_status, cudaStream_t stream) {
  if (!clip_mma_eligible(dt, in, N, kCG) || nf < 1 || nf > kMaxClip) return cudaErrorInvalidValue;
  if ((reinterpret_cast<uintptr_t>(W) & 15) != 0 || (reinterpret_cast<uintptr_t>(X) & 15) != 0)
    return cudaErrorInvalidValue;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  float* ss = reinterpret_cast<float*>(wsb);
  float* xf = reinterpret_cast<float*>(wsb + align_up((size_t)in * 4, 256));
  // control area (256 bytes): ctl floats [0, 2), max|W| and max|X| bits at
  // words 16 and 17, four words of wait diagnostics from word 18
  float* ctl = reinterpret_cast<float*>(wsb + 2 * align_up((size_t)in * 4, 256));
  uint32_t* absmax = reinterpret_cast<uint32_t*>(ctl) + 16;
  void* xs = wsb + 2 * align_up((size_t)in * 4, 256) + 256;
  cudaError_t e = cudaMemsetAsync(ctl, 0, 256, stream);
  if (e == cudaSuccess) e = launch_absmax(W, dt, out * in, absmax, stream);
  if (e == cudaSuccess) e = launch_absmax(X, dt, N * in, absmax + 1, stream);
  if (e == cudaSuccess) e = launch_pdl(clip_prep_kernel, 1, 1024, 0, stream, s, in, absmax, ss, xf, ctl);
  if (e != cudaSuccess) return e;
  const int64_t n8 = N * in / 8;
  const unsigned xgrid = (unsigned)std::max<int64_t>(1, std::min<int64_t>((n8 + 255) / 256,
                                                                          device_sm_count() * 8));
  if (dt == kDtF16)
    e = launch_pdl(clip_xcopy_kernel<__half>, xgrid, 256, 0, stream, static_cast<const __half*>(X),
                   N, in, xf, static_cast<uint4*>(xs));
  else
    e = launch_pdl(clip_xcopy_kernel<__nv_bfloat16>, xgrid, 256, 0, stream,
                   static_cast<const __nv_bfloat16*>(X), N, in, xf, static_cast<uint4*>(xs));
  if (e != cudaSuccess) return e;

  const int T = (int)((N + 31) / 32 * 32);
  CUtensorMap mw, mx;
  const CUtensorMapDataType wt =
      dt == kDtF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (!tensor_map_sw128(&mw, wt, W, (uint64_t)in, (uint64_t)out, (uint64_t)in * 2, kCKB, kCRows) ||
      !tensor_map_sw128(&mx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xs, (uint64_t)in, (uint64_t)N,
                        (uint64_t)in * 2, kCKB, (uint32_t)T))
    return cudaErrorInvalidValue;
  ClipMmaArgs a{};
  a.out = (int)out;
  a.in = (int)in;
  a.T = T;
  a.ngroups = (int)(in / kCG);
  const int n_rt = (int)((out + kCRows - 1) / kCRows);
  a.n_items = n_rt * a.ngroups;
  a.nf = nf;
  for (int i = 0; i < kMaxClip; ++i) a.factors[i] = cf.c[i];
  a.Lf = (float)((1 << (bits - 1)) - 1);
  a.maxqf = (float)((1 << bits) - 1);
  a.ss = ss;
  a.ctl = ctl;
  a.clip = clip;
  a.errs = errs;
  a.status = dev_status;
  a.diag = absmax + 2;
  a.wait_limit_ns = 2000000000ull;
  const size_t smem = kCCtrl + 1024 + kCSW * kCW_TILE + kCSlots * kCD_SLOT + kCSX * (size_t)T * 128;
  using Kern = void (*)(const CUtensorMap, const CUtensorMap, const ClipMmaArgs);
  Kern k;
  if (dt == kDtF16)
    k = sym ? clip_mma_kernel<__half, true> : clip_mma_kernel<__half, false>;
  else
    k = sym ? clip_mma_kernel<__nv_bfloat16, true> : clip_mma_kernel<__nv_bfloat16, false>;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = std::max(1, std::min(a.n_items, device_sm_count()));
  return launch_pdl(k, dim3((unsigned)grid), dim3(kCThreads), smem, stream, mw, mx, a);
}

}  // namespace awq
