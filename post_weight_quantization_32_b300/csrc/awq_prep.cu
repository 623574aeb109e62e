// The alpha grid and its scale tables, and the final reduction and argmin.
//
// alpha_k = linspace(0, 1, grid + 1)[k] = k * (1 / grid) for k < grid, 1 at k = grid
// s_k     = s_X ** alpha_k,  s_k /= sqrt(max(s_k) * min(s_k))
// ("AWQ (activation-aware weight quantization)", "The code, line by line",
//  bullets on the grid and on centring), all in float64, then rounded to
// float32 for the quantizer.  Float64 transcendentals are costly on this
// GPU, so the powers are running products of s_X^(1/grid) (write_powers):
// one float64 product per entry, within a few float64 ulps of the power,
// far below the float32 rounding that follows.
//
// err_k = sum of the search's per-tile partial sums / (N * out), times the
// exact power of two that undoes the fp16 operand scaling; the kept alpha is
// the first one with the smallest error under a strict comparison, so NaN
// errors are never kept ("Source code": if err < best_err).
#include <math.h>

#include <algorithm>

#include "awq_alpha.cuh"
#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

constexpr int kPrepChunk = kChunkCols;  // columns per CTA of the root launch (one chunk)

// CTA b: root r = sx^(1 / grid) in float64 of the 32 columns 32 b .. 32 b +
// 31 (warp 0), the chunk's max and min of sx with their roots, and the
// columns' powers u[k][j] = sx^(k / grid) (write_powers, warps 0..3); CTA 0
// sets pow2_s[k] = 1.  (The statistics launch does the same when it
// computes sx itself; this kernel serves a caller-given sx.)
__global__ void __launch_bounds__(128) alpha_root_kernel(const double* __restrict__ sx, int64_t in,
                                                        CentreArgs ca) {
  pdl_wait();
  pdl_trigger();
  __shared__ double sh_v[kPrepChunk], sh_r[kPrepChunk];
  if (blockIdx.x == 0)
    for (int k = threadIdx.x; k <= ca.grid; k += blockDim.x) ca.pow2_s[k] = 1;
  if (threadIdx.x < kPrepChunk) {
    SxExt x;
    x.init();
    const int64_t j = (int64_t)blockIdx.x * kPrepChunk + threadIdx.x;
    if (j < in) {
      const double v = sx[j];
      const double r = exp(log(v) / (double)ca.grid);
      sh_v[threadIdx.x] = v;
      sh_r[threadIdx.x] = r;
      x.take(v, r);
    }
    x.warp_merge();
    if (threadIdx.x == 0) x.store(ca.minmax + 4 * blockIdx.x);
  }
  __syncthreads();
  write_powers(sh_v, sh_r, (int64_t)blockIdx.x * kPrepChunk, in, ca.grid, ca.u);
}

// CTA (x, k): alpha k of the 256 columns 256 x .. 256 x + 255, one column
// a thread.  Each CTA reduces the chunk extremes and centres alpha k
// (centre_alpha), forms its scalings from q and the max|W| / max|X| bits
// (alpha_scalings; CTA x = 0 stores escale[k] and unscale[k]), then
// s32[k][j] = f = fp32(u[k][j] * ic) and inv_s32[k][j] = 2^e_k / f;
// pow2_s[k] is cleared when some entry is not a power of two.
constexpr int kTabCols = 256;
__global__ void __launch_bounds__(kTabCols) alpha_table_kernel(
    const double* __restrict__ u, const double* __restrict__ minmax,
    const uint32_t* __restrict__ absmax, int x_scaled, int64_t in, int grid,
    float* __restrict__ s32, float* __restrict__ inv_s32, float* __restrict__ escale,
    double* __restrict__ unscale, int32_t* __restrict__ pow2_s) {
  pdl_wait();
  pdl_trigger();
  const int k = blockIdx.y;
  const int64_t j = (int64_t)blockIdx.x * kTabCols + threadIdx.x;
  const double uk = j < in ? u[(int64_t)k * in + j] : 1.0;
  double ic, q;
  centre_alpha(minmax, chunk_count(in), k, grid, ic, q);
  int e, m;
  alpha_scalings(q, __uint_as_float(absmax[0]), __uint_as_float(absmax[1]), false, x_scaled != 0,
                 e, m);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    escale[k] = exp2i_f32(e);
    unscale[k] = exp2i_f64(-2 * (e + m));
  }
  bool np2 = false;
  if (j < in) {
    const float f = __double2float_rn(uk * ic);
    s32[(int64_t)k * in + j] = f;
    inv_s32[(int64_t)k * in + j] = __frcp_rn(f) * exp2i_f32(e);
    np2 = (__float_as_uint(f) & 0x007FFFFFu) != 0u;
  }
  if (__syncthreads_or(np2) && threadIdx.x == 0) atomicAnd(&pow2_s[k], 0);
}

// The pre-divided mode's scalings, CTA (x, k) as alpha_table_kernel:
// ss32[k][j] = s32[k][j] * 2^e_k (exact), escale[k] = 2^e_k and
// unscale[k] = 2^-2(e_k + m_k) from qk[k], max|W| and max|X|.
__global__ void __launch_bounds__(kTabCols) scale_table_xs_kernel(
    const float* __restrict__ s32, const double* __restrict__ qk,
    const uint32_t* __restrict__ absmax, int64_t in, float* __restrict__ ss32,
    float* __restrict__ escale, double* __restrict__ unscale) {
  pdl_wait();
  pdl_trigger();
  const int k = blockIdx.y;
  int e, m;
  alpha_scalings(qk[k], __uint_as_float(absmax[0]), __uint_as_float(absmax[1]), true, false, e, m);
  const float es = exp2i_f32(e);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    escale[k] = es;
    unscale[k] = exp2i_f64(-2 * (e + m));
  }
  const int64_t j = (int64_t)blockIdx.x * kTabCols + threadIdx.x;
  if (j < in) ss32[(int64_t)k * in + j] = s32[(int64_t)k * in + j] * es;
}

// One CTA: per-alpha fixed-order sums, strict argmin, copy of the kept scales.
// err_k = unscale[k] * sum_t partials[k][t] / denom, the tiles added in
// order; with parts > 0 (the finish of a row-split search) err_k is instead
// sum_{p < parts} partials[p][k] / denom, added in part order, and unscale
// is not read.
//
// One thread per alpha: the SM's float64 pipe takes a warp instruction
// about every 19 cycles however few lanes are active, so the sums and the
// division run as few warp instructions as possible (for up to 32 alphas,
// the lanes of warp 0, which then also takes the argmin by shuffles).
__device__ __forceinline__ double alpha_error(const double* __restrict__ partials,
                                              const double* __restrict__ unscale, int k,
                                              int n_alpha, int n_tiles, int parts, double denom) {
  double s = 0.0;
  if (parts > 0) {
    for (int q = 0; q < parts; ++q) s += __ldcg(partials + (int64_t)q * n_alpha + k);
    return s / denom;
  }
  const double* row = partials + (int64_t)k * n_tiles;
  for (int t = 0; t < n_tiles; ++t) s += row[t];
  return s * unscale[k] / denom;
}

// Strict-< keep over (key, index) pairs: the smaller error, then the smaller index.
__device__ __forceinline__ void keep_smaller(unsigned long long& bk, int& best,
                                             unsigned long long ok, int ob) {
  if (ob >= 0 && (best < 0 || ok < bk || (ok == bk && ob < best))) {
    bk = ok;
    best = ob;
  }
}

constexpr int kStageDoubles = 4096;  // partial sums staged in shared memory (32 KB)
__global__ void __launch_bounds__(1024) reduce_argmin_kernel(const double* __restrict__ partials,
                                                            const double* __restrict__ unscale,
                                                            int n_alpha, int n_tiles, double denom,
                                                            const float* __restrict__ s32,
                                                            int64_t in, double* __restrict__ err,
                                                            int32_t* __restrict__ best_out,
                                                            float* __restrict__ s_best,
                                                            int32_t* dev_status, int parts) {
  pdl_wait();
  pdl_trigger();
  __shared__ int best_sh;
  __shared__ double stage[kStageDoubles];
  extern __shared__ double err_sh[];  // [n_alpha] (more than 32 alphas)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the first index of the smallest error under strict <, starting from
  // +inf, on total-order keys of the errors (integer compares): NaN is never
  // kept, -0 counts as +0
  const unsigned long long kinf = f64_key(INFINITY);
  auto key_of = [](double e) {
    return f64_is_nan(e) ? ~0ull : f64_key(f64_drop_sign_of_zero(e));
  };
  // tiles mode: the partial sums staged in shared memory by every thread in
  // one coalesced pass (one load round trip), then summed per alpha there
  const int64_t n_part = (int64_t)n_alpha * n_tiles;
  const bool staged = parts == 0 && n_part <= kStageDoubles;
  if (staged) {
    for (int i = threadIdx.x; i < n_part; i += blockDim.x) stage[i] = __ldcg(partials + i);
    __syncthreads();
  }
  const double* psrc = staged ? stage : partials;
  if (n_alpha <= 32) {
    if (warp == 0) {
      unsigned long long bk = kinf;
      int best = -1;
      if (lane < n_alpha) {
        const double e = alpha_error(psrc, unscale, lane, n_alpha, n_tiles, parts, denom);
        err[lane] = e;
        const unsigned long long k = key_of(e);
        if (k < kinf) {
          bk = k;
          best = lane;
        }
      }
      for (int o = 16; o > 0; o >>= 1)
        keep_smaller(bk, best, __shfl_xor_sync(0xffffffffu, bk, o),
                     __shfl_xor_sync(0xffffffffu, best, o));
      if (lane == 0) {
        if (best < 0) set_status(dev_status, ST_NONFINITE);
        *best_out = best;
        best_sh = best;
      }
    }
  } else {
    for (int k = threadIdx.x; k < n_alpha; k += blockDim.x) {
      const double e = alpha_error(psrc, unscale, k, n_alpha, n_tiles, parts, denom);
      err[k] = e;
      err_sh[k] = e;
    }
    __syncthreads();
    if (warp == 0) {
      // each lane scans its own alphas in order, then lanes merge
      int best = -1;
      unsigned long long bk = kinf;
      for (int k = lane; k < n_alpha; k += 32) {
        const unsigned long long ek = key_of(err_sh[k]);
        if (ek < bk) {
          bk = ek;
          best = k;
        }
      }
      for (int o = 16; o > 0; o >>= 1)
        keep_smaller(bk, best, __shfl_xor_sync(0xffffffffu, bk, o),
                     __shfl_xor_sync(0xffffffffu, best, o));
      if (lane == 0) {
        if (best < 0) set_status(dev_status, ST_NONFINITE);
        *best_out = best;
        best_sh = best;
      }
    }
  }
  __syncthreads();
  const int best = best_sh;
  const float* src = s32 + (int64_t)(best >= 0 ? best : 0) * in;
  if ((in & 3) == 0 && ((reinterpret_cast<uintptr_t>(s_best) & 15) == 0)) {
    const float4 nan4 = make_float4(__int_as_float(0x7fc00000), __int_as_float(0x7fc00000),
                                    __int_as_float(0x7fc00000), __int_as_float(0x7fc00000));
    for (int64_t j = threadIdx.x; j < in / 4; j += blockDim.x)
      reinterpret_cast<float4*>(s_best)[j] =
          best >= 0 ? reinterpret_cast<const float4*>(src)[j] : nan4;
  } else {
    for (int64_t j = threadIdx.x; j < in; j += blockDim.x)
      s_best[j] = best >= 0 ? src[j] : __int_as_float(0x7fc00000);
  }
}

// One row of a bit-width / group-size sweep (one thread): the kept alpha's
// value on the grid (linspace(0, 1, grid + 1)[best], R2 of the readings),
// RTN's error (alpha = 0), AWQ's error, and both relative to the output power.
__global__ void sweep_summary_kernel(const double* __restrict__ err, const int32_t* __restrict__ best,
                                     const double* __restrict__ power, int grid,
                                     double* __restrict__ row) {
  pdl_wait();
  const int b = *best;
  const double nan = __longlong_as_double(0x7FF8000000000000ll);
  const double p = *power;
  const double e0 = err[0];
  const double eb = b >= 0 ? err[b] : nan;
  row[0] = b < 0 ? nan : (b == grid ? 1.0 : (double)b * (1.0 / (double)grid));
  row[1] = e0;
  row[2] = eb;
  row[3] = e0 / p;
  row[4] = eb / p;
}

// Sum of squares of D in a fixed order: each thread of a fixed grid adds
// the entries it strides over, the CTA adds its threads in a tree, and the
// last CTA to finish (a ticket) adds the CTAs' sums in order.
constexpr int kPowBlocks = 512;
__global__ void __launch_bounds__(256) power_reduce_kernel(const float* __restrict__ D, int64_t n,
                                                           double denom, uint32_t* ticket,
                                                           double* __restrict__ part,
                                                           double* __restrict__ power) {
  pdl_wait();
  pdl_trigger();
  double acc = 0.0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const double v = (double)D[i];
    acc = fma(v, v, acc);
  }
  __shared__ double red[256];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  __shared__ bool last;
  if (threadIdx.x == 0) {
    part[blockIdx.x] = red[0];
    __threadfence();
    last = atomicAdd(ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (last && threadIdx.x == 0) {
    __threadfence();
    double s = 0.0;
    for (unsigned b = 0; b < gridDim.x; ++b) s += __ldcg(part + b);
    *power = s / denom;
  }
}

}  // namespace

size_t power_reduce_scratch_bytes() { return 256 + (size_t)kPowBlocks * 8; }

cudaError_t launch_power_reduce(const float* D, int64_t n, double denom, void* scratch,
                                double* power, cudaStream_t s) {
  uint8_t* b = static_cast<uint8_t*>(scratch);
  return launch_pdl(power_reduce_kernel, kPowBlocks, 256, 0, s, D, n, denom,
                    reinterpret_cast<uint32_t*>(b), reinterpret_cast<double*>(b + 256), power);
}

cudaError_t launch_sweep_summary(const double* err, const int32_t* best, const double* power,
                                 int grid, double* row, cudaStream_t s) {
  return launch_pdl(sweep_summary_kernel, 1, 1, 0, s, err, best, power, grid, row);
}

size_t prep_chunks(int64_t in) { return (size_t)((in + kPrepChunk - 1) / kPrepChunk); }

cudaError_t launch_alpha_root(const double* sx, int64_t in, const CentreArgs& ca, cudaStream_t s) {
  if (ca.grid < 1 || ca.grid > kMaxGrid) return cudaErrorInvalidValue;
  return launch_pdl(alpha_root_kernel, (unsigned)((in + kPrepChunk - 1) / kPrepChunk), 128, 0, s,
                    sx, in, ca);
}

cudaError_t launch_alpha_table(const double* u, const double* minmax, const uint32_t* absmax,
                               int x_scaled, int64_t in, int grid, float* s32, float* inv_s32,
                               float* escale, double* unscale, int32_t* pow2_s, cudaStream_t s) {
  if (grid < 1 || grid > kMaxGrid) return cudaErrorInvalidValue;
  const dim3 g((unsigned)((in + kTabCols - 1) / kTabCols), (unsigned)(grid + 1));
  return launch_pdl(alpha_table_kernel, g, kTabCols, 0, s, u, minmax, absmax, x_scaled, in, grid,
                    s32, inv_s32, escale, unscale, pow2_s);
}

cudaError_t launch_scale_table_xs(const float* s32, const double* qk, const uint32_t* absmax,
                                  int64_t in, int grid, float* ss32, float* escale,
                                  double* unscale, cudaStream_t s) {
  if (grid < 1 || grid > kMaxGrid) return cudaErrorInvalidValue;
  const dim3 g((unsigned)((in + kTabCols - 1) / kTabCols), (unsigned)(grid + 1));
  return launch_pdl(scale_table_xs_kernel, g, kTabCols, 0, s, s32, qk, absmax, in, ss32, escale,
                    unscale);
}

cudaError_t launch_reduce_argmin(const double* partials, const double* unscale, int n_alpha,
                                 int n_tiles, double denom, const float* s32, int64_t in,
                                 double* err, int32_t* best, float* s_best, int32_t* dev_status,
                                 cudaStream_t s) {
  if (n_alpha < 1 || n_alpha > kMaxGrid + 1) return cudaErrorInvalidValue;
  return launch_pdl(reduce_argmin_kernel, 1, 1024, n_alpha > 32 ? (size_t)n_alpha * sizeof(double) : 0,
                    s, partials, unscale, n_alpha, n_tiles, denom, s32, in, err, best, s_best,
                    dev_status, 0);
}

cudaError_t launch_search_finish(const double* sums, int parts, int n_alpha, double denom,
                                 const float* s_table, int64_t in, double* err, int32_t* best,
                                 float* s_best, int32_t* dev_status, cudaStream_t s) {
  if (n_alpha < 1 || n_alpha > kMaxGrid + 1 || parts < 1) return cudaErrorInvalidValue;
  return launch_pdl(reduce_argmin_kernel, 1, 1024, n_alpha > 32 ? (size_t)n_alpha * sizeof(double) : 0,
                    s, sums, static_cast<const double*>(nullptr), n_alpha, 0, denom, s_table, in,
                    err, best, s_best, dev_status, parts);
}

}  // namespace awq
