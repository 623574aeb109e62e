// The alpha grid and its scale tables, and the final reduction and argmin.
//
// alpha_k = linspace(0, 1, grid + 1)[k] = k * (1 / grid) for k < grid, 1 at k = grid
// s_k     = s_X ** alpha_k,  s_k /= sqrt(max(s_k) * min(s_k))
// ("AWQ (activation-aware weight quantization)", "The code, line by line",
//  bullets on the grid and on centring), all in float64, then rounded to
// float32 for the quantizer.  Float64 transcendentals are costly on this
// GPU, so the table entries are running products of s_X^(1/grid): one
// float64 multiplication per entry, within a few float64 ulps of the power,
// far below the float32 rounding that follows.
//
// err_k = sum of the search's per-tile partial sums / (N * out), times the
// exact power of two that undoes the fp16 operand scaling; the kept alpha is
// the first one with the smallest error under a strict comparison, so NaN
// errors are never kept ("Source code": if err < best_err).
#include <math.h>

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

constexpr int kPrepChunk = 64;   // columns per CTA of the per-column kernels

// grid = chunks: root[j] = sx[j] ^ (1 / grid) in float64 and each chunk's
// max and min of sx.
__global__ void __launch_bounds__(kPrepChunk) alpha_root_kernel(const double* __restrict__ sx,
                                                                int64_t in, int grid,
                                                                double* __restrict__ root,
                                                                double* __restrict__ minmax) {
  double mx = -INFINITY, mn = INFINITY;
  const int64_t j = (int64_t)blockIdx.x * kPrepChunk + threadIdx.x;
  if (j < in) {
    const double v = sx[j];
    root[j] = exp(log(v) / (double)grid);
    mx = v;
    mn = v;
  }
  __shared__ double smx[kPrepChunk / 32], smn[kPrepChunk / 32];
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = fmin(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  if ((threadIdx.x & 31) == 0) {
    smx[threadIdx.x >> 5] = mx;
    smn[threadIdx.x >> 5] = mn;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 0; w < kPrepChunk / 32; ++w) {
      mx = fmax(mx, smx[w]);
      mn = fmin(mn, smn[w]);
    }
    minmax[2 * blockIdx.x + 0] = mx;
    minmax[2 * blockIdx.x + 1] = mn;
  }
}

// One CTA, thread k per alpha (strided).  The largest and smallest s_k over
// the columns are s_k at the largest and smallest s_X (the power is
// monotone); from them the centring factor inv_c[k] = 1 / sqrt(max * min),
// and the fp16 scaling of the weight changes: one entry's change is
// |q*scale - w*s| / s <= (group step) / s, and the group step is at most
// max|W| * max(s) (either quantizer), so max|W| * max(s) / min(s) bounds
// |dW| for the whole alpha; its power-of-two exponent sets e_k, folded into
// the 1/s table, and unscale[k] = 2^-2(e_k + m_x) undoes both operand
// scalings on the squared sums.  pow2_s[k] starts at 1 here.
__global__ void __launch_bounds__(256) alpha_centre_kernel(
    const double* __restrict__ minmax, int64_t nch, int grid,
    const uint32_t* __restrict__ absmax, int x_scaled, double* __restrict__ inv_c,
    float* __restrict__ escale, double* __restrict__ unscale, int32_t* __restrict__ pow2_s) {
  __shared__ double smx[8], smn[8];
  double mx = -INFINITY, mn = INFINITY;
  for (int64_t ch = threadIdx.x; ch < nch; ch += blockDim.x) {
    mx = fmax(mx, minmax[2 * ch + 0]);
    mn = fmin(mn, minmax[2 * ch + 1]);
  }
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    mn = fmin(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  }
  if ((threadIdx.x & 31) == 0) {
    smx[threadIdx.x >> 5] = mx;
    smn[threadIdx.x >> 5] = mn;
  }
  __syncthreads();
  mx = smx[0];
  mn = smn[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
    mx = fmax(mx, smx[w]);
    mn = fmin(mn, smn[w]);
  }
  const double lmx = log(mx) / (double)grid, lmn = log(mn) / (double)grid;
  const int m = x_scaled ? pow2_exponent_for((double)__uint_as_float(absmax[1])) : 0;
  for (int k = threadIdx.x; k <= grid; k += blockDim.x) {
    double smax, smin;
    if (k == 0) {
      smax = smin = 1.0;
    } else if (k == grid) {
      smax = mx;
      smin = mn;
    } else {
      smax = exp(k * lmx);
      smin = exp(k * lmn);
    }
    inv_c[k] = 1.0 / sqrt(smax * smin);
    const int e = pow2_exponent_for((double)__uint_as_float(absmax[0]) * (smax / smin));
    escale[k] = ldexpf(1.0f, e);
    unscale[k] = ldexp(1.0, -2 * (e + m));
    pow2_s[k] = 1;
  }
}

// grid = chunks, one thread per column, looping over the alphas: s_k =
// sx ^ (k / grid) as the running product root^k (exactly 1 at k = 0 and
// exactly sx at k = grid), centred, rounded to float32; inv_s32 = 2^e_k / s.
// pow2_s[k] is cleared when some entry of the chunk is not a power of two.
__global__ void __launch_bounds__(kPrepChunk) alpha_table_kernel(
    const double* __restrict__ sx, const double* __restrict__ root,
    const double* __restrict__ inv_c, const float* __restrict__ escale, int64_t in, int grid,
    float* __restrict__ s32, float* __restrict__ inv_s32, int32_t* __restrict__ pow2_s) {
  const int64_t j = (int64_t)blockIdx.x * kPrepChunk + threadIdx.x;
  const bool live = j < in;
  const double sxj = live ? sx[j] : 1.0, r = live ? root[j] : 1.0;
  double v = 1.0;
  for (int k = 0; k <= grid; ++k) {
    if (k > 0) v = k == grid ? sxj : v * r;
    const float f = __double2float_rn(v * inv_c[k]);
    if (live) {
      s32[(int64_t)k * in + j] = f;
      inv_s32[(int64_t)k * in + j] = __frcp_rn(f) * escale[k];
    }
    const int p2 = (!live || (__float_as_uint(f) & 0x007FFFFFu) == 0u) ? 1 : 0;
    if (!__syncthreads_and(p2) && threadIdx.x == 0) atomicAnd(&pow2_s[k], 0);
  }
}

// One CTA: per-alpha fixed-order sums, strict argmin, copy of the kept scales.
__global__ void __launch_bounds__(1024) reduce_argmin_kernel(const double* __restrict__ partials,
                                                            const double* __restrict__ unscale,
                                                            int n_alpha, int n_tiles, double denom,
                                                            const float* __restrict__ s32,
                                                            int64_t in, double* __restrict__ err,
                                                            int32_t* __restrict__ best_out,
                                                            float* __restrict__ s_best,
                                                            int32_t* dev_status) {
  __shared__ int best_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int k = warp; k < n_alpha; k += blockDim.x >> 5) {
    double s = 0.0;
    for (int t = lane; t < n_tiles; t += 32) s += partials[(int64_t)k * n_tiles + t];
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) err[k] = s * unscale[k] / denom;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int best = -1;
    double be = INFINITY;
    for (int k = 0; k < n_alpha; ++k) {
      const double e = err[k];
      if (e < be) {
        be = e;
        best = k;
      }
    }
    if (best < 0) set_status(dev_status, ST_NONFINITE);
    *best_out = best;
    best_sh = best;
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

}  // namespace

size_t prep_chunks(int64_t in) { return (size_t)((in + kPrepChunk - 1) / kPrepChunk); }

cudaError_t launch_alpha_prep(const double* sx, int64_t in, int grid, const uint32_t* absmax,
                              int x_scaled, double* root, double* minmax, double* inv_c,
                              float* escale, float* s32, float* inv_s32, double* unscale,
                              int32_t* pow2_s, cudaStream_t s) {
  const unsigned nch = (unsigned)prep_chunks(in);
  alpha_root_kernel<<<nch, kPrepChunk, 0, s>>>(sx, in, grid, root, minmax);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  alpha_centre_kernel<<<1, 256, 0, s>>>(minmax, nch, grid, absmax, x_scaled, inv_c, escale,
                                        unscale, pow2_s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  alpha_table_kernel<<<nch, kPrepChunk, 0, s>>>(sx, root, inv_c, escale, in, grid, s32, inv_s32,
                                                pow2_s);
  return cudaGetLastError();
}

cudaError_t launch_reduce_argmin(const double* partials, const double* unscale, int n_alpha,
                                 int n_tiles, double denom, const float* s32, int64_t in,
                                 double* err, int32_t* best, float* s_best, int32_t* dev_status,
                                 cudaStream_t s) {
  reduce_argmin_kernel<<<1, 1024, 0, s>>>(partials, unscale, n_alpha, n_tiles, denom, s32, in, err,
                                          best, s_best, dev_status);
  return cudaGetLastError();
}

}  // namespace awq
