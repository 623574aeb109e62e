// The alpha grid and its scale tables, and the final reduction and argmin.
//
// alpha_k = linspace(0, 1, grid + 1)[k] = k * (1 / grid) for k < grid, 1 at k = grid
// s_k     = s_X ** alpha_k,  s_k /= sqrt(max(s_k) * min(s_k))
// ("AWQ (activation-aware weight quantization)", "The code, line by line",
//  bullets on the grid and on centring), all in float64, then rounded to
// float32 for the quantizer.
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

constexpr int kPrepChunk = 1024;  // columns per CTA

__device__ __forceinline__ double alpha_at(int k, int grid) {
  return k == grid ? 1.0 : (double)k * (1.0 / (double)grid);
}

// grid = (n_alpha, chunks): powers and per-chunk max/min.
__global__ void __launch_bounds__(256) alpha_pow_kernel(const double* __restrict__ sx, int64_t in,
                                                        int grid, double* __restrict__ s64,
                                                        double* __restrict__ minmax) {
  const int k = blockIdx.x;
  const double a = alpha_at(k, grid);
  double mx = -INFINITY, mn = INFINITY;
  for (int i = threadIdx.x; i < kPrepChunk; i += blockDim.x) {
    const int64_t j = (int64_t)blockIdx.y * kPrepChunk + i;
    if (j < in) {
      const double v = pow(sx[j], a);
      s64[(int64_t)k * in + j] = v;
      mx = fmax(mx, v);
      mn = fmin(mn, v);
    }
  }
  __shared__ double smx[8], smn[8];
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
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
      mx = fmax(mx, smx[w]);
      mn = fmin(mn, smn[w]);
    }
    const int64_t nch = (in + kPrepChunk - 1) / kPrepChunk;
    minmax[((int64_t)k * nch + blockIdx.y) * 2 + 0] = mx;
    minmax[((int64_t)k * nch + blockIdx.y) * 2 + 1] = mn;
  }
}

// grid = (n_alpha, chunks): centring, float32 rounding, and the fp16 scaling
// of the weight changes.  One entry's change is |q*scale - w*s| / s <= (group
// step) / s, and the group step is at most max|w| * max(s) (either
// quantizer), so max|W| * max(s) / min(s) bounds |dW| for the whole alpha;
// its power-of-two exponent sets the scaling e_k of this alpha's dW.
__global__ void __launch_bounds__(256) alpha_centre_kernel(const double* __restrict__ s64,
                                                           const double* __restrict__ minmax,
                                                           int64_t in,
                                                           const uint32_t* __restrict__ absmax,
                                                           int x_scaled, float* __restrict__ s32,
                                                           float* __restrict__ inv_s32,
                                                           double* __restrict__ unscale,
                                                           int32_t* __restrict__ pow2_s) {
  const int k = blockIdx.x;
  const int64_t nch = (in + kPrepChunk - 1) / kPrepChunk;
  __shared__ double c_sh;
  __shared__ int e_sh;
  if (threadIdx.x == 0) {
    double mx = -INFINITY, mn = INFINITY;
    for (int64_t c = 0; c < nch; ++c) {
      mx = fmax(mx, minmax[(k * nch + c) * 2 + 0]);
      mn = fmin(mn, minmax[(k * nch + c) * 2 + 1]);
    }
    c_sh = sqrt(mx * mn);
    const int e = pow2_exponent_for((double)__uint_as_float(absmax[0]) * (mx / mn));
    const int m = x_scaled ? pow2_exponent_for((double)__uint_as_float(absmax[1])) : 0;
    e_sh = e;
    if (blockIdx.y == 0) unscale[k] = ldexp(1.0, -2 * (e + m));
  }
  __syncthreads();
  const double c = c_sh;
  const float f2 = ldexpf(1.0f, e_sh);
  int all_pow2 = 1;
  for (int i = threadIdx.x; i < kPrepChunk; i += blockDim.x) {
    const int64_t j = (int64_t)blockIdx.y * kPrepChunk + i;
    if (j < in) {
      const float f = __double2float_rn(s64[(int64_t)k * in + j] / c);
      s32[(int64_t)k * in + j] = f;
      inv_s32[(int64_t)k * in + j] = __frcp_rn(f) * f2;
      all_pow2 &= ((__float_as_uint(f) & 0x007FFFFFu) == 0u) ? 1 : 0;
    }
  }
  all_pow2 = __syncthreads_and(all_pow2);
  if (threadIdx.x == 0 && !all_pow2) atomicAnd(&pow2_s[k], 0);
}

// One CTA: per-alpha fixed-order sums, strict argmin, copy of the kept scales.
__global__ void __launch_bounds__(256) reduce_argmin_kernel(const double* __restrict__ partials,
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
  for (int64_t j = threadIdx.x; j < in; j += blockDim.x)
    s_best[j] = best >= 0 ? s32[(int64_t)best * in + j] : __int_as_float(0x7fc00000);
}

}  // namespace

size_t prep_chunks(int64_t in) { return (size_t)((in + kPrepChunk - 1) / kPrepChunk); }

cudaError_t launch_alpha_prep(const double* sx, int64_t in, int grid, const uint32_t* absmax,
                              int x_scaled, double* s64, double* minmax, float* s32,
                              float* inv_s32, double* unscale, int32_t* pow2_s, cudaStream_t s) {
  const dim3 g(grid + 1, (unsigned)prep_chunks(in));
  alpha_pow_kernel<<<g, 256, 0, s>>>(sx, in, grid, s64, minmax);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  alpha_centre_kernel<<<g, 256, 0, s>>>(s64, minmax, in, absmax, x_scaled, s32, inv_s32, unscale,
                                        pow2_s);
  return cudaGetLastError();
}

cudaError_t launch_reduce_argmin(const double* partials, const double* unscale, int n_alpha,
                                 int n_tiles, double denom, const float* s32, int64_t in,
                                 double* err, int32_t* best, float* s_best, int32_t* dev_status,
                                 cudaStream_t s) {
  reduce_argmin_kernel<<<1, 256, 0, s>>>(partials, unscale, n_alpha, n_tiles, denom, s32, in, err,
                                         best, s_best, dev_status);
  return cudaGetLastError();
}

}  // namespace awq
