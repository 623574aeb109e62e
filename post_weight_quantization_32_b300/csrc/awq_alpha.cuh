// Per-alpha centring values of the scale search, formed by the last CTA of
// whichever launch produced the channel statistics (see CentreArgs).
//
// s_k = s_X ** alpha_k is centred by 1 / sqrt(max(s_k) * min(s_k))
// ("AWQ (activation-aware weight quantization)", "The code, line by line",
// centring bullet).  The power is monotone in s_X, so the extremes of s_k
// are the powers of the extremes of s_X, and only those two are needed.
#pragma once

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

// Extremes of s_X over a set of columns, each with its s_X^(1 / grid).
// Comparisons are strict, so NaN entries are never taken.
struct SxExt {
  double mx, rmx, mn, rmn;
  __device__ __forceinline__ void init() {
    mx = -INFINITY;
    mn = INFINITY;
    rmx = rmn = 1.0;
  }
  __device__ __forceinline__ void take(double v, double r) {
    if (v > mx) mx = v, rmx = r;
    if (v < mn) mn = v, rmn = r;
  }
  __device__ __forceinline__ void merge(const SxExt& o) {
    if (o.mx > mx) mx = o.mx, rmx = o.rmx;
    if (o.mn < mn) mn = o.mn, rmn = o.rmn;
  }
  __device__ __forceinline__ void warp_merge() {
    for (int o = 16; o > 0; o >>= 1) {
      SxExt t;
      t.mx = __shfl_xor_sync(0xffffffffu, mx, o);
      t.rmx = __shfl_xor_sync(0xffffffffu, rmx, o);
      t.mn = __shfl_xor_sync(0xffffffffu, mn, o);
      t.rmn = __shfl_xor_sync(0xffffffffu, rmn, o);
      merge(t);
    }
  }
  __device__ __forceinline__ void store(double* p) const {
    p[0] = mx;
    p[1] = rmx;
    p[2] = mn;
    p[3] = rmn;
  }
  __device__ __forceinline__ void load_cg(const double* p) {
    mx = __ldcg(p);
    rmx = __ldcg(p + 1);
    mn = __ldcg(p + 2);
    rmn = __ldcg(p + 3);
  }
};

// r^k by binary powering: at most 2 * log2(k) float64 products.
__device__ __forceinline__ double pow_int(double r, int k) {
  double acc = 1.0;
  while (k > 0) {
    if (k & 1) acc *= r;
    r *= r;
    k >>= 1;
  }
  return acc;
}

// For every alpha k: max(s_k) = max(s_X)^(k/grid) = rmx^k, and likewise the
// minimum (exactly s_X's extremes at k = grid, 1 at k = 0);
// inv_c[k] = 1 / sqrt(max * min).  The fp16 scaling of the weight changes:
// one entry's change is |q*scale - w*s| / s <= (group step) / s, and the
// group step is at most max|W| * max(s) (either quantizer), so
// max|W| * max(s) / min(s) bounds |dW| for the whole alpha; its
// power-of-two exponent sets e_k (folded into the 1/s table), and
// unscale[k] = 2^-2(e_k + m_x) undoes both operand scalings on the squared
// sums (the pre-divided mode scales the weights and X / s separately, see
// CentreArgs).  pow2_s[k] starts at 1 here.  Threads stride over the alphas; only
// products and one reciprocal square root per alpha, no logarithms.
__device__ __forceinline__ void alpha_centre(const SxExt& x, float wmax, float xmax, int m_x,
                                             const CentreArgs& ca) {
  const int grid = ca.grid;
  for (int k = threadIdx.x; k <= grid; k += blockDim.x) {
    double smax, smin;
    if (k == 0) {
      smax = smin = 1.0;
    } else if (k == grid) {
      smax = x.mx;
      smin = x.mn;
    } else {
      smax = pow_int(x.rmx, k);
      smin = pow_int(x.rmn, k);
    }
    const double ic = k == 0 ? 1.0 : rsqrt(smax * smin);
    ca.inv_c[k] = ic;
    const double q = smax * ic;  // sqrt(max / min)
    if (ca.xs) {
      // pre-divided mode: the weights' rounding errors are at most
      // max|W| * max(s) = max|W| * q, and |X / s| at most max|X| / min(s) =
      // max|X| * q
      const int e = pow2_exponent_for((double)wmax * q);
      const int m = pow2_exponent_for((double)xmax * q);
      ca.escale[k] = ldexpf(1.0f, e);
      ca.xscale[k] = ldexpf(1.0f, m);
      ca.unscale[k] = ldexp(1.0, -2 * (e + m));
    } else {
      const int e = pow2_exponent_for((double)wmax * (q * q));
      ca.escale[k] = ldexpf(1.0f, e);
      ca.unscale[k] = ldexp(1.0, -2 * (e + m_x));
    }
    ca.pow2_s[k] = 1;
  }
}

// Called by every thread of every CTA of the launch, after the CTA has
// written its chunk's extremes (SxExt::store at ca.minmax + 4c) and folded
// its part of max|W| / max|X| into ca.absmax: the last CTA to arrive (a
// ticket counter, zero on entry) reduces the nchunks extremes and forms the
// centring values.
__device__ __forceinline__ void centre_if_last(const CentreArgs& ca, unsigned nchunks) {
  __shared__ bool last;
  __shared__ SxExt sext[32];
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last = atomicAdd(ca.ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  SxExt x;
  x.init();
  for (unsigned ch = threadIdx.x; ch < nchunks; ch += blockDim.x) {
    SxExt t;
    t.load_cg(ca.minmax + 4 * ch);
    x.merge(t);
  }
  x.warp_merge();
  if ((threadIdx.x & 31) == 0) sext[threadIdx.x >> 5] = x;
  __syncthreads();
  x = sext[0];
  for (unsigned w = 1; w < (blockDim.x + 31) / 32; ++w) x.merge(sext[w]);
  const float wmax = __uint_as_float(__ldcg(ca.absmax));
  const float xmax = __uint_as_float(__ldcg(ca.absmax + 1));
  const int m_x = ca.x_scaled ? pow2_exponent_for((double)xmax) : 0;
  alpha_centre(x, wmax, xmax, m_x, ca);
}

}  // namespace awq
