// Per-alpha centring values of the scale search.
//
// s_k = s_X ** alpha_k is centred by 1 / sqrt(max(s_k) * min(s_k))
// ("AWQ (activation-aware weight quantization)", "The code, line by line",
// centring bullet).  The power is monotone in s_X, so the extremes of s_k
// are the powers of the extremes of s_X, and only those two are needed.
//
// Float64 arithmetic is slow on this GPU (dependent float64 operations take
// tens of cycles each, a comparison or a division hundreds, and the float64
// pipe issues a warp instruction about every 19 cycles), and a global
// memory round trip costs microseconds while another launch streams the
// weights.  So the statistics launch writes every column's powers s_X^(k /
// grid) with one float64 product each and its chunk's extremes, with no
// cross-CTA step; each CTA of the table launches then reduces the chunk
// extremes itself (integer comparisons) and centres its own alpha, and the
// max|W| / max|X| scalings come from exponent arithmetic on bit patterns.
#pragma once

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

// Total-order key of a float64: the integer order of the keys is the value
// order of non-NaN doubles (negative values included).
__device__ __forceinline__ unsigned long long f64_key(double v) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(v);
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}
__device__ __forceinline__ double f64_from_key(unsigned long long k) {
  return __longlong_as_double((long long)((k >> 63) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k));
}
__device__ __forceinline__ bool f64_is_nan(double v) {
  return ((unsigned long long)__double_as_longlong(v) & 0x7FFFFFFFFFFFFFFFull) >
         0x7FF0000000000000ull;
}

// v with -0 replaced by +0 (bit test, no float64 comparison).
__device__ __forceinline__ double f64_drop_sign_of_zero(double v) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(v);
  return (b & 0x7FFFFFFFFFFFFFFFull) == 0ull ? 0.0 : v;
}

// Extremes of s_X over a set of columns, each with its s_X^(1 / grid), as
// keys (kmx = 0 and kmn = ~0 mean none yet).  NaN entries are never taken,
// and an entry replaces the current one only when strictly beyond it.
struct SxExt {
  unsigned long long kmx, kmn;
  double rmx, rmn;
  __device__ __forceinline__ void init() {
    kmx = 0ull;
    kmn = ~0ull;
    rmx = rmn = 1.0;
  }
  __device__ __forceinline__ void take(double v, double r) {
    if (f64_is_nan(v)) return;
    const unsigned long long k = f64_key(v);
    if (k > kmx) kmx = k, rmx = r;
    if (k < kmn) kmn = k, rmn = r;
  }
  __device__ __forceinline__ void merge(const SxExt& o) {
    if (o.kmx > kmx) kmx = o.kmx, rmx = o.rmx;
    if (o.kmn < kmn) kmn = o.kmn, rmn = o.rmn;
  }
  __device__ __forceinline__ void warp_merge() {
    for (int o = 16; o > 0; o >>= 1) {
      SxExt t;
      t.kmx = __shfl_xor_sync(0xffffffffu, kmx, o);
      t.rmx = __shfl_xor_sync(0xffffffffu, rmx, o);
      t.kmn = __shfl_xor_sync(0xffffffffu, kmn, o);
      t.rmn = __shfl_xor_sync(0xffffffffu, rmn, o);
      merge(t);
    }
  }
  // max and min of s_X (-inf / +inf when no entry was taken)
  __device__ __forceinline__ double mx() const { return kmx ? f64_from_key(kmx) : -INFINITY; }
  __device__ __forceinline__ double mn() const { return ~kmn ? f64_from_key(kmn) : INFINITY; }
  __device__ __forceinline__ void store(double* p) const {
    reinterpret_cast<unsigned long long*>(p)[0] = kmx;
    p[1] = rmx;
    reinterpret_cast<unsigned long long*>(p)[2] = kmn;
    p[3] = rmn;
  }
  __device__ __forceinline__ void load_cg(const double* p) {
    kmx = __ldcg(reinterpret_cast<const unsigned long long*>(p));
    rmx = __ldcg(p + 1);
    kmn = __ldcg(reinterpret_cast<const unsigned long long*>(p) + 2);
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

// pow2_exponent_for on the bit pattern: m such that v * 2^m < 2^14, clamped
// to [-60, 60]; 0 for zero, negative, non-finite or huge (>= 1e300) v.
__device__ __forceinline__ int pow2_exponent_bits(double v) {
  const unsigned long long b = (unsigned long long)__double_as_longlong(v);
  if (b == 0ull || (b >> 63) || b >= 0x7E37E43C8800759Cull) return 0;  // 1e300
  const int e = (int)((b >> 52) & 0x7FF) - 1022;  // v = f * 2^e, f in [0.5, 1), normal v
  const int m = 14 - e;
  return m < -60 ? -60 : (m > 60 ? 60 : m);
}
__device__ __forceinline__ float exp2i_f32(int n) { return __int_as_float((127 + n) << 23); }
__device__ __forceinline__ double exp2i_f64(int n) {
  return __longlong_as_double((long long)(1023 + n) << 52);
}

// Columns per chunk record of s_X's extremes (the statistics and root
// launches write one record per chunk).
constexpr int kChunkCols = 32;
__host__ __device__ constexpr int chunk_count(int64_t in) {
  return (int)((in + kChunkCols - 1) / kChunkCols);
}

// The powers u[k][j] = s_X[j]^(k / grid), k = 0..grid, of the 32 columns
// j0 .. j0 + 31 (v = s_X and r = s_X^(1/grid) of column j0 + l in sh_v[l],
// sh_r[l]), by warps 0..3 of the calling CTA: warp q takes k = q, q + 4,
// q + 8, ... as running products by r^4 from r^q (binary powering), so
// each entry costs one float64 product and the chains are a quarter of
// the grid long; u[0][j] = 1 and u[grid][j] = s_X[j] exactly.
constexpr int kPowSlices = 4;
__device__ __forceinline__ void write_powers(const double* sh_v, const double* sh_r, int64_t j0,
                                             int64_t in, int grid, double* __restrict__ u) {
  const int q = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t j = j0 + lane;
  if (q >= kPowSlices || j >= in) return;
  const double v = sh_v[lane], r = sh_r[lane];
  const double step = pow_int(r, kPowSlices);
  double w = pow_int(r, q);
  for (int k = q; k <= grid; k += kPowSlices) {
    u[(int64_t)k * in + j] = k == grid ? v : w;
    w *= step;
  }
}

// Every thread of the CTA calls this: the extremes of s_X (nchunks chunk
// records SxExt::store'd by the statistics or root launch) and alpha k's
// centring, formed by thread 0 and returned to all: max(s_k) =
// max(s_X)^(k/grid) = rmx^k and likewise the minimum (exactly s_X's
// extremes at k = grid, 1 at k = 0); ic = 1 / sqrt(max * min) and q =
// sqrt(max / min) = max * ic.
__device__ __forceinline__ void centre_alpha(const double* __restrict__ minmax, int nchunks, int k,
                                             int grid, double& ic, double& q) {
  __shared__ SxExt sext[32];
  __shared__ double sh[2];
  SxExt x;
  x.init();
  for (int ch = threadIdx.x; ch < nchunks; ch += blockDim.x) {
    SxExt t;
    t.load_cg(minmax + 4 * ch);
    x.merge(t);
  }
  x.warp_merge();
  if ((threadIdx.x & 31) == 0) sext[threadIdx.x >> 5] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (unsigned w = 1; w < (blockDim.x + 31) / 32; ++w) x.merge(sext[w]);
    double smax, smin;
    if (k == 0) {
      smax = smin = 1.0;
    } else if (k == grid) {
      smax = x.mx();
      smin = x.mn();
    } else {
      smax = pow_int(x.rmx, k);
      smin = pow_int(x.rmn, k);
    }
    const double c = k == 0 ? 1.0 : rsqrt(smax * smin);
    sh[0] = c;
    sh[1] = smax * c;
  }
  __syncthreads();
  ic = sh[0];
  q = sh[1];
}

// The power-of-two operand scalings of alpha k from q (centre_alpha),
// max|W| and max|X|.  The fp16 scaling of the weight changes: one entry's
// change is |q*scale - w*s| / s <= (group step) / s, and the group step is
// at most max|W| * max(s) (either quantizer), so max|W| * max(s) / min(s)
// = max|W| * q^2 bounds |dW| for the whole alpha; its exponent e sets
// escale = 2^e (folded into the 1/s table), and X, when copied to fp16, is
// scaled by 2^m with m from max|X| (m = 0 when X is read as it is).  In the
// pre-divided mode (xs) the weights' rounding errors are at most max|W| *
// max(s) = max|W| * q and |X / s| at most max|X| / min(s) = max|X| * q,
// each with its own exponent.  unscale = 2^-2(e + m) undoes both on the
// squared sums.
__device__ __forceinline__ void alpha_scalings(double q, float wmax, float xmax, bool xs,
                                               bool x_scaled, int& e, int& m) {
  if (xs) {
    e = pow2_exponent_bits((double)wmax * q);
    m = pow2_exponent_bits((double)xmax * q);
  } else {
    e = pow2_exponent_bits((double)wmax * (q * q));
    m = x_scaled ? pow2_exponent_bits((double)xmax) : 0;
  }
}

}  // namespace awq
