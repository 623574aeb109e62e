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

#include <algorithm>

#include "awq_alpha.cuh"
#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

constexpr int kPrepChunk = 64;   // columns per CTA of the per-column kernels
constexpr int kMaxGrid = 4096;   // largest grid the C ABI accepts

// grid = chunks: root[j] = sx[j] ^ (1 / grid) in float64 and each chunk's
// max and min of sx; the last CTA to finish reduces the chunk extremes and
// forms the per-alpha centring values.  (The statistics launch does the same
// when it computes sx itself; this kernel serves a caller-given sx.)
__global__ void __launch_bounds__(kPrepChunk) alpha_root_kernel(const double* __restrict__ sx,
                                                               int64_t in, CentreArgs ca) {
  pdl_wait();
  pdl_trigger();
  SxExt x;
  x.init();
  const int64_t j = (int64_t)blockIdx.x * kPrepChunk + threadIdx.x;
  if (j < in) {
    const double v = sx[j];
    const double r = exp(log(v) / (double)ca.grid);
    ca.root[j] = r;
    x.take(v, r);
  }
  __shared__ SxExt sext[kPrepChunk / 32];
  x.warp_merge();
  if ((threadIdx.x & 31) == 0) sext[threadIdx.x >> 5] = x;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kPrepChunk / 32; ++w) x.merge(sext[w]);
    x.store(ca.minmax + 4 * blockIdx.x);
  }
  centre_if_last(ca, gridDim.x);
}

// One CTA per kTabCols columns; warp q of the CTA takes the alphas k = q,
// q + kTabSlices, q + 2 kTabSlices, ... of every column, so the float64
// product chains are kTabSlices times shorter than one chain per column.
// s_k = sx ^ (k / grid) = root^k: root^q by binary powering, then running
// products by root^kTabSlices (exactly 1 at k = 0 and exactly sx at
// k = grid), centred, rounded to float32; inv_s32 = 2^e_k / s.  pow2_s[k]
// is cleared when some entry of the chunk is not a power of two (a bit per
// alpha in shared memory, applied once per alpha at the end).
constexpr int kTabCols = 32, kTabSlices = 4;

//
// With ss32 != nullptr (the pre-divided search): inv_s32[k][j] = xscale[k] /
// s32 (the factor X is multiplied by) and ss32[k][j] = s32 * escale[k].
__global__ void __launch_bounds__(kTabCols * kTabSlices) alpha_table_kernel(
    const double* __restrict__ sx, const double* __restrict__ root,
    const double* __restrict__ inv_c, const float* __restrict__ escale,
    const float* __restrict__ xscale, int64_t in, int grid, float* __restrict__ s32,
    float* __restrict__ inv_s32, float* __restrict__ ss32, int32_t* __restrict__ pow2_s) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint32_t not_pow2[(kMaxGrid + 1 + 31) / 32];
  const int nwords = (grid + 1 + 31) / 32;
  for (int i = threadIdx.x; i < nwords; i += blockDim.x) not_pow2[i] = 0u;
  __syncthreads();
  const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
  const int64_t j = (int64_t)blockIdx.x * kTabCols + lane;
  const bool live = j < in;
  const double sxj = live ? sx[j] : 1.0, r = live ? root[j] : 1.0;
  const double step = pow_int(r, kTabSlices);
  double v = pow_int(r, q);
  for (int k = q; k <= grid; k += kTabSlices) {
    const double sk = k == grid ? sxj : v;
    const float f = __double2float_rn(sk * inv_c[k]);
    bool np2 = false;
    if (live) {
      s32[(int64_t)k * in + j] = f;
      if (ss32 != nullptr) {
        inv_s32[(int64_t)k * in + j] = __frcp_rn(f) * xscale[k];
        ss32[(int64_t)k * in + j] = f * escale[k];
      } else {
        inv_s32[(int64_t)k * in + j] = __frcp_rn(f) * escale[k];
      }
      np2 = (__float_as_uint(f) & 0x007FFFFFu) != 0u;
    }
    if (__any_sync(0xffffffffu, np2) && lane == 0) atomicOr(&not_pow2[k / 32], 1u << (k % 32));
    v *= step;
  }
  __syncthreads();
  for (int k = threadIdx.x; k <= grid; k += blockDim.x)
    if ((not_pow2[k / 32] >> (k % 32)) & 1u) atomicAnd(&pow2_s[k], 0);
}

// One CTA: per-alpha fixed-order sums, strict argmin, copy of the kept scales.
// With parts > 0 (the finish of a row-split search) err_k is instead
// sum_{p < parts} partials[p][k] / denom, added in part order, and unscale
// is not read.
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
  __shared__ double err_sh[kMaxGrid + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (parts > 0) {
    for (int k = threadIdx.x; k < n_alpha; k += blockDim.x) {
      double s = 0.0;
      for (int q = 0; q < parts; ++q) s += partials[(int64_t)q * n_alpha + k];
      const double e = s / denom;
      err[k] = e;
      err_sh[k] = e;
    }
  } else {
    for (int k = warp; k < n_alpha; k += blockDim.x >> 5) {
      double s = 0.0;
      for (int t = lane; t < n_tiles; t += 32) s += __ldcg(partials + (int64_t)k * n_tiles + t);
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (lane == 0) {
        const double e = s * unscale[k] / denom;
        err[k] = e;
        err_sh[k] = e;
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    // first index of the smallest error under strict <, starting from +inf:
    // each lane scans its own alphas in order, then lanes merge preferring
    // the smaller error and, on equal errors, the smaller index
    int best = -1;
    double be = INFINITY;
    for (int k = lane; k < n_alpha; k += 32) {
      const double e = err_sh[k];
      if (e < be) {
        be = e;
        best = k;
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      const double oe = __shfl_xor_sync(0xffffffffu, be, o);
      const int ob = __shfl_xor_sync(0xffffffffu, best, o);
      if (ob >= 0 && (best < 0 || oe < be || (oe == be && ob < best))) {
        be = oe;
        best = ob;
      }
    }
    if (lane == 0) {
      if (best < 0) set_status(dev_status, ST_NONFINITE);
      *best_out = best;
      best_sh = best;
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

size_t prep_chunks(int64_t in) { return (size_t)((in + 31) / 32); }  // the finer of the two chunkings

cudaError_t launch_alpha_root(const double* sx, int64_t in, const CentreArgs& ca, cudaStream_t s) {
  if (ca.grid < 1 || ca.grid > kMaxGrid) return cudaErrorInvalidValue;
  return launch_pdl(alpha_root_kernel, (unsigned)((in + kPrepChunk - 1) / kPrepChunk), kPrepChunk,
                    0, s, sx, in, ca);
}

cudaError_t launch_alpha_table(const double* sx, const double* root, const double* inv_c,
                               const float* escale, int64_t in, int grid, float* s32,
                               float* inv_s32, int32_t* pow2_s, cudaStream_t s) {
  if (grid < 1 || grid > kMaxGrid) return cudaErrorInvalidValue;
  return launch_pdl(alpha_table_kernel, (unsigned)((in + kTabCols - 1) / kTabCols),
                    kTabCols * kTabSlices, 0, s, sx, root, inv_c, escale,
                    static_cast<const float*>(nullptr), in, grid, s32, inv_s32,
                    static_cast<float*>(nullptr), pow2_s);
}

cudaError_t launch_alpha_table_xs(const double* sx, const double* root, const double* inv_c,
                                  const float* escale, const float* xscale, int64_t in, int grid,
                                  float* s32, float* inv_s32, float* ss32, int32_t* pow2_s,
                                  cudaStream_t s) {
  if (grid < 1 || grid > kMaxGrid || ss32 == nullptr || xscale == nullptr)
    return cudaErrorInvalidValue;
  return launch_pdl(alpha_table_kernel, (unsigned)((in + kTabCols - 1) / kTabCols),
                    kTabCols * kTabSlices, 0, s, sx, root, inv_c, escale, xscale, in, grid, s32,
                    inv_s32, ss32, pow2_s);
}

cudaError_t launch_reduce_argmin(const double* partials, const double* unscale, int n_alpha,
                                 int n_tiles, double denom, const float* s32, int64_t in,
                                 double* err, int32_t* best, float* s_best, int32_t* dev_status,
                                 cudaStream_t s) {
  return launch_pdl(reduce_argmin_kernel, 1, 1024, 0, s, partials, unscale, n_alpha, n_tiles, denom,
                    s32, in, err, best, s_best, dev_status, 0);
}

cudaError_t launch_search_finish(const double* sums, int parts, int n_alpha, double denom,
                                 const float* s_table, int64_t in, double* err, int32_t* best,
                                 float* s_best, int32_t* dev_status, cudaStream_t s) {
  if (n_alpha < 1 || n_alpha > kMaxGrid + 1 || parts < 1) return cudaErrorInvalidValue;
  return launch_pdl(reduce_argmin_kernel, 1, 1024, 0, s, sums, static_cast<const double*>(nullptr),
                    n_alpha, 0, denom, s_table, in, err, best, s_best, dev_status, parts);
}

}  // namespace awq
