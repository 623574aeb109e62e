// Channel statistics s_X[j] = mean_n |X[n, j]| + 1e-8 ("AWQ (activation-aware
// weight quantization)", "How it works" step 1), the max |.| reductions that
// set the power-of-two operand scalings, and the fp16 copy of X that the
// tensor-core error GEMM reads when X is not fp16 already.
//
// All are HBM-bound passes.  The statistic is accumulated in a fixed order
// (exactly, as an integer, for fp16 X), so repeated calls give identical
// results.
#include <algorithm>
#include <climits>
#include <type_traits>

#include "awq_alpha.cuh"
#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

constexpr int kStatCols = kChunkCols;  // columns per CTA of the vector path (4 lanes x 8 columns)
constexpr int kStatSlices = 64;  // row slices per CTA of the vector path
constexpr int kScalarCols = 64;  // columns per CTA of the scalar path

// max(|v|) over a CTA as the bit pattern of a non-negative float, folded into
// *out with one atomicMax (the integer order of such patterns is the float
// order, so the result does not depend on the order of the CTAs).  NaN is
// ignored.
__device__ __forceinline__ void block_absmax(float m, uint32_t* out) {
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float wm[32];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, wm[w]);
    atomicMax(out, __float_as_uint(m));
  }
}

// Column sums of |x| over 8 columns.  For fp16 the sum is kept exactly as an
// integer count of 2^-24 (every |x| is an integer multiple of 2^-24 below
// 2^16, so sums of up to 2^24 rows stay below 2^64), which makes the mean
// identical to the correctly rounded float64 one and independent of the
// order of addition; infinities and NaN are tracked apart so the result is
// what a float64 sum would give.  Other types accumulate in float64.
template <typename T>
struct ColSum {
  using Part = double;
  double acc[8];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0;
  }
  __device__ __forceinline__ void add(const T* p, float& m) {
    float v[8];
    load8_f32<T>(p, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      acc[e] += (double)fabsf(v[e]);
      m = fmaxf(m, fabsf(v[e]));
    }
  }
  __device__ __forceinline__ Part part(int e) const { return acc[e]; }
  __device__ __forceinline__ void flag_specials(uint32_t*) const {}
  __device__ __forceinline__ void finish_max(float&) const {}
  static __device__ __forceinline__ double total(Part a, uint32_t) { return a; }
};

template <>
struct ColSum<__half> {
  using Part = unsigned long long;
  unsigned long long acc[8];
  uint32_t special;  // bit e: column e saw an infinity; bit 8 + e: a NaN
  uint32_t mbits;    // largest |x| seen (NaN excluded) as fp16 bits: their integer order is the value order
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0ull;
    special = 0u;
    mbits = 0u;
  }
  __device__ __forceinline__ void add(const __half* p, float&) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t h = (w[e >> 1] >> ((e & 1) * 16)) & 0x7FFFu;
      const uint32_t ex = h >> 10, mant = h & 0x3FFu;
      if (!(ex == 31u && mant != 0u)) mbits = max(mbits, h);
      if (ex == 31u) {
        special |= mant ? (1u << (8 + e)) : (1u << e);
      } else {
        acc[e] += ex == 0u ? (unsigned long long)mant
                           : ((unsigned long long)(mant | 0x400u) << (ex - 1u));
      }
    }
  }
  __device__ __forceinline__ Part part(int e) const { return acc[e]; }
  __device__ __forceinline__ void finish_max(float& m) const {
    m = __half2float(__ushort_as_half((unsigned short)mbits));
  }
  // per column of the CTA: bit 0 = an infinity was seen, bit 1 = a NaN
  __device__ __forceinline__ void flag_specials(uint32_t* spec) const {
    if (special == 0u) return;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t f = ((special >> e) & 1u) | (((special >> (8 + e)) & 1u) << 1);
      if (f) atomicOr(spec + e, f);
    }
  }
  static __device__ __forceinline__ double total(Part a, uint32_t spec) {
    if (spec & 2u) return __longlong_as_double(0x7FF8000000000000ll);
    if (spec & 1u) return INFINITY;
    return (double)a * 0x1p-24;  // exact: a power of two
  }
};

// Vector path: in % 8 == 0 and 16-byte aligned rows.  Thread (c, r) of CTA
// b sums the 8 columns c*8..c*8+7 of the CTA's 32 over rows r, r+64,
// r+128, ..., four 16-byte loads in flight at a time; the 64 slices are
// then added in a fixed order.  With xmax != nullptr the pass also folds
// max|X| into *xmax.  With ca.grid != 0 the CTA also writes its columns'
// powers s_X^(k / grid) and its chunk's extremes of s_X with their roots
// (CentreArgs; no step crosses CTAs).  Each CTA lets the next launch start
// once it has read its part of X: that launch streams W, and X's loads
// would otherwise queue behind W's.
template <typename T>
__global__ void __launch_bounds__(256) stats_vec_kernel(const T* __restrict__ X, int64_t N,
                                                        int64_t in, double* __restrict__ sx,
                                                        uint32_t* __restrict__ xmax,
                                                        CentreArgs ca) {
  using Part = typename ColSum<T>::Part;
  __shared__ Part red[kStatSlices][kStatCols + 1];
  __shared__ Part red2[kStatSlices / 8][kStatCols + 1];
  __shared__ uint32_t spec[kStatCols];
  __shared__ double sh_v[kStatCols], sh_r[kStatCols];
  if (threadIdx.x < kStatCols) spec[threadIdx.x] = 0u;
  if (ca.grid != 0 && blockIdx.x == 0)
    for (int k = threadIdx.x; k <= ca.grid; k += blockDim.x) ca.pow2_s[k] = 1;
  __syncthreads();
  const int c = threadIdx.x % 4, r = threadIdx.x / 4;
  const int64_t col0 = (int64_t)blockIdx.x * kStatCols + c * 8;
  ColSum<T> cs;
  cs.init();
  float m = 0.0f;
  if (col0 < in) {
    int64_t n = r;
    for (; n + 3 * kStatSlices < N; n += 4 * kStatSlices) {
#pragma unroll
      for (int u = 0; u < 4; ++u) cs.add(X + (n + u * kStatSlices) * in + col0, m);
    }
    for (; n < N; n += kStatSlices) cs.add(X + n * in + col0, m);
  }
  pdl_trigger();
#pragma unroll
  for (int e = 0; e < 8; ++e) red[r][c * 8 + e] = cs.part(e);
  cs.flag_specials(spec + c * 8);
  cs.finish_max(m);
  if (xmax != nullptr) block_absmax(m, xmax);  // contains __syncthreads
  __syncthreads();
  {  // the 64 slices in a fixed two-level order: 8 runs of 8, then the 8 run sums
    const int cc = threadIdx.x % kStatCols, pp = threadIdx.x / kStatCols;
    Part a = red[pp * 8][cc];
#pragma unroll
    for (int k = 1; k < 8; ++k) a += red[pp * 8 + k][cc];
    red2[pp][cc] = a;
  }
  __syncthreads();
  if (threadIdx.x < kStatCols) {  // warp 0
    const int64_t j = (int64_t)blockIdx.x * kStatCols + threadIdx.x;
    SxExt x;
    x.init();
    if (j < in) {
      Part a = red2[0][threadIdx.x];
#pragma unroll
      for (int k = 1; k < kStatSlices / 8; ++k) a += red2[k][threadIdx.x];
      const double v = ColSum<T>::total(a, spec[threadIdx.x]) / (double)N + 1e-8;
      sx[j] = v;
      if (ca.grid != 0) {
        const double rt = exp(log(v) / (double)ca.grid);
        sh_v[threadIdx.x] = v;
        sh_r[threadIdx.x] = rt;
        x.take(v, rt);
      }
    }
    if (ca.grid != 0) {
      x.warp_merge();
      if (threadIdx.x == 0) x.store(ca.minmax + 4 * blockIdx.x);
    }
  }
  if (ca.grid == 0) return;
  __syncthreads();
  write_powers(sh_v, sh_r, (int64_t)blockIdx.x * kStatCols, in, ca.grid, ca.u);
}

// fp16(v[i] * f[i]) for i < 8, packed into 16 bytes.
__device__ __forceinline__ uint4 scaled_f16x8(const float (&v)[8], const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    __half2 h = __floats2half2_rn(v[2 * p] * f[2 * p], v[2 * p + 1] * f[2 * p + 1]);
    w[p] = *reinterpret_cast<uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// max|W| (CTAs [0, nw)) and, with xs != nullptr, the pre-divided search's
// table and X copies (CTAs [nw, gridDim.x)) in one launch, so that the
// copies are formed while the weights stream.
//
// A max|W| CTA: eight 16-byte loads in flight per thread, folded into *wmax.
//
// A copy CTA (x, k) (x fastest) owns columns 256 x .. 256 x + 255 and alpha
// k.  Once the statistics launch is done it reduces the chunk extremes and
// centres alpha k (centre_alpha; CTA x = 0 stores qk[k]); thread i forms
// the table entry f = fp32(u[k][j] * ic) of column j = 256 x + i, writes
// s32[k][j] = f and leaves the factor 2^m_k / f that X is multiplied by in
// shared memory; pow2_s[k] is cleared when some entry is not a power of
// two.  Lane l of every warp then owns the eight columns 8 (32 x + l) .. + 7
// (a warp covers 512 contiguous bytes of a row) and the eight warps walk
// the rows, four rows in flight: xs[k][n][j] = fp16(X[n][j] * factor[j]).
//
// Every CTA waits for the launch before it before finishing, so this launch
// ends after the statistics launch whatever it does.
template <typename T>
__global__ void __launch_bounds__(256, 5) wmax_xs_kernel(
    const T* __restrict__ W, int64_t nW, uint32_t* __restrict__ wmax, int nw,
    const T* __restrict__ X, int N, int in, int grid, const double* __restrict__ u,
    const double* __restrict__ minmax, const uint32_t* __restrict__ xmax_bits,
    float* __restrict__ s32, double* __restrict__ qk, int32_t* __restrict__ pow2_s,
    uint4* __restrict__ xs) {
  pdl_trigger();
  if ((int)blockIdx.x < nw) {
    float m = 0.0f;
    const int64_t n8 = nW / 8;
    const int64_t stride = (int64_t)nw * blockDim.x;
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i < n8; i += 8 * stride) {  // eight 16-byte loads in flight
      float v[8][8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (i + q * stride < n8) {
          load8_f32<T>(W + (i + q * stride) * 8, v[q]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[q][e] = 0.0f;
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q)
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[q][e]));
    }
    block_absmax(m, wmax);
    pdl_wait();
    return;
  }
  pdl_wait();
  __shared__ __align__(16) float fac[256];
  const int b = (int)blockIdx.x - nw;
  const int nxb = (in + 255) / 256;
  const int k = b / nxb, xb = b % nxb;
  const int j = xb * 256 + (int)threadIdx.x;
  const double uk = j < in ? u[(int64_t)k * in + j] : 1.0;
  double ic, q;
  centre_alpha(minmax, chunk_count(in), k, grid, ic, q);
  if (xb == 0 && threadIdx.x == 0) qk[k] = q;
  int e, mexp;
  alpha_scalings(q, 0.0f, __uint_as_float(*xmax_bits), true, false, e, mexp);
  bool np2 = false;
  if (j < in) {
    const float f = __double2float_rn(uk * ic);
    s32[(int64_t)k * in + j] = f;
    fac[threadIdx.x] = __frcp_rn(f) * exp2i_f32(mexp);
    np2 = (__float_as_uint(f) & 0x007FFFFFu) != 0u;
  }
  if (__syncthreads_or(np2) && threadIdx.x == 0) atomicAnd(&pow2_s[k], 0);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j8 = xb * 32 + lane;
  const int n8 = in / 8;
  if (j8 >= n8) return;
  float f[8];
  {
    const float4 a = reinterpret_cast<const float4*>(fac + lane * 8)[0];
    const float4 c4 = reinterpret_cast<const float4*>(fac + lane * 8)[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = c4.x; f[5] = c4.y; f[6] = c4.z; f[7] = c4.w;
  }
  const T* src = X + (int64_t)j8 * 8;
  uint4* dst = xs + (int64_t)k * N * n8 + j8;
  int n = warp;
  for (; n + 24 < N; n += 32) {  // rows n, n + 8, n + 16, n + 24: four loads in flight
    float v[4][8];
#pragma unroll
    for (int p = 0; p < 4; ++p) load8_f32<T>(src + (int64_t)(n + 8 * p) * in, v[p]);
#pragma unroll
    for (int p = 0; p < 4; ++p) dst[(int64_t)(n + 8 * p) * n8] = scaled_f16x8(v[p], f);
  }
  for (; n < N; n += 8) {
    float v[8];
    load8_f32<T>(src + (int64_t)n * in, v);
    dst[(int64_t)n * n8] = scaled_f16x8(v, f);
  }
}

// Scalar path for any shape: thread (c, r) sums column c over rows r, r+4, ...
template <typename T>
__global__ void __launch_bounds__(256) stats_scalar_kernel(const T* __restrict__ X, int64_t N,
                                                           int64_t in, double* __restrict__ sx) {
  __shared__ double red[4][kScalarCols];
  const int c = threadIdx.x % kScalarCols, r = threadIdx.x / kScalarCols;
  const int64_t j = (int64_t)blockIdx.x * kScalarCols + c;
  double acc = 0.0;
  if (j < in)
    for (int64_t n = r; n < N; n += 4) acc += (double)fabsf(Elt<T>::to_f32(X[n * in + j]));
  red[r][c] = acc;
  __syncthreads();
  if (r == 0 && j < in)
    sx[j] = (((red[0][c] + red[1][c]) + red[2][c]) + red[3][c]) / (double)N + 1e-8;
}

// max |x| over n values into *out (see block_absmax), four 16-byte loads in
// flight per thread.
template <typename T>
__global__ void __launch_bounds__(256) absmax_kernel(const T* __restrict__ p, int64_t n, bool vec,
                                                     uint32_t* __restrict__ out) {
  float m = 0.0f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (vec) {
    const int64_t n8 = n / 8;
    int64_t i = i0;
    for (; i + 3 * stride < n8; i += 4 * stride) {
      float v[4][8];
#pragma unroll
      for (int u = 0; u < 4; ++u) load8_f32<T>(p + (i + u * stride) * 8, v[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[u][e]));
    }
    for (; i < n8; i += stride) {
      float v[8];
      load8_f32<T>(p + i * 8, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[e]));
    }
  } else {
    for (int64_t i = i0; i < n; i += stride) m = fmaxf(m, fabsf(Elt<T>::to_f32(p[i])));
  }
  block_absmax(m, out);
}

// dst = fp16(X * 2^m), m from max|X| (pow2_exponent_for): an exact
// power-of-two scaling, then one rounding to fp16.
template <typename T>
__global__ void __launch_bounds__(256) to_f16_kernel(const T* __restrict__ X, int64_t n8,
                                                     const uint32_t* __restrict__ xmax_bits,
                                                     uint4* __restrict__ dst) {
  pdl_wait();
  pdl_trigger();
  const float sc = ldexpf(1.0f, pow2_exponent_for((double)__uint_as_float(*xmax_bits)));
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v[8];
    load8_f32<T>(X + i * 8, v);
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      __half2 h = __floats2half2_rn(v[2 * k] * sc, v[2 * k + 1] * sc);
      w[k] = *reinterpret_cast<uint32_t*>(&h);
    }
    dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

unsigned grid_for(int64_t work);

template <typename T>
cudaError_t stats_dispatch(const void* X, int64_t N, int64_t in, double* sx, uint32_t* xmax,
                           const CentreArgs& ca, cudaStream_t s) {
  const bool vec = (in % 8 == 0) && ((reinterpret_cast<uintptr_t>(X) & 15) == 0);
  if (vec) {
    const int nx = (int)((in + kStatCols - 1) / kStatCols);
    stats_vec_kernel<T><<<(unsigned)nx, 256, 0, s>>>(static_cast<const T*>(X), N, in, sx, xmax,
                                                     ca);
  } else {
    if (xmax != nullptr || ca.grid != 0) return cudaErrorInvalidValue;
    stats_scalar_kernel<T><<<(unsigned)((in + kScalarCols - 1) / kScalarCols), 256, 0, s>>>(
        static_cast<const T*>(X), N, in, sx);
  }
  return cudaGetLastError();
}

template <typename T>
cudaError_t wmax_xs_dispatch(const void* W, int64_t nW, uint32_t* wmax, const void* X, int64_t N,
                             int64_t in, int grid, const double* u, const double* minmax,
                             const uint32_t* xmax_bits, float* s32, double* qk, int32_t* pow2_s,
                             void* xs, cudaStream_t s) {
  if (nW % 8 != 0 || (reinterpret_cast<uintptr_t>(W) & 15) != 0) return cudaErrorInvalidValue;
  // max|W| CTAs: eight 16-byte loads in flight per thread, at most three
  // per SM (five fit), so that copy CTAs find room beside them
  const int nw = (int)std::max<int64_t>(
      1, std::min<int64_t>((nW / 8 + 2047) / 2048, (int64_t)device_sm_count() * 3));
  int64_t ncopy = 0;
  if (xs != nullptr) {
    if (in % 8 != 0 || (reinterpret_cast<uintptr_t>(X) & 15) != 0 || N > (1 << 24) ||
        in > (1 << 24) || grid < 1 || grid > kMaxGrid)
      return cudaErrorInvalidValue;
    ncopy = ((in + 255) / 256) * (int64_t)(grid + 1);
  }
  if (nw + ncopy > INT_MAX) return cudaErrorInvalidValue;
  return launch_pdl(wmax_xs_kernel<T>, (unsigned)(nw + ncopy), 256, 0, s, static_cast<const T*>(W),
                    nW, wmax, nw, static_cast<const T*>(X), (int)N, (int)in, grid, u, minmax,
                    xmax_bits, s32, qk, pow2_s, static_cast<uint4*>(xs));
}

unsigned grid_for(int64_t work) {
  const int64_t want = (work + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 4;
  return (unsigned)std::max<int64_t>(1, std::min(want, cap));
}

}  // namespace

cudaError_t launch_channel_stats(const void* X, int dt, int64_t N, int64_t in, double* sx,
                                 uint32_t* xmax, const CentreArgs& ca, cudaStream_t s) {
  switch (dt) {
    case kDtF32: return stats_dispatch<float>(X, N, in, sx, xmax, ca, s);
    case kDtF16: return stats_dispatch<__half>(X, N, in, sx, xmax, ca, s);
    default: return stats_dispatch<__nv_bfloat16>(X, N, in, sx, xmax, ca, s);
  }
}

cudaError_t launch_wmax_xs(const void* W, int dt, int64_t nW, uint32_t* wmax, const void* X,
                           int64_t N, int64_t in, int grid, const double* u,
                           const double* minmax, const uint32_t* xmax_bits, float* s32,
                           double* qk, int32_t* pow2_s, void* xs, cudaStream_t s) {
  switch (dt) {
    case kDtF32:
      return wmax_xs_dispatch<float>(W, nW, wmax, X, N, in, grid, u, minmax, xmax_bits, s32, qk,
                                     pow2_s, xs, s);
    case kDtF16:
      return wmax_xs_dispatch<__half>(W, nW, wmax, X, N, in, grid, u, minmax, xmax_bits, s32, qk,
                                      pow2_s, xs, s);
    default:
      return wmax_xs_dispatch<__nv_bfloat16>(W, nW, wmax, X, N, in, grid, u, minmax, xmax_bits,
                                             s32, qk, pow2_s, xs, s);
  }
}

cudaError_t launch_absmax(const void* p, int dt, int64_t n, uint32_t* out, cudaStream_t s) {
  const bool vec = (n % 8 == 0) && ((reinterpret_cast<uintptr_t>(p) & 15) == 0);
  const unsigned grid = grid_for(vec ? n / 8 : n);
  switch (dt) {
    case kDtF32:
      absmax_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(p), n, vec, out);
      break;
    case kDtF16:
      absmax_kernel<__half><<<grid, 256, 0, s>>>(static_cast<const __half*>(p), n, vec, out);
      break;
    default:
      absmax_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(p), n,
                                                        vec, out);
  }
  return cudaGetLastError();
}

cudaError_t launch_to_f16(const void* X, int dt, int64_t n, const uint32_t* xmax_bits, void* dst,
                          cudaStream_t s) {
  const int64_t n8 = n / 8;
  const unsigned grid = grid_for(n8);
  uint4* d = static_cast<uint4*>(dst);
  if (dt == kDtF32)
    return launch_pdl(to_f16_kernel<float>, grid, 256, 0, s, static_cast<const float*>(X), n8,
                      xmax_bits, d);
  return launch_pdl(to_f16_kernel<__nv_bfloat16>, grid, 256, 0, s,
                    static_cast<const __nv_bfloat16*>(X), n8, xmax_bits, d);
}

}  // namespace awq
