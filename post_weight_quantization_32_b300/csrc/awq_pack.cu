// Final quantization at the chosen scales and bit packing.
//
// Per group of `group` columns of a row, in IEEE float32 with
// round-to-nearest on every operation ("GPTQ and AWQ weight quantisation",
// rtn_nbit; "AWQ vs GPTQ ...", group_params and rtn):
//   t = w * s
//   symmetric:  scale = max(max|t| / L, 1e-8), L = 2^(b-1) - 1,
//               q = clamp(round(t / scale), -L-1, L), stored u = q + 2^(b-1)
//   asymmetric: lo = min(min t, 0), hi = max(max t, 0),
//               scale = max((hi - lo) / maxq, 1e-8), maxq = 2^b - 1,
//               zero = round(-lo / scale), u = clamp(round(t / scale) + zero, 0, maxq)
// round() is half-to-even.  Code i of a row goes to bit i*b of the row's
// little-endian uint32 stream.
//
// The quotient t / scale is formed as t * (1/scale) and replaced by the
// correctly rounded quotient whenever it lies within 2^-21 (relative) of a
// half-integer, the only place where the two could round differently: the
// multiply-by-reciprocal result is within 3 float32 ulps of the true
// quotient.  Codes therefore equal those of true division exactly.
#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

struct QParams {
  float Lf;     // symmetric: 2^(b-1) - 1
  float maxqf;  // asymmetric: 2^b - 1
  int bits;
  int sym;
};

constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

// round(t / scale) as an integer.  r = t * (1/scale) is rounded to the
// nearest integer (ties to even) by adding and subtracting 1.5 * 2^23, exact
// for |r| < 2^22, and the integer is read off the bits of r + 1.5 * 2^23.
// Where r lies within 2^-21 (relative) of a half-integer the correctly
// rounded quotient is formed by true division instead, so the result is
// that of rounding fl32(t / scale).
__device__ __forceinline__ int round_quotient(float t, float scale, float rcp) {
  const float r = __fmul_rn(t, rcp);
  const float rm = __fadd_rn(r, kMagic);
  const float k = __fsub_rn(rm, kMagic);
  const float fr = fabsf(__fsub_rn(r, k));
  if (fabsf(__fsub_rn(fr, 0.5f)) <= __fmul_rn(fabsf(r), 4.76837158203125e-7f))  // 2^-21
    return (int)rintf(__fdiv_rn(t, scale));
  return __float_as_int(rm) - __float_as_int(kMagic);
}

__device__ __forceinline__ void group_params_sym(float m, const QParams& qp, float& scale,
                                                 int& zero) {
  scale = fmaxf(__fdiv_rn(m, qp.Lf), 1e-8f);
  zero = 1 << (qp.bits - 1);
}
__device__ __forceinline__ void group_params_asym(float lo, float hi, const QParams& qp,
                                                  float& scale, int& zero) {
  scale = fmaxf(__fdiv_rn(__fsub_rn(hi, lo), qp.maxqf), 1e-8f);
  zero = (int)rintf(__fdiv_rn(-lo, scale));
}

// Unsigned storage code of one value: symmetric q + 2^(b-1) with q clamped
// to [-2^(b-1), 2^(b-1) - 1]; asymmetric q + zero clamped to [0, 2^b - 1].
// Both are clamp(q + zero, lo, hi) with (lo, hi) = (0, 2^b - 1).
__device__ __forceinline__ uint32_t code_of(float t, float scale, float rcp, int zero, int maxq) {
  const int q = round_quotient(t, scale, rcp) + zero;
  return (uint32_t)min(max(q, 0), maxq);
}

// Fast path: group = 8 * LPG columns, LPG lanes per group (a power of two
// <= 32).  A warp handles 256 consecutive columns of one row per step, eight
// per lane, and writes 8*b whole words (256 codes of b bits).
template <typename T, int LPG>
__global__ void __launch_bounds__(256) pack_warp_kernel(const T* __restrict__ W, int64_t out,
                                                        int64_t in, const float* __restrict__ s,
                                                        QParams qp, uint32_t* __restrict__ qweight,
                                                        int64_t nwords, float* __restrict__ scales,
                                                        uint8_t* __restrict__ zeros,
                                                        int32_t* dev_status) {
  const int lane = threadIdx.x & 31;
  const int64_t segs = (in + 255) / 256;
  const int64_t total = out * segs;
  const int64_t ngroups = in / (8 * LPG);
  const int bits = qp.bits;
  const int lane_bits = 8 * bits;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; w < total;
       w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int64_t row = w / segs, seg = w % segs;
    const int64_t c0 = seg * 256 + lane * 8;
    const bool valid = c0 < in;
    float t[8];
    bool nan = false;
    if (valid) {
      float v[8], sv[8];
      load8_f32<T>(W + row * in + c0, v);
      load8_f32<float>(s + c0, sv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        t[e] = __fmul_rn(v[e], sv[e]);
        nan |= (t[e] != t[e]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) t[e] = 0.0f;
    }
    if (__any_sync(0xffffffffu, nan) && lane == 0) set_status(dev_status, ST_NONFINITE);
    float scale;
    int zero;
    if (qp.sym) {
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(t[e]));
#pragma unroll
      for (int o = 1; o < LPG; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      group_params_sym(m, qp, scale, zero);
    } else {
      float lo = 0.0f, hi = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        lo = fminf(lo, t[e]);
        hi = fmaxf(hi, t[e]);
      }
#pragma unroll
      for (int o = 1; o < LPG; o <<= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      }
      group_params_asym(lo, hi, qp, scale, zero);
    }
    const float rcp = __frcp_rn(scale);
    const int maxq = (1 << bits) - 1;
    uint64_t chunk = 0;
    if (valid) {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        chunk |= (uint64_t)code_of(t[e], scale, rcp, zero, maxq) << (e * bits);
      if ((lane & (LPG - 1)) == 0) {
        const int64_t g = c0 / (8 * LPG);
        scales[row * ngroups + g] = scale;
        zeros[row * ngroups + g] = (uint8_t)zero;
      }
    }
    // word k of this segment (8*b words) covers bits [32k, 32k + 32): at most two lanes
    for (int k0 = 0; k0 < lane_bits; k0 += 32) {
      const int k = k0 + lane;
      const int la = (32 * k) / lane_bits;
      const int lb = (32 * k + 31) / lane_bits;
      const uint64_t va = __shfl_sync(0xffffffffu, chunk, la & 31);
      const uint64_t vb = __shfl_sync(0xffffffffu, chunk, lb & 31);
      if (k < lane_bits) {
        uint64_t word = va >> (32 * k - lane_bits * la);
        if (lb != la) word |= vb << (lane_bits * lb - 32 * k);
        const int64_t wi = seg * lane_bits + k;
        if (wi < nwords) qweight[row * nwords + wi] = (uint32_t)word;
      }
    }
  }
}

// General path (any group size): one warp per (row, group), lanes strided
// over the group's columns; codes are OR-ed into the zeroed output words
// (OR is exact and order-independent, so the result is deterministic).
template <typename T>
__global__ void __launch_bounds__(256) pack_general_kernel(const T* __restrict__ W, int64_t out,
                                                           int64_t in, const float* __restrict__ s,
                                                           int group, QParams qp,
                                                           uint32_t* __restrict__ qweight,
                                                           int64_t nwords,
                                                           float* __restrict__ scales,
                                                           uint8_t* __restrict__ zeros,
                                                           int32_t* dev_status) {
  const int lane = threadIdx.x & 31;
  const int64_t ngroups = in / group;
  const int64_t total = out * ngroups;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; w < total;
       w += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int64_t row = w / ngroups, g = w % ngroups;
    const T* wr = W + row * in + g * group;
    const float* sr = s + g * group;
    float m = 0.0f, lo = 0.0f, hi = 0.0f;
    bool nan = false;
    for (int j = lane; j < group; j += 32) {
      const float t = __fmul_rn(Elt<T>::to_f32(wr[j]), sr[j]);
      nan |= (t != t);
      m = fmaxf(m, fabsf(t));
      lo = fminf(lo, t);
      hi = fmaxf(hi, t);
    }
    for (int o = 16; o > 0; o >>= 1) {
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
      lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
      hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (__any_sync(0xffffffffu, nan) && lane == 0) set_status(dev_status, ST_NONFINITE);
    float scale;
    int zero;
    if (qp.sym)
      group_params_sym(m, qp, scale, zero);
    else
      group_params_asym(lo, hi, qp, scale, zero);
    const float rcp = __frcp_rn(scale);
    const int maxq = (1 << qp.bits) - 1;
    if (lane == 0) {
      scales[row * ngroups + g] = scale;
      zeros[row * ngroups + g] = (uint8_t)zero;
    }
    for (int j = lane; j < group; j += 32) {
      const float t = __fmul_rn(Elt<T>::to_f32(wr[j]), sr[j]);
      const uint32_t u = code_of(t, scale, rcp, zero, maxq);
      const int64_t bit = (g * group + j) * (int64_t)qp.bits;
      const int64_t wi = bit >> 5;
      const int sh = (int)(bit & 31);
      uint32_t* dst = qweight + row * nwords + wi;
      atomicOr(dst, u << sh);
      if (sh + qp.bits > 32) atomicOr(dst + 1, u >> (32 - sh));
    }
  }
}

unsigned pack_grid(int64_t warps) {
  const int64_t blocks = (warps + 7) / 8;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  return (unsigned)(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

template <typename T, int LPG>
void launch_warp(const void* W, int64_t out, int64_t in, const float* s, QParams qp, uint32_t* qw,
                 int64_t nwords, float* sc, uint8_t* z, int32_t* st, cudaStream_t stream) {
  pack_warp_kernel<T, LPG><<<pack_grid(out * ((in + 255) / 256)), 256, 0, stream>>>(
      static_cast<const T*>(W), out, in, s, qp, qw, nwords, sc, z, st);
}

template <typename T>
cudaError_t pack_dispatch(const void* W, int64_t out, int64_t in, const float* s, int group,
                          QParams qp, uint32_t* qw, int64_t nwords, float* sc, uint8_t* z,
                          int32_t* st, cudaStream_t stream) {
  bool vec = (in % 8 == 0) && ((reinterpret_cast<uintptr_t>(W) & 15) == 0) &&
             ((reinterpret_cast<uintptr_t>(s) & 15) == 0);
  if (vec) {
    switch (group) {
      case 8: launch_warp<T, 1>(W, out, in, s, qp, qw, nwords, sc, z, st, stream); break;
      case 16: launch_warp<T, 2>(W, out, in, s, qp, qw, nwords, sc, z, st, stream); break;
      case 32: launch_warp<T, 4>(W, out, in, s, qp, qw, nwords, sc, z, st, stream); break;
      case 64: launch_warp<T, 8>(W, out, in, s, qp, qw, nwords, sc, z, st, stream); break;
      case 128: launch_warp<T, 16>(W, out, in, s, qp, qw, nwords, sc, z, st, stream); break;
      case 256: launch_warp<T, 32>(W, out, in, s, qp, qw, nwords, sc, z, st, stream); break;
      default: vec = false;
    }
  }
  if (!vec) {
    cudaError_t e = cudaMemsetAsync(qw, 0, (size_t)out * nwords * sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
    pack_general_kernel<T><<<pack_grid(out * (in / group)), 256, 0, stream>>>(
        static_cast<const T*>(W), out, in, s, group, qp, qw, nwords, sc, z, st);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_pack(const void* W, int dt, int64_t out, int64_t in, const float* s,
                                 int bits, int group, int sym, uint32_t* qweight, float* scales,
                                 uint8_t* zeros, int32_t* dev_status, cudaStream_t st) {
  QParams qp;
  qp.bits = bits;
  qp.sym = sym ? 1 : 0;
  qp.Lf = (float)((1 << (bits - 1)) - 1);
  qp.maxqf = (float)((1 << bits) - 1);
  const int64_t nwords = (in * bits + 31) / 32;
  switch (dt) {
    case kDtF32:
      return pack_dispatch<float>(W, out, in, s, group, qp, qweight, nwords, scales, zeros,
                                  dev_status, st);
    case kDtF16:
      return pack_dispatch<__half>(W, out, in, s, group, qp, qweight, nwords, scales, zeros,
                                   dev_status, st);
    default:
      return pack_dispatch<__nv_bfloat16>(W, out, in, s, group, qp, qweight, nwords, scales,
                                          zeros, dev_status, st);
  }
}

}  // namespace awq
