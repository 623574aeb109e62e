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
// With per-group clip factors c (the clipping search's result) the range is
// scaled first: m = fl32(c * m), or lo = fl32(c * lo), hi = fl32(c * hi),
// and values beyond it take the clamped end codes.
//
// The quotient t / scale is formed as t * (1/scale) and replaced by the
// correctly rounded quotient whenever it lies within 2^-21 (relative) of a
// half-integer, the only place where the two could round differently: the
// multiply-by-reciprocal result is within 3 float32 ulps of the true
// quotient.  Codes therefore equal those of true division exactly.
#include <algorithm>
#include <type_traits>

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

struct QParams {
  float Lf;     // symmetric: 2^(b-1) - 1
  float maxqf;  // asymmetric: 2^b - 1
  int bits;
  int sym;
  const float* clip;  // null, or [out][in/group] factors scaling each group's range
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
  pdl_wait();
  pdl_trigger();
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
        nan |= !(fabsf(t[e]) <= 3.402823466e38f);  // NaN or infinite
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
      if (qp.clip != nullptr && valid) m = __fmul_rn(qp.clip[row * ngroups + c0 / (8 * LPG)], m);
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
      if (qp.clip != nullptr && valid) {
        const float f = qp.clip[row * ngroups + c0 / (8 * LPG)];
        lo = __fmul_rn(f, lo);
        hi = __fmul_rn(f, hi);
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

// NaN-propagating max / min (the plain fmaxf / fminf drop NaN operands).
__device__ __forceinline__ float max_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float min_nan(float a, float b) {
  float d;
  asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float max3_nan(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3_nan(float a, float b, float c) {
  float d;
  asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Sixteen consecutive elements of a row as loaded (raw bits), widened later,
// so that several rows' loads are in flight before any arithmetic.
template <typename T>
struct Raw16 {
  uint4 u[2];
  __device__ __forceinline__ void load(const T* p) {
    u[0] = __ldg(reinterpret_cast<const uint4*>(p));
    u[1] = __ldg(reinterpret_cast<const uint4*>(p) + 1);
  }
  __device__ __forceinline__ void widen(float (&v)[16]) const {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t w[4] = {u[h].x, u[h].y, u[h].z, u[h].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 f;
        if constexpr (std::is_same<T, __half>::value) {
          f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
        } else {
          f = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
        }
        v[8 * h + 2 * i] = f.x;
        v[8 * h + 2 * i + 1] = f.y;
      }
    }
  }
};
template <>
struct Raw16<float> {
  float4 u[4];
  __device__ __forceinline__ void load(const float* p) {
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = __ldg(reinterpret_cast<const float4*>(p) + i);
  }
  __device__ __forceinline__ void widen(float (&v)[16]) const {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[4 * i] = u[i].x;
      v[4 * i + 1] = u[i].y;
      v[4 * i + 2] = u[i].z;
      v[4 * i + 3] = u[i].w;
    }
  }
};

// 16-byte asynchronous copy global -> shared (bypassing L1), and the
// per-thread group bookkeeping of those copies.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Fast path for b in {2, 4, 8} and group in {32, 64, ..., 1024} (lpg =
// group / 32 lanes per group).  CTA (x, y) works on the 1024-column segment
// y; its warps take rows (warp w: row x*8 + w, then every gridDim.x*8
// rows), 32 columns per lane, so each lane's 32 codes fill b whole words and
// are stored without exchange.  Each thread streams its own slice of W
// through a kPackStages-deep ring in shared memory with cp.async (no
// barriers: a thread reads only what it copied), so the loads of the next
// rows are in flight while the current one is quantized.
//
// Rounding as in round_quotient, with the screen for half-integers taken
// once per lane: |t / scale| < 2^B for every finite group (the group's own
// extreme sets the scale), so the multiply-by-reciprocal error stays below
// 2^(B-21) and only a lane with some |r - round(r)| >= 0.5 - 2^(B-21)
// re-forms its codes by true division (clamped).  Away from half-integers
// the codes need no clamp: symmetric ones lie in [1, 2^B - 1] by
// construction, and an asymmetric code can only exceed 2^B - 1 when both
// t / scale and -lo / scale sit on half-integers, which the screen catches.
// So a word is formed as sum_i bits(r_i + 1.5 * 2^23) << (i * B) plus one
// constant that removes the magic number and adds the zero point to every
// field.  A NaN or infinite product sends the row's lanes down the
// clamped path (codes unspecified but within [0, 2^B - 1]) and sets the
// status.
constexpr int kPackSeg = 1024;
constexpr int kPackStages = 3;
constexpr int kPackThreads = 256;
constexpr int kPackCtasPerSm = 3;

template <typename T>
constexpr int pack_chunks() {  // 16-byte chunks of one lane's 32 weights
  return 32 * (int)sizeof(T) / 16;
}
template <typename T>
constexpr size_t pack_smem_bytes() {
  return (size_t)kPackStages * pack_chunks<T>() * kPackThreads * 16;
}

template <typename T, int B>
__global__ void __launch_bounds__(kPackThreads, kPackCtasPerSm) pack_fast_kernel(
    const T* __restrict__ W, int64_t out, int64_t in, const float* __restrict__ s, QParams qp,
    int lpg, uint32_t* __restrict__ qweight, int64_t nwords, float* __restrict__ scales,
    uint8_t* __restrict__ zeros, int32_t* dev_status) {
  // W is an input of the call, so the first rows' copies start before the
  // launch that forms s has finished; s is read only after pdl_wait
  pdl_trigger();
  bool waited = false;
  constexpr int kChunks = pack_chunks<T>();
  constexpr int kPerWord = 32 / B;  // codes per 32-bit word
  constexpr uint32_t kMaxq = (1u << B) - 1u;
  // sum over one word's fields of 2^(i * B)
  constexpr uint32_t kRep = B == 2 ? 0x55555555u : (B == 4 ? 0x11111111u : 0x01010101u);
  extern __shared__ uint4 ring[];  // [stage][chunk][thread]
  __shared__ float4 s_seg[8][32];
  const float thr = 0.5f - ldexpf(1.0f, B - 21);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t segs = (in + kPackSeg - 1) / kPackSeg;
  const int64_t ngroups = in / (32 * lpg);
  const int64_t rstep = (int64_t)gridDim.x * 8;
  for (int64_t seg = blockIdx.y; seg < segs; seg += gridDim.y) {
    const int64_t c0 = seg * kPackSeg + lane * 32;
    const bool live = c0 < in;  // in is a multiple of the group, so all 32 columns are live
    const int64_t r0 = (int64_t)blockIdx.x * 8 + warp;
    // copies of row r0 + i * rstep into ring stage i % kPackStages (one group per row)
    auto issue = [&](int64_t i) {
      const int64_t row = r0 + i * rstep;
      if (row < out && live) {
        uint4* st = ring + (size_t)(i % kPackStages) * kChunks * kPackThreads + threadIdx.x;
        const uint4* src = reinterpret_cast<const uint4*>(W + row * in + c0);
#pragma unroll
        for (int h = 0; h < kChunks; ++h) cp_async16(st + (size_t)h * kPackThreads, src + h);
      }
      cp_async_commit();
    };
#pragma unroll
    for (int i = 0; i < kPackStages - 1; ++i) issue(i);
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    // the segment's scales, shared by every warp of the CTA: [i][lane] holds
    // s[c0 + 4i .. c0 + 4i + 3] of that lane, so a warp's reads of one i are
    // 32 consecutive 16-byte words
    if (warp == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        s_seg[i][lane] = live ? __ldg(reinterpret_cast<const float4*>(s + c0) + i)
                              : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    __syncthreads();
    for (int64_t i = 0; r0 + i * rstep < out; ++i) {
      issue(i + kPackStages - 1);
      cp_async_wait<kPackStages - 1>();
      const int64_t row = r0 + i * rstep;
      const uint4* st = ring + (size_t)(i % kPackStages) * kChunks * kPackThreads + threadIdx.x;
      // t = w * s (zero on lanes past the end of the row)
      float t[32];
      if (live) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float sv[16];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 x = s_seg[4 * h + q][lane];
            sv[4 * q] = x.x;
            sv[4 * q + 1] = x.y;
            sv[4 * q + 2] = x.z;
            sv[4 * q + 3] = x.w;
          }
          Raw16<T> raw;
#pragma unroll
          for (int c = 0; c < (int)sizeof(Raw16<T>) / 16; ++c)
            reinterpret_cast<uint4*>(&raw)[c] =
                st[(size_t)(h * (int)sizeof(Raw16<T>) / 16 + c) * kPackThreads];
          float v[16];
          raw.widen(v);
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float2 p =
                __fmul2_rn(make_float2(v[e], v[e + 1]), make_float2(sv[e], sv[e + 1]));
            t[16 * h + e] = p.x;
            t[16 * h + e + 1] = p.y;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) t[e] = 0.0f;
      }
      // group parameters (NaN-propagating extremes: a NaN marks the row bad)
      float scale;
      int zero;
      bool bad;
      if (qp.sym) {
        float m = 0.0f;
#pragma unroll
        for (int e = 0; e < 32; e += 2) m = max3_nan(m, fabsf(t[e]), fabsf(t[e + 1]));
        for (int o = 1; o < lpg; o <<= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
        bad = !(m <= 3.402823466e38f);
        scale = fmaxf(__fdiv_rn(m, qp.Lf), 1e-8f);
        zero = 1 << (B - 1);
      } else {
        float lo = 0.0f, hi = 0.0f;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          lo = min3_nan(lo, t[e], t[e + 1]);
          hi = max3_nan(hi, t[e], t[e + 1]);
        }
        for (int o = 1; o < lpg; o <<= 1) {
          lo = min_nan(lo, __shfl_xor_sync(0xffffffffu, lo, o));
          hi = max_nan(hi, __shfl_xor_sync(0xffffffffu, hi, o));
        }
        const float span = __fsub_rn(hi, lo);
        bad = !(span <= 3.402823466e38f);
        scale = fmaxf(__fdiv_rn(span, qp.maxqf), 1e-8f);
        zero = (int)rintf(__fdiv_rn(-lo, scale));
      }
      const bool row_bad = __any_sync(0xffffffffu, bad);
      if (row_bad && lane == 0) set_status(dev_status, ST_NONFINITE);
      if (!live) continue;
      // codes: each word is a sum of shifted magic-number bit patterns plus
      // one constant (see above)
      const float rcp = __frcp_rn(scale);
      const uint32_t cw = (uint32_t)(zero - __float_as_int(kMagic)) * kRep;
      uint32_t wd[B];
      float dmax = 0.0f;
#pragma unroll
      for (int w = 0; w < B; ++w) {
        uint32_t acc = cw;
#pragma unroll
        for (int e = 0; e < kPerWord; e += 2) {
          const int x = w * kPerWord + e;
          const float2 rr = __fmul2_rn(make_float2(t[x], t[x + 1]), make_float2(rcp, rcp));
          const float2 rm = __fadd2_rn(rr, make_float2(kMagic, kMagic));
          const float2 k = __fadd2_rn(rm, make_float2(-kMagic, -kMagic));
          const float2 d = __fadd2_rn(rr, make_float2(-k.x, -k.y));
          dmax = fmax3f(dmax, fabsf(d.x), fabsf(d.y));
          acc += (uint32_t)__float_as_int(rm.x) << (e * B);
          acc += (uint32_t)__float_as_int(rm.y) << ((e + 1) * B);
        }
        wd[w] = acc;
      }
      if (dmax >= thr || row_bad) {  // rare: a quotient close to a half-integer, or NaN / inf
#pragma unroll
        for (int w = 0; w < B; ++w) {
          uint32_t acc = 0u;
#pragma unroll
          for (int e = 0; e < kPerWord; ++e) {
            const uint32_t q = min(
                (uint32_t)((int)rintf(__fdiv_rn(t[w * kPerWord + e], scale)) + zero), kMaxq);
            acc |= q << (e * B);
          }
          wd[w] = acc;
        }
      }
      uint32_t* dst = qweight + row * nwords + seg * (kPackSeg * B / 32) + lane * B;
      if constexpr (B == 2) {
        *reinterpret_cast<uint2*>(dst) = make_uint2(wd[0], wd[1]);
      } else {
#pragma unroll
        for (int w = 0; w < B; w += 4)
          *reinterpret_cast<uint4*>(dst + w) = make_uint4(wd[w], wd[w + 1], wd[w + 2], wd[w + 3]);
      }
      if ((lane & (lpg - 1)) == 0) {
        const int64_t g = c0 / (32 * lpg);
        scales[row * ngroups + g] = scale;
        zeros[row * ngroups + g] = (uint8_t)zero;
      }
    }
    cp_async_wait<0>();  // no copy may still target the ring when it is reused
    __syncthreads();     // nor any warp still read the segment's scales
  }
  if (!waited) pdl_wait();
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
      nan |= !(fabsf(t) <= 3.402823466e38f);  // NaN or infinite
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
    if (qp.clip != nullptr) {
      const float f = qp.clip[row * ngroups + g];
      m = __fmul_rn(f, m);
      lo = __fmul_rn(f, lo);
      hi = __fmul_rn(f, hi);
    }
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
  launch_pdl(pack_warp_kernel<T, LPG>, pack_grid(out * ((in + 255) / 256)), 256, 0, stream,
             static_cast<const T*>(W), out, in, s, qp, qw, nwords, sc, z, st);
}

template <typename T, int B>
cudaError_t launch_fast(const void* W, int64_t out, int64_t in, const float* s, QParams qp,
                        int lpg, uint32_t* qw, int64_t nwords, float* sc, uint8_t* z, int32_t* st,
                        cudaStream_t stream) {
  const size_t smem = pack_smem_bytes<T>();
  static bool attr_set[64] = {false};  // per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(pack_fast_kernel<T, B>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  // about kPackCtasPerSm CTAs per SM in all, spread over the segments
  const int64_t segs = (in + kPackSeg - 1) / kPackSeg;
  const int64_t ys = segs < 65535 ? segs : 65535;
  int64_t xs = (kPackCtasPerSm * (int64_t)device_sm_count() + ys - 1) / ys;
  xs = std::min<int64_t>(std::max<int64_t>(xs, 1), (out + 7) / 8);
  return launch_pdl(pack_fast_kernel<T, B>, dim3((unsigned)xs, (unsigned)ys), kPackThreads, smem,
                    stream, static_cast<const T*>(W), out, in, s, qp, lpg, qw, nwords, sc, z, st);
}

template <typename T>
cudaError_t pack_dispatch(const void* W, int64_t out, int64_t in, const float* s, int group,
                          QParams qp, uint32_t* qw, int64_t nwords, float* sc, uint8_t* z,
                          int32_t* st, cudaStream_t stream) {
  bool vec = (in % 8 == 0) && ((reinterpret_cast<uintptr_t>(W) & 15) == 0) &&
             ((reinterpret_cast<uintptr_t>(s) & 15) == 0);
  const bool fast_shape = (qp.bits == 2 || qp.bits == 4 || qp.bits == 8) && group >= 32 &&
                          group <= 1024 && (group & (group - 1)) == 0;
  if (vec && fast_shape && qp.clip == nullptr &&
      (reinterpret_cast<uintptr_t>(qw) & (uintptr_t)(qp.bits == 2 ? 7 : 15)) == 0) {
    const int lpg = group / 32;
    switch (qp.bits) {
      case 2: return launch_fast<T, 2>(W, out, in, s, qp, lpg, qw, nwords, sc, z, st, stream);
      case 4: return launch_fast<T, 4>(W, out, in, s, qp, lpg, qw, nwords, sc, z, st, stream);
      default: return launch_fast<T, 8>(W, out, in, s, qp, lpg, qw, nwords, sc, z, st, stream);
    }
  }
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
                                 int bits, int group, int sym, const float* clip,
                                 uint32_t* qweight, float* scales, uint8_t* zeros,
                                 int32_t* dev_status, cudaStream_t st) {
  QParams qp;
  qp.clip = clip;
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
