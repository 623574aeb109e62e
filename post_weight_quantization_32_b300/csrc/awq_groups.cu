// Group ranges computed ahead of the search, for groups that the search
// kernel's producer jobs do not contain: wider than a job (a multiple of 256
// columns, or one group per row), or not aligned with the 64-column jobs
// (another multiple of 8, e.g. 24, 48, 96).
//
// For every alpha k, row r and group g the quantizer needs the extremes of
// t = fl32(w * s_k) over the group ("AWQ vs GPTQ ...", group_params;
// "GPTQ and AWQ weight quantisation", rtn_nbit): max|t| for the symmetric
// quantizer, min(min t, 0) and max(max t, 0) for the asymmetric one.  When a
// group spans several of the search kernel's 128-column jobs, no producer
// sees the whole group, so this pass forms the extremes first and the
// search reads them.
//
// ext is zeroed by the caller.  Every value folded in is non-negative (max|t|,
// -min(t, 0), max(t, 0)), so the bit patterns order like the values and
// atomicMax on them gives the exact maximum whatever the order of the CTAs.
#include <algorithm>

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

constexpr int kExtRows = 4;     // rows per warp task
constexpr int kExtAlphas = 4;   // alphas per inner step
constexpr int kExtChunk = 256;  // columns per warp task (8 per lane)

__device__ __forceinline__ void fold_max(float* p, float v) {
  atomicMax(reinterpret_cast<unsigned int*>(p), __float_as_uint(v) & 0x7FFFFFFFu);
}

// Warp task (row block rb, 256-column chunk ch).  Each lane's 8 columns lie
// in one group (the group is a multiple of 8).  Each lane keeps its 8
// weights of kExtRows rows in registers and runs through the alphas
// kExtAlphas at a time; per (row, alpha) the partial extremes of the lanes
// of one group are combined (a max over the lanes with the same group, on
// the bit patterns of the non-negative values) and the group's first lane
// folds them into ext.
template <typename WT, bool SYM>
__global__ void __launch_bounds__(256) group_extremes_kernel(const WT* __restrict__ W, int64_t out,
                                                             int64_t in, const float* __restrict__ s32,
                                                             int n_alpha, int64_t group,
                                                             float* __restrict__ ext) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t nchunk = (in + kExtChunk - 1) / kExtChunk;
  const int64_t ntask = (out + kExtRows - 1) / kExtRows * nchunk;
  const int64_t ngroups = in / group;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t task = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); task < ntask;
       task += wstride) {
    const int64_t rb = task / nchunk, ch = task % nchunk;
    const int64_t c0 = ch * kExtChunk + lane * 8;
    const bool live = c0 < in;  // in % 8 == 0, so all 8 columns are live
    // lanes past the last column join the last lane's group with zeros
    const int64_t g = (live ? c0 : in - 8) / group;
    const unsigned same = __match_any_sync(0xffffffffu, (unsigned long long)g);
    const bool leader = (int)(__ffs(same) - 1) == lane;
    float w[kExtRows][8];
#pragma unroll
    for (int r = 0; r < kExtRows; ++r) {
      const int64_t row = rb * kExtRows + r;
      if (live && row < out) {
        load8_f32<WT>(W + row * in + c0, w[r]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) w[r][e] = 0.0f;
      }
    }
    for (int k0 = 0; k0 < n_alpha; k0 += kExtAlphas) {
      float sv[kExtAlphas][8];
#pragma unroll
      for (int a = 0; a < kExtAlphas; ++a) {
        if (live && k0 + a < n_alpha) {
          load8_f32<float>(s32 + (int64_t)(k0 + a) * in + c0, sv[a]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) sv[a][e] = 0.0f;
        }
      }
      float hi[kExtRows][kExtAlphas], nlo[kExtRows][kExtAlphas];
#pragma unroll
      for (int r = 0; r < kExtRows; ++r)
#pragma unroll
        for (int a = 0; a < kExtAlphas; ++a) {
          float h = 0.0f, l = 0.0f;
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const float2 t =
                __fmul2_rn(make_float2(w[r][e], w[r][e + 1]), make_float2(sv[a][e], sv[a][e + 1]));
            if (SYM) {
              h = fmax3f(h, fabsf(t.x), fabsf(t.y));
            } else {
              h = fmax3f(h, t.x, t.y);
              l = fmin3f(l, t.x, t.y);
            }
          }
          hi[r][a] = h;
          nlo[r][a] = -l;
        }
      // (hi and nlo are >= 0 or -0 and never NaN: the running max ignores
      // NaN and starts at 0; with the sign bit cleared the bit patterns order
      // like the values)
#pragma unroll
      for (int r = 0; r < kExtRows; ++r)
#pragma unroll
        for (int a = 0; a < kExtAlphas; ++a) {
          hi[r][a] = __uint_as_float(
              __reduce_max_sync(same, __float_as_uint(hi[r][a]) & 0x7FFFFFFFu));
          if (!SYM)
            nlo[r][a] = __uint_as_float(
                __reduce_max_sync(same, __float_as_uint(nlo[r][a]) & 0x7FFFFFFFu));
        }
      if (leader) {
#pragma unroll
        for (int r = 0; r < kExtRows; ++r)
#pragma unroll
          for (int a = 0; a < kExtAlphas; ++a) {
            const int64_t row = rb * kExtRows + r;
            if (row >= out || k0 + a >= n_alpha) continue;
            const int64_t idx = ((int64_t)(k0 + a) * out + row) * ngroups + g;
            if (SYM) {
              fold_max(ext + idx, hi[r][a]);
            } else {
              fold_max(ext + 2 * idx, nlo[r][a]);
              fold_max(ext + 2 * idx + 1, hi[r][a]);
            }
          }
      }
    }
  }
}

template <typename WT>
cudaError_t launch_ext(const void* W, int64_t out, int64_t in, const float* s32, int n_alpha,
                       int64_t group, int sym, float* ext, cudaStream_t s) {
  const int64_t ntask = (out + kExtRows - 1) / kExtRows * ((in + kExtChunk - 1) / kExtChunk);
  const int64_t blocks = std::min<int64_t>((ntask + 7) / 8, (int64_t)device_sm_count() * 8);
  const unsigned grid = (unsigned)std::max<int64_t>(1, blocks);
  if (sym)
    return launch_pdl(group_extremes_kernel<WT, true>, grid, 256, 0, s, static_cast<const WT*>(W),
                      out, in, s32, n_alpha, group, ext);
  return launch_pdl(group_extremes_kernel<WT, false>, grid, 256, 0, s, static_cast<const WT*>(W),
                    out, in, s32, n_alpha, group, ext);
}

}  // namespace

cudaError_t launch_group_extremes(const void* W, int dt, int64_t out, int64_t in,
                                  const float* s32, int n_alpha, int64_t group, int sym,
                                  float* ext, cudaStream_t s) {
  if (in % 8 != 0 || group < 8 || in % group != 0 || (group % 8 != 0 && group != in))
    return cudaErrorInvalidValue;
  switch (dt) {
    case kDtF32: return launch_ext<float>(W, out, in, s32, n_alpha, group, sym, ext, s);
    case kDtF16: return launch_ext<__half>(W, out, in, s32, n_alpha, group, sym, ext, s);
    default: return launch_ext<__nv_bfloat16>(W, out, in, s32, n_alpha, group, sym, ext, s);
  }
}

}  // namespace awq
