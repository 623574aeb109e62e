// Per-group clipping search at fixed scales ("AWQ (activation-aware weight
// quantization)", "Simplifications": the method "also searches a clipping
// threshold per group, shrinking the max range"; "AWQ vs GPTQ ...", "AWQ:
// move the error away from what matters": the second search "shrinks each
// group's clipping range a little when that lowers output error").
//
// For each row r and group G of W * diag(s) and each shrink factor c of the
// group's range, the group's own share of the row's output error is
//   e(r, G, c) = sum_n (sum_{j in G} X[n, j] d_c[j])^2 = d_c^T H_G d_c,
//   d_c = Q_c(W * s)[r, G] / s - W[r, G],   H_G = X_G^T X_G,
// so one Gram matrix per group (g x g, formed once from X) replaces the N
// token products of every (row, factor).  The kept factor is the first with
// the smallest share (strict <).
//
// gram_kernel: CTA (group, token split) accumulates its tokens' X_G^T X_G in
// fp32, 8 x 8 outputs per thread; the splits are added in a fixed order by
// the next kernel, so the result does not depend on scheduling.
// clip_kernel: CTA (group, row block) stages H_G in shared memory (each lane's
// columns contiguous), one warp per row: the warp forms d_c for every factor
// (each lane holds g/32 columns, codes by true division with the quantizer's
// clamps, d = w_hat * (1/s) - w), writes them to shared memory, and
// accumulates H_G d_c over k with one 16-byte load of H and one per four
// factors' d per step (fp32 FMA-bound), then reduces d_c . (H_G d_c) across
// the warp.
#include <algorithm>

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

constexpr int kClipWarps = 8;
constexpr int kGramTok = 32;  // tokens staged per step of gram_kernel

template <typename T, int G>
__global__ void __launch_bounds__((G / 8) * (G / 8)) gram_kernel(const T* __restrict__ X, int64_t N,
                                                                int64_t in, int nsplit,
                                                                float* __restrict__ H) {
  pdl_wait();
  pdl_trigger();
  constexpr int TB = G / 8;  // thread blocks of 8 x 8 outputs per side
  __shared__ float xs[kGramTok][G + 4];
  const int g = blockIdx.x, sp = blockIdx.y;
  const int ti = threadIdx.x / TB, tj = threadIdx.x % TB;
  const int64_t per = (N + nsplit - 1) / nsplit;
  const int64_t n0 = (int64_t)sp * per, n1 = min(N, n0 + per);
  float acc[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.0f;
  for (int64_t nb = n0; nb < n1; nb += kGramTok) {
    __syncthreads();
    for (int i = threadIdx.x; i < kGramTok * G; i += blockDim.x) {
      const int r = i / G, c = i % G;
      const int64_t n = nb + r;
      xs[r][c] = n < n1 ? Elt<T>::to_f32(X[n * in + (int64_t)g * G + c]) : 0.0f;
    }
    __syncthreads();
    for (int r = 0; r < kGramTok; ++r) {
      float u[8], v[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) {
        u[a] = xs[r][ti * 8 + a];
        v[a] = xs[r][tj * 8 + a];
      }
#pragma unroll
      for (int a = 0; a < 8; ++a)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(u[a], v[b], acc[a][b]);
    }
  }
  float* Hg = H + ((int64_t)sp * (in / G) + g) * G * G;
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) Hg[(ti * 8 + a) * G + tj * 8 + b] = acc[a][b];
}

template <typename T, int G, bool SYM, int NCQ>
__global__ void __launch_bounds__(kClipWarps * 32) clip_kernel(
    const T* __restrict__ W, const float* __restrict__ s, const float* __restrict__ H, int nsplit,
    int64_t out, int64_t in, float Lf, float maxqf, int nc, ClipFactors cf,
    float* __restrict__ clip, float* __restrict__ errs, int32_t* dev_status) {
  pdl_wait();
  pdl_trigger();
  constexpr int CPL = G / 32;  // columns per lane: j = lane + 32 i
  constexpr int NCP = 4 * NCQ;  // factors carried through the quadratic forms (>= nc)
  extern __shared__ float4 csm[];
  // Hs[k][lane] holds H[k][lane + 32 i], i < CPL (a float4 slot each)
  float4* Hs = csm;
  float* dsm = reinterpret_cast<float*>(csm + G * 32);  // [warp][k][kMaxClip]
  const int g = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t ng = in / G;
  for (int i = threadIdx.x; i < G * 32; i += blockDim.x) {
    const int k = i / 32, l = i % 32;
    float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int sp = 0; sp < nsplit; ++sp) {  // the token splits in a fixed order
      const float* Hg = H + ((int64_t)sp * ng + g) * G * G + (int64_t)k * G;
#pragma unroll
      for (int c = 0; c < CPL; ++c) v[c] += Hg[l + 32 * c];
    }
    Hs[i] = make_float4(v[0], v[1], v[2], v[3]);
  }
  for (int i = threadIdx.x; i < kClipWarps * G * kMaxClip; i += blockDim.x) dsm[i] = 0.0f;
  __syncthreads();
  float* dw = dsm + (size_t)warp * G * kMaxClip;
  float sv[CPL], inv_s[CPL];  // the group's scales are the same for every row
#pragma unroll
  for (int i = 0; i < CPL; ++i) {
    sv[i] = s[(int64_t)g * G + lane + 32 * i];
    inv_s[i] = 1.0f / sv[i];
  }
  for (int64_t row = (int64_t)blockIdx.y * kClipWarps + warp; row < out;
       row += (int64_t)gridDim.y * kClipWarps) {
    float w[CPL], t[CPL];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int64_t j = (int64_t)g * G + lane + 32 * i;
      w[i] = Elt<T>::to_f32(W[row * in + j]);
      t[i] = __fmul_rn(w[i], sv[i]);
    }
    float r0 = 0.0f, r1 = 0.0f;  // sym: max|t|; asym: min(min t, 0), max(max t, 0)
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      if (SYM) {
        r0 = fmaxf(r0, fabsf(t[i]));
      } else {
        r0 = fminf(r0, t[i]);
        r1 = fmaxf(r1, t[i]);
      }
    }
    for (int o = 16; o > 0; o >>= 1) {
      if (SYM) {
        r0 = fmaxf(r0, __shfl_xor_sync(0xffffffffu, r0, o));
      } else {
        r0 = fminf(r0, __shfl_xor_sync(0xffffffffu, r0, o));
        r1 = fmaxf(r1, __shfl_xor_sync(0xffffffffu, r1, o));
      }
    }
    if (!(fabsf(r0) <= 3.402823466e38f) || !(fabsf(r1) <= 3.402823466e38f)) {
      if (lane == 0) set_status(dev_status, ST_NONFINITE);
    }
    // d_c for every factor, into this warp's shared buffer [k][c]
    for (int c = 0; c < nc; ++c) {
      const float f = cf.c[c];
      float scale, zero;
      if (SYM) {
        scale = fmaxf(__fdiv_rn(__fmul_rn(f, r0), Lf), 1e-8f);
        zero = 0.0f;
      } else {
        const float lo = __fmul_rn(f, r0), hi = __fmul_rn(f, r1);
        scale = fmaxf(__fdiv_rn(__fsub_rn(hi, lo), maxqf), 1e-8f);
        zero = rintf(__fdiv_rn(-lo, scale));
      }
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        float q = rintf(__fdiv_rn(t[i], scale));
        float what;
        if (SYM) {
          q = fminf(fmaxf(q, -Lf - 1.0f), Lf);
          what = __fmul_rn(q, scale);
        } else {
          q = fminf(fmaxf(__fadd_rn(q, zero), 0.0f), maxqf);
          what = __fmul_rn(scale, __fsub_rn(q, zero));
        }
        dw[(lane + 32 * i) * kMaxClip + c] = fmaf(what, inv_s[i], -w[i]);
      }
    }
    __syncwarp();
    // v_c = H_G d_c for this lane's columns
    float v[NCP][CPL];
#pragma unroll
    for (int c = 0; c < NCP; ++c)
#pragma unroll
      for (int i = 0; i < CPL; ++i) v[c][i] = 0.0f;
    for (int k = 0; k < G; ++k) {
      const float4 h = Hs[k * 32 + lane];
      const float hv[4] = {h.x, h.y, h.z, h.w};
      const float4* dk = reinterpret_cast<const float4*>(dw + k * kMaxClip);
      float dv[NCP];
#pragma unroll
      for (int q = 0; q < NCQ; ++q) {
        const float4 x = dk[q];
        dv[4 * q] = x.x;
        dv[4 * q + 1] = x.y;
        dv[4 * q + 2] = x.z;
        dv[4 * q + 3] = x.w;
      }
#pragma unroll
      for (int c = 0; c < NCP; ++c)
#pragma unroll
        for (int i = 0; i < CPL; ++i) v[c][i] = fmaf(hv[i], dv[c], v[c][i]);
    }
    // e_c = d_c . v_c across the warp; lane 0 keeps the first smallest
    float best_e = INFINITY;
    int best = 0;
#pragma unroll
    for (int c = 0; c < NCP; ++c) {
      if (c >= nc) break;
      float e = 0.0f;
#pragma unroll
      for (int i = 0; i < CPL; ++i) e = fmaf(dw[(lane + 32 * i) * kMaxClip + c], v[c][i], e);
      for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
      if (e < best_e) {
        best_e = e;
        best = c;
      }
      if (lane == 0 && errs != nullptr) errs[(row * ng + g) * nc + c] = e;
    }
    if (lane == 0) clip[row * ng + g] = cf.c[best];
    __syncwarp();  // the buffer is rewritten for the next row
  }
}

template <typename T, int G>
cudaError_t launch_clip_g(const void* W, const void* X, int64_t out, int64_t in, int64_t N,
                          const float* s, int bits, int sym, int nc, const ClipFactors& cf,
                          float* H, int nsplit, float* clip, float* errs, int32_t* st,
                          cudaStream_t stream) {
  const int64_t ng = in / G;
  cudaError_t e = launch_pdl(gram_kernel<T, G>, dim3((unsigned)ng, (unsigned)nsplit),
                             dim3((G / 8) * (G / 8)), 0, stream, static_cast<const T*>(X), N, in,
                             nsplit, H);
  if (e != cudaSuccess) return e;
  const size_t smem = (size_t)G * 32 * sizeof(float4) + (size_t)kClipWarps * G * kMaxClip * 4;
  using Kern = void (*)(const T*, const float*, const float*, int, int64_t, int64_t, float, float,
                        int, ClipFactors, float*, float*, int32_t*);
  const Kern table[2][3] = {{clip_kernel<T, G, false, 1>, clip_kernel<T, G, false, 2>,
                             clip_kernel<T, G, false, 3>},
                            {clip_kernel<T, G, true, 1>, clip_kernel<T, G, true, 2>,
                             clip_kernel<T, G, true, 3>}};
  static_assert(kMaxClip == 12, "three groups of four factors");
  const Kern kern = table[sym ? 1 : 0][(nc + 3) / 4 - 1];
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int64_t rb = (out + kClipWarps - 1) / kClipWarps;
  const int64_t per_group = std::max<int64_t>(1, (int64_t)device_sm_count() * 2 / ng);
  const unsigned gy = (unsigned)std::min<int64_t>(std::min<int64_t>(rb, per_group), 65535);
  const float Lf = (float)((1 << (bits - 1)) - 1), maxqf = (float)((1 << bits) - 1);
  return launch_pdl(kern, dim3((unsigned)ng, gy), dim3(kClipWarps * 32), smem, stream,
                    static_cast<const T*>(W), s, H, nsplit, out, in, Lf, maxqf, nc, cf, clip, errs,
                    st);
}

template <typename T>
cudaError_t launch_clip_t(const void* W, const void* X, int64_t out, int64_t in, int64_t N,
                          const float* s, int bits, int group, int sym, int nc,
                          const ClipFactors& cf, float* H, int nsplit, float* clip, float* errs,
                          int32_t* st, cudaStream_t stream) {
  switch (group) {
    case 32:
      return launch_clip_g<T, 32>(W, X, out, in, N, s, bits, sym, nc, cf, H, nsplit, clip, errs,
                                  st, stream);
    case 64:
      return launch_clip_g<T, 64>(W, X, out, in, N, s, bits, sym, nc, cf, H, nsplit, clip, errs,
                                  st, stream);
    default:
      return launch_clip_g<T, 128>(W, X, out, in, N, s, bits, sym, nc, cf, H, nsplit, clip, errs,
                                   st, stream);
  }
}

}  // namespace

int clip_splits(int64_t N) { return (int)std::min<int64_t>(8, std::max<int64_t>(1, (N + 255) / 256)); }

cudaError_t launch_clip_search(const void* W, const void* X, int dt, int64_t out, int64_t in,
                               int64_t N, const float* s, int bits, int group, int sym, int nc,
                               const ClipFactors& cf, float* H, float* clip, float* errs,
                               int32_t* dev_status, cudaStream_t stream) {
  if (group != 32 && group != 64 && group != 128) return cudaErrorInvalidValue;
  if (nc < 1 || nc > kMaxClip || in % group != 0) return cudaErrorInvalidValue;
  const int nsplit = clip_splits(N);
  switch (dt) {
    case kDtF32:
      return launch_clip_t<float>(W, X, out, in, N, s, bits, group, sym, nc, cf, H, nsplit, clip,
                                  errs, dev_status, stream);
    case kDtF16:
      return launch_clip_t<__half>(W, X, out, in, N, s, bits, group, sym, nc, cf, H, nsplit, clip,
                                   errs, dev_status, stream);
    default:
      return launch_clip_t<__nv_bfloat16>(W, X, out, in, N, s, bits, group, sym, nc, cf, H,
                                          nsplit, clip, errs, dev_status, stream);
  }
}

}  // namespace awq
