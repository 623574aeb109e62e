// Host-side interfaces between the C ABI (awq_api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace awq {

constexpr int kDtF32 = 0, kDtF16 = 1, kDtBF16 = 2;

inline size_t dtype_size(int dt) { return dt == kDtF32 ? 4 : 2; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Number of SMs of the current device (cached per device).
int device_sm_count();

// ---- statistics and conversions (awq_stats.cu)
// sx[j] = sum_n |X[n, j]| / N + 1e-8, float64.  With xmax != nullptr the same
// pass folds max|X| into *xmax (the bits of a non-negative float; *xmax must
// start at 0; needs in % 8 == 0 and X 16-byte aligned).
cudaError_t launch_channel_stats(const void* X, int dt, int64_t N, int64_t in, double* sx,
                                 uint32_t* xmax, cudaStream_t s);
// *out = max(*out, bits of max_i |p[i]|); *out must start at 0.
cudaError_t launch_absmax(const void* p, int dt, int64_t n, uint32_t* out, cudaStream_t s);
// dst = fp16(X * 2^m) with m = pow2_exponent_for(max|X|) read from *xmax_bits;
// n elements, n % 8 == 0, 16-byte aligned.  dt is AWQ_F32 or AWQ_BF16.
cudaError_t launch_to_f16(const void* X, int dt, int64_t n, const uint32_t* xmax_bits, void* dst,
                          cudaStream_t s);

// ---- alpha tables, reduction and argmin (awq_prep.cu)
// For k = 0..grid: s = sx^alpha_k / sqrt(max * min), written as float32
// s32[k][j], and inv_s32[k][j] = 2^e_k / s32[k][j] where 2^e_k scales the
// weight changes of alpha k into the fp16 range of the error GEMM
// (absmax[0] = max|W| bits).  unscale[k] = 2^-2(e_k + m_x) undoes both
// operand scalings on the squared sums (absmax[1] = max|X| bits; m_x = 0
// when x_scaled == 0).  pow2_s[k] ends nonzero iff every s32[k][j] is a
// power of two.  root ([in] doubles) holds sx^(1/grid), minmax
// (prep_chunks(in) pairs) the per-chunk max and min of sx, inv_c and escale
// ([grid + 1] each) the centring factors and 2^e_k.
size_t prep_chunks(int64_t in);
cudaError_t launch_alpha_prep(const double* sx, int64_t in, int grid, const uint32_t* absmax,
                              int x_scaled, double* root, double* minmax, double* inv_c,
                              float* escale, float* s32, float* inv_s32, double* unscale,
                              int32_t* pow2_s, cudaStream_t s);
// err[k] = unscale[k] * sum_t partials[k][t] / denom (fixed order),
// best = strict-< argmin, s_best = s32[best].
cudaError_t launch_reduce_argmin(const double* partials, const double* unscale, int n_alpha,
                                 int n_tiles, double denom, const float* s32, int64_t in,
                                 double* err, int32_t* best, float* s_best, int32_t* dev_status,
                                 cudaStream_t s);

// ---- the fused search (awq_search.cu)
struct SearchPlan {
  int T;        // token tile (multiple of 32, <= 256) = MMA N
  int n_tt;     // token tiles
  int a_per;    // alphas per work unit (accumulators in tensor memory)
  int n_ag;     // alpha groups
  int n_rt;     // 128-row tiles
  int n_kb;     // 64-column K blocks
  int n_units;  // n_rt * n_ag * n_tt
  int n_tiles;  // partial sums per alpha = n_rt * n_tt
  int sw, sx;   // W and X ring depths
  size_t w_stage;  // bytes of one W ring stage (W tile + the alphas' scale-table columns)
  size_t smem;  // dynamic shared memory bytes
  int grid;     // persistent CTAs
};
bool search_supported(int dt, int64_t out, int64_t in, int64_t N, int bits, int group, int grid);
SearchPlan plan_search(int dt, int64_t out, int64_t in, int64_t N, int n_alpha, int group,
                       int sms);
cudaError_t launch_search(const void* W, const void* Xf16, int dt, int64_t out, int64_t in,
                          int64_t N, int bits, int group, int sym, int n_alpha,
                          const float* s32, const float* inv_s32, const int32_t* pow2_s,
                          double* partials, const SearchPlan& plan, int64_t wait_limit_ns,
                          int test_timeout, int32_t* dev_status, uint32_t* diag, cudaStream_t s,
                          cudaEvent_t ev0, cudaEvent_t ev1);

// ---- final quantization and packing (awq_pack.cu)
cudaError_t launch_quantize_pack(const void* W, int dt, int64_t out, int64_t in, const float* s,
                                 int bits, int group, int sym, uint32_t* qweight, float* scales,
                                 uint8_t* zeros, int32_t* dev_status, cudaStream_t st);

}  // namespace awq
