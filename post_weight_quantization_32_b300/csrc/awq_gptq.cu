// GPTQ's rounding of W * diag(s) against the inputs X / s: AWQ's scaling
// first, then GPTQ's choice of integers ("AWQ vs GPTQ Quantization
// Architectures Compared", "GPTQ: compensate the error you just made" and
// "Failure modes and combining the two").
//
//   H  = 2 Xs^T Xs + damp * mean(diag) * I,   Xs = X / s
//   U  = upper Cholesky factor of H^-1 (U^T U = H^-1)
//   for each column i (natural order): at a group's first column fit the
//   group's step and zero on the corrected weights; round column i with the
//   float32 quantizer; err = (w - w_hat) / U[i][i]; w[:, j>i] -= err U[i][j]
//
// Everything runs in fp32 (the GEMMs in cuBLAS, float32 emulated on the
// tensor cores; the rest on the CUDA cores), in this order:
//  1. Xr = X / s with its columns reversed (Xr = Xs J, J the exchange matrix).
//  2. A = 2 Xr^T Xr = J H J (a GEMM), dampened on its diagonal.
//  3. A = M M^T, M lower (blocked right-looking Cholesky: a one-CTA factor of
//     each 32 x 32 diagonal block, a row-parallel triangular solve for the
//     panel below it, a GEMM for the trailing matrix).
//  4. Y = M^-1 (blocked: the inverse of each diagonal block in one CTA, then
//     Y[i, :i] = -Y[i, i] (M[i, :i] Y[:i, :i]) by two GEMMs).
//  5. U = J Y J: with H = J M M^T J = R R^T, R = J M J upper, H^-1 = R^-T R^-1,
//     so U = R^-1 = J M^-1 J (upper, positive diagonal: the Cholesky factor).
//  6. The sweep in blocks of 128 columns: one thread per row runs the block's
//     columns in order with the block's rows of U and the row's block of
//     weights in shared memory, writing codes and the scaled errors; a GEMM
//     then applies the block's errors to all later columns.
//  7. The codes are packed as awq_quantize_pack packs them.
#include <algorithm>
#include <mutex>

#include <cublas_v2.h>

#include "awq_device.cuh"
#include "awq_internal.h"

namespace awq {

namespace {

// ---------------------------------------------------------------- fp32 GEMM
// C[m][n] = alpha * sum_k A(m, k) B(k, n) + beta * C[m][n] (row-major); A(m,
// k) is A[m * lda + k] (or A[k * lda + m] when ta), B(k, n) is B[k * ldb + n]
// (or B[n * ldb + k] when tb).  These are plain GEMMs, so they go to cuBLAS
// with its float32 result emulated on the bf16 tensor cores (each float32
// operand split into three bf16 parts, products accumulated in float32):
// float32 accuracy at tensor-core speed.  cuBLAS is column-major: the
// row-major product is computed as C^T = B^T A^T.
}  // namespace

namespace {
std::mutex g_blas_mu;
cublasHandle_t g_blas[64] = {nullptr};

cublasHandle_t blas_handle() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_blas_mu);
  if (g_blas[dev] == nullptr) {
    cublasHandle_t h = nullptr;
    if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return nullptr;
    g_blas[dev] = h;
  }
  return g_blas[dev];
}
}  // namespace

cudaError_t blas_gemm(cudaStream_t s, int m, int n, int k, float alpha, const void* A, int64_t lda,
                      int ta, const void* B, int64_t ldb, int tb, float beta, float* C, int64_t ldc,
                      int dt) {
  if (m <= 0 || n <= 0 || k <= 0) return cudaSuccess;
  cublasHandle_t h = blas_handle();
  if (h == nullptr || cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  const cudaDataType_t t = dt == kDtF16 ? CUDA_R_16F : (dt == kDtBF16 ? CUDA_R_16BF : CUDA_R_32F);
  // 16-bit operands: their products are exact in float32 and accumulate in
  // float32; float32 operands: float32 emulated on the bf16 tensor cores
  const cublasComputeType_t ct =
      dt == kDtF32 ? CUBLAS_COMPUTE_32F_EMULATED_16BFX9 : CUBLAS_COMPUTE_32F;
  const cublasStatus_t r =
      cublasGemmEx(h, tb ? CUBLAS_OP_T : CUBLAS_OP_N, ta ? CUBLAS_OP_T : CUBLAS_OP_N, n, m, k,
                   &alpha, B, t, (int)ldb, A, t, (int)lda, &beta, C, CUDA_R_32F, (int)ldc, ct,
                   CUBLAS_GEMM_DEFAULT);
  return r == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

namespace {


cudaError_t sgemm(cudaStream_t s, int m, int n, int k, float alpha, const float* A, int64_t lda,
                  int ta, const float* B, int64_t ldb, int tb, float beta, float* C, int64_t ldc) {
  return blas_gemm(s, m, n, k, alpha, A, lda, ta, B, ldb, tb, beta, C, ldc, kDtF32);
}

// batch row-major products C_i = alpha A_i B_i + beta C_i (no transposes),
// operand i at A + i * sa, B + i * sb, C + i * sc; float32 emulated as above
cudaError_t sgemm_batched(cudaStream_t s, int m, int n, int k, float alpha, const float* A,
                          int64_t lda, int64_t sa, const float* B, int64_t ldb, int64_t sb,
                          float beta, float* C, int64_t ldc, int64_t sc, int batch) {
  if (m <= 0 || n <= 0 || k <= 0 || batch <= 0) return cudaSuccess;
  cublasHandle_t h = blas_handle();
  if (h == nullptr || cublasSetStream(h, s) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  const cublasStatus_t r = cublasGemmStridedBatchedEx(
      h, CUBLAS_OP_N, CUBLAS_OP_N, n, m, k, &alpha, B, CUDA_R_32F, (int)ldb, sb, A, CUDA_R_32F,
      (int)lda, sa, &beta, C, CUDA_R_32F, (int)ldc, sc, batch, CUBLAS_COMPUTE_32F_EMULATED_16BFX9,
      CUBLAS_GEMM_DEFAULT);
  return r == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

// ------------------------------------------------------- inputs and Hessian
// Xr[t][j] = X[t][in - 1 - j] / s[in - 1 - j] (fp32)
template <typename T>
__global__ void __launch_bounds__(256) scale_reverse_kernel(const T* __restrict__ X, int64_t N,
                                                            int64_t in, const float* __restrict__ s,
                                                            float* __restrict__ Xr) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = N * in;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / in, j = i % in, src = in - 1 - j;
    const float sv = s != nullptr ? s[src] : 1.0f;
    Xr[i] = Elt<T>::to_f32(X[t * in + src]) / sv;
  }
}

// A[i][i] += damp * mean(diag A); one CTA
__global__ void __launch_bounds__(1024) damp_kernel(float* __restrict__ A, int64_t n, float damp) {
  pdl_wait();
  pdl_trigger();
  __shared__ double part[32];
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) acc += (double)A[i * n + i];
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += part[w];
    part[0] = t;
  }
  __syncthreads();
  const float add = damp * (float)(part[0] / (double)n);
  __syncthreads();
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) A[i * n + i] += add;
}

// ------------------------------------------------------- blocked Cholesky
constexpr int kCB = 64;  // Cholesky / inverse block
constexpr int kDiagThreads = 1024;
constexpr int kDiagPer = kCB * kCB / kDiagThreads;  // entries of the diagonal block per thread

// Factor the diagonal block A[k0:k0+b, k0:k0+b] = L L^T in place (lower).
// A non-positive pivot sets the status (the matrix is not positive definite).
// Right-looking, one thread per entry: at step j the pivot is taken, column
// j is divided by it and the trailing lower triangle loses L[r][j] L[c][j].
// Every entry sees the same subtractions in the same order (t = 0, 1, ...)
// as a column-by-column (left-looking) factorisation.
__global__ void __launch_bounds__(kDiagThreads) chol_diag_kernel(float* __restrict__ A, int64_t n,
                                                                 int64_t k0, int b,
                                                                 int32_t* dev_status) {
  pdl_wait();
  pdl_trigger();
  __shared__ float L[kCB][kCB + 1];
  // thread t holds entries t, t + kDiagThreads, ... of the block (row-major)
  int r[kDiagPer], c[kDiagPer];
#pragma unroll
  for (int e = 0; e < kDiagPer; ++e) {
    const int idx = (int)threadIdx.x + kDiagThreads * e;
    r[e] = idx / kCB;
    c[e] = idx % kCB;
    if (r[e] < b && c[e] < b) L[r[e]][c[e]] = A[(k0 + r[e]) * n + k0 + c[e]];
  }
  __syncthreads();
  for (int j = 0; j < b; ++j) {
    if (threadIdx.x == 0) {
      float d = L[j][j];
      if (!(d > 0.0f)) {
        set_status(dev_status, ST_NONFINITE);
        d = 1e-30f;
      }
      L[j][j] = sqrtf(d);
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kDiagPer; ++e)
      if (c[e] == j && r[e] > j && r[e] < b) L[r[e]][j] = L[r[e]][j] / L[j][j];
    __syncthreads();
#pragma unroll
    for (int e = 0; e < kDiagPer; ++e)
      if (c[e] > j && r[e] >= c[e] && r[e] < b) L[r[e]][c[e]] -= L[r[e]][j] * L[c[e]][j];
    __syncthreads();
  }
#pragma unroll
  for (int e = 0; e < kDiagPer; ++e)
    if (r[e] < b && c[e] < b) A[(k0 + r[e]) * n + k0 + c[e]] = c[e] <= r[e] ? L[r[e]][c[e]] : 0.0f;
}

// Rows i >= k0 + b: solve x L11^T = A[i, k0:k0+b] (one thread per row).
__global__ void __launch_bounds__(128) chol_panel_kernel(float* __restrict__ A, int64_t n,
                                                        int64_t k0, int b) {
  pdl_wait();
  pdl_trigger();
  __shared__ float L[kCB][kCB + 1];
  {  // thread t loads column t % kCB of rows t / kCB, t / kCB + 2, ...: all loads in flight
    const int c = (int)threadIdx.x % kCB, r0 = (int)threadIdx.x / kCB;
#pragma unroll
    for (int k = 0; k < kCB / 2; ++k) {
      const int r = r0 + 2 * k;
      if (r < b && c < b) L[r][c] = A[(k0 + r) * n + k0 + c];
    }
  }
  __syncthreads();
  const int64_t row = k0 + b + blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (row >= n) return;
  float x[kCB];
  float* a = A + row * n + k0;
#pragma unroll
  for (int j = 0; j < kCB; ++j) {
    if (j < b) {
      float v = a[j];
#pragma unroll
      for (int t = 0; t < j; ++t) v -= x[t] * L[j][t];  // both loops unrolled: x stays in registers
      x[j] = v / L[j][j];
      a[j] = x[j];
    }
  }
}

// ------------------------------------------------- blocked lower inverse
// Y[i0:i0+b, i0:i0+b] = inverse of the lower block M[i0:i0+b, i0:i0+b],
// i0 = blockIdx.x * kCB (every diagonal block in one launch: each needs only
// its own block of M): thread c solves M y = e_c by forward substitution.
__global__ void __launch_bounds__(kCB) tri_inv_diag_kernel(const float* __restrict__ M,
                                                           float* __restrict__ Y, int64_t n) {
  pdl_wait();
  pdl_trigger();
  const int64_t i0 = (int64_t)blockIdx.x * kCB;
  const int b = (int)min((int64_t)kCB, n - i0);
  __shared__ float L[kCB][kCB + 1];
#pragma unroll
  for (int r = 0; r < kCB; ++r)  // thread c loads column c: all loads in flight
    if (r < b && (int)threadIdx.x < b) L[r][threadIdx.x] = M[(i0 + r) * n + i0 + threadIdx.x];
  __syncthreads();
  const int c = threadIdx.x;
  if (c >= b) return;
  float y[kCB];
#pragma unroll
  for (int r = 0; r < kCB; ++r) {
    if (r < b) {
      float v = r == c ? 1.0f : 0.0f;
#pragma unroll
      for (int t = 0; t < r; ++t) v -= L[r][t] * y[t];  // both loops unrolled: y stays in registers
      y[r] = v / L[r][r];
      Y[(i0 + r) * n + i0 + c] = y[r];
    }
  }
}

// U[r][c] = Y[n-1-r][n-1-c]
__global__ void __launch_bounds__(256) reverse_kernel(const float* __restrict__ Y,
                                                      float* __restrict__ U, int64_t n) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = n * n;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / n, c = i % n;
    U[i] = Y[(n - 1 - r) * n + (n - 1 - c)];
  }
}

// Ws = W * s (fp32 working copy)
template <typename T>
__global__ void __launch_bounds__(256) scale_weights_kernel(const T* __restrict__ W, int64_t out,
                                                            int64_t in, const float* __restrict__ s,
                                                            float* __restrict__ Ws) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = out * in;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float w = Elt<T>::to_f32(W[i]);
    Ws[i] = s != nullptr ? __fmul_rn(w, s[i % in]) : w;
  }
}

// ------------------------------------------------------------ the sweep
constexpr int kSB = 128;                  // columns per sweep block
constexpr int kSLanes = 8;                // threads per row
constexpr int kSOwn = kSB / kSLanes;      // columns a thread holds (16)
constexpr int kSRows = 32;                // rows per CTA (256 threads)

// Eight threads per row run columns b0 .. b0+bw-1 in order; thread q of a
// row holds columns q, q + 8, q + 16, ... of the block in registers.  For
// column i every thread of the row takes the column's current value from
// its holder (a shuffle) and forms the same code and scaled error, and
// each thread takes that error off the columns it holds beyond i (the
// updates of a column arrive in column order, as in a one-thread sweep).
// At a group's first column the group is fitted on the corrected weights
// (extremes over the row's eight threads).  Codes and errors are staged in
// shared memory and stored row by row.  Shared memory: U[b0:b0+bw,
// b0:b0+bw], then the codes [32][128] and errors [32][128] of the CTA.
// Writes the storage codes, the group steps and zero points, and
// Err[row][i - b0] = (w - w_hat) / U[i][i].
__global__ void __launch_bounds__(kSRows * kSLanes, 2) sweep_block_kernel(
    float* __restrict__ Ws, const float* __restrict__ U, int64_t out, int64_t in, int64_t b0,
    int bw, int group, int bits, int sym, uint8_t* __restrict__ codes, float* __restrict__ scales,
    uint8_t* __restrict__ zeros, float* __restrict__ Err) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float sm[];
  float* Ub = sm;                                                    // [kSB][kSB]
  float* est = sm + kSB * kSB;                                       // [kSRows][kSB]
  uint8_t* cst = reinterpret_cast<uint8_t*>(est + kSRows * kSB);     // [kSRows][kSB]
  {  // thread t loads columns 4 (t % 32) .. + 3 of rows t / 32, t / 32 + 8, ...: all in flight
    const int c4 = 4 * ((int)threadIdx.x % 32), r0 = (int)threadIdx.x / 32;
#pragma unroll
    for (int k = 0; k < kSB / 8; ++k) {
      const int r = r0 + 8 * k;
      if (r < bw) {
        const float* src = U + (b0 + r) * in + b0 + c4;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c4 + e < bw) Ub[r * kSB + c4 + e] = src[e];
      }
    }
  }
  const int rl = (int)threadIdx.x / kSLanes, q = (int)threadIdx.x % kSLanes;
  const int lane = (int)threadIdx.x & 31, base = lane & ~(kSLanes - 1);
  const int64_t row = (int64_t)blockIdx.x * kSRows + rl;
  const bool live = row < out;
  float w[kSOwn];
#pragma unroll
  for (int k = 0; k < kSOwn; ++k) {
    const int j = q + kSLanes * k;
    w[k] = (live && j < bw) ? Ws[row * in + b0 + j] : 0.0f;
  }
  __syncthreads();
  const float Lf = (float)((1 << (bits - 1)) - 1), maxqf = (float)((1 << bits) - 1);
  const int64_t ng = in / group;
  // group is 32, 64 or 128 and b0 a multiple of kSB (128), so column b0 + i
  // starts a group exactly when i is a multiple of group: a mask test per
  // column instead of a 64-bit remainder
  const int gmask = group - 1;
  const int64_t g0 = b0 / group;
  float scale = 1.0f, zero = 0.0f;
  constexpr unsigned FULL = 0xffffffffu;
#pragma unroll
  for (int ki = 0; ki < kSOwn; ++ki) {
#pragma unroll
    for (int o = 0; o < kSLanes; ++o) {
      const int i = kSLanes * ki + o;
      if (i < bw) {
        if ((i & gmask) == 0) {  // fit the group on the corrected weights
          float m = 0.0f, lo = 0.0f, hi = 0.0f;
#pragma unroll
          for (int k = ki; k < kSOwn; ++k) {
            const int j = q + kSLanes * k;
            if (j >= i && j < i + group && j < bw) {
              m = fmaxf(m, fabsf(w[k]));
              lo = fminf(lo, w[k]);
              hi = fmaxf(hi, w[k]);
            }
          }
#pragma unroll
          for (int x = 1; x < kSLanes; x <<= 1) {
            m = fmaxf(m, __shfl_xor_sync(FULL, m, x));
            lo = fminf(lo, __shfl_xor_sync(FULL, lo, x));
            hi = fmaxf(hi, __shfl_xor_sync(FULL, hi, x));
          }
          if (sym) {
            scale = fmaxf(__fdiv_rn(m, Lf), 1e-8f);
            zero = 0.0f;
          } else {
            scale = fmaxf(__fdiv_rn(__fsub_rn(hi, lo), maxqf), 1e-8f);
            zero = rintf(__fdiv_rn(-lo, scale));
          }
          if (live && q == 0) {
            const int64_t gi = row * ng + g0 + i / group;
            scales[gi] = scale;
            zeros[gi] = (uint8_t)(sym ? (1 << (bits - 1)) : (int)zero);
          }
        }
        const float wi = __shfl_sync(FULL, w[ki], base | o);
        float qv, what;
        uint8_t code;
        if (sym) {
          qv = fminf(fmaxf(rintf(__fdiv_rn(wi, scale)), -Lf - 1.0f), Lf);
          what = __fmul_rn(qv, scale);
          code = (uint8_t)((int)qv + (1 << (bits - 1)));
        } else {
          qv = fminf(fmaxf(__fadd_rn(rintf(__fdiv_rn(wi, scale)), zero), 0.0f), maxqf);
          what = __fmul_rn(scale, __fsub_rn(qv, zero));
          code = (uint8_t)qv;
        }
        const float err = (wi - what) / Ub[i * kSB + i];
        if (q == o) {
          est[rl * kSB + i] = err;
          cst[rl * kSB + i] = code;
        }
        const float* ur = Ub + i * kSB + q;
#pragma unroll
        for (int k = ki; k < kSOwn; ++k) {
          const int j = q + kSLanes * k;
          if ((k > ki || q > o) && j < bw) w[k] -= err * ur[kSLanes * k];
        }
      }
    }
  }
  __syncthreads();
  // the CTA's codes and errors, row by row
  for (int idx = threadIdx.x; idx < kSRows * bw; idx += blockDim.x) {
    const int r = idx / bw, i = idx % bw;
    const int64_t gr = (int64_t)blockIdx.x * kSRows + r;
    if (gr < out) {
      codes[gr * in + b0 + i] = cst[r * kSB + i];
      Err[gr * kSB + i] = est[r * kSB + i];
    }
  }
}

// qweight[row][k]: bits [32k, 32k + 32) of the row's little-endian stream of
// b-bit codes.
__global__ void __launch_bounds__(256) pack_codes_kernel(const uint8_t* __restrict__ codes,
                                                         int64_t out, int64_t in, int bits,
                                                         uint32_t* __restrict__ qweight,
                                                         int64_t nwords) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = out * nwords;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / nwords, k = i % nwords;
    uint32_t word = 0u;
    const int64_t c0 = (32 * k) / bits, c1 = std::min<int64_t>(in, (32 * k + 31) / bits + 1);
    for (int64_t c = c0; c < c1; ++c) {
      const int64_t bit = c * bits - 32 * k;  // may be negative for a code straddling in
      const uint32_t u = codes[row * in + c];
      if (bit >= 0)
        word |= u << bit;
      else
        word |= u >> (-bit);
    }
    qweight[i] = word;
  }
}

unsigned grid_for_elems(int64_t n) {
  return (unsigned)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256,
                                                          (int64_t)device_sm_count() * 8));
}

}  // namespace

GptqLayout gptq_layout(int64_t out, int64_t in, int64_t N) {
  GptqLayout w{};
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  w.xr = take((size_t)N * in * 4);
  w.h = take((size_t)in * in * 4);
  w.y = take((size_t)in * in * 4);
  w.t = take((size_t)kCB * in * 4);
  w.ws = take((size_t)out * in * 4);
  w.err = take((size_t)out * kSB * 4);
  w.codes = take((size_t)out * in);
  w.total = o;
  return w;
}

cudaError_t launch_gptq(const void* W, const void* X, int dt, int64_t out, int64_t in, int64_t N,
                        const float* s, int bits, int group, int sym, float damp, void* workspace,
                        uint32_t* qweight, float* scales, uint8_t* zeros, int32_t* dev_status,
                        cudaStream_t st) {
  const GptqLayout L = gptq_layout(out, in, N);
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  float* Xr = reinterpret_cast<float*>(wsb + L.xr);
  float* A = reinterpret_cast<float*>(wsb + L.h);     // J H J, then M, later U
  float* Y = reinterpret_cast<float*>(wsb + L.y);     // M^-1
  float* T = reinterpret_cast<float*>(wsb + L.t);
  float* Ws = reinterpret_cast<float*>(wsb + L.ws);
  float* Err = reinterpret_cast<float*>(wsb + L.err);
  uint8_t* codes = wsb + L.codes;
  cudaError_t e;
#define AWQ_TRY(x)                      \
  do {                                  \
    if ((e = (x)) != cudaSuccess) return e; \
  } while (0)
  // 1-2: Xr = (X / s) J, A = 2 Xr^T Xr + damping
  switch (dt) {
    case kDtF32:
      AWQ_TRY(launch_pdl(scale_reverse_kernel<float>, grid_for_elems(N * in), 256, 0, st,
                         static_cast<const float*>(X), N, in, s, Xr));
      AWQ_TRY(launch_pdl(scale_weights_kernel<float>, grid_for_elems(out * in), 256, 0, st,
                         static_cast<const float*>(W), out, in, s, Ws));
      break;
    case kDtF16:
      AWQ_TRY(launch_pdl(scale_reverse_kernel<__half>, grid_for_elems(N * in), 256, 0, st,
                         static_cast<const __half*>(X), N, in, s, Xr));
      AWQ_TRY(launch_pdl(scale_weights_kernel<__half>, grid_for_elems(out * in), 256, 0, st,
                         static_cast<const __half*>(W), out, in, s, Ws));
      break;
    default:
      AWQ_TRY(launch_pdl(scale_reverse_kernel<__nv_bfloat16>, grid_for_elems(N * in), 256, 0, st,
                         static_cast<const __nv_bfloat16*>(X), N, in, s, Xr));
      AWQ_TRY(launch_pdl(scale_weights_kernel<__nv_bfloat16>, grid_for_elems(out * in), 256, 0,
                         st, static_cast<const __nv_bfloat16*>(W), out, in, s, Ws));
      break;
  }
  AWQ_TRY(sgemm(st, (int)in, (int)in, (int)N, 2.0f, Xr, in, 1, Xr, in, 0, 0.0f, A, in));
  AWQ_TRY(launch_pdl(damp_kernel, 1, 1024, 0, st, A, in, damp));
  // 3: A = M M^T
  for (int64_t k0 = 0; k0 < in; k0 += kCB) {
    const int b = (int)std::min<int64_t>(kCB, in - k0);
    AWQ_TRY(launch_pdl(chol_diag_kernel, 1, kDiagThreads, 0, st, A, in, k0, b, dev_status));
    const int64_t rest = in - k0 - b;
    if (rest > 0) {
      AWQ_TRY(launch_pdl(chol_panel_kernel, (unsigned)((rest + 127) / 128), 128, 0, st, A, in, k0,
                         b));
      AWQ_TRY(sgemm(st, (int)rest, (int)rest, b, -1.0f, A + (k0 + b) * in + k0, in, 0,
                    A + (k0 + b) * in + k0, in, 1, 1.0f, A + (k0 + b) * in + k0 + b, in));
    }
  }
  // 4: Y = M^-1 (Y starts at zero above the diagonal): every diagonal block
  // inverted in one launch, then each block row's off-diagonal part from the
  // rows above it
  AWQ_TRY(cudaMemsetAsync(Y, 0, (size_t)in * in * 4, st));
  AWQ_TRY(launch_pdl(tri_inv_diag_kernel, (unsigned)((in + kCB - 1) / kCB), kCB, 0, st, A, Y,
                     in));
  const int64_t nblk = (in + kCB - 1) / kCB;
  if (in % kCB == 0 && (nblk & (nblk - 1)) == 0) {
    // a power-of-two count of blocks: recursive doubling.  With the inverses
    // Y_A, Y_C of two neighbouring sz x sz lower triangles and the block B of
    // M below the first, inv([[A, 0], [B, C]]) = [[Y_A, 0], [-Y_C B Y_A,
    // Y_C]]; every pair of a level in one batched call (pairs 2 sz (in + 1)
    // elements apart along the diagonal).  B Y_A goes to the upper triangle
    // of A's storage, unused until U is written there.
    for (int64_t sz = kCB; sz < in; sz *= 2) {
      const int batch = (int)(in / (2 * sz));
      const int64_t stride = 2 * sz * (in + 1);
      float* Tb = A + sz;                  // rows [0, sz), columns [sz, 2 sz): scratch
      AWQ_TRY(sgemm_batched(st, (int)sz, (int)sz, (int)sz, 1.0f, A + sz * in, in, stride, Y, in,
                            stride, 0.0f, Tb, in, stride, batch));
      AWQ_TRY(sgemm_batched(st, (int)sz, (int)sz, (int)sz, -1.0f, Y + sz * in + sz, in, stride,
                            Tb, in, stride, 0.0f, Y + sz * in, in, stride, batch));
    }
  }
  for (int64_t i0 = 0; i0 < in && (in % kCB != 0 || (nblk & (nblk - 1)) != 0); i0 += kCB) {
    const int b = (int)std::min<int64_t>(kCB, in - i0);
    if (i0 > 0) {
      AWQ_TRY(sgemm(st, b, (int)i0, (int)i0, 1.0f, A + i0 * in, in, 0, Y, in, 0, 0.0f, T, i0));
      AWQ_TRY(sgemm(st, b, (int)i0, b, -1.0f, Y + i0 * in + i0, in, 0, T, i0, 0, 0.0f,
                    Y + i0 * in, in));
    }
  }
  // 5: U = J Y J, into A's storage
  AWQ_TRY(launch_pdl(reverse_kernel, grid_for_elems(in * in), 256, 0, st, Y, A, in));
  const float* U = A;
  // 6: the sweep
  const size_t smem = (size_t)(kSB * kSB + kSB * kSRows) * 4 + (size_t)kSB * kSRows;
  AWQ_TRY(cudaFuncSetAttribute(sweep_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem));
  for (int64_t b0 = 0; b0 < in; b0 += kSB) {
    const int bw = (int)std::min<int64_t>(kSB, in - b0);
    AWQ_TRY(launch_pdl(sweep_block_kernel, (unsigned)((out + kSRows - 1) / kSRows), kSRows * kSLanes, smem,
                       st, Ws, U, out, in, b0, bw, group, bits, sym, codes, scales, zeros, Err));
    const int64_t rest = in - b0 - bw;
    if (rest > 0)
      AWQ_TRY(sgemm(st, (int)out, (int)rest, bw, -1.0f, Err, kSB, 0, U + b0 * in + b0 + bw, in, 0,
                    1.0f, Ws + b0 + bw, in));
  }
  // 7: pack
  const int64_t nwords = (in * bits + 31) / 32;
  AWQ_TRY(launch_pdl(pack_codes_kernel, grid_for_elems(out * nwords), 256, 0, st, codes, out, in,
                     bits, qweight, nwords));
#undef AWQ_TRY
  return cudaSuccess;
}

}  // namespace awq
