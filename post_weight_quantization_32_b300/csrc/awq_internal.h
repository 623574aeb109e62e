// Host-side interfaces between the C ABI (awq_api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace awq {

constexpr int kDtF32 = 0, kDtF16 = 1, kDtBF16 = 2;

inline size_t dtype_size(int dt) { return dt == kDtF32 ? 4 : 2; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Number of SMs of the current device (cached per device).
int device_sm_count();

// 2-D tensor map of a row-major matrix [rows][cols] (row_bytes apart) with
// box_cols x box_rows boxes in the 128-byte swizzled layout of a K-major
// MMA operand; out-of-range elements read as zero.  False when the driver's
// encoder is missing or rejects the arguments.
bool tensor_map_sw128(CUtensorMap* m, CUtensorMapDataType t, const void* ptr, uint64_t cols,
                      uint64_t rows, uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows);

// Launch with the programmatic-stream-serialization attribute: the kernel
// may begin while the previous kernel in the stream is still running, and
// must call pdl_wait() before touching anything that kernel writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// launch_pdl for a grid of thread-block clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, unsigned cluster, dim3 block,
                               size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Largest alpha grid (grid + 1 alphas) the C ABI accepts.
constexpr int kMaxGrid = 4096;

// ---- statistics and conversions (awq_stats.cu)
// Where a statistics (or root) launch puts what the table launches need
// (grid == 0: nothing).  u[k][j] = s_X[j]^(k / grid) for k = 0..grid
// (float64, [grid + 1][in]; exactly 1 at k = 0 and s_X at k = grid);
// minmax holds each 32-column chunk's max and min of s_X with their roots
// s_X^(1 / grid) (4 words per chunk, prep_chunks(in) chunks); pow2_s[k] is
// set to 1 for k = 0..grid (the table launches clear it).
struct CentreArgs {
  int grid;
  double* u;
  double* minmax;
  int32_t* pow2_s;
};

// sx[j] = sum_n |X[n, j]| / N + 1e-8, float64.  With xmax != nullptr the same
// pass folds max|X| into *xmax (bits of a non-negative float; must start at
// 0).  With ca.grid != 0 the launch also writes the powers and chunk
// extremes of CentreArgs (needs in % 8 == 0 and a 16-byte aligned X, as
// does xmax).  The launch lets the next one in the stream start
// (programmatic dependent launch) as soon as its CTAs have read X.
cudaError_t launch_channel_stats(const void* X, int dt, int64_t N, int64_t in, double* sx,
                                 uint32_t* xmax, const CentreArgs& ca, cudaStream_t s);
// Fold max|W| (nW values, nW % 8 == 0, 16-byte aligned) into *wmax, and
// finish only after the launch before it in the stream.  With xs != nullptr
// the same launch forms the pre-divided search's table and X copies once
// that earlier launch is done: for k = 0..grid, s32[k][j] = fp32(u[k][j] *
// ic_k) (ic_k the centring of alpha k from the chunk extremes), qk[k] (see
// launch_alpha_table), and xs[k][n][j] = fp16(X[n][j] * 2^m_k / s32[k][j])
// (m_k from max|X| in xmax_bits; X of dtype dt, in % 8 == 0, 16-byte
// aligned); pow2_s[k] is cleared when some s32[k][j] is not a power of two.
cudaError_t launch_wmax_xs(const void* W, int dt, int64_t nW, uint32_t* wmax, const void* X,
                           int64_t N, int64_t in, int grid, const double* u,
                           const double* minmax, const uint32_t* xmax_bits, float* s32,
                           double* qk, int32_t* pow2_s, void* xs, cudaStream_t s);
// *out = max(*out, bits of max_i |p[i]|); *out must start at 0.
cudaError_t launch_absmax(const void* p, int dt, int64_t n, uint32_t* out, cudaStream_t s);
// dst = fp16(X * 2^m) with m = pow2_exponent_for(max|X|) read from *xmax_bits;
// n elements, n % 8 == 0, 16-byte aligned.  dt is AWQ_F32 or AWQ_BF16.
cudaError_t launch_to_f16(const void* X, int dt, int64_t n, const uint32_t* xmax_bits, void* dst,
                          cudaStream_t s);

// ---- alpha tables, reduction and argmin (awq_prep.cu)
// Column chunks of the statistics / root launches (32 columns each):
// minmax needs 4 * prep_chunks(in) words.
size_t prep_chunks(int64_t in);
// The powers and chunk extremes of CentreArgs from a given sx.
cudaError_t launch_alpha_root(const double* sx, int64_t in, const CentreArgs& ca, cudaStream_t s);
// For k = 0..grid: s32[k][j] = fp32(u[k][j] * ic_k), where ic_k = 1 /
// sqrt(max(s_k) * min(s_k)) comes from the chunk extremes, and inv_s32[k][j]
// = escale[k] / s32[k][j]; escale[k] = 2^e_k (which scales the weight
// changes of alpha k into the fp16 range of the error GEMM) and unscale[k]
// are formed from qk = sqrt(max(s_k) / min(s_k)) and the max|W|, max|X|
// bits in absmax (X copied to fp16 with a scaling when x_scaled).
// pow2_s[k] (1 on entry) ends nonzero iff every s32[k][j] is a power of two.
cudaError_t launch_alpha_table(const double* u, const double* minmax, const uint32_t* absmax,
                               int x_scaled, int64_t in, int grid, float* s32, float* inv_s32,
                               float* escale, double* unscale, int32_t* pow2_s, cudaStream_t s);
// The pre-divided mode's scalings, after launch_wmax_xs: ss32[k][j] =
// s32[k][j] * escale[k] (exact: a power of two), and escale[k], unscale[k]
// from qk[k] and the max|W|, max|X| bits in absmax.
cudaError_t launch_scale_table_xs(const float* s32, const double* qk, const uint32_t* absmax,
                                  int64_t in, int grid, float* ss32, float* escale,
                                  double* unscale, cudaStream_t s);
// err[k] = unscale[k] * sum_t partials[k][t] / denom (fixed order),
// best = strict-< argmin, s_best = s32[best].
cudaError_t launch_reduce_argmin(const double* partials, const double* unscale, int n_alpha,
                                 int n_tiles, double denom, const float* s32, int64_t in,
                                 double* err, int32_t* best, float* s_best, int32_t* dev_status,
                                 cudaStream_t s);

// row[0..4] = alpha value of best, err[0], err[best], err[0] / *power,
// err[best] / *power (NaN where best < 0); one thread.
cudaError_t launch_sweep_summary(const double* err, const int32_t* best, const double* power,
                                 int grid, double* row, cudaStream_t s);

// The finish of a row-split search: err[k] = (sum over parts p, in order,
// of sums[p][k]) / denom, then best and s_best = s_table[best] as
// launch_reduce_argmin.
cudaError_t launch_search_finish(const double* sums, int parts, int n_alpha, double denom,
                                 const float* s_table, int64_t in, double* err, int32_t* best,
                                 float* s_best, int32_t* dev_status, cudaStream_t s);

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
// Groups whose ranges are formed by launch_group_extremes ahead of the
// search: a multiple of 256 columns (wider than one 128-column producer
// job), or one group per row (group == in, any width).  Needs in % 8 == 0.
bool search_wide_group(int64_t group, int64_t in);
// Group widths whose ranges come from launch_group_extremes: the wide ones,
// and any other multiple of 8 outside {8, 16, 32, 64, 128} (e.g. 24, 48,
// 96), which 64-column producer jobs do not align with.  Needs in % 8 == 0.
bool search_needs_ranges(int64_t group, int64_t in);
bool search_supported(int dt, int64_t out, int64_t in, int64_t N, int bits, int group, int grid);
// Whether the search may read X already divided by s (launch_search with
// ss32): one alpha per work unit, group 8, 16, 32, 64 or 128, 16-bit W, and
// the n_alpha fp16 copies of X / s small enough to stay in L2.
bool search_xs_eligible(int dt, int64_t in, int64_t N, int group, int grid);
// The smallest workspace awq_search accepts (without the pre-divided mode's
// regions); awq_search_workspace_bytes may return more.
size_t search_workspace_min_bytes(int dtype, int64_t out, int64_t in, int64_t N, int group,
                                  int grid);
// gp: the group extremes come precomputed (launch_search with gext); xs: X
// arrives divided by s (launch_search with ss32).
SearchPlan plan_search(int dt, int64_t out, int64_t in, int64_t N, int n_alpha, int group,
                       bool gp, int sms, bool xs = false);
// With gext != nullptr the group extremes are read from gext (layout of
// launch_group_extremes) instead of being formed per job; group must then be
// in or a multiple of 128 (and must be when search_wide_group holds).
// With ss32 != nullptr (the pre-divided mode, see search_xs_eligible):
// Xf16 holds the n_alpha copies X * 2^m_k / s_k ([n_alpha][N][in] fp16),
// ss32 the table s_k * 2^e_k ([n_alpha][in]) that the weights are scaled
// by, escale[k] = 2^e_k; inv_s32 is not read.
cudaError_t launch_search(const void* W, const void* Xf16, int dt, int64_t out, int64_t in,
                          int64_t N, int bits, int group, int sym, int n_alpha,
                          const float* s32, const float* inv_s32, const int32_t* pow2_s,
                          const float* gext, const float* ss32, const float* escale,
                          double* partials, const SearchPlan& plan, int64_t wait_limit_ns,
                          int test_timeout, int32_t* dev_status, uint32_t* diag, cudaStream_t s,
                          cudaEvent_t ev0, cudaEvent_t ev1);

// ---- group extremes for wide groups (awq_groups.cu)
// For every alpha k < n_alpha, row and group: the extremes of
// t = fl32(W[row][j] * s32[k][j]) over the group's columns, folded into ext
// (zeroed by the caller): symmetric ext[(k*out + row)*ngroups + g] = max|t|;
// asymmetric ext[2i] = -min(min t, 0), ext[2i + 1] = max(max t, 0).
// group is a multiple of 8 (or equal to in); in % 8 == 0; W 16-byte aligned.
cudaError_t launch_group_extremes(const void* W, int dt, int64_t out, int64_t in,
                                  const float* s32, int n_alpha, int64_t group, int sym,
                                  float* ext, cudaStream_t s);

// ---- final quantization and packing (awq_pack.cu)
// clip: null, or [out][in/group] factors scaling each group's range (the
// codes then take the quantizer's clamps).
cudaError_t launch_quantize_pack(const void* W, int dt, int64_t out, int64_t in, const float* s,
                                 int bits, int group, int sym, const float* clip,
                                 uint32_t* qweight, float* scales, uint8_t* zeros,
                                 int32_t* dev_status, cudaStream_t st);

// ---- per-group clipping search (awq_clip.cu)
constexpr int kMaxClip = 12;  // shrink factors per search (a multiple of 4)
struct ClipFactors {
  float c[kMaxClip];
};
// Token splits of the Gram-matrix pass: the workspace holds
// clip_splits(N) * in * group floats.
int clip_splits(int64_t N);
// For every row and group (group in {32, 64, 128}) of W * diag(s): the
// group's share of the row's output error for each of the nc factors of cf,
// and clip[row][group] = the first factor with the smallest share; errs
// ([out][in/group][nc], may be null) receives the shares.
// The tensor-core clipping search (awq_clip_mma.cu): 16-bit W and X, group
// 128, 32 to 256 tokens.  workspace: clip_mma_workspace_bytes(in, N).
bool clip_mma_eligible(int dt, int64_t in, int64_t N, int group);
size_t clip_mma_workspace_bytes(int64_t in, int64_t N);
cudaError_t launch_clip_search_mma(const void* W, const void* X, int dt, int64_t out, int64_t in,
                                   int64_t N, const float* s, int bits, int sym, int nf,
                                   const ClipFactors& cf, void* workspace, float* clip, float* errs,
                                   int32_t* dev_status, cudaStream_t stream);
cudaError_t launch_clip_search(const void* W, const void* X, int dt, int64_t out, int64_t in,
                               int64_t N, const float* s, int bits, int group, int sym, int nc,
                               const ClipFactors& cf, float* H, float* clip, float* errs,
                               int32_t* dev_status, cudaStream_t stream);

// ---- GPTQ rounding after AWQ scaling (awq_gptq.cu)
// Workspace regions (byte offsets, 256-aligned): X / s reversed (N x in),
// the Hessian / its factors (in x in twice), a 32 x in scratch, the fp32
// working weights (out x in), the errors of one sweep block (out x 128) and
// the byte codes (out x in).
struct GptqLayout {
  size_t xr, h, y, t, ws, err, codes, total;
};
GptqLayout gptq_layout(int64_t out, int64_t in, int64_t N);
// s may be null (plain GPTQ).  group in {32, 64, 128}.  Outputs as
// launch_quantize_pack.  A Hessian that is not positive definite after
// dampening sets ST_NONFINITE.
cudaError_t launch_gptq(const void* W, const void* X, int dt, int64_t out, int64_t in, int64_t N,
                        const float* s, int bits, int group, int sym, float damp, void* workspace,
                        uint32_t* qweight, float* scales, uint8_t* zeros, int32_t* dev_status,
                        cudaStream_t st);

// ---- plain GEMMs (cuBLAS; awq_gptq.cu)
// Row-major C[m][n] (float32) = alpha * A(m, k) B(k, n) + beta * C, A(m, k) =
// A[m * lda + k] (or A[k * lda + m] when ta), B(k, n) = B[k * ldb + n] (or
// B[n * ldb + k] when tb); A and B of dtype dt.  16-bit operands accumulate
// in float32; float32 operands use float32 emulated on the bf16 tensor cores.
cudaError_t blas_gemm(cudaStream_t s, int m, int n, int k, float alpha, const void* A, int64_t lda,
                      int ta, const void* B, int64_t ldb, int tb, float beta, float* C, int64_t ldc,
                      int dt);

// mean((X W^T)^2) by tcgen05 with the square sum in the epilogue (16-bit
// W and X, in a multiple of 8, 16-byte aligned operands).  workspace:
// power_mma_workspace_bytes(out, N), 256-byte aligned; its first 256 bytes
// are zeroed by the launch.
bool power_mma_eligible(int dt, int64_t out, int64_t in, int64_t N, const void* W, const void* X);
size_t power_mma_workspace_bytes(int64_t out, int64_t N);
cudaError_t launch_power_mma(const void* W, const void* X, int dt, int64_t out, int64_t in,
                             int64_t N, void* workspace, double* power, int32_t* dev_status,
                             cudaStream_t stream);
// ---- output power (awq_prep.cu)
// *power = sum over the n floats of D of D^2 (float64, a fixed order: the
// grid's threads' strided sums, each CTA's tree, then the CTAs in order) /
// denom.  scratch: power_reduce_scratch_bytes(n), its first word zeroed.
size_t power_reduce_scratch_bytes();
cudaError_t launch_power_reduce(const float* D, int64_t n, double denom, void* scratch,
                                double* power, cudaStream_t s);

// ---- checkpoint export (awq_export.cu)
// From quantize_pack's row-major outputs (bits divides 32, in % (32/bits) ==
// 0): qweight_t [in*bits/32][out] (transposed words), scales_h [in/g][out]
// fp16 (rounded to nearest; overflow sets ST_NONFINITE), qzeros
// [in/g][ceil(out*bits/32)] (zero points packed along the output axis).
cudaError_t launch_export_checkpoint(const uint32_t* qweight, const float* scales,
                                     const uint8_t* zeros, int64_t out, int64_t in, int bits,
                                     int group, uint32_t* qweight_t, void* scales_h,
                                     uint32_t* qzeros, int32_t* dev_status, cudaStream_t s);

}  // namespace awq
