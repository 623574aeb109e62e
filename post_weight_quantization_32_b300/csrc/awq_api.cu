// The C ABI of libawq (declared in include/awq.h): argument checks,
// workspace layout, and the order of launches on the caller's stream.
// Every entry point is an NVTX range named after it (header-only NVTX: a
// no-op unless a profiler attaches), so timelines group the launches by call.
#include <algorithm>
#include <nvtx3/nvToolsExt.h>

#include "awq.h"
#include "awq_internal.h"

namespace awq {

int device_sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = v > 0 ? v : 1;
  }
  return cache[dev];
}

namespace {


// Byte offsets of the workspace regions of awq_search (each 256-aligned).
struct WsLayout {
  size_t ctl, pow2, unscale, escale, qk, sx64, u64, minmax, s32, inv_s32, ss32, xf16,
      gext, gext_bytes, partials, sbest, total;
};

// xs: the pre-divided search (search_xs_eligible), which adds the scaled s
// table and the n_alpha copies of X / s and needs no fp16 copy of X.
WsLayout ws_layout(int dt, int64_t out, int64_t in, int64_t N, int group, int grid,
                   bool xs = false) {
  WsLayout w{};
  const int64_t n_alpha = grid + 1;
  const int64_t n_tiles = ((out + 127) / 128) * ((N + 255) / 256);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  // max|W|, max|X| bits, a ticket, the kept alpha (row split), 4 words of
  // wait diagnostics
  w.ctl = take(8 * sizeof(uint32_t));
  w.pow2 = take((size_t)n_alpha * 4);
  w.unscale = take((size_t)n_alpha * 8);
  w.escale = take((size_t)n_alpha * 4);
  w.qk = take((size_t)n_alpha * 8);
  w.sx64 = take((size_t)in * 8);
  w.u64 = take((size_t)n_alpha * in * 8);          // s_X ^ (k / grid)
  w.minmax = take(prep_chunks(in) * 32);           // per-chunk extremes of s_X with their roots
  w.s32 = take((size_t)n_alpha * in * 4);
  w.inv_s32 = take((size_t)n_alpha * in * 4);
  w.ss32 = take(xs ? (size_t)n_alpha * in * 4 : 0);
  // fp16 copy of a bf16/fp32 X, or the n_alpha copies of X / s
  w.xf16 = take(xs ? (size_t)n_alpha * N * in * 2 : (dt == kDtF16 ? 0 : (size_t)N * in * 2));
  // extremes of groups wider than a producer job: two floats per (alpha, row, group)
  w.gext_bytes = search_needs_ranges(group, in) ? (size_t)n_alpha * out * (in / group) * 8 : 0;
  w.gext = take(w.gext_bytes);
  w.partials = take((size_t)n_alpha * n_tiles * 8);
  w.sbest = take((size_t)in * 4);  // awq_search_rows: the reduction's kept-scale output
  w.total = o;
  return w;
}

bool dtype_ok(int dt) { return dt == kDtF32 || dt == kDtF16 || dt == kDtBF16; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? AWQ_OK : AWQ_ERR_CUDA; }

// NVTX range for the lifetime of one entry-point call.
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

}  // namespace

size_t search_workspace_min_bytes(int dtype, int64_t out, int64_t in, int64_t N, int group,
                                  int grid) {
  if (!dtype_ok(dtype) || out < 1 || in < 1 || N < 1 || grid < 1 || grid > kMaxGrid ||
      group < 1 || in % group != 0)
    return 0;
  return ws_layout(dtype, out, in, N, group, grid).total;
}

}  // namespace awq

using namespace awq;

extern "C" {

const char* awq_status_string(int status) {
  switch (status) {
    case AWQ_OK: return "ok";
    case AWQ_ERR_INVALID_ARG: return "invalid argument";
    case AWQ_ERR_UNSUPPORTED: return "unsupported by this build";
    case AWQ_ERR_NONFINITE: return "non-finite values: no alpha has a finite error";
    case AWQ_ERR_TIMEOUT: return "a bounded device wait ran out";
    case AWQ_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown status";
  }
}

int awq_channel_stats(const void* X, int dtype, int64_t N, int64_t in, double* sx,
                      int32_t* dev_status, awq_stream_t stream) {
  const Range range("awq_channel_stats");
  (void)dev_status;  // no device-side errors in this kernel
  if (!X || !sx || !dtype_ok(dtype) || N < 1 || in < 1) return AWQ_ERR_INVALID_ARG;
  return cuda_status(
      launch_channel_stats(X, dtype, N, in, sx, nullptr, CentreArgs{}, (cudaStream_t)stream));
}

size_t awq_search_workspace_bytes(int dtype, int64_t out, int64_t in, int64_t N, int group,
                                  int grid) {
  if (!dtype_ok(dtype) || out < 1 || in < 1 || N < 1 || grid < 1 || grid > kMaxGrid ||
      group < 1 || in % group != 0)
    return 0;
  return ws_layout(dtype, out, in, N, group, grid,
                   search_xs_eligible(dtype, in, N, group, grid)).total;
}

size_t awq_search_workspace_min_bytes(int dtype, int64_t out, int64_t in, int64_t N, int group,
                                      int grid) {
  return search_workspace_min_bytes(dtype, out, in, N, group, grid);
}

}  // extern "C"

namespace {

// The search; rows_mode: err receives the per-alpha sums over these rows,
// unnormalised (denominator 1), best and s_best go to workspace scratch, and
// s_table (if given) receives the per-alpha scale table.
int search_impl(const void* W, const void* X, int dtype, int64_t out, int64_t in, int64_t N,
                const double* sx, int bits, int group, int sym, int grid, void* workspace,
                size_t workspace_bytes, double* err, int32_t* best, float* s_best,
                int32_t* dev_status, awq_stream_t stream, const awq_search_opts* opts,
                bool rows_mode, float* s_table) {
  if (!W || !X || !workspace || !err || (!rows_mode && (!best || !s_best)) || !dtype_ok(dtype))
    return AWQ_ERR_INVALID_ARG;
  if (out < 1 || in < 1 || N < 1 || bits < 2 || bits > 8 || grid < 1 || grid > kMaxGrid ||
      group < 1 || in % group != 0)
    return AWQ_ERR_INVALID_ARG;
  // the pre-divided search where it applies and the workspace has room for it
  const bool xs = search_xs_eligible(dtype, in, N, group, grid) &&
                  workspace_bytes >= ws_layout(dtype, out, in, N, group, grid, true).total;
  const WsLayout ws = ws_layout(dtype, out, in, N, group, grid, xs);
  if (workspace_bytes < ws.total || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return AWQ_ERR_INVALID_ARG;
  if (!search_supported(dtype, out, in, N, bits, group, grid)) return AWQ_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(W) & 15) != 0 || (reinterpret_cast<uintptr_t>(X) & 15) != 0)
    return AWQ_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  const int n_alpha = grid + 1;

  // max|W| and max|X| set the exact power-of-two scalings of the fp16 GEMM operands
  uint32_t* absmax = reinterpret_cast<uint32_t*>(wsb + ws.ctl);
  uint32_t* diag = (opts && opts->diag) ? opts->diag : absmax + 4;
  cudaError_t e = cudaMemsetAsync(absmax, 0, 8 * sizeof(uint32_t), s);
  if (e == cudaSuccess && opts && opts->diag)
    e = cudaMemsetAsync(opts->diag, 0, 4 * sizeof(uint32_t), s);
  float* gext = ws.gext_bytes ? reinterpret_cast<float*>(wsb + ws.gext) : nullptr;
  if (e == cudaSuccess && gext) e = cudaMemsetAsync(gext, 0, ws.gext_bytes, s);
  if (e != cudaSuccess) return AWQ_ERR_CUDA;
  int32_t* pow2_s = reinterpret_cast<int32_t*>(wsb + ws.pow2);
  float* s32 = reinterpret_cast<float*>(wsb + ws.s32);
  float* inv_s32 = reinterpret_cast<float*>(wsb + ws.inv_s32);
  double* unscale = reinterpret_cast<double*>(wsb + ws.unscale);
  const bool x_copy = dtype != kDtF16 && !xs;
  const bool need_xmax = x_copy || xs;
  float* ss32 = xs ? reinterpret_cast<float*>(wsb + ws.ss32) : nullptr;
  float* escale = reinterpret_cast<float*>(wsb + ws.escale);
  double* qk = reinterpret_cast<double*>(wsb + ws.qk);
  CentreArgs ca{};
  ca.grid = grid;
  ca.u = reinterpret_cast<double*>(wsb + ws.u64);
  ca.minmax = reinterpret_cast<double*>(wsb + ws.minmax);
  ca.pow2_s = pow2_s;
  // The statistics launch: s_X (unless given), max|X| where it sets a
  // scaling, every column's powers s_X^(k / grid) and the chunk extremes of
  // s_X.  Then one launch streams W for max|W| -- in the pre-divided mode
  // forming the s table and the n_alpha fp16 copies of X / s meanwhile --
  // and a table launch folds max|W| and max|X| into the power-of-two
  // scalings.  A bf16 / fp32 X is copied to fp16 (scaled by a power of two)
  // for the tensor cores.
  const double* sxp = sx;
  if (!sxp) {
    e = launch_channel_stats(X, dtype, N, in, reinterpret_cast<double*>(wsb + ws.sx64),
                             need_xmax ? absmax + 1 : nullptr, ca, s);
    sxp = reinterpret_cast<const double*>(wsb + ws.sx64);
  } else {
    if (need_xmax) e = launch_absmax(X, dtype, N * in, absmax + 1, s);
    if (e == cudaSuccess) e = launch_alpha_root(sxp, in, ca, s);
  }
  if (e == cudaSuccess)
    e = launch_wmax_xs(W, dtype, out * in, absmax, X, N, in, grid, ca.u, ca.minmax, absmax + 1, s32,
                       qk, pow2_s, xs ? wsb + ws.xf16 : nullptr, s);
  if (e == cudaSuccess && x_copy) e = launch_to_f16(X, dtype, N * in, absmax + 1, wsb + ws.xf16, s);
  if (e == cudaSuccess && xs)
    e = launch_scale_table_xs(s32, qk, absmax, in, grid, ss32, escale, unscale, s);
  else if (e == cudaSuccess)
    e = launch_alpha_table(ca.u, ca.minmax, absmax, x_copy ? 1 : 0, in, grid, s32, inv_s32, escale,
                           unscale, pow2_s, s);
  if (e == cudaSuccess && gext)
    e = launch_group_extremes(W, dtype, out, in, s32, n_alpha, group, sym, gext, s);
  if (e != cudaSuccess) return AWQ_ERR_CUDA;
  const void* xh = (x_copy || xs) ? static_cast<const void*>(wsb + ws.xf16) : X;

  const SearchPlan pl =
      plan_search(dtype, out, in, N, n_alpha, group, gext != nullptr && search_wide_group(group, in),
                  device_sm_count(), xs);
  double* partials = reinterpret_cast<double*>(wsb + ws.partials);
  e = launch_search(W, xh, dtype, out, in, N, bits, group, sym ? 1 : 0, n_alpha, s32, inv_s32,
                    pow2_s, gext, ss32, xs ? escale : nullptr, partials, pl,
                    opts ? opts->wait_limit_ns : 0,
                    opts ? opts->test_timeout : 0, dev_status, diag, s,
                    opts ? (cudaEvent_t)opts->ev_search_start : nullptr,
                    opts ? (cudaEvent_t)opts->ev_search_stop : nullptr);
  if (e == cudaErrorInvalidValue) return AWQ_ERR_UNSUPPORTED;
  if (e != cudaSuccess) return AWQ_ERR_CUDA;
  if (rows_mode) {
    best = reinterpret_cast<int32_t*>(absmax + 3);
    s_best = reinterpret_cast<float*>(wsb + ws.sbest);
  }
  e = launch_reduce_argmin(partials, unscale, n_alpha, pl.n_tiles,
                           rows_mode ? 1.0 : (double)N * (double)out, s32, in, err, best, s_best,
                           dev_status, s);
  if (e == cudaSuccess && s_table)
    e = cudaMemcpyAsync(s_table, s32, (size_t)n_alpha * in * sizeof(float),
                        cudaMemcpyDeviceToDevice, s);
  return cuda_status(e);
}

}  // namespace

extern "C" {

int awq_search_ex(const void* W, const void* X, int dtype, int64_t out, int64_t in, int64_t N,
                  const double* sx, int bits, int group, int sym, int grid, void* workspace,
                  size_t workspace_bytes, double* err, int32_t* best, float* s_best,
                  int32_t* dev_status, awq_stream_t stream, const awq_search_opts* opts) {
  const Range range("awq_search_ex");
  return search_impl(W, X, dtype, out, in, N, sx, bits, group, sym, grid, workspace,
                     workspace_bytes, err, best, s_best, dev_status, stream, opts, false, nullptr);
}

int awq_search_rows(const void* W, const void* X, int dtype, int64_t rows, int64_t in, int64_t N,
                    const double* sx, int bits, int group, int sym, int grid, void* workspace,
                    size_t workspace_bytes, double* sums, float* s_table, int32_t* dev_status,
                    awq_stream_t stream) {
  const Range range("awq_search_rows");
  return search_impl(W, X, dtype, rows, in, N, sx, bits, group, sym, grid, workspace,
                     workspace_bytes, sums, nullptr, nullptr, dev_status, stream, nullptr, true,
                     s_table);
}

int awq_search_finish(const double* sums, int n_parts, int grid, int64_t N, int64_t out,
                      const float* s_table, int64_t in, double* err, int32_t* best, float* s_best,
                      int32_t* dev_status, awq_stream_t stream) {
  const Range range("awq_search_finish");
  if (!sums || !s_table || !err || !best || !s_best || n_parts < 1 || grid < 1 ||
      grid > kMaxGrid || N < 1 || out < 1 || in < 1)
    return AWQ_ERR_INVALID_ARG;
  return cuda_status(launch_search_finish(sums, n_parts, grid + 1, (double)N * (double)out, s_table,
                                          in, err, best, s_best, dev_status,
                                          (cudaStream_t)stream));
}

int awq_search(const void* W, const void* X, int dtype, int64_t out, int64_t in, int64_t N,
               const double* sx, int bits, int group, int sym, int grid, void* workspace,
               size_t workspace_bytes, double* err, int32_t* best, float* s_best,
               int32_t* dev_status, awq_stream_t stream) {
  return awq_search_ex(W, X, dtype, out, in, N, sx, bits, group, sym, grid, workspace,
                       workspace_bytes, err, best, s_best, dev_status, stream, nullptr);
}

size_t awq_output_power_workspace_bytes(int dtype, int64_t out, int64_t in, int64_t N) {
  if (!dtype_ok(dtype) || out < 1 || in < 1 || N < 1) return 0;
  return align_up((size_t)N * out * sizeof(float), 256) + align_up(power_reduce_scratch_bytes(), 256);
}

int awq_output_power(const void* W, const void* X, int dtype, int64_t out, int64_t in, int64_t N,
                     void* workspace, size_t workspace_bytes, double* power, int32_t* dev_status,
                     awq_stream_t stream) {
  const Range range("awq_output_power");
  if (!W || !X || !workspace || !power || !dtype_ok(dtype)) return AWQ_ERR_INVALID_ARG;
  if (out < 1 || in < 1 || N < 1) return AWQ_ERR_INVALID_ARG;
  if (workspace_bytes < awq_output_power_workspace_bytes(dtype, out, in, N) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return AWQ_ERR_INVALID_ARG;
  if (out >= (1ll << 31) || N >= (1ll << 31) || in >= (1ll << 31)) return AWQ_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (power_mma_eligible(dtype, out, in, N, W, X) &&
      workspace_bytes >= power_mma_workspace_bytes(out, N))
    return cuda_status(launch_power_mma(W, X, dtype, out, in, N, workspace, power, dev_status, s));
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  // D = X W^T ([N][out] float32, a plain GEMM), then mean(D^2) in float64
  float* D = reinterpret_cast<float*>(wsb);
  void* scratch = wsb + align_up((size_t)N * out * sizeof(float), 256);
  cudaError_t e = cudaMemsetAsync(scratch, 0, 256, s);
  if (e == cudaSuccess)
    e = blas_gemm(s, (int)N, (int)out, (int)in, 1.0f, X, in, 0, W, in, 1, 0.0f, D, out, dtype);
  if (e == cudaSuccess)
    e = launch_power_reduce(D, N * out, (double)N * (double)out, scratch, power, s);
  return cuda_status(e);
}

int awq_sweep_summary(const double* err, const int32_t* best, const double* power, int grid,
                      double* row, awq_stream_t stream) {
  const Range range("awq_sweep_summary");
  if (!err || !best || !power || !row || grid < 1 || grid > kMaxGrid) return AWQ_ERR_INVALID_ARG;
  return cuda_status(launch_sweep_summary(err, best, power, grid, row, (cudaStream_t)stream));
}

int awq_quantize_pack(const void* W, int dtype, int64_t out, int64_t in, const float* s, int bits,
                      int group, int sym, uint32_t* qweight, float* scales, uint8_t* zeros,
                      int32_t* dev_status, awq_stream_t stream) {
  const Range range("awq_quantize_pack");
  if (!W || !s || !qweight || !scales || !zeros || !dtype_ok(dtype)) return AWQ_ERR_INVALID_ARG;
  if (out < 1 || in < 1 || bits < 2 || bits > 8 || group < 1 || in % group != 0)
    return AWQ_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_pack(W, dtype, out, in, s, bits, group, sym ? 1 : 0, nullptr,
                                          qweight, scales, zeros, dev_status,
                                          (cudaStream_t)stream));
}

int awq_quantize_pack_clipped(const void* W, int dtype, int64_t out, int64_t in, const float* s,
                              int bits, int group, int sym, const float* clip, uint32_t* qweight,
                              float* scales, uint8_t* zeros, int32_t* dev_status,
                              awq_stream_t stream) {
  const Range range("awq_quantize_pack_clipped");
  if (!W || !s || !clip || !qweight || !scales || !zeros || !dtype_ok(dtype))
    return AWQ_ERR_INVALID_ARG;
  if (out < 1 || in < 1 || bits < 2 || bits > 8 || group < 1 || in % group != 0)
    return AWQ_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_pack(W, dtype, out, in, s, bits, group, sym ? 1 : 0, clip,
                                          qweight, scales, zeros, dev_status,
                                          (cudaStream_t)stream));
}

size_t awq_clip_search_workspace_bytes(int64_t in, int64_t N, int group) {
  if (in < 1 || N < 1 || (group != 32 && group != 64 && group != 128) || in % group != 0)
    return 0;
  // the Gram matrices of the FMA path, or what the tensor-core path needs
  // (16-bit inputs, group 128, at most 256 tokens), whichever is larger
  const size_t gram = align_up((size_t)clip_splits(N) * in * group * sizeof(float), 256);
  const size_t mma = clip_mma_eligible(kDtF16, in, N, group) ? clip_mma_workspace_bytes(in, N) : 0;
  return std::max(gram, mma);
}

int awq_clip_search(const void* W, const void* X, int dtype, int64_t out, int64_t in, int64_t N,
                    const float* s, int bits, int group, int sym, int n_grid, int max_shrink_steps,
                    void* workspace, size_t workspace_bytes, float* clip, float* errs,
                    int32_t* dev_status, awq_stream_t stream) {
  const Range range("awq_clip_search");
  if (!W || !X || !s || !workspace || !clip || !dtype_ok(dtype)) return AWQ_ERR_INVALID_ARG;
  if (out < 1 || in < 1 || N < 1 || bits < 2 || bits > 8 || group < 1 || in % group != 0)
    return AWQ_ERR_INVALID_ARG;
  if (n_grid < 1 || max_shrink_steps < 0 || max_shrink_steps >= n_grid) return AWQ_ERR_INVALID_ARG;
  if (group != 32 && group != 64 && group != 128) return AWQ_ERR_UNSUPPORTED;
  if (max_shrink_steps + 1 > kMaxClip) return AWQ_ERR_UNSUPPORTED;
  if (workspace_bytes < awq_clip_search_workspace_bytes(in, N, group) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return AWQ_ERR_INVALID_ARG;
  ClipFactors cf{};
  for (int i = 0; i <= max_shrink_steps; ++i) cf.c[i] = (float)(1.0 - (double)i / n_grid);
  if (clip_mma_eligible(dtype, in, N, group) && out <= (1 << 24) &&
      (reinterpret_cast<uintptr_t>(W) & 15) == 0 && (reinterpret_cast<uintptr_t>(X) & 15) == 0)
    return cuda_status(launch_clip_search_mma(W, X, dtype, out, in, N, s, bits, sym ? 1 : 0,
                                              max_shrink_steps + 1, cf, workspace, clip, errs,
                                              dev_status, (cudaStream_t)stream));
  return cuda_status(launch_clip_search(W, X, dtype, out, in, N, s, bits, group, sym ? 1 : 0,
                                        max_shrink_steps + 1, cf, static_cast<float*>(workspace),
                                        clip, errs, dev_status, (cudaStream_t)stream));
}

size_t awq_gptq_workspace_bytes(int64_t out, int64_t in, int64_t N) {
  if (out < 1 || in < 1 || N < 1) return 0;
  return gptq_layout(out, in, N).total;
}

int awq_gptq(const void* W, const void* X, int dtype, int64_t out, int64_t in, int64_t N,
             const float* s, int bits, int group, int sym, double damp, void* workspace,
             size_t workspace_bytes, uint32_t* qweight, float* scales, uint8_t* zeros,
             int32_t* dev_status, awq_stream_t stream) {
  const Range range("awq_gptq");
  if (!W || !X || !workspace || !qweight || !scales || !zeros || !dtype_ok(dtype))
    return AWQ_ERR_INVALID_ARG;
  if (out < 1 || in < 1 || N < 1 || bits < 2 || bits > 8 || group < 1 || in % group != 0 ||
      !(damp >= 0.0))
    return AWQ_ERR_INVALID_ARG;
  if (group != 32 && group != 64 && group != 128) return AWQ_ERR_UNSUPPORTED;
  if (in > (1 << 30) / in || out > (1 << 24) || N > (1 << 24)) return AWQ_ERR_UNSUPPORTED;
  if (workspace_bytes < gptq_layout(out, in, N).total ||
      (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
    return AWQ_ERR_INVALID_ARG;
  return cuda_status(launch_gptq(W, X, dtype, out, in, N, s, bits, group, sym ? 1 : 0,
                                 (float)damp, workspace, qweight, scales, zeros, dev_status,
                                 (cudaStream_t)stream));
}

int awq_export_checkpoint(const uint32_t* qweight, const float* scales, const uint8_t* zeros,
                          int64_t out, int64_t in, int bits, int group, uint32_t* qweight_t,
                          void* scales_h, uint32_t* qzeros, int32_t* dev_status,
                          awq_stream_t stream) {
  const Range range("awq_export_checkpoint");
  if (!qweight || !scales || !zeros || !qweight_t || !scales_h || !qzeros)
    return AWQ_ERR_INVALID_ARG;
  if (out < 1 || in < 1 || group < 1 || in % group != 0) return AWQ_ERR_INVALID_ARG;
  if (bits != 2 && bits != 4 && bits != 8) return AWQ_ERR_INVALID_ARG;
  if (in % (32 / bits) != 0) return AWQ_ERR_INVALID_ARG;
  return cuda_status(launch_export_checkpoint(qweight, scales, zeros, out, in, bits, group,
                                              qweight_t, scales_h, qzeros, dev_status,
                                              (cudaStream_t)stream));
}

}  // extern "C"
