/*
 * awq.h - C ABI of libawq: AWQ's per-layer activation-aware scale search on
 * one NVIDIA B300 (sm_103a).
 *
 * The method (stated in "AWQ (activation-aware weight quantization)",
 * sections "How it works" and "The code, line by line"): for one linear
 * layer W (out x in) with calibration inputs X (N x in),
 *
 *   s_X[j]  = mean_n |X[n, j]| + 1e-8
 *   for alpha in linspace(0, 1, grid + 1):
 *       s   = s_X ** alpha,  s /= sqrt(max(s) * min(s))
 *       Wq  = Q(W * s) / s            Q = group round-to-nearest
 *       err = mean((X Wq^T - X W^T)^2)
 *   keep the alpha with the smallest err (strict <, first wins)
 *
 * then the weights are quantized once more at the kept scales and packed
 * ("AWQ vs GPTQ Quantization Architectures Compared", "What lands on disk").
 *
 * Conventions for every entry point:
 *  - All array pointers are DEVICE pointers owned by the caller, contiguous
 *    and row-major.  The library never allocates device memory; scratch
 *    comes from the caller's workspace.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and runs asynchronously.  Nothing synchronises the host.
 *  - The return value reports host-side argument checks and launch errors
 *    (awq_status).  Errors found on the device are written to *dev_status
 *    (an int32 in device memory, may be NULL): a call sets it to its error
 *    code only if it is still 0, and never clears it.  Read it after
 *    synchronising the stream.
 *  - dtype applies to both W and X: AWQ_F32, AWQ_F16 or AWQ_BF16.
 */
#ifndef AWQ_H
#define AWQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same types as cudaStream_t / cudaEvent_t; declared here so that the
 * header needs no CUDA include. */
typedef struct CUstream_st* awq_stream_t;
typedef struct CUevent_st* awq_event_t;

typedef enum {
    AWQ_F32 = 0,
    AWQ_F16 = 1,
    AWQ_BF16 = 2
} awq_dtype;

typedef enum {
    AWQ_OK = 0,
    AWQ_ERR_INVALID_ARG = 1,  /* a size, pointer or parameter is out of range */
    AWQ_ERR_UNSUPPORTED = 2,  /* valid for the method, not handled by this build */
    AWQ_ERR_NONFINITE = 3,    /* every alpha's error was NaN/inf, or a NaN product in pack */
    AWQ_ERR_TIMEOUT = 4,      /* a bounded device-side wait ran out; outputs are invalid */
    AWQ_ERR_CUDA = 5          /* a CUDA runtime call failed */
} awq_status;

/* Text for a status code (static storage). */
const char* awq_status_string(int status);

/*
 * awq_channel_stats - per-input-channel activation size.
 *   sx[j] = (1/N) * sum_n |X[n, j]| + 1e-8, accumulated in float64.
 * ["AWQ (activation-aware weight quantization)", "How it works" step 1 and
 *  "The code, line by line", first bullet.]
 *
 *   X   [N][in] of `dtype`          (read)
 *   sx  [in] double                 (written)
 * N >= 1, in >= 1.  The sums are taken in a fixed order, so repeated calls
 * give identical results.  For fp16 X (with 8 | in and X 16-byte aligned)
 * the column sum is formed exactly, as an integer multiple of 2^-24, so sx
 * then equals the correctly rounded float64 mean plus 1e-8.
 */
int awq_channel_stats(const void* X, int dtype, int64_t N, int64_t in,
                      double* sx, int32_t* dev_status, awq_stream_t stream);

/*
 * Bytes of device workspace for awq_search's fastest path at these sizes (0
 * on invalid sizes).  The workspace must be 256-byte aligned.  Where the
 * problem allows it (more than 128 tokens, group 8, 16, 32, 64 or 128, fp16
 * or bf16, and (grid + 1) * N * in * 2 <= 64 MiB) this includes room for
 * grid + 1 fp16 copies of X / s, which the search then reads instead of
 * dividing every weight change by s.
 */
size_t awq_search_workspace_bytes(int dtype, int64_t out, int64_t in, int64_t N,
                                  int group, int grid);

/*
 * The smallest workspace awq_search accepts for these sizes (0 on invalid
 * sizes): without the copies of X / s.  A workspace between this and
 * awq_search_workspace_bytes gives the same results within the search's
 * tolerance, by the other path.
 */
size_t awq_search_workspace_min_bytes(int dtype, int64_t out, int64_t in, int64_t N,
                                      int group, int grid);

/*
 * awq_search - the alpha-grid scale search.
 * ["AWQ (activation-aware weight quantization)", "Source code";
 *  "AWQ vs GPTQ ...", "AWQ: move the error away from what matters"]
 *
 *   W      [out][in] of `dtype`   layer weights (read)
 *   X      [N][in]   of `dtype`   calibration inputs (read)
 *   sx     [in] double or NULL    channel sizes; NULL = computed here as
 *                                 awq_channel_stats does
 *   bits   2..8                   code width
 *   group  columns per quantization group; divides `in`.  group == in is the
 *          pages' "one group per row".  This build's search handles group
 *          in {8, 16, 32, 64, 128}, any other multiple of 8 (24, 48, 96,
 *          256, ...) and group == in (those need in % 8 == 0); others return
 *          AWQ_ERR_UNSUPPORTED.  Groups outside {8, ..., 128} get their
 *          ranges from a pass over W ahead of the search.
 *   sym    1: symmetric, scale = max|w| / (2^(b-1) - 1), codes in
 *             [-2^(b-1), 2^(b-1) - 1]
 *             ["GPTQ and AWQ weight quantisation", "Output MSE vs bit width"]
 *          0: asymmetric, scale = (max(hi,0) - min(lo,0)) / (2^b - 1),
 *             zero = round(-min/scale), codes in [0, 2^b - 1]
 *             ["AWQ vs GPTQ ...", "The shared problem: one layer, sixteen levels"]
 *   grid   1..4096; the search tries the grid + 1 alphas k/grid, k = 0..grid
 *   workspace, workspace_bytes  >= awq_search_workspace_min_bytes(...);
 *          with >= awq_search_workspace_bytes(...) the faster path runs
 *   err    [grid + 1] double      (written) mean((X (Wq - W)^T)^2) per alpha
 *   best   [1] int32              (written) index of the kept alpha; -1 and
 *                                 AWQ_ERR_NONFINITE in *dev_status if every
 *                                 error is NaN or infinite
 *   s_best [in] float             (written) the kept centred scale vector,
 *                                 rounded to float32
 *
 * The error is formed as X (Wq - W)^T, which equals the pages' X Wq^T - X W^T;
 * the GEMM runs on the tensor cores with fp16 operands (X and the weight
 * change each scaled by an exact power of two chosen from max|X| and max|W|)
 * and fp32 accumulation, the per-alpha sum in float64.  On the faster path
 * the same sum is formed as (X / s)(W^ s - W s)^T, with X / s rounded to
 * fp16 once per alpha.  Rows, tokens and
 * alphas are summed in a fixed order: repeated calls give bit-identical
 * results.  Shared-input layer groups (q/k/v) are searched by passing their
 * weights concatenated along `out` with the common X: one s, one error.
 * Requirements beyond the method's: W and X 16-byte aligned, out, in, N
 * <= 2^24.
 */
int awq_search(const void* W, const void* X, int dtype,
               int64_t out, int64_t in, int64_t N,
               const double* sx, int bits, int group, int sym, int grid,
               void* workspace, size_t workspace_bytes,
               double* err, int32_t* best, float* s_best,
               int32_t* dev_status, awq_stream_t stream);

/*
 * awq_output_power - the size of the layer's exact output,
 *   power = mean((X W^T)^2) over the N x out entries, float64,
 * the denominator of the relative output error ||X W^T - X Wq^T||^2 /
 * ||X W^T||^2 ["AWQ (activation-aware weight quantization)", "What the
 * simulations show"]: with err from awq_search (a mean over the same
 * entries), err / power is that ratio.
 *
 *   W, X, dtype, out, in, N   as for awq_search
 *   workspace, workspace_bytes >= awq_output_power_workspace_bytes(dtype,
 *                               out, in, N) (256-byte aligned)
 *   power  [1] double (written)
 * 16-bit W and X (in a multiple of 8, 16-byte aligned) take one tcgen05
 * kernel: 128-row tiles of W against tiles of tokens, accumulated over all
 * of `in` in tensor memory (float32), each entry squared as it leaves it and
 * never stored; rows are summed in float64 and the tiles' sums added in a
 * fixed order.  Other calls form X W^T as a plain GEMM (cuBLAS: float32
 * operands emulated to float32 accuracy) in the workspace and sum its
 * squares in float64 in a fixed order.  Either way repeated calls give
 * identical results, and a NaN or infinite product shows in power.
 * dev_status (may be NULL) is set to AWQ_ERR_TIMEOUT when a wait inside the
 * tensor-core kernel runs past its limit.
 */
size_t awq_output_power_workspace_bytes(int dtype, int64_t out, int64_t in, int64_t N);

int awq_output_power(const void* W, const void* X, int dtype,
                     int64_t out, int64_t in, int64_t N,
                     void* workspace, size_t workspace_bytes,
                     double* power, int32_t* dev_status, awq_stream_t stream);

/*
 * awq_search_rows / awq_search_finish - the search split by output rows
 * ["AWQ (activation-aware weight quantization)", "Source code": the error
 * is a mean over every output entry, so it splits into sums over slices of
 * the output rows; s depends on X alone, so every slice sees the same s].
 *
 * awq_search_rows runs the search on `rows` consecutive rows of a layer
 * (W points at the first of them, [rows][in]); arguments as awq_search
 * (workspace sized by awq_search_workspace_bytes(dtype, rows, in, N, group,
 * grid)), except:
 *   sums    [grid + 1] double (written)  per alpha, the sum over these rows
 *           and all N tokens of (X (Wq - W)^T)^2, not divided by anything
 *   s_table [grid + 1][in] float or NULL (written)  the centred scale
 *           vector of every alpha, rounded to float32 (the same on every
 *           slice: it depends on X only)
 * awq_search_finish combines the slices' sums:
 *   sums    [n_parts][grid + 1] double (read)  the slices' sums, in slice
 *           order; they are added in that order, so the result does not
 *           depend on which device or process produced which slice
 *   N, out  tokens, and rows of the whole layer (the sum of the slices' rows)
 *   s_table [grid + 1][in] float (read)  any slice's s_table
 *   err, best, s_best  as awq_search's outputs for the whole layer
 * A layer can be searched slice by slice on several devices: gather the
 * slices' sums (every device the same, in slice order) and finish anywhere.
 */
int awq_search_rows(const void* W, const void* X, int dtype,
                    int64_t rows, int64_t in, int64_t N,
                    const double* sx, int bits, int group, int sym, int grid,
                    void* workspace, size_t workspace_bytes,
                    double* sums, float* s_table,
                    int32_t* dev_status, awq_stream_t stream);

int awq_search_finish(const double* sums, int n_parts, int grid, int64_t N, int64_t out,
                      const float* s_table, int64_t in,
                      double* err, int32_t* best, float* s_best,
                      int32_t* dev_status, awq_stream_t stream);

/*
 * awq_sweep_summary - one row of a bit-width / group-size sweep
 * ["AWQ (activation-aware weight quantization)", "What the simulations
 * show": RTN beside AWQ at each setting, as relative output errors;
 * "GPTQ and AWQ weight quantisation", "Output MSE vs bit width"].
 *
 *   err    [grid + 1] double (read)  awq_search's per-alpha errors
 *   best   [1] int32 (read)          awq_search's kept index
 *   power  [1] double (read)         awq_output_power of the same W and X
 *   grid   the search's grid (1..4096)
 *   row    [5] double (written): the kept alpha's value on the grid
 *          (linspace(0, 1, grid + 1)[best]), RTN's error err[0] (alpha = 0,
 *          which is plain round-to-nearest), AWQ's error err[best], and the
 *          two relative errors err[0] / power and err[best] / power.  With
 *          best = -1 (no finite error) the alpha and AWQ entries are NaN.
 * All pointers are device memory; the call enqueues one small kernel.
 */
int awq_sweep_summary(const double* err, const int32_t* best, const double* power, int grid,
                      double* row, awq_stream_t stream);

/* Options for awq_search_ex; zero-initialise, then set what you need. */
typedef struct {
    awq_event_t ev_search_start;  /* recorded on `stream` right before the fused search kernel */
    awq_event_t ev_search_stop;   /* recorded right after it (both or neither) */
    int64_t wait_limit_ns;        /* bound of each device-side wait; 0 = 2 s */
    int test_timeout;             /* nonzero: the search kernel also waits on a barrier that
                                     nothing arrives at, so the bounded wait runs out and the
                                     call reports AWQ_ERR_TIMEOUT (tests of the error path) */
    uint32_t* diag;               /* NULL, or 4 device words, cleared by the call: when a wait
                                     runs out they receive {site, block, sequence, parity} of
                                     the first wait that gave up (site 0 = none) */
} awq_search_opts;

/* awq_search with options (opts may be NULL). */
int awq_search_ex(const void* W, const void* X, int dtype,
                  int64_t out, int64_t in, int64_t N,
                  const double* sx, int bits, int group, int sym, int grid,
                  void* workspace, size_t workspace_bytes,
                  double* err, int32_t* best, float* s_best,
                  int32_t* dev_status, awq_stream_t stream,
                  const awq_search_opts* opts);

/*
 * awq_quantize_pack - quantize W * s once and pack the codes.
 * ["AWQ vs GPTQ ...", "What lands on disk"; "GPTQ and AWQ weight
 *  quantisation", "Storage math"]
 *
 *   W        [out][in] of `dtype`       (read)
 *   s        [in] float                 column scales (e.g. s_best)
 *   qweight  [out][ceil(in*bits/32)] uint32 (written)  code i of a row sits
 *            at bit i*bits of the row's little-endian bit stream; high bits
 *            of the last word are zero
 *   scales   [out][in/group] float      (written) group step
 *   zeros    [out][in/group] uint8      (written) zero point
 * Codes are unsigned: symmetric codes are stored as q + 2^(b-1) with zero
 * 2^(b-1), so that every code decodes as scale * (u - zero).
 * Arithmetic is IEEE float32 with round-to-nearest on every operation and
 * round-half-to-even for the codes: t = w*s, scale = max(m/L, 1e-8) or
 * max((hi-lo)/maxq, 1e-8), code = round(t/scale) (+ zero, clamped).
 * Any group size dividing `in` is accepted.  A NaN or infinite product w*s
 * sets AWQ_ERR_NONFINITE; the codes, scale and zero of its group are then
 * unspecified (codes stay within [0, 2^b - 1]).
 */
int awq_quantize_pack(const void* W, int dtype, int64_t out, int64_t in,
                      const float* s, int bits, int group, int sym,
                      uint32_t* qweight, float* scales, uint8_t* zeros,
                      int32_t* dev_status, awq_stream_t stream);

/*
 * awq_clip_search - per-group clipping search at fixed scales.
 * ["AWQ (activation-aware weight quantization)", "Simplifications": the
 *  method also searches a clipping threshold per group, shrinking the max
 *  range to cut rounding error; "AWQ vs GPTQ ...", "AWQ: move the error away
 *  from what matters": a second search shrinks each group's clipping range
 *  when that lowers output error.]
 *
 * For every row r and group G of W * diag(s) and each factor
 *   c_i = 1 - i / n_grid,  i = 0 .. max_shrink_steps   (rounded to float32)
 * the group's range is scaled by c_i (symmetric: max|t|; asymmetric: the
 * min(min t, 0) and max(max t, 0) ends), the group is quantized with the
 * quantizer's clamps, and the group's own share of the row's output error
 *   e = sum_n (sum_{j in G} X[n, j] (Wq[r, j] - W[r, j]))^2
 * is formed.  clip[r][G] receives the first factor with the smallest share
 * (strict <; c_0 = 1, no clipping, is kept unless clipping lowers it).
 *
 *   W, X, dtype, out, in, N   as for awq_search; s [in] float (e.g. s_best)
 *   bits, group, sym          as for awq_quantize_pack; group in {32, 64, 128}
 *                             (others: AWQ_ERR_UNSUPPORTED)
 *   n_grid >= 1, 0 <= max_shrink_steps < n_grid, max_shrink_steps <= 11
 *   workspace, workspace_bytes >= awq_clip_search_workspace_bytes(in, N, group)
 *   clip   [out][in/group] float (written): the kept factors
 *   errs   [out][in/group][max_shrink_steps + 1] float (written) or NULL
 * The shares are formed as d^T H_G d with the group's Gram matrix
 * H_G = X_G^T X_G (fp32 sums in a fixed order), d = Wq - W in fp32.
 * Pass clip to awq_quantize_pack_clipped for the codes.
 */
size_t awq_clip_search_workspace_bytes(int64_t in, int64_t N, int group);

int awq_clip_search(const void* W, const void* X, int dtype,
                    int64_t out, int64_t in, int64_t N, const float* s,
                    int bits, int group, int sym, int n_grid, int max_shrink_steps,
                    void* workspace, size_t workspace_bytes,
                    float* clip, float* errs, int32_t* dev_status, awq_stream_t stream);

/*
 * awq_quantize_pack_clipped - awq_quantize_pack with each group's range
 * scaled by clip[out][in/group] (float, e.g. from awq_clip_search) before its
 * step and zero point are formed: symmetric m = fl32(c * max|t|), asymmetric
 * lo = fl32(c * min(min t, 0)), hi = fl32(c * max(max t, 0)); values beyond
 * the shrunk range take the end codes.  Same outputs and errors as
 * awq_quantize_pack.
 */
int awq_quantize_pack_clipped(const void* W, int dtype, int64_t out, int64_t in,
                              const float* s, int bits, int group, int sym,
                              const float* clip, uint32_t* qweight, float* scales,
                              uint8_t* zeros, int32_t* dev_status, awq_stream_t stream);

/*
 * awq_gptq - GPTQ's rounding after AWQ's scaling.
 * ["AWQ vs GPTQ ...", "GPTQ: compensate the error you just made" (the
 *  column-by-column rounding with error compensation through the Cholesky
 *  factor of the inverse Hessian, dampening, lazily fitted group parameters)
 *  and "Failure modes and combining the two" (AWQ's scaling, then GPTQ's
 *  rounding).]
 *
 * Rounds W * diag(s) against the inputs X / s (s NULL: plain GPTQ):
 *   H = 2 (X/s)^T (X/s) + damp * mean(diag) * I,  U^T U = H^-1 (U upper),
 *   for each column i in natural order: at a group's first column its step
 *   and zero point are fitted on the weights as corrected so far; column i
 *   is rounded with awq_quantize_pack's quantizer; its error divided by
 *   U[i][i] is taken off the later columns through row i of U.
 *
 *   W, X, dtype, out, in, N   as for awq_search
 *   s       [in] float or NULL
 *   bits, group, sym          as for awq_quantize_pack; group in {32, 64, 128}
 *   damp    >= 0 (the pages' default is 0.01)
 *   workspace, workspace_bytes >= awq_gptq_workspace_bytes(out, in, N)
 *           (about 8 in^2 + 5 out*in + 4 N*in bytes)
 *   qweight, scales, zeros   as awq_quantize_pack writes them (the codes of
 *           W * s; decode as scale * (code - zero), then divide by s)
 * Arithmetic is fp32 (the Hessian, its factors and the running weights), so
 * codes can differ from a float64 evaluation where a corrected weight sits
 * within rounding of a decision boundary.  A Hessian that is not positive
 * definite after dampening sets AWQ_ERR_NONFINITE.
 */
size_t awq_gptq_workspace_bytes(int64_t out, int64_t in, int64_t N);

int awq_gptq(const void* W, const void* X, int dtype,
             int64_t out, int64_t in, int64_t N, const float* s,
             int bits, int group, int sym, double damp,
             void* workspace, size_t workspace_bytes,
             uint32_t* qweight, float* scales, uint8_t* zeros,
             int32_t* dev_status, awq_stream_t stream);

/*
 * awq_export_checkpoint - the tensors a quantized checkpoint stores for one
 * linear layer, from awq_quantize_pack's outputs.
 * ["AWQ vs GPTQ ...", "What lands on disk": qweight int32 words packing
 *  4-bit values; FP16 scales, one per group per output channel, shape
 *  [in/g, out]; qzeros, packed 4-bit zero points, one per group per output
 *  channel.  "Sizes are easy to predict": 4 bits plus a 16-bit scale and a
 *  4-bit zero per 128 weights is about 4.16 bits per weight.]
 *
 *   qweight, scales, zeros   awq_quantize_pack's outputs (read), out x in
 *                            layer, `bits` in {2, 4, 8}, in % (32/bits) == 0
 *   qweight_t [in*bits/32][out] uint32 (written): word (k, o) holds the codes
 *            of inputs (32/bits)k .. (32/bits)k + 32/bits - 1 of output o,
 *            the lowest input in the lowest bits
 *   scales_h  [in/group][out] IEEE binary16 (written): the float32 steps
 *            rounded to nearest (ties to even); a step beyond the binary16
 *            range (or NaN) sets AWQ_ERR_NONFINITE
 *   qzeros    [in/group][ceil(out*bits/32)] uint32 (written): word (g, w)
 *            holds the zero points of outputs (32/bits)w .. of group g, the
 *            lowest output in the lowest bits, stored as they are (no offset)
 * The pages leave the packing axis and the nibble order to the format; these
 * are this library's.  The weights are those of W * diag(s): the scales s
 * (s_best) are folded into whatever produces the layer's input.  Every code
 * decodes as scale * (code - zero).
 */
int awq_export_checkpoint(const uint32_t* qweight, const float* scales, const uint8_t* zeros,
                          int64_t out, int64_t in, int bits, int group,
                          uint32_t* qweight_t, void* scales_h, uint32_t* qzeros,
                          int32_t* dev_status, awq_stream_t stream);

/*
 * awq_search_noalloc - awq_search for callers that cannot allocate device
 * memory.  (The method itself has no counterpart of this: it is a calling
 * convenience of this library.)
 *
 * Some callers have no way to obtain scratch memory: a plug-in whose host
 * application owns every device allocation and offers no workspace hook,
 * real-time code that forbids cudaMalloc because it can synchronise the
 * device and take unbounded time, or code that must not grow its memory
 * footprint after start-up.  This entry point needs no workspace argument:
 * its scratch is a fixed device array inside the library of
 * AWQ_NOALLOC_SCRATCH_BYTES (32 MiB), reserved on every GPU that loads this
 * part of the library and held until the process exits.  The call makes no
 * cudaMalloc, cudaFree or other allocating call.
 *
 * Arguments, outputs, numerics and errors are those of awq_search, except:
 *  - the sizes must satisfy awq_search_workspace_min_bytes(dtype, out, in, N,
 *    group, grid) <= AWQ_NOALLOC_SCRATCH_BYTES; larger problems return
 *    AWQ_ERR_UNSUPPORTED before anything is enqueued (use awq_search with
 *    your own workspace for those);
 *  - the first call on each device looks up the device address of the
 *    array (with that device current) and caches it; make that first call
 *    before any stream capture begins;
 *  - every call on a device shares the one array, which keeps the previous
 *    call's contents (the call clears what must start at zero).  Calls whose
 *    work overlaps on the GPU (for example on two streams without ordering
 *    between them) race on the array and give wrong results: order them on
 *    one stream or with events.
 */
#define AWQ_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

int awq_search_noalloc(const void* W, const void* X, int dtype,
                       int64_t out, int64_t in, int64_t N,
                       const double* sx, int bits, int group, int sym, int grid,
                       double* err, int32_t* best, float* s_best,
                       int32_t* dev_status, awq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* AWQ_H */
