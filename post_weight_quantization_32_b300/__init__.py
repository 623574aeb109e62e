"""AWQ per-layer activation-aware scale search on one B300 (sm_103a).

A thin ctypes binding over ``libawq.so`` (C ABI in include/awq.h).  Every
step of the computation runs in the library's CUDA kernels; this module only
checks tensor shapes and dtypes, allocates outputs and workspace with
PyTorch, and passes pointers and the current CUDA stream.  Importing it
fails loudly if the library has not been built.

Entry points (same names as the C ABI):

* ``awq_channel_stats(X)`` -> s_X (float64, [in])
* ``awq_search(W, X, bits, group, sym, grid)`` -> (err float64 [grid+1],
  best int32 [1], s_best float32 [in])
* ``awq_quantize_pack(W, s, bits, group, sym)`` -> (qweight, scales, zeros):
  qweight int32 [out, ceil(in*bits/32)] holding the uint32 words (view it
  as unsigned), scales float32 [out, in/group], zeros uint8 [out, in/group]
* ``awq_search_noalloc(W, X, bits, group, sym, grid)`` -> as ``awq_search``,
  but the library's fixed scratch array (``NOALLOC_SCRATCH_BYTES``) stands
  in for the workspace, for callers that cannot allocate device memory
* ``awq_output_power(W, X)`` -> mean((X W^T)^2) (float64 [1]), the
  denominator of the relative output error; ``awq_sweep(W, X, settings)``
  runs the search over (bits, group) settings and reports RTN beside AWQ,
  absolute and relative (each row from ``awq_sweep_summary`` on the device)
* ``awq_clip_search(W, X, s, bits, group, sym)`` -> (clip factors
  [out, in/group], shares or None); ``awq_quantize_pack_clipped(W, s, clip,
  ...)`` packs at those factors
* ``awq_gptq(W, X, s, bits, group, sym, damp)`` -> (qweight, scales, zeros)
  from GPTQ's rounding of W * diag(s) against X / s
* ``awq_export_checkpoint(qweight, scales, zeros, in, bits, group)`` ->
  (qweight [in*b/32, out], fp16 scales [in/g, out], packed zeros)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

__all__ = [
    "AWQError", "SearchOpts", "lib", "awq_channel_stats", "awq_search",
    "awq_search_workspace_bytes", "awq_search_workspace_min_bytes", "awq_quantize_pack",
    "new_status", "check_status", "STATUS",
    "DTYPE", "awq_search_noalloc", "NOALLOC_SCRATCH_BYTES", "awq_output_power", "awq_sweep",
    "awq_export_checkpoint", "awq_clip_search", "awq_clip_search_workspace_bytes",
    "awq_quantize_pack_clipped", "awq_gptq", "awq_gptq_workspace_bytes", "awq_sweep_summary",
    "awq_search_rows", "awq_search_finish", "gather_row_sums",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libawq.so")

DTYPE = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
STATUS = {0: "AWQ_OK", 1: "AWQ_ERR_INVALID_ARG", 2: "AWQ_ERR_UNSUPPORTED", 3: "AWQ_ERR_NONFINITE",
          4: "AWQ_ERR_TIMEOUT", 5: "AWQ_ERR_CUDA"}

EXPORTS = ("awq_status_string", "awq_channel_stats", "awq_search_workspace_bytes",
           "awq_search_workspace_min_bytes", "awq_search",
           "awq_search_ex", "awq_quantize_pack", "awq_search_noalloc", "awq_output_power",
           "awq_export_checkpoint", "awq_clip_search", "awq_clip_search_workspace_bytes",
           "awq_quantize_pack_clipped", "awq_gptq", "awq_gptq_workspace_bytes",
           "awq_sweep_summary", "awq_search_rows", "awq_search_finish",
           "awq_output_power_workspace_bytes")

# Size of the library's fixed scratch array used by awq_search_noalloc.
NOALLOC_SCRATCH_BYTES = 32 << 20


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError("libawq.so is not built (run `python post_weight_quantization_32_b300/build.py`)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.awq_status_string.restype = ctypes.c_char_p
    L.awq_status_string.argtypes = [i32]
    L.awq_channel_stats.restype = i32
    L.awq_channel_stats.argtypes = [vp, i32, i64, i64, vp, vp, vp]
    L.awq_search_workspace_bytes.restype = sz
    L.awq_search_workspace_bytes.argtypes = [i32, i64, i64, i64, i32, i32]
    L.awq_search_rows.restype = i32
    L.awq_search_rows.argtypes = [vp, vp, i32, i64, i64, i64, vp, i32, i32, i32, i32, vp, sz, vp,
                                  vp, vp, vp]
    L.awq_search_finish.restype = i32
    L.awq_search_finish.argtypes = [vp, i32, i32, i64, i64, vp, i64, vp, vp, vp, vp, vp]
    L.awq_output_power_workspace_bytes.restype = sz
    L.awq_output_power_workspace_bytes.argtypes = [i32, i64, i64, i64]
    L.awq_sweep_summary.restype = i32
    L.awq_sweep_summary.argtypes = [vp, vp, vp, i32, vp, vp]
    L.awq_search_workspace_min_bytes.restype = sz
    L.awq_search_workspace_min_bytes.argtypes = [i32, i64, i64, i64, i32, i32]
    L.awq_search.restype = i32
    L.awq_search.argtypes = [vp, vp, i32, i64, i64, i64, vp, i32, i32, i32, i32, vp, sz, vp, vp, vp,
                             vp, vp]
    L.awq_search_ex.restype = i32
    L.awq_search_ex.argtypes = L.awq_search.argtypes + [vp]
    L.awq_quantize_pack.restype = i32
    L.awq_quantize_pack.argtypes = [vp, i32, i64, i64, vp, i32, i32, i32, vp, vp, vp, vp, vp]
    L.awq_output_power.restype = i32
    L.awq_output_power.argtypes = [vp, vp, i32, i64, i64, i64, vp, sz, vp, vp, vp]
    L.awq_export_checkpoint.restype = i32
    L.awq_export_checkpoint.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp, vp, vp, vp, vp]
    L.awq_clip_search_workspace_bytes.restype = sz
    L.awq_clip_search_workspace_bytes.argtypes = [i64, i64, i32]
    L.awq_clip_search.restype = i32
    L.awq_clip_search.argtypes = [vp, vp, i32, i64, i64, i64, vp, i32, i32, i32, i32, i32, vp, sz,
                                  vp, vp, vp, vp]
    L.awq_quantize_pack_clipped.restype = i32
    L.awq_quantize_pack_clipped.argtypes = [vp, i32, i64, i64, vp, i32, i32, i32, vp, vp, vp, vp,
                                            vp, vp]
    L.awq_gptq_workspace_bytes.restype = sz
    L.awq_gptq_workspace_bytes.argtypes = [i64, i64, i64]
    L.awq_gptq.restype = i32
    L.awq_gptq.argtypes = [vp, vp, i32, i64, i64, i64, vp, i32, i32, i32, ctypes.c_double, vp, sz,
                           vp, vp, vp, vp, vp]
    L.awq_search_noalloc.restype = i32
    L.awq_search_noalloc.argtypes = [vp, vp, i32, i64, i64, i64, vp, i32, i32, i32, i32, vp, vp, vp,
                                     vp, vp]
    return L


lib = _load()


class AWQError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (%s)" % (where, STATUS.get(code, code),
                                          lib.awq_status_string(int(code)).decode()))


class SearchOpts(ctypes.Structure):
    """awq_search_opts of the C ABI."""
    _fields_ = [("ev_search_start", ctypes.c_void_p), ("ev_search_stop", ctypes.c_void_p),
                ("wait_limit_ns", ctypes.c_int64), ("test_timeout", ctypes.c_int),
                ("diag", ctypes.c_void_p)]


def _env_opts() -> Optional["SearchOpts"]:
    """Search options from the environment: AWQ_WAIT_LIMIT_MS bounds every
    device-side wait of the search kernel (the library's default is 2000 ms).
    None when it is not set."""
    v = os.environ.get("AWQ_WAIT_LIMIT_MS")
    if not v:
        return None
    o = SearchOpts()
    o.wait_limit_ns = int(float(v) * 1e6)
    return o


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(code: int, where: str) -> None:
    if code != 0:
        raise AWQError(code, where)


def _need(t: torch.Tensor, name: str, ndim: int) -> None:
    if not t.is_cuda or not t.is_contiguous() or t.dim() != ndim:
        raise ValueError("%s must be a contiguous %d-D CUDA tensor" % (name, ndim))
    # the library launches on the current device (and awq_search_noalloc uses
    # that device's scratch array): tensors elsewhere would be read through
    # pointers of another device
    if t.device.index != torch.cuda.current_device():
        raise ValueError("%s is on %s but the current CUDA device is %d: call under "
                         "torch.cuda.device(%s)" % (name, t.device, torch.cuda.current_device(),
                                                    t.device))


def new_status(device=None) -> torch.Tensor:
    """A zeroed device status word."""
    return torch.zeros(1, dtype=torch.int32, device=device or "cuda")


def check_status(dev_status: torch.Tensor, where: str = "device") -> None:
    """Synchronise and raise if a kernel reported an error."""
    code = int(dev_status.item())
    if code != 0:
        raise AWQError(code, where)


def awq_channel_stats(X: torch.Tensor, sx: Optional[torch.Tensor] = None, stream=None,
                      dev_status: Optional[torch.Tensor] = None) -> torch.Tensor:
    _need(X, "X", 2)
    N, n_in = X.shape
    if sx is None:
        sx = torch.empty(n_in, dtype=torch.float64, device=X.device)
    _check(lib.awq_channel_stats(_ptr(X), DTYPE[X.dtype], N, n_in, _ptr(sx), _ptr(dev_status),
                                 _stream(stream)), "awq_channel_stats")
    return sx


def awq_search_workspace_bytes(dtype: torch.dtype, out: int, n_in: int, N: int, group: int,
                               grid: int) -> int:
    """Workspace bytes for the search's fastest path (see the C header)."""
    return int(lib.awq_search_workspace_bytes(DTYPE[dtype], out, n_in, N, group, grid))


def awq_search_workspace_min_bytes(dtype: torch.dtype, out: int, n_in: int, N: int, group: int,
                                   grid: int) -> int:
    """The smallest workspace the search accepts."""
    return int(lib.awq_search_workspace_min_bytes(DTYPE[dtype], out, n_in, N, group, grid))


def awq_search(W: torch.Tensor, X: torch.Tensor, bits: int = 4, group: Optional[int] = None,
               sym: bool = True, grid: int = 20, sx: Optional[torch.Tensor] = None,
               workspace: Optional[torch.Tensor] = None, out_tensors=None, stream=None,
               dev_status: Optional[torch.Tensor] = None, opts: Optional[SearchOpts] = None,
               check: bool = True) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Alpha-grid search; returns (err [grid+1] f64, best [1] i32, s_best [in] f32).

    ``group=None`` means one group per row (group = in).  With ``check``
    the call synchronises and raises on a device-reported error.
    """
    _need(W, "W", 2)
    _need(X, "X", 2)
    if W.dtype != X.dtype or W.shape[1] != X.shape[1]:
        raise ValueError("W and X must share dtype and the input dimension")
    out, n_in = W.shape
    N = X.shape[0]
    g = n_in if group is None else int(group)
    if workspace is None:
        need = awq_search_workspace_bytes(W.dtype, out, n_in, N, g, grid)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=W.device)
    if out_tensors is None:
        err = torch.empty(grid + 1, dtype=torch.float64, device=W.device)
        best = torch.empty(1, dtype=torch.int32, device=W.device)
        s_best = torch.empty(n_in, dtype=torch.float32, device=W.device)
    else:
        err, best, s_best = out_tensors
    st = dev_status if dev_status is not None else new_status(W.device)
    args = (_ptr(W), _ptr(X), DTYPE[W.dtype], out, n_in, N, _ptr(sx), bits, g, 1 if sym else 0,
            grid, _ptr(workspace), workspace.numel(), _ptr(err), _ptr(best), _ptr(s_best), _ptr(st),
            _stream(stream))
    if opts is None:
        opts = _env_opts()
    if opts is None:
        code = lib.awq_search(*args)
    else:
        code = lib.awq_search_ex(*args, ctypes.byref(opts))
    _check(code, "awq_search")
    if check:
        check_status(st, "awq_search")
    return err, best, s_best


def awq_search_rows(W_rows: torch.Tensor, X: torch.Tensor, bits: int = 4,
                    group: Optional[int] = None, sym: bool = True, grid: int = 20,
                    sx: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream=None, dev_status: Optional[torch.Tensor] = None, check: bool = True):
    """The search on a slice of a layer's output rows; returns (sums [grid+1]
    f64: per alpha the unnormalised sum of squared output errors over these
    rows, s_table [grid+1, in] f32: every alpha's scale vector)."""
    _need(W_rows, "W_rows", 2)
    _need(X, "X", 2)
    if W_rows.dtype != X.dtype or W_rows.shape[1] != X.shape[1]:
        raise ValueError("W_rows and X must share dtype and the input dimension")
    rows, n_in = W_rows.shape
    N = X.shape[0]
    g = n_in if group is None else int(group)
    if workspace is None:
        need = awq_search_workspace_bytes(W_rows.dtype, rows, n_in, N, g, grid)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=W_rows.device)
    sums = torch.empty(grid + 1, dtype=torch.float64, device=W_rows.device)
    s_table = torch.empty((grid + 1, n_in), dtype=torch.float32, device=W_rows.device)
    st = dev_status if dev_status is not None else new_status(W_rows.device)
    _check(lib.awq_search_rows(_ptr(W_rows), _ptr(X), DTYPE[W_rows.dtype], rows, n_in, N, _ptr(sx),
                               bits, g, 1 if sym else 0, grid, _ptr(workspace), workspace.numel(),
                               _ptr(sums), _ptr(s_table), _ptr(st), _stream(stream)),
           "awq_search_rows")
    if check:
        check_status(st, "awq_search_rows")
    return sums, s_table


def awq_search_finish(sums: torch.Tensor, N: int, out: int, s_table: torch.Tensor,
                      stream=None, dev_status: Optional[torch.Tensor] = None, check: bool = True):
    """Whole-layer (err, best, s_best) from the slices' sums ([n_parts,
    grid+1] f64, slice order), the layer's N and out, and any slice's s_table."""
    _need(sums, "sums", 2)
    _need(s_table, "s_table", 2)
    n_parts, n_alpha = sums.shape
    n_in = s_table.shape[1]
    err = torch.empty(n_alpha, dtype=torch.float64, device=sums.device)
    best = torch.empty(1, dtype=torch.int32, device=sums.device)
    s_best = torch.empty(n_in, dtype=torch.float32, device=sums.device)
    st = dev_status if dev_status is not None else new_status(sums.device)
    _check(lib.awq_search_finish(_ptr(sums), n_parts, n_alpha - 1, N, out, _ptr(s_table), n_in,
                                 _ptr(err), _ptr(best), _ptr(s_best), _ptr(st), _stream(stream)),
           "awq_search_finish")
    if check:
        check_status(st, "awq_search_finish")
    return err, best, s_best


def gather_row_sums(sums: torch.Tensor, group=None) -> torch.Tensor:
    """Every rank's row-slice sums ([grid+1] f64), stacked in rank order on
    every rank ([world, grid+1]): the input of awq_search_finish when rank r
    searched slice r.  Only moves data (torch.distributed.all_gather); the
    sums are added in awq_search_finish, in rank order, so every rank gets
    the same answer."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(sums) for _ in range(world)]
    dist.all_gather(parts, sums.contiguous(), group=group)
    return torch.stack(parts, 0)


def awq_quantize_pack(W: torch.Tensor, s: torch.Tensor, bits: int = 4, group: Optional[int] = None,
                      sym: bool = True, out_tensors=None, stream=None,
                      dev_status: Optional[torch.Tensor] = None, check: bool = True):
    """Quantize W * s per group and pack; returns (qweight, scales, zeros)."""
    _need(W, "W", 2)
    _need(s, "s", 1)
    if s.dtype != torch.float32 or s.numel() != W.shape[1]:
        raise ValueError("s must be float32 with one entry per input column")
    out, n_in = W.shape
    g = n_in if group is None else int(group)
    if out_tensors is None:
        nwords = (n_in * bits + 31) // 32
        qweight = torch.empty((out, nwords), dtype=torch.int32, device=W.device)
        scales = torch.empty((out, max(n_in // g, 1)), dtype=torch.float32, device=W.device)
        zeros = torch.empty((out, max(n_in // g, 1)), dtype=torch.uint8, device=W.device)
    else:
        qweight, scales, zeros = out_tensors
    st = dev_status if dev_status is not None else new_status(W.device)
    _check(lib.awq_quantize_pack(_ptr(W), DTYPE[W.dtype], out, n_in, _ptr(s), bits, g,
                                 1 if sym else 0, _ptr(qweight), _ptr(scales), _ptr(zeros), _ptr(st),
                                 _stream(stream)), "awq_quantize_pack")
    if check:
        check_status(st, "awq_quantize_pack")
    return qweight, scales, zeros


def awq_search_noalloc(W: torch.Tensor, X: torch.Tensor, bits: int = 4, group: Optional[int] = None,
                       sym: bool = True, grid: int = 20, sx: Optional[torch.Tensor] = None,
                       out_tensors=None, stream=None, dev_status: Optional[torch.Tensor] = None,
                       check: bool = True) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """``awq_search`` without a workspace: the library's fixed scratch array
    is used instead, so the C call allocates nothing.  Output tensors are
    still the caller's (pass ``out_tensors`` to reuse preallocated ones).
    Problems whose smallest workspace (``awq_search_workspace_min_bytes``)
    would exceed ``NOALLOC_SCRATCH_BYTES`` raise AWQError with
    AWQ_ERR_UNSUPPORTED."""
    _need(W, "W", 2)
    _need(X, "X", 2)
    if W.dtype != X.dtype or W.shape[1] != X.shape[1]:
        raise ValueError("W and X must share dtype and the input dimension")
    out, n_in = W.shape
    N = X.shape[0]
    g = n_in if group is None else int(group)
    if out_tensors is None:
        err = torch.empty(grid + 1, dtype=torch.float64, device=W.device)
        best = torch.empty(1, dtype=torch.int32, device=W.device)
        s_best = torch.empty(n_in, dtype=torch.float32, device=W.device)
    else:
        err, best, s_best = out_tensors
    st = dev_status if dev_status is not None else new_status(W.device)
    _check(lib.awq_search_noalloc(_ptr(W), _ptr(X), DTYPE[W.dtype], out, n_in, N, _ptr(sx), bits, g,
                                  1 if sym else 0, grid, _ptr(err), _ptr(best), _ptr(s_best),
                                  _ptr(st), _stream(stream)), "awq_search_noalloc")
    if check:
        check_status(st, "awq_search_noalloc")
    return err, best, s_best


def awq_output_power(W: torch.Tensor, X: torch.Tensor, workspace: Optional[torch.Tensor] = None,
                     out: Optional[torch.Tensor] = None, stream=None,
                     dev_status: Optional[torch.Tensor] = None, check: bool = True) -> torch.Tensor:
    """mean((X W^T)^2) as a [1] float64 tensor: the denominator of the
    relative output error err / power (err from ``awq_search``)."""
    _need(W, "W", 2)
    _need(X, "X", 2)
    if W.dtype != X.dtype or W.shape[1] != X.shape[1]:
        raise ValueError("W and X must share dtype and the input dimension")
    n_out, n_in = W.shape
    N = X.shape[0]
    if workspace is None:
        need = int(lib.awq_output_power_workspace_bytes(DTYPE[W.dtype], n_out, n_in, N))
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=W.device)
    power = out if out is not None else torch.empty(1, dtype=torch.float64, device=W.device)
    st = dev_status if dev_status is not None else new_status(W.device)
    _check(lib.awq_output_power(_ptr(W), _ptr(X), DTYPE[W.dtype], n_out, n_in, N, _ptr(workspace),
                                workspace.numel(), _ptr(power), _ptr(st), _stream(stream)),
           "awq_output_power")
    if check:
        check_status(st, "awq_output_power")
    return power


def awq_sweep_summary(err: torch.Tensor, best: torch.Tensor, power: torch.Tensor, grid: int,
                      stream=None) -> torch.Tensor:
    """One sweep row from a search's (err, best) and the layer's output power:
    float64 [5] = (alpha value, RTN error, AWQ error, RTN relative error, AWQ
    relative error), computed on the device."""
    row = torch.empty(5, dtype=torch.float64, device=err.device)
    _check(lib.awq_sweep_summary(_ptr(err), _ptr(best), _ptr(power), grid, _ptr(row),
                                 _stream(stream)), "awq_sweep_summary")
    return row


def awq_sweep(W: torch.Tensor, X: torch.Tensor, settings, sym: bool = True, grid: int = 20):
    """The search at several (bits, group) settings of one layer, with RTN
    (alpha = 0, the first grid point) beside AWQ and both errors also relative
    to mean((X W^T)^2).  ``group=None`` means one group per row.  Returns one
    dict per setting: bits, group, best (alpha index), alpha, err_rtn,
    err_awq, rel_rtn, rel_awq."""
    power = awq_output_power(W, X)
    rows = []
    for bits, group in settings:
        err, best, _ = awq_search(W, X, bits=bits, group=group, sym=sym, grid=grid)
        r = awq_sweep_summary(err, best, power, grid).cpu().tolist()
        rows.append(dict(bits=bits, group=group, best=int(best.item()), alpha=r[0], err_rtn=r[1],
                         err_awq=r[2], rel_rtn=r[3], rel_awq=r[4]))
    return rows


def awq_export_checkpoint(qweight: torch.Tensor, scales: torch.Tensor, zeros: torch.Tensor,
                          n_in: int, bits: int = 4, group: Optional[int] = None, stream=None,
                          dev_status: Optional[torch.Tensor] = None, check: bool = True):
    """Checkpoint tensors of one layer from ``awq_quantize_pack``'s outputs:
    (qweight [in*b/32, out] int32, scales [in/g, out] float16, qzeros
    [in/g, ceil(out*b/32)] int32); see awq_export_checkpoint in awq.h for the
    bit layout."""
    _need(qweight, "qweight", 2)
    n_out = qweight.shape[0]
    g = n_in if group is None else int(group)
    dev = qweight.device
    qw_t = torch.empty((n_in * bits // 32, n_out), dtype=torch.int32, device=dev)
    sc_h = torch.empty((n_in // g, n_out), dtype=torch.float16, device=dev)
    qz = torch.empty((n_in // g, (n_out * bits + 31) // 32), dtype=torch.int32, device=dev)
    st = dev_status if dev_status is not None else new_status(dev)
    _check(lib.awq_export_checkpoint(_ptr(qweight), _ptr(scales), _ptr(zeros), n_out, n_in, bits,
                                     g, _ptr(qw_t), _ptr(sc_h), _ptr(qz), _ptr(st),
                                     _stream(stream)), "awq_export_checkpoint")
    if check:
        check_status(st, "awq_export_checkpoint")
    return qw_t, sc_h, qz


def awq_clip_search_workspace_bytes(n_in: int, N: int, group: int) -> int:
    return int(lib.awq_clip_search_workspace_bytes(n_in, N, group))


def awq_clip_search(W: torch.Tensor, X: torch.Tensor, s: torch.Tensor, bits: int = 4,
                    group: int = 128, sym: bool = True, n_grid: int = 20,
                    max_shrink_steps: int = 10, want_errs: bool = False, stream=None,
                    dev_status: Optional[torch.Tensor] = None, check: bool = True):
    """Per-group clipping search at scales s; returns (clip [out, in/g] f32,
    errs [out, in/g, steps + 1] f32 or None)."""
    _need(W, "W", 2)
    _need(X, "X", 2)
    if W.dtype != X.dtype or W.shape[1] != X.shape[1]:
        raise ValueError("W and X must share dtype and the input dimension")
    n_out, n_in = W.shape
    N = X.shape[0]
    need = awq_clip_search_workspace_bytes(n_in, N, group)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=W.device)
    clip = torch.empty((n_out, n_in // group), dtype=torch.float32, device=W.device)
    errs = (torch.empty((n_out, n_in // group, max_shrink_steps + 1), dtype=torch.float32,
                        device=W.device) if want_errs else None)
    st = dev_status if dev_status is not None else new_status(W.device)
    _check(lib.awq_clip_search(_ptr(W), _ptr(X), DTYPE[W.dtype], n_out, n_in, N, _ptr(s), bits,
                               group, 1 if sym else 0, n_grid, max_shrink_steps, _ptr(ws),
                               ws.numel(), _ptr(clip), _ptr(errs), _ptr(st), _stream(stream)),
           "awq_clip_search")
    if check:
        check_status(st, "awq_clip_search")
    return clip, errs


def awq_quantize_pack_clipped(W: torch.Tensor, s: torch.Tensor, clip: torch.Tensor, bits: int = 4,
                              group: int = 128, sym: bool = True, stream=None,
                              dev_status: Optional[torch.Tensor] = None, check: bool = True):
    """``awq_quantize_pack`` with each group's range scaled by clip [out, in/g]."""
    _need(W, "W", 2)
    n_out, n_in = W.shape
    nwords = (n_in * bits + 31) // 32
    dev = W.device
    qw = torch.empty((n_out, nwords), dtype=torch.int32, device=dev)
    sc = torch.empty((n_out, n_in // group), dtype=torch.float32, device=dev)
    z = torch.empty((n_out, n_in // group), dtype=torch.uint8, device=dev)
    st = dev_status if dev_status is not None else new_status(dev)
    _check(lib.awq_quantize_pack_clipped(_ptr(W), DTYPE[W.dtype], n_out, n_in, _ptr(s), bits,
                                         group, 1 if sym else 0, _ptr(clip), _ptr(qw), _ptr(sc),
                                         _ptr(z), _ptr(st), _stream(stream)),
           "awq_quantize_pack_clipped")
    if check:
        check_status(st, "awq_quantize_pack_clipped")
    return qw, sc, z


def awq_gptq_workspace_bytes(n_out: int, n_in: int, N: int) -> int:
    return int(lib.awq_gptq_workspace_bytes(n_out, n_in, N))


def awq_gptq(W: torch.Tensor, X: torch.Tensor, s: Optional[torch.Tensor] = None, bits: int = 4,
             group: int = 128, sym: bool = True, damp: float = 0.01, stream=None,
             dev_status: Optional[torch.Tensor] = None, check: bool = True):
    """GPTQ's rounding of W * diag(s) against X / s (s None: plain GPTQ);
    returns (qweight, scales, zeros) laid out as ``awq_quantize_pack``'s."""
    _need(W, "W", 2)
    _need(X, "X", 2)
    if W.dtype != X.dtype or W.shape[1] != X.shape[1]:
        raise ValueError("W and X must share dtype and the input dimension")
    n_out, n_in = W.shape
    N = X.shape[0]
    dev = W.device
    ws = torch.empty(max(awq_gptq_workspace_bytes(n_out, n_in, N), 256), dtype=torch.uint8,
                     device=dev)
    qw = torch.empty((n_out, (n_in * bits + 31) // 32), dtype=torch.int32, device=dev)
    sc = torch.empty((n_out, n_in // group), dtype=torch.float32, device=dev)
    z = torch.empty((n_out, n_in // group), dtype=torch.uint8, device=dev)
    st = dev_status if dev_status is not None else new_status(dev)
    _check(lib.awq_gptq(_ptr(W), _ptr(X), DTYPE[W.dtype], n_out, n_in, N, _ptr(s), bits, group,
                        1 if sym else 0, float(damp), _ptr(ws), ws.numel(), _ptr(qw), _ptr(sc),
                        _ptr(z), _ptr(st), _stream(stream)), "awq_gptq")
    if check:
        check_status(st, "awq_gptq")
    return qw, sc, z
