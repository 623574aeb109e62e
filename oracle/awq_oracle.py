"""Plain CPU oracle for AWQ's per-layer activation-aware scale search.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's ``smoke()`` check and
the benchmark's CPU-baseline leg may import this module.  The product path
(the CUDA library and its binding) never calls it, and it calls nothing of
the product: the two share no code.

What it computes is the method as the pages state it, step by step, in
float64 numpy (the group quantizer in float32, see below):

* s_X[j] = mean_n |X[n, j]| + 1e-8
      [AWQ guide, "How it works" step 1 and "The code, line by line"]
* for alpha in linspace(0, 1, grid + 1):
      s = s_X ** alpha;  s = s / sqrt(max(s) * min(s))
      [AWQ guide, "How it works" step 2 and "The code, line by line"]
      Wq = Q(W * s) / s                       (columns scaled, rounded, unscaled)
      err = mean((X @ Wq.T - X @ W.T) ** 2)
      keep alpha when err < best (strict, first wins)
      [AWQ guide, "Source code"; "AWQ vs GPTQ ...", section "AWQ: move the
       error away from what matters"]
* Q is round-to-nearest per group of ``group`` input columns of each row:
    - symmetric: scale = max|w| / (2^(b-1) - 1), clamped at 1e-8,
      q = clamp(round(w / scale), -2^(b-1), 2^(b-1) - 1), w_hat = q * scale
      ["GPTQ and AWQ weight quantisation", "Per-group symmetric int4 (RTN)"
       and "Output MSE vs bit width"]
    - asymmetric: lo = min(min w, 0), hi = max(max w, 0),
      scale = max((hi - lo) / (2^b - 1), 1e-8), zero = round(-lo / scale),
      q = clamp(round(w / scale) + zero, 0, 2^b - 1), w_hat = scale * (q - zero)
      ["AWQ vs GPTQ Quantization Architectures Compared", "The shared
       problem: one layer, sixteen levels" and the group_params / rtn code in
       "GPTQ: compensate the error you just made"]
  round() is round-half-to-even (numpy's and torch's rounding).

Readings taken where the pages leave a step open (each is listed with its
reason in the design notes):

* The quantizer runs in IEEE float32 with round-to-nearest on every
  operation: t = fl32(w * s32), scale = fl32(m / L) (asym:
  fl32(fl32(hi - lo) / maxq)), r = fl32(t / scale), zero = round(fl32(-lo /
  scale)).  s32 = float32(s) is the scale vector that parity is pinned to.
  Everything else (statistics, powers, centring, the error) is float64.
* The asymmetric code is round(t / scale) + zero, as written, not
  round(t / scale + zero).
* If every alpha's error is NaN the search has no answer (the pages' loop
  would return None); ``awq_search`` reports ``best = -1``.

Storage convention (the pages leave packing open: "What lands on disk"):
codes are b-bit unsigned, symmetric codes stored offset-binary
u = q + 2^(b-1) with zero = 2^(b-1); code i of a row sits at bit i*b of that
row's little-endian uint32 bitstream; scales float32 [out][in/g]; zeros
uint8 [out][in/g].

Beyond the search itself, each from the page and section it cites:
output_power / sweep (relative output error, bit-width and group-size
sweeps), clip_search / quantize_pack_clipped (the per-group clipping
search), export_checkpoint / dequantize_checkpoint (the checkpoint
tensors) and gptq (GPTQ's rounding after AWQ's scaling).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "channel_salience", "alpha_grid", "centred_scales", "quantize_groups",
    "quantize_groups_f64", "fake_quant", "output_mse", "awq_search", "SearchResult",
    "stored_codes", "pack_bits", "unpack_bits", "quantize_pack", "rtn_fake_quant",
    "output_power", "sweep", "Checkpoint", "export_checkpoint", "dequantize_checkpoint",
    "clip_factors", "quantize_groups_clipped", "ClipResult", "clip_search",
    "quantize_pack_clipped", "GptqResult", "inverse_hessian_factor", "gptq",
]

_EPS_SALIENCE = 1e-8          # added to the mean |X| [AWQ guide, "The code, line by line"]
_EPS_SCALE = np.float32(1e-8)  # lower clamp of the group step (notebook RTN, group_params)


def channel_salience(X: np.ndarray) -> np.ndarray:
    """s_X[j] = mean over tokens of |X[:, j]|, plus 1e-8, in float64.

    [AWQ guide, "How it works" step 1; "The code, line by line", first bullet]
    """
    X64 = np.asarray(X, dtype=np.float64)
    return np.abs(X64).mean(0) + _EPS_SALIENCE


def alpha_grid(grid: int) -> np.ndarray:
    """grid + 1 exponents evenly spaced on [0, 1], both ends included.

    [AWQ guide, "The code, line by line": with grid = 20 that is 21 values]
    """
    return np.linspace(0.0, 1.0, grid + 1)


def centred_scales(sx: np.ndarray, alpha: float):
    """s = s_X ** alpha, divided by sqrt(max(s) * min(s)).

    Returns the float64 vector and its float32 rounding s32 (the vector the
    float32 quantizer multiplies by).
    [AWQ guide, "The code, line by line", bullets on the grid and on centring]
    """
    s = np.asarray(sx, dtype=np.float64) ** float(alpha)
    s = s / np.sqrt(s.max() * s.min())
    return s, s.astype(np.float32)


@dataclasses.dataclass
class GroupQuant:
    q: np.ndarray        # integer codes as float32 (sym: signed; asym: 0..2^b-1)
    scale: np.ndarray    # float32 [out, in/g]
    zero: np.ndarray     # float32 [out, in/g] (sym: zeros)
    w_hat: np.ndarray    # float32 [out, in], reconstructed (still scaled) weights


def quantize_groups(t: np.ndarray, bits: int, group: int, sym: bool) -> GroupQuant:
    """Round-to-nearest of each group of ``group`` consecutive columns, in float32.

    Symmetric: ["GPTQ and AWQ weight quantisation", rtn_nbit in "Output MSE vs
    bit width"; the int4 form in "Per-group symmetric int4 (RTN)"].
    Asymmetric: ["AWQ vs GPTQ ...", group_params and rtn, with the fake_quant
    loop over column groups in "AWQ: move the error away from what matters"].
    """
    t = np.asarray(t, dtype=np.float32)
    out, n_in = t.shape
    if n_in % group != 0:
        raise ValueError("in must be a multiple of group")
    tg = t.reshape(out, n_in // group, group)
    if sym:
        L = np.float32(2 ** (bits - 1) - 1)
        m = np.abs(tg).max(axis=-1)
        scale = np.maximum(m / L, _EPS_SCALE)
        q = np.clip(np.round(tg / scale[..., None]), -L - np.float32(1), L)
        w_hat = q * scale[..., None]
        zero = np.zeros_like(scale)
    else:
        maxq = np.float32(2 ** bits - 1)
        lo = np.minimum(tg.min(axis=-1), np.float32(0))
        hi = np.maximum(tg.max(axis=-1), np.float32(0))
        scale = np.maximum((hi - lo) / maxq, _EPS_SCALE)
        zero = np.round(-lo / scale)
        q = np.clip(np.round(tg / scale[..., None]) + zero[..., None], np.float32(0), maxq)
        w_hat = scale[..., None] * (q - zero[..., None])
    assert q.dtype == np.float32 and scale.dtype == np.float32 and w_hat.dtype == np.float32
    return GroupQuant(q.reshape(out, n_in), scale, zero.astype(np.float32), w_hat.reshape(out, n_in))


def quantize_groups_f64(t: np.ndarray, bits: int, group: int, sym: bool) -> GroupQuant:
    """The same quantizer carried out in float64 (a diagnostic, not the spec).

    Used only to count how many codes an all-float64 evaluation would round
    the other way; such codes sit at near-ties of t / scale.
    """
    t = np.asarray(t, dtype=np.float64)
    out, n_in = t.shape
    tg = t.reshape(out, n_in // group, group)
    if sym:
        L = float(2 ** (bits - 1) - 1)
        scale = np.maximum(np.abs(tg).max(axis=-1) / L, 1e-8)
        q = np.clip(np.round(tg / scale[..., None]), -L - 1, L)
        w_hat = q * scale[..., None]
        zero = np.zeros_like(scale)
    else:
        maxq = float(2 ** bits - 1)
        lo = np.minimum(tg.min(axis=-1), 0.0)
        hi = np.maximum(tg.max(axis=-1), 0.0)
        scale = np.maximum((hi - lo) / maxq, 1e-8)
        zero = np.round(-lo / scale)
        q = np.clip(np.round(tg / scale[..., None]) + zero[..., None], 0, maxq)
        w_hat = scale[..., None] * (q - zero[..., None])
    return GroupQuant(q.reshape(out, n_in), scale, zero, w_hat.reshape(out, n_in))


def fake_quant(W32: np.ndarray, s32: np.ndarray, bits: int, group: int, sym: bool):
    """Wq = Q(W * s) / s: scale columns by s, round, divide by s again.

    [AWQ guide, "The code, line by line", the Wq bullet; "AWQ vs GPTQ ...",
    awq_scales: fake_quant(W * s, group) / s]
    Returns (Wq in float64, the GroupQuant of W * s).
    """
    W32 = np.asarray(W32, dtype=np.float32)
    s32 = np.asarray(s32, dtype=np.float32)
    t = W32 * s32[None, :]                       # fl32(w * s)
    gq = quantize_groups(t, bits, group, sym)
    Wq = gq.w_hat.astype(np.float64) / s32.astype(np.float64)[None, :]
    return Wq, gq


def rtn_fake_quant(W32: np.ndarray, bits: int, group: int, sym: bool) -> np.ndarray:
    """Plain RTN of W (no scaling), float64 result.  The alpha = 0 baseline."""
    return quantize_groups(np.asarray(W32, np.float32), bits, group, sym).w_hat.astype(np.float64)


def output_mse(X64: np.ndarray, Wq: np.ndarray, ref: np.ndarray) -> float:
    """mean((X @ Wq.T - ref) ** 2) with ref = X @ W.T, in float64.

    [AWQ guide, "Source code" (err line); "AWQ vs GPTQ ...", awq_scales]
    """
    return float(np.mean((X64 @ Wq.T - ref) ** 2))


@dataclasses.dataclass
class SearchResult:
    alphas: np.ndarray     # float64 [n_alpha]
    errs: np.ndarray       # float64 [n_alpha]
    best: int              # index of the kept alpha, -1 if none
    sx: np.ndarray         # float64 [in]
    s32: np.ndarray        # float32 [n_alpha, in], the centred scales per alpha
    s32_best: Optional[np.ndarray]


def awq_search(W, X, bits: int = 4, group: Optional[int] = None, grid: int = 20,
               sym: bool = True, alpha_index=None) -> SearchResult:
    """The per-layer alpha-grid search, literally as the pages give it.

    W: (out, in) real values (any float dtype, used exactly as float32);
    X: (N, in) calibration inputs.  ``group=None`` means one group per row.
    ``alpha_index`` (optional) restricts the evaluated grid points; the
    others get err = NaN and the argmin runs over the evaluated ones only.

    [AWQ guide, "Source code" and "The code, line by line"]
    """
    W32 = np.asarray(W, dtype=np.float32)
    X64 = np.asarray(X, dtype=np.float64)
    n_in = W32.shape[1]
    g = n_in if group is None else int(group)
    sx = channel_salience(X64)
    ref = X64 @ W32.astype(np.float64).T
    alphas = alpha_grid(grid)
    errs = np.full(alphas.shape, np.nan)
    s32_all = np.empty((alphas.size, n_in), dtype=np.float32)
    best, best_err = -1, np.inf
    for k, a in enumerate(alphas):
        _, s32 = centred_scales(sx, a)
        s32_all[k] = s32
        if alpha_index is not None and k not in alpha_index:
            continue
        Wq, _ = fake_quant(W32, s32, bits, g, sym)
        err = output_mse(X64, Wq, ref)
        errs[k] = err
        if err < best_err:
            best, best_err = k, err
    return SearchResult(alphas, errs, best, sx, s32_all, s32_all[best] if best >= 0 else None)


def output_power(W, X) -> float:
    """mean((X @ W.T) ** 2) in float64: the size of the layer's exact output.

    The relative output error of the pages is ||h W - h Wq||^2 / ||h W||^2
    [AWQ guide, "What the simulations show"]; err (a mean over the same
    N * out entries) divided by this mean is that ratio.
    """
    X64 = np.asarray(X, dtype=np.float64)
    W64 = np.asarray(W, dtype=np.float32).astype(np.float64)
    return float(np.mean((X64 @ W64.T) ** 2))


def sweep(W, X, settings, sym: bool = True, grid: int = 20):
    """The search at several (bits, group) settings of one layer, RTN (the
    alpha = 0 point of the grid) beside AWQ, both also relative to
    output_power.  [AWQ guide, "What the simulations show" and "Try this";
    "GPTQ and AWQ weight quantisation", "Output MSE vs bit width" and its
    group-size exercise]
    """
    power = output_power(W, X)
    rows = []
    for bits, group in settings:
        res = awq_search(W, X, bits=bits, group=group, grid=grid, sym=sym)
        b = res.best
        rows.append(dict(bits=bits, group=group, best=b, alpha=float(res.alphas[b]),
                         errs=res.errs, err_rtn=float(res.errs[0]), err_awq=float(res.errs[b]),
                         rel_rtn=float(res.errs[0]) / power, rel_awq=float(res.errs[b]) / power))
    return rows


def stored_codes(q: np.ndarray, bits: int, sym: bool) -> np.ndarray:
    """Unsigned b-bit storage codes: symmetric codes offset by 2^(b-1).

    ["AWQ vs GPTQ ...", "The shared problem": symmetric variants fix the zero
    point at the middle level]
    """
    qi = np.asarray(q).astype(np.int64)
    if sym:
        qi = qi + (1 << (bits - 1))
    assert qi.min(initial=0) >= 0 and qi.max(initial=0) < (1 << bits)
    return qi.astype(np.uint32)


def pack_bits(u: np.ndarray, bits: int) -> np.ndarray:
    """Code i of each row at bit offset i*bits of the row's little-endian
    uint32 stream; ceil(in*bits/32) words per row, unused high bits zero."""
    u = np.asarray(u, dtype=np.uint32)
    out, n = u.shape
    nwords = -(-(n * bits) // 32)
    words = np.zeros((out, nwords), dtype=np.uint32)
    shifts = np.arange(bits, dtype=np.uint32)
    weights = np.uint64(1) << np.arange(32, dtype=np.uint64)
    step = 512
    for r0 in range(0, out, step):   # row chunks bound the temporary bit array
        blk = u[r0:r0 + step]
        bitarr = ((blk[..., None] >> shifts) & np.uint32(1)).astype(np.uint8)
        bitarr = bitarr.reshape(blk.shape[0], n * bits)
        bitarr = np.pad(bitarr, ((0, 0), (0, nwords * 32 - n * bits)))
        bitarr = bitarr.reshape(blk.shape[0], nwords, 32).astype(np.uint64)
        words[r0:r0 + step] = (bitarr * weights).sum(-1).astype(np.uint32)
    return words


def unpack_bits(words: np.ndarray, bits: int, n: int) -> np.ndarray:
    """Inverse of ``pack_bits``: the first n codes of each row."""
    words = np.asarray(words, dtype=np.uint32)
    out, nwords = words.shape
    bitarr = ((words[..., None] >> np.arange(32, dtype=np.uint32)) & np.uint32(1)).astype(np.uint32)
    bitarr = bitarr.reshape(out, nwords * 32)[:, : n * bits].reshape(out, n, bits)
    return (bitarr << np.arange(bits, dtype=np.uint32)).sum(-1).astype(np.uint32)


def quantize_pack(W, s32, bits: int, group: int, sym: bool):
    """Final quantization at the chosen scales, then packing.

    Returns (qweight uint32 [out, ceil(in*b/32)], scales float32 [out, in/g],
    zeros uint8 [out, in/g]).  ["AWQ vs GPTQ ...", "What lands on disk";
    "GPTQ and AWQ weight quantisation", "Storage math"]
    """
    W32 = np.asarray(W, dtype=np.float32)
    t = W32 * np.asarray(s32, dtype=np.float32)[None, :]
    gq = quantize_groups(t, bits, group, sym)
    u = stored_codes(gq.q, bits, sym)
    if sym:
        zeros = np.full(gq.scale.shape, 1 << (bits - 1), dtype=np.uint8)
    else:
        zeros = gq.zero.astype(np.uint8)
    return pack_bits(u, bits), gq.scale.copy(), zeros


@dataclasses.dataclass
class Checkpoint:
    qweight: np.ndarray   # uint32 [in * b / 32, out]
    scales: np.ndarray    # float16 [in / g, out]
    qzeros: np.ndarray    # uint32 [in / g, out * b / 32]


def export_checkpoint(qweight, scales, zeros, n_in: int, bits: int) -> Checkpoint:
    """The checkpoint tensors of one quantized layer, from quantize_pack's
    outputs.  ["AWQ vs GPTQ ...", "What lands on disk": qweight int32 words
    packing 4-bit values, FP16 scales one per group per output channel of
    shape [in/g, out], qzeros packed 4-bit zero points one per group per
    output channel.]  The pages leave the packing axis and the nibble order
    open; taken here: qweight packs 32/b consecutive input channels of one
    output channel per word, qzeros 32/b consecutive output channels of one
    group per word, lowest index in the lowest bits; the zero points are
    stored as they are (no offset); scales are the float32 steps rounded to
    float16 (nearest, ties to even).
    """
    if 32 % bits != 0:
        raise ValueError("bits must divide 32")
    per = 32 // bits
    if n_in % per != 0:
        raise ValueError("in must be a multiple of 32 / bits")
    u = unpack_bits(qweight, bits, n_in)               # [out, in] codes
    # word k of output o: inputs per*k .. per*k + per - 1, lowest in the lowest bits
    qw = np.ascontiguousarray(pack_bits(u, bits).T)    # [in / per, out]
    sc = np.asarray(scales, dtype=np.float32).T.astype(np.float16)
    qz = pack_bits(np.ascontiguousarray(np.asarray(zeros, dtype=np.uint32).T), bits)
    return Checkpoint(qw, sc, qz)


def dequantize_checkpoint(ck: Checkpoint, n_out: int, n_in: int, bits: int, group: int):
    """W_hat[o, i] = scale * (code - zero) from the checkpoint tensors, float64
    [out, in] (of W * diag(s): the scales s are folded elsewhere)."""
    per = 32 // bits
    codes = unpack_bits(ck.qweight.T.copy(), bits, per * ck.qweight.shape[0])  # [out, in]
    zeros = unpack_bits(ck.qzeros, bits, n_out)                                # [in/g, out]
    scale = ck.scales.astype(np.float64)                                       # [in/g, out]
    gi = np.arange(n_in) // group
    return scale[gi, :].T * (codes[:, :n_in].astype(np.float64) - zeros[gi, :].T.astype(np.float64))


# --------------------------------------------------------------------------
# Per-group clipping search at fixed scales
# --------------------------------------------------------------------------

def clip_factors(n_grid: int = 20, max_shrink: float = 0.5) -> np.ndarray:
    """The shrink factors tried for each group's range: 1, 1 - 1/n_grid, ...,
    down to 1 - max_shrink, as float32.  c = 1 (no clipping) comes first, so
    with a strict comparison clipping is kept only when it lowers the error.

    The pages give the step in words only ("searches a clipping threshold
    per group, shrinking the max range to cut rounding error", AWQ guide,
    "Simplifications"; "a second search then shrinks each group's clipping
    range a little when that lowers output error", comparison page, "AWQ:
    move the error away from what matters"); the grid is this library's
    reading.
    """
    k = int(round(max_shrink * n_grid))
    return np.array([1.0 - i / n_grid for i in range(k + 1)], dtype=np.float32)


def quantize_groups_clipped(t: np.ndarray, bits: int, group: int, sym: bool,
                            c: np.ndarray) -> GroupQuant:
    """The float32 group quantizer with each group's range scaled by its
    factor c[row, group] (float32): symmetric m = fl32(c * max|t|); asymmetric
    lo = fl32(c * min(min t, 0)), hi = fl32(c * max(max t, 0)).  Values
    beyond the shrunk range take the end codes (the clamps of the quantizer).
    With c = 1 this is quantize_groups exactly.
    """
    t = np.asarray(t, dtype=np.float32)
    out, n_in = t.shape
    ng = n_in // group
    tg = t.reshape(out, ng, group)
    c = np.asarray(c, dtype=np.float32).reshape(out, ng)
    if sym:
        L = np.float32((1 << (bits - 1)) - 1)
        m = (c * np.abs(tg).max(-1)).astype(np.float32)
        scale = np.maximum((m / L).astype(np.float32), _EPS_SCALE)
        q = np.clip(np.round((tg / scale[..., None]).astype(np.float32)), -L - 1, L)
        zero = np.zeros_like(scale)
        w_hat = (q * scale[..., None]).astype(np.float32)
    else:
        maxq = np.float32((1 << bits) - 1)
        lo = (c * np.minimum(tg.min(-1), np.float32(0))).astype(np.float32)
        hi = (c * np.maximum(tg.max(-1), np.float32(0))).astype(np.float32)
        scale = np.maximum(((hi - lo).astype(np.float32) / maxq).astype(np.float32), _EPS_SCALE)
        zero = np.round((-lo / scale).astype(np.float32))
        q = np.clip(np.round((tg / scale[..., None]).astype(np.float32)) + zero[..., None], 0, maxq)
        w_hat = (scale[..., None] * (q - zero[..., None])).astype(np.float32)
    return GroupQuant(q.reshape(out, n_in), scale, zero, w_hat.reshape(out, n_in))


@dataclasses.dataclass
class ClipResult:
    factors: np.ndarray   # float32 [n_c]
    errs: np.ndarray      # float64 [out, in/g, n_c]: each group's share of its row's output error
    best: np.ndarray      # int [out, in/g]: index of the kept factor


def clip_search(W, X, s32, bits: int, group: int, sym: bool, n_grid: int = 20,
                max_shrink: float = 0.5) -> ClipResult:
    """For each row r and group G of W * s (s fixed, e.g. the kept AWQ
    scales) and each shrink factor c, the group's own share of the row's
    output error, sum_n (sum_{j in G} X[n, j] * (Wq[r, j] - W[r, j]))^2 with
    Wq = Q_c(W * s) / s, in float64; the kept factor is the first with the
    smallest share (strict <).  The shares of different groups of a row do
    not add up to the row's error (cross terms), which is why each group is
    judged on its own share.
    """
    W32 = np.asarray(W, dtype=np.float32)
    X64 = np.asarray(X, dtype=np.float64)
    s32 = np.asarray(s32, dtype=np.float32)
    out, n_in = W32.shape
    ng = n_in // group
    t = W32 * s32[None, :]
    cs = clip_factors(n_grid, max_shrink)
    errs = np.empty((out, ng, cs.size))
    for i, c in enumerate(cs):
        gq = quantize_groups_clipped(t, bits, group, sym, np.full((out, ng), c, np.float32))
        dW = gq.w_hat.astype(np.float64) / s32.astype(np.float64)[None, :] - W32.astype(np.float64)
        for g in range(ng):
            sl = slice(g * group, (g + 1) * group)
            errs[:, g, i] = np.sum((X64[:, sl] @ dW[:, sl].T) ** 2, axis=0)
    best = np.zeros((out, ng), dtype=np.int64)
    best_err = np.full((out, ng), np.inf)
    for i in range(cs.size):
        better = errs[:, :, i] < best_err
        best[better] = i
        best_err[better] = errs[:, :, i][better]
    return ClipResult(cs, errs, best)


def quantize_pack_clipped(W, s32, bits: int, group: int, sym: bool, clip):
    """quantize_pack with each group's range scaled by clip[row, group]
    (float32) first, as the clipping search keeps it."""
    W32 = np.asarray(W, dtype=np.float32)
    t = W32 * np.asarray(s32, dtype=np.float32)[None, :]
    gq = quantize_groups_clipped(t, bits, group, sym, clip)
    u = stored_codes(gq.q, bits, sym)
    if sym:
        zeros = np.full(gq.scale.shape, 1 << (bits - 1), dtype=np.uint8)
    else:
        zeros = gq.zero.astype(np.uint8)
    return pack_bits(u, bits), gq.scale.copy(), zeros


# --------------------------------------------------------------------------
# GPTQ rounding after AWQ scaling
# --------------------------------------------------------------------------

@dataclasses.dataclass
class GptqResult:
    q: np.ndarray        # codes [out, in] (signed for the symmetric quantizer, as quantize_groups)
    scale: np.ndarray    # float32 [out, in/g], fitted on the corrected weights at each group start
    zero: np.ndarray     # float32 [out, in/g]
    w_hat: np.ndarray    # float64 [out, in]: dequantized weights of W * s
    Wq: np.ndarray       # float64 [out, in]: w_hat / s


def inverse_hessian_factor(Xs, damp: float = 0.01) -> np.ndarray:
    """The upper-triangular U with U^T U = H^-1, H = 2 Xs^T Xs plus `damp`
    times the mean of its diagonal on the diagonal.  ["AWQ vs GPTQ ...",
    "GPTQ: compensate the error you just made": H = 2 X X^T for one row of
    weights, dampening by 1% of the mean diagonal, rows of H^-1 read from one
    Cholesky factorisation.]  Xs: (N, in) inputs of the layer, float64."""
    H = 2.0 * (Xs.T @ Xs)
    H[np.diag_indices_from(H)] += damp * np.mean(np.diag(H))
    Hinv = np.linalg.inv(H)
    return np.linalg.cholesky(Hinv).T


def gptq(W, X, bits: int, group: int, sym: bool, s32=None, damp: float = 0.01) -> GptqResult:
    """GPTQ's rounding of W * diag(s) against the inputs X / s (AWQ's scaling
    first, then GPTQ's choice of integers: "AWQ vs GPTQ ...", "Failure modes
    and combining the two"; without s, plain GPTQ).

    Columns are rounded in their natural order (no act-order).  At the first
    column of each group the group's step and zero point are fitted on the
    weights as they stand then, corrections from earlier columns included;
    each column is rounded with the float32 quantizer of this module
    (quantize_groups' arithmetic on fl32 of the corrected weight); the
    rounding error, divided by U[i, i], is spread over the later columns of
    every row through row i of U.  The running weights are float64.
    ["AWQ vs GPTQ ...", "GPTQ: compensate the error you just made" and the
    production details after it]
    """
    W32 = np.asarray(W, dtype=np.float32)
    out, n_in = W32.shape
    s32 = np.ones(n_in, np.float32) if s32 is None else np.asarray(s32, dtype=np.float32)
    Ws = (W32 * s32[None, :]).astype(np.float64)          # W * s, as the quantizer sees it
    Xs = np.asarray(X, dtype=np.float64) / s32.astype(np.float64)[None, :]
    U = inverse_hessian_factor(Xs, damp)
    ng = n_in // group
    q = np.zeros((out, n_in))
    w_hat = np.zeros((out, n_in))
    scale = np.zeros((out, ng), np.float32)
    zero = np.zeros((out, ng), np.float32)
    for i in range(n_in):
        g = i // group
        if i % group == 0:
            gq = quantize_groups(Ws[:, i:i + group].astype(np.float32), bits, group, sym)
            scale[:, g], zero[:, g] = gq.scale[:, 0], gq.zero[:, 0]
        col = Ws[:, i].astype(np.float32)
        sc = scale[:, g]
        if sym:
            L = np.float32((1 << (bits - 1)) - 1)
            qi = np.clip(np.round((col / sc).astype(np.float32)), -L - 1, L)
            wh = (qi * sc).astype(np.float32)
        else:
            maxq = np.float32((1 << bits) - 1)
            z = zero[:, g]
            qi = np.clip(np.round((col / sc).astype(np.float32)) + z, 0, maxq)
            wh = (sc * (qi - z)).astype(np.float32)
        q[:, i] = qi
        w_hat[:, i] = wh
        err = (Ws[:, i] - wh.astype(np.float64)) / U[i, i]
        Ws[:, i + 1:] -= np.outer(err, U[i, i + 1:])
    return GptqResult(q, scale, zero, w_hat, w_hat / s32.astype(np.float64)[None, :])
