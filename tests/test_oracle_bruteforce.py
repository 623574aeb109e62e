"""Exact brute force on tiny layers, independent of the oracle's code.

For every weight the nearest allowed integer level is found by enumerating
the candidates and comparing distances exactly in rationals
(``fractions.Fraction``); every float32 rounding the quantizer specifies is
done by an explicit correctly-rounded float32 search; the output error is
summed exactly over tokens, rows and columns.  The oracle must agree:
codes, scales and zero points bit for bit, the float64 error within 1e-12
relative, and the same argmin over the alpha grid.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import awq_oracle as O

F32_EPS = np.float32(1e-8)


def round_f32(fr: Fraction) -> np.float32:
    """Correctly rounded (ties to even) float32 of an exact rational."""
    x = np.float32(float(fr))
    cands = {x, np.nextafter(x, np.float32(-np.inf)), np.nextafter(x, np.float32(np.inf))}
    best = None
    for c in cands:
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - fr)
        key = (d, int(np.array(c, dtype=np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return np.float32(best[1])


def nearest_int_even(r: Fraction) -> int:
    """Nearest integer to r, ties to the even one, by enumeration."""
    lo = math.floor(r)
    cands = [lo - 1, lo, lo + 1, lo + 2]
    return min(cands, key=lambda k: (abs(r - k), k % 2))


def brute_quantize(t32, bits, group, sym):
    """Returns codes (ints), scales (float32), zeros (ints), w_hat (float32)."""
    out, n_in = t32.shape
    ng = n_in // group
    q = np.zeros((out, n_in), dtype=np.int64)
    w_hat = np.zeros((out, n_in), dtype=np.float32)
    scales = np.zeros((out, ng), dtype=np.float32)
    zeros = np.zeros((out, ng), dtype=np.int64)
    near_ties = 0
    for r in range(out):
        for gi in range(ng):
            cols = range(gi * group, (gi + 1) * group)
            tv = [Fraction(float(t32[r, j])) for j in cols]
            if sym:
                L = 2 ** (bits - 1) - 1
                m = max(abs(v) for v in tv)
                scale = max(round_f32(m / L), F32_EPS)
                z = 0
                allowed = range(-L - 1, L + 1)
            else:
                maxq = 2 ** bits - 1
                lo = min(min(tv), Fraction(0))
                hi = max(max(tv), Fraction(0))
                d = round_f32(hi - lo)
                scale = max(round_f32(Fraction(float(d)) / maxq), F32_EPS)
                z = nearest_int_even(Fraction(float(round_f32(-lo / Fraction(float(scale))))))
                allowed = range(0, maxq + 1)
            S = Fraction(float(scale))
            scales[r, gi] = scale
            zeros[r, gi] = z
            for j, v in zip(cols, tv):
                r_exact = v / S
                r32 = Fraction(float(round_f32(r_exact)))
                # nearest integer of the float32 quotient, plus the zero point,
                # then the nearest allowed code (= clamping)
                k = nearest_int_even(r32) + z
                code = min(allowed, key=lambda c: abs(c - k))
                k_exact = nearest_int_even(r_exact) + z
                if min(allowed, key=lambda c: abs(c - k_exact)) != code:
                    near_ties += 1
                q[r, j] = code
                w_hat[r, j] = round_f32(S * (code - z))
    return q, scales, zeros, w_hat, near_ties


def brute_err(X, W32, w_hat, s32):
    """Exact mean of (X (Wq - W)^T)^2 with Wq = w_hat / s."""
    N, n_in = X.shape
    out = W32.shape[0]
    Xf = [[Fraction(float(X[n, j])) for j in range(n_in)] for n in range(N)]
    D = [[Fraction(float(w_hat[r, j])) / Fraction(float(s32[j])) - Fraction(float(W32[r, j]))
          for j in range(n_in)] for r in range(out)]
    tot = Fraction(0)
    for n in range(N):
        for r in range(out):
            y = sum(Xf[n][j] * D[r][j] for j in range(n_in))
            tot += y * y
    return tot / (N * out)


CASES = list(itertools.product(
    [(2, 4, 2), (3, 8, 3), (4, 6, 1), (1, 8, 2)],   # (out, in, N)
    [2, 3, 4],                                     # bits
    [True, False],                                 # sym
))


@pytest.mark.parametrize("shape,bits,sym", CASES)
def test_bruteforce_tiny_layer(shape, bits, sym):
    out, n_in, N = shape
    seed = out * 1000 + n_in * 100 + N * 10 + bits + (7 if sym else 0)
    rng = np.random.default_rng(seed)
    W32 = (rng.standard_normal((out, n_in)) * 0.05).astype(np.float32)
    X = rng.standard_normal((N, n_in)) * rng.uniform(0.2, 30.0, size=n_in)
    for group in sorted({2, n_in // 2 if n_in % 4 == 0 else 2, n_in}):
        if n_in % group:
            continue
        grid = 5
        res = O.awq_search(W32, X, bits=bits, group=group, grid=grid, sym=sym)
        exact_errs = []
        for k in range(grid + 1):
            s32 = res.s32[k]
            t32 = W32 * s32[None, :]
            q, scales, zeros, w_hat, _ = brute_quantize(t32, bits, group, sym)
            _, gq = O.fake_quant(W32, s32, bits, group, sym)
            codes = gq.q.astype(np.int64)
            assert np.array_equal(codes, q)
            assert np.array_equal(gq.scale, scales)
            assert np.array_equal(gq.zero.astype(np.int64), zeros)
            assert np.array_equal(gq.w_hat, w_hat)
            e = brute_err(X, W32, w_hat, s32)
            exact_errs.append(e)
            assert abs(res.errs[k] - float(e)) <= 1e-12 * float(e) + 1e-300
        best_exact = min(range(grid + 1), key=lambda k: (exact_errs[k], k))
        assert res.best == best_exact


def test_bruteforce_scales_from_salience():
    """The grid's scale vectors recomputed with plain Python floats."""
    rng = np.random.default_rng(11)
    X = rng.standard_normal((3, 6)) * rng.uniform(0.1, 40.0, size=6)
    res = O.awq_search(np.zeros((1, 6), np.float32), X, bits=4, group=6, grid=4, sym=True)
    for k in range(5):
        a = k / 4
        sx = [sum(abs(float(X[n, j])) for n in range(3)) / 3 + 1e-8 for j in range(6)]
        s = [v ** a for v in sx]
        c = math.sqrt(max(s) * min(s))
        want = np.array([x / c for x in s], dtype=np.float64)
        assert np.allclose(res.s32[k].astype(np.float64), want, rtol=1e-7, atol=0)


def test_near_tie_rounding_follows_float32_quotient():
    """A code whose exact quotient sits within an ulp of k + 1/2 follows the
    float32 quotient, as specified; count how often that can matter."""
    rng = np.random.default_rng(12)
    t32 = (rng.standard_normal((4, 16)) * 0.05).astype(np.float32)
    q, *_, near = brute_quantize(t32, 4, 8, True)
    assert near <= 1
    assert np.array_equal(O.quantize_groups(t32, 4, 8, True).q.astype(np.int64), q)
