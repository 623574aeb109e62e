"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests retypes the oracle's formulas to compare it with itself:
they check printed values of the pages' worked example, closed forms,
invariants the pages state, and exact (rational) brute force on tiny layers
(the latter lives in test_oracle_bruteforce.py).
"""
import os

import numpy as np
import pytest

from oracle import awq_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = line.split("=", 1)
            vals[k.strip()] = [float(x) for x in v.split()]
    return vals


def _tol(printed):
    """Half a unit in the last digit the page printed."""
    s = repr(printed)
    if "." not in s:
        return 0.5
    return 0.5 * 10.0 ** -(len(s.split(".")[1]))


WE = _read_golden("worked_example_two_channel.txt")


def _close_printed(actual, printed_list):
    for a, p in zip(np.ravel(actual), printed_list):
        assert abs(a - p) <= _tol(p) + 1e-12, (a, p)


# --------------------------------------------------------------------------
# Worked example ("AWQ > Worked Example: Tracing AWQ Through a Two-Channel Layer")
# --------------------------------------------------------------------------

def test_worked_example_quantizer_with_page_scales():
    """The page's own normalisation s = (abar / max abar) ** alpha."""
    w = np.array([WE["w"]], dtype=np.float32)
    s = np.array(WE["s_page"], dtype=np.float32)
    bits = int(WE["bits"][0])
    Wq, gq = O.fake_quant(w, s, bits, group=2, sym=True)
    _close_printed(w * s, WE["w_scaled"])
    _close_printed(gq.scale, WE["step_awq"])
    assert list(gq.q.ravel()) == WE["codes_awq"]
    _close_printed(Wq, WE["w_eff_awq"])
    abar = np.array(WE["abar"])
    _close_printed(np.abs(w[0] - Wq[0]) * abar, WE["err_awq"])


def test_worked_example_rtn():
    w = np.array([WE["w"]], dtype=np.float32)
    bits = int(WE["bits"][0])
    gq = O.quantize_groups(w, bits, group=2, sym=True)
    _close_printed(gq.scale, WE["step_rtn"])
    assert list(gq.q.ravel()) == WE["codes_rtn"]
    _close_printed(gq.w_hat, WE["w_rtn"])
    abar = np.array(WE["abar"])
    _close_printed(np.abs(w[0] - gq.w_hat[0]) * abar, WE["err_rtn"])


def test_worked_example_through_search():
    """Full search path with one calibration token X = abar (so mean|X| = abar).

    The search centres s by sqrt(max*min) instead of the page's max: both are
    alpha-independent factors, so codes, effective weights and the output
    error are the page's.  grid = 2 puts alpha = 0.5 on the grid.
    """
    w = np.array([WE["w"]], dtype=np.float32)
    X = np.array([WE["abar"]], dtype=np.float64)
    res = O.awq_search(w, X, bits=3, group=2, grid=2, sym=True)
    assert res.alphas[1] == WE["alpha"][0]
    # output error |X (Wq - W)^T| = sum over channels of the page's weighted errors
    _close_printed(np.sqrt(res.errs[1]), [sum(WE["err_awq"])])
    _close_printed(np.sqrt(res.errs[0]), [sum(WE["err_rtn"])])
    Wq, gq = O.fake_quant(w, res.s32[1], 3, 2, True)
    assert list(gq.q.ravel()) == WE["codes_awq"]
    _close_printed(Wq, WE["w_eff_awq"])
    # the search keeps the smallest error; AWQ at alpha=0.5 beats RTN here
    assert res.errs[res.best] <= res.errs[1] < res.errs[0]


# --------------------------------------------------------------------------
# Closed forms and invariants stated on the pages
# --------------------------------------------------------------------------

def test_salience_closed_form():
    X = np.array([[1.0, -2.0, 0.0], [3.0, 4.0, 0.0]])
    sx = O.channel_salience(X)
    assert sx[0] == 2.0 + 1e-8 and sx[1] == 3.0 + 1e-8
    assert sx[2] == 1e-8          # always-zero channel keeps a nonzero scale


def test_alpha_grid():
    a = O.alpha_grid(20)
    assert a.size == 21 and a[0] == 0.0 and a[-1] == 1.0
    assert np.allclose(np.diff(a), 0.05, atol=1e-15)
    a41 = O.alpha_grid(40)
    assert a41.size == 41 and np.allclose(np.diff(a41), 0.025, atol=1e-15)


def test_centring_is_geometric():
    rng = np.random.default_rng(1)
    sx = rng.uniform(0.3, 80.0, size=257)
    for a in (0.0, 0.25, 0.5, 1.0):
        s, s32 = O.centred_scales(sx, a)
        assert abs(s.max() * s.min() - 1.0) < 1e-14
        # monotone in s_X: larger salience never gets a smaller scale
        order = np.argsort(sx)
        assert np.all(np.diff(s[order]) >= 0)
        assert s32.dtype == np.float32


def test_alpha_zero_is_plain_rtn():
    """alpha = 0 gives s = 1 exactly, so the search starts from plain RTN."""
    rng = np.random.default_rng(2)
    W = (rng.standard_normal((16, 64)) * 0.02).astype(np.float32)
    X = rng.standard_normal((8, 64))
    sx = O.channel_salience(X)
    s, s32 = O.centred_scales(sx, 0.0)
    assert np.all(s == 1.0) and np.all(s32 == np.float32(1.0))
    for sym in (True, False):
        Wq, _ = O.fake_quant(W, s32, 4, 32, sym)
        assert np.array_equal(Wq, O.rtn_fake_quant(W, 4, 32, sym))
        res = O.awq_search(W, X, bits=4, group=32, grid=20, sym=sym)
        ref = X @ W.astype(np.float64).T
        assert res.errs[0] == O.output_mse(X, O.rtn_fake_quant(W, 4, 32, sym), ref)
        assert res.errs[res.best] <= res.errs[0]


def test_flat_salience_reduces_to_rtn():
    """Equal mean |X| in every channel: s = 1 for every alpha, all errors tie,
    and the strict comparison keeps the first alpha (plain RTN)."""
    rng = np.random.default_rng(3)
    W = (rng.standard_normal((8, 32)) * 0.02).astype(np.float32)
    X = np.where(rng.random((5, 32)) < 0.5, -1.0, 1.0) * 0.37
    res = O.awq_search(W, X, bits=3, group=16, grid=20, sym=False)
    assert np.all(res.s32 == np.float32(1.0))
    assert np.all(res.errs == res.errs[0])
    assert res.best == 0


def test_scaling_identity_before_rounding():
    """(W diag(s)) (diag(s)^-1 X) = W X, and the oracle's Wq is the deployed
    computation: X @ Wq^T = (X / s) @ Q(W s)^T."""
    rng = np.random.default_rng(4)
    W = rng.standard_normal((12, 48)) * 0.02
    X = rng.standard_normal((7, 48)) * rng.uniform(0.5, 50, size=48)
    s = rng.uniform(0.1, 10.0, size=48)
    lhs = (X / s) @ (W * s).T
    rhs = X @ W.T
    assert np.max(np.abs(lhs - rhs)) <= 1e-12 * np.max(np.abs(rhs))
    s32 = s.astype(np.float32)
    Wq, gq = O.fake_quant(W.astype(np.float32), s32, 4, 16, True)
    deployed = (X / s32.astype(np.float64)) @ gq.w_hat.astype(np.float64).T
    assert np.max(np.abs(X @ Wq.T - deployed)) <= 1e-12 * np.max(np.abs(deployed))
    # the error is linear in the weight change: X Wq^T - X W^T = X (Wq - W)^T
    W32 = W.astype(np.float32).astype(np.float64)
    d1 = X @ Wq.T - X @ W32.T
    d2 = X @ (Wq - W32).T
    assert np.max(np.abs(d1 - d2)) <= 1e-12 * np.max(np.abs(X @ W32.T))


def test_power_of_two_homogeneity():
    """Scaling t by 2^k leaves codes and zero points unchanged and scales
    every group step by exactly 2^k (both quantizers are positively
    homogeneous, and multiplying by 2^k is exact)."""
    rng = np.random.default_rng(5)
    t = (rng.standard_normal((9, 64)) * 0.05).astype(np.float32)
    for sym in (True, False):
        base = O.quantize_groups(t, 4, 16, sym)
        for k in (-3, 1, 5):
            f = np.float32(2.0 ** k)
            g = O.quantize_groups(t * f, 4, 16, sym)
            assert np.array_equal(g.q, base.q)
            assert np.array_equal(g.zero, base.zero)
            assert np.array_equal(g.scale, base.scale * f)


@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_quantizer_bounds(sym, bits):
    rng = np.random.default_rng(6 + bits)
    t = (rng.standard_normal((20, 128)) * 0.03).astype(np.float32)
    t[0, :32] = np.abs(t[0, :32])       # an all-positive group
    t[1, :32] = -np.abs(t[1, :32])      # an all-negative group
    t[2, :32] = 0.0                     # an all-zero group
    g = O.quantize_groups(t, bits, 32, sym)
    if sym:
        L = 2 ** (bits - 1) - 1
        assert g.q.min() >= -L - 1 and g.q.max() <= L
        # scale = max/L means the clamp never fires: codes stay in [-L, L]
        assert g.q.min() >= -L
    else:
        maxq = 2 ** bits - 1
        assert g.q.min() >= 0 and g.q.max() <= maxq
        assert g.zero.min() >= 0 and g.zero.max() <= maxq
        assert np.all(g.zero[0, 0] == 0)            # all-positive: lo = 0
        assert g.zero[1, 0] == maxq                 # all-negative: hi = 0
    # rounding error at most half a step (relative slack for float32 rounding)
    step = np.repeat(g.scale, 32, axis=1)
    err = np.abs(g.w_hat.astype(np.float64) - t)
    assert np.all(err <= 0.5 * step * (1 + 1e-5) + 1e-30)
    assert np.all(g.w_hat[2, :32] == 0)
    assert np.all(g.scale[2, 0] == np.float32(1e-8))


def test_fp64_quantizer_differs_only_at_near_ties():
    rng = np.random.default_rng(7)
    t = (rng.standard_normal((64, 512)) * 0.02).astype(np.float32)
    for sym in (True, False):
        a = O.quantize_groups(t, 4, 128, sym)
        b = O.quantize_groups_f64(t, 4, 128, sym)
        diff = a.q != b.q
        assert diff.sum() <= 3
        if diff.any():
            r = t.astype(np.float64) / np.repeat(b.scale, 128, axis=1)
            frac = np.abs(np.abs(r - np.floor(r)) - 0.5)
            assert np.all(frac[diff] < 1e-5)


def test_awq_beats_rtn_on_outlier_layer():
    """The notebook's check: with a few high-activation channels the searched
    scales give a lower output MSE than RTN ("GPTQ and AWQ weight
    quantisation", awq_beats_rtn_on_output_mse), and the error is finite and
    positive (awq_outputs_finite)."""
    rng = np.random.default_rng(8)
    W = (rng.standard_normal((256, 512)) * 0.02).astype(np.float16).astype(np.float32)
    X = rng.standard_normal((64, 512))
    X[:, rng.permutation(512)[:8]] *= 6.0
    res = O.awq_search(W, X, bits=4, group=128, grid=20, sym=True)
    assert res.best > 0
    assert res.errs[res.best] < res.errs[0]
    assert np.isfinite(res.errs).all() and res.errs[res.best] > 0


def test_nonfinite_input_has_no_answer():
    W = np.ones((2, 4), dtype=np.float32)
    X = np.ones((3, 4))
    X[0, 0] = np.nan
    res = O.awq_search(W, X, bits=4, group=4, grid=4, sym=True)
    assert res.best == -1 and np.all(np.isnan(res.errs))


# --------------------------------------------------------------------------
# Storage and packing
# --------------------------------------------------------------------------

def test_pack_layout_by_hand():
    u = np.array([[1, 2, 3, 4, 5, 6, 7, 8, 9]], dtype=np.uint32)
    w = O.pack_bits(u, 4)
    assert w.shape == (1, 2)
    assert w[0, 0] == 0x87654321 and w[0, 1] == 0x9
    u3 = np.full((1, 11), 7, dtype=np.uint32)
    w3 = O.pack_bits(u3, 3)
    assert w3.shape == (1, 2) and w3[0, 0] == 0xFFFFFFFF and w3[0, 1] == 0x1
    u3b = np.array([[1, 0, 0, 0, 0, 0, 0, 0, 0, 0, 6]], dtype=np.uint32)
    w3b = O.pack_bits(u3b, 3)
    # code 10 (value 0b110) sits at bits 30..32: bit 31 of word 0 and bit 0 of word 1
    assert w3b[0, 0] == 0x80000001 and w3b[0, 1] == 0x1


@pytest.mark.parametrize("bits", [2, 3, 4, 5, 8])
def test_pack_roundtrip(bits):
    rng = np.random.default_rng(bits)
    u = rng.integers(0, 2 ** bits, size=(5, 77)).astype(np.uint32)
    assert np.array_equal(O.unpack_bits(O.pack_bits(u, bits), bits, 77), u)


def test_storage_ratio_notebook_layer():
    """4096 x 4096 layer at 4 bits: 8 MiB of codes; with one fp16 scale per
    group of 128 the notebook gets 8.25 MiB, "4x" within 5 %
    ("GPTQ and AWQ weight quantisation", "Storage math")."""
    out = n_in = 4096
    rng = np.random.default_rng(9)
    W = (rng.standard_normal((out, n_in)) * 0.02).astype(np.float32)
    s32 = np.ones(n_in, dtype=np.float32)
    qweight, scales, zeros = O.quantize_pack(W, s32, 4, 128, True)
    assert qweight.dtype == np.uint32 and qweight.nbytes == 8 * 2 ** 20
    assert scales.shape == (out, n_in // 128) and zeros.shape == scales.shape
    assert np.all(zeros == 8)
    bytes_int4 = qweight.nbytes + scales.size * 2
    assert bytes_int4 == int(8.25 * 2 ** 20)
    ratio = (out * n_in * 2) / bytes_int4
    assert abs(ratio - 4.0) <= 0.05 * 4.0
    # decoding the packed words gives back the symmetric codes
    codes = O.unpack_bits(qweight[:4], 4, n_in).astype(np.int64) - 8
    assert np.array_equal(codes, O.quantize_groups(W[:4], 4, 128, True).q.astype(np.int64))


def test_asym_code_formula_at_exact_ties():
    """The code is round(w / scale) + zero, as the page writes it ("AWQ vs GPTQ
    ...", "The shared problem"), not round(w / scale + zero): the two differ
    when w / scale is exactly k + 1/2 and the zero point is odd.  A group with
    lo = -3, hi = 12 has scale (12 + 3) / 15 = 1 and zero 3 exactly."""
    t = np.array([[-3.0, 12.0, 0.5, 1.5, -2.5, 2.0, 0.0, 4.5]], dtype=np.float32)
    g = O.quantize_groups(t, 4, 8, sym=False)
    assert g.scale[0, 0] == 1.0 and g.zero[0, 0] == 3.0
    # half-to-even of the quotient first: 0.5 -> 0, 1.5 -> 2, -2.5 -> -2, 4.5 -> 4
    assert list(g.q[0]) == [0.0, 15.0, 3.0, 5.0, 1.0, 5.0, 3.0, 7.0]
    # symmetric ties: scale = 3.5 / 7 = 0.5, so 0.25 / 0.5 = 0.5 -> 0 and 0.75 -> 2
    ts = np.array([[3.5, 0.25, 0.75, -0.25, -0.75, 1.25, 0.0, -3.5]], dtype=np.float32)
    gs = O.quantize_groups(ts, 4, 8, sym=True)
    assert gs.scale[0, 0] == 0.5
    assert list(gs.q[0]) == [7.0, 0.0, 2.0, -0.0, -2.0, 2.0, 0.0, -7.0]


# --------------------------------------------------------------------------
# Output power and relative error (AWQ guide, "What the simulations show":
# error is ||h W - h Wq||^2 / ||h W||^2)
# --------------------------------------------------------------------------

def test_output_power_closed_forms():
    W = np.array([[1.0, 2.0], [3.0, 4.0]])
    # one token of ones: the outputs are the row sums 3 and 7
    assert O.output_power(W, np.array([[1.0, 1.0]])) == (9.0 + 49.0) / 2
    # the identity as calibration set: the outputs are W^T itself
    rng = np.random.default_rng(3)
    W = rng.normal(size=(5, 8)).astype(np.float32)
    assert np.isclose(O.output_power(W, np.eye(8)), np.mean(W.astype(np.float64) ** 2),
                      rtol=1e-15, atol=0)


def test_relative_error_of_dropping_the_layer_is_one():
    rng = np.random.default_rng(4)
    W = rng.normal(size=(6, 16)).astype(np.float32)
    X = rng.normal(size=(9, 16))
    ref = X @ W.astype(np.float64).T
    assert O.output_mse(X, np.zeros(W.shape), ref) / O.output_power(W, X) == pytest.approx(1.0, rel=1e-15)


def test_worked_example_relative_errors():
    # the page's two-channel layer: exact output 10 * 0.5 + 0.1 * 2.0 = 5.2;
    # AWQ (alpha = 0.5) misses it by the printed 0.033, RTN by the printed 1.67
    W = np.array([WE["w"]], dtype=np.float32)
    X = np.array([WE["abar"]])
    rows = O.sweep(W, X, [(int(WE["bits"][0]), None)], grid=2)
    r = rows[0]
    assert r["best"] == 1 and r["alpha"] == WE["alpha"][0]
    y = float(np.dot(WE["w"], WE["abar"]))
    assert O.output_power(W, X) == pytest.approx(y * y, rel=1e-12)
    for key, printed in (("rel_awq", WE["err_awq"][1]), ("rel_rtn", WE["err_rtn"][0])):
        lo = ((printed - _tol(printed)) / y) ** 2
        hi = ((printed + _tol(printed)) / y) ** 2
        assert lo <= r[key] <= hi, (key, r[key], lo, hi)


def test_sweep_rtn_column_is_plain_rtn():
    rng = np.random.default_rng(5)
    W = rng.normal(0, 0.02, size=(8, 64)).astype(np.float32)
    X = rng.normal(size=(12, 64))
    X[:, 3] *= 20.0
    ref = X @ W.astype(np.float64).T
    for bits, group in ((4, 32), (3, None), (8, 64)):
        r = O.sweep(W, X, [(bits, group)], grid=4)[0]
        g = 64 if group is None else group
        assert r["err_rtn"] == O.output_mse(X, O.rtn_fake_quant(W, bits, g, True), ref)
        assert r["err_awq"] <= r["err_rtn"]


def test_relative_error_is_scale_free():
    # W -> 2W leaves s_X alone and doubles every fl32(w * s), group step and
    # dequantized weight exactly, so err and power both grow by exactly 4
    rng = np.random.default_rng(6)
    W = rng.normal(0, 0.02, size=(8, 64)).astype(np.float32)
    X = rng.normal(size=(12, 64))
    a = O.sweep(W, X, [(4, 32)], grid=4)[0]
    b = O.sweep(2 * W, X, [(4, 32)], grid=4)[0]
    assert a["best"] == b["best"]
    assert a["rel_awq"] == b["rel_awq"] and a["rel_rtn"] == b["rel_rtn"]
    # X -> 2X also scales s_X, up to its 1e-8 floor: equal to ~1e-7
    c = O.sweep(W, 2 * X, [(4, 32)], grid=4)[0]
    assert a["best"] == c["best"]
    assert c["rel_awq"] == pytest.approx(a["rel_awq"], rel=1e-6)


# --------------------------------------------------------------------------
# Checkpoint tensors ("AWQ vs GPTQ ...", "What lands on disk")
# --------------------------------------------------------------------------

def test_checkpoint_layout_by_hand():
    # two output channels of eight inputs, 4-bit codes 0..7 and 15..8
    u = np.array([list(range(8)), list(range(15, 7, -1))], dtype=np.uint32)
    qw = O.pack_bits(u, 4)
    ck = O.export_checkpoint(qw, np.array([[0.5], [2.0]], np.float32),
                             np.array([[3], [12]], np.uint8), 8, 4)
    assert ck.qweight.shape == (1, 2)
    assert int(ck.qweight[0, 0]) == 0x76543210 and int(ck.qweight[0, 1]) == 0x89ABCDEF
    assert ck.scales.dtype == np.float16 and ck.scales.tolist() == [[0.5, 2.0]]
    assert ck.qzeros.shape == (1, 1) and int(ck.qzeros[0, 0]) == 0xC3


def test_checkpoint_size_matches_the_pages_arithmetic():
    # 4 bits plus a 16-bit scale and a 4-bit zero per 128 weights: "about 4.16
    # bits per weight"; 6.98B decoder weights then take "3.63 GB"
    out, n_in, g = 256, 1024, 128
    rng = np.random.default_rng(7)
    W = rng.normal(0, 0.02, size=(out, n_in)).astype(np.float32)
    qw, sc, z = O.quantize_pack(W, np.ones(n_in, np.float32), 4, g, False)
    ck = O.export_checkpoint(qw, sc, z, n_in, 4)
    nbytes = ck.qweight.nbytes + ck.scales.nbytes + ck.qzeros.nbytes
    bpw = nbytes * 8 / (out * n_in)
    assert bpw == 4 + 16 / 128 + 4 / 128
    assert abs(bpw - 4.16) <= 0.005
    # half a unit of the printed 3.63, plus what half a unit of 6.98B moves it
    assert abs(6.98e9 * bpw / 8 / 1e9 - 3.63) <= 0.005 + 0.005e9 * bpw / 8 / 1e9


@pytest.mark.parametrize("sym", [True, False])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_checkpoint_dequantizes_to_the_quantized_weights(sym, bits):
    out, n_in, g = 24, 256, 64
    rng = np.random.default_rng(bits)
    W = rng.normal(0, 0.02, size=(out, n_in)).astype(np.float32)
    s32 = rng.uniform(0.5, 4.0, size=n_in).astype(np.float32)
    qw, sc, z = O.quantize_pack(W, s32, bits, g, sym)
    ck = O.export_checkpoint(qw, sc, z, n_in, bits)
    Wh = O.dequantize_checkpoint(ck, out, n_in, bits, g)
    gq = O.quantize_groups(W * s32[None, :], bits, g, sym)
    # equal but for the rounding of each step to float16 (relative 2^-11)
    levels = np.abs(gq.q.astype(np.float64) - (0 if sym else gq.zero.repeat(g, axis=1)))
    bound = levels * np.repeat(gq.scale, g, axis=1) * 2.0 ** -11 + 1e-12
    assert np.all(np.abs(Wh - gq.w_hat) <= bound)


# --------------------------------------------------------------------------
# Per-group clipping search (AWQ guide, "Simplifications"; comparison page,
# "AWQ: move the error away from what matters")
# --------------------------------------------------------------------------

@pytest.mark.parametrize("sym", [True, False])
def test_clip_factor_one_is_the_plain_quantizer(sym):
    rng = np.random.default_rng(8)
    t = rng.normal(0, 0.05, size=(6, 96)).astype(np.float32)
    a = O.quantize_groups(t, 3, 32, sym)
    b = O.quantize_groups_clipped(t, 3, 32, sym, np.ones((6, 3), np.float32))
    for x, y in ((a.q, b.q), (a.scale, b.scale), (a.zero, b.zero), (a.w_hat, b.w_hat)):
        assert np.array_equal(x, y)


def test_clip_search_by_hand_keeps_no_clipping():
    # one group [1.0, 0.4], X = I, 3-bit symmetric (L = 3):
    #   c = 1:    step 1/3,    codes [3, 1] -> [1, 1/3],       share (0.4 - 1/3)^2
    #   c = 0.95: step 0.95/3, codes [3, 1] -> [0.95, 0.95/3], share 0.05^2 + (0.4 - 0.95/3)^2
    #   c = 0.8:  step 0.8/3,  codes [3 (3.75 clamped), 2]    share 0.2^2 + (0.4 - 1.6/3)^2
    W = np.array([[1.0, 0.4]], np.float32)
    r = O.clip_search(W, np.eye(2), np.ones(2, np.float32), 3, 2, True)
    e = r.errs[0, 0]
    assert e[0] == pytest.approx((0.4 - 1 / 3) ** 2, rel=1e-6)
    assert e[1] == pytest.approx(0.05 ** 2 + (0.4 - 0.95 / 3) ** 2, rel=1e-5)
    assert e[4] == pytest.approx(0.2 ** 2 + (0.4 - 1.6 / 3) ** 2, rel=1e-5)
    assert r.best[0, 0] == 0


def test_clip_search_by_hand_clips_an_outlier():
    # one group [1.0, 0.5, 0.5], X = I, 2-bit symmetric (L = 1): without
    # clipping the step is 1 and both 0.5 round to 0 (ties to even), share
    # 0.5; with 0.5 < c < 1 every value lands on the code for c, share
    # (1 - c)^2 + 2 (0.5 - c)^2, least on the grid at c = 0.65 (0.1675)
    W = np.array([[1.0, 0.5, 0.5]], np.float32)
    r = O.clip_search(W, np.eye(3), np.ones(3, np.float32), 2, 3, True)
    c = r.factors.astype(np.float64)
    e = r.errs[0, 0]
    assert e[0] == pytest.approx(0.5, rel=1e-12)
    for i in range(1, 10):
        assert e[i] == pytest.approx((1 - c[i]) ** 2 + 2 * (0.5 - c[i]) ** 2, rel=1e-6)
    assert r.factors[r.best[0, 0]] == np.float32(0.65)


def test_asymmetric_clipped_group_by_hand():
    # one group t = [-1.0, 0.25, 3.0], 2 bits (maxq = 3), factor c = 0.5:
    #   lo = c * min(min t, 0) = -0.5,  hi = c * max(max t, 0) = 1.5
    #   step = fl32((hi - lo) / 3) = fl32(2/3),  zero = round(fl32(0.5 / step)) = round(0.74999994) = 1
    #   codes: -1.0 / step = -1.5 -> -2 + 1 = -1 -> clamped to 0   (either neighbour of the
    #          tie gives a code <= 0, so the clamp decides)
    #          0.25 / step = 0.37499998 -> 0 + 1 = 1
    #          3.0 / step = 4.4999998 -> 4 + 1 = 5 -> clamped to 3
    #   w_hat = step * (code - zero) = [-step, 0, 2 step]
    # Shrinking only hi would give step fl32(2.5/3); taking the zero point from
    # the unclipped lo would give zero 2 and code 2 for 0.25.
    t = np.array([[-1.0, 0.25, 3.0]], np.float32)
    g = O.quantize_groups_clipped(t, 2, 3, False, np.array([[0.5]], np.float32))
    step = np.float32(2.0) / np.float32(3.0)
    assert g.scale[0, 0] == step and g.zero[0, 0] == 1.0
    assert g.q.tolist() == [[0.0, 1.0, 3.0]]
    assert g.w_hat.tolist() == [[float(-step), 0.0, float(np.float32(2) * step)]]
    # an all-positive group [0.5, 1.0, 2.0] at c = 0.75: lo = c * 0 = 0, hi = 1.5,
    # step 0.5, zero 0, codes [1, 2, 4 -> 3], w_hat [0.5, 1.0, 1.5]
    t = np.array([[0.5, 1.0, 2.0]], np.float32)
    g = O.quantize_groups_clipped(t, 2, 3, False, np.array([[0.75]], np.float32))
    assert g.scale[0, 0] == np.float32(0.5) and g.zero[0, 0] == 0.0
    assert g.q.tolist() == [[1.0, 2.0, 3.0]] and g.w_hat.tolist() == [[0.5, 1.0, 1.5]]


@pytest.mark.parametrize("sym", [True, False])
def test_clip_share_of_a_whole_row_group_is_the_row_error(sym):
    # with one group per row the group's share is the row's whole output error
    rng = np.random.default_rng(9)
    W = rng.normal(0, 0.02, size=(5, 64)).astype(np.float32)
    X = rng.normal(size=(7, 64))
    s32 = rng.uniform(0.5, 2.0, size=64).astype(np.float32)
    r = O.clip_search(W, X, s32, 3, 64, sym, n_grid=10, max_shrink=0.3)
    ref = X @ W.astype(np.float64).T
    for i, c in enumerate(r.factors):
        gq = O.quantize_groups_clipped(W * s32[None, :], 3, 64, sym, np.full((5, 1), c, np.float32))
        Wq = gq.w_hat.astype(np.float64) / s32.astype(np.float64)[None, :]
        per_row = np.sum((X @ Wq.T - ref) ** 2, axis=0)
        assert np.allclose(r.errs[:, 0, i], per_row, rtol=1e-10, atol=0)


# --------------------------------------------------------------------------
# GPTQ rounding after AWQ scaling ("AWQ vs GPTQ ...", "GPTQ: compensate the
# error you just made" and "Failure modes and combining the two")
# --------------------------------------------------------------------------

def test_inverse_hessian_factor_is_the_upper_cholesky_of_the_inverse():
    rng = np.random.default_rng(10)
    X = rng.normal(size=(40, 12))
    X[:, 3] *= 15.0
    U = O.inverse_hessian_factor(X, damp=0.01)
    H = 2.0 * X.T @ X
    H[np.diag_indices_from(H)] += 0.01 * np.mean(np.diag(H))
    assert np.allclose(np.triu(U), U) and np.all(np.diag(U) > 0)
    assert np.allclose(U.T @ U @ H, np.eye(12), atol=1e-9)


@pytest.mark.parametrize("sym", [True, False])
def test_gptq_with_uncorrelated_inputs_is_rtn(sym):
    # X = 3 I: H is diagonal, so is U, and no error is passed on
    rng = np.random.default_rng(11)
    W = rng.normal(0, 0.02, size=(6, 64)).astype(np.float32)
    r = O.gptq(W, 3.0 * np.eye(64), 4, 32, sym)
    gq = O.quantize_groups(W, 4, 32, sym)
    assert np.array_equal(r.q, gq.q) and np.array_equal(r.w_hat, gq.w_hat.astype(np.float64))


def test_gptq_second_column_is_the_best_code_given_the_first():
    # one row, two columns, one group: after column 0 is rounded, the
    # quadratic error (w_hat - w)^T H (w_hat - w) is a parabola in column 1
    # alone, so the nearest code to its minimum is the best code, found here
    # by trying every code
    rng = np.random.default_rng(12)
    for trial in range(200):
        X = rng.normal(size=(5, 2)) * rng.uniform(0.2, 3.0, size=2)
        W = rng.normal(0, 0.5, size=(1, 2)).astype(np.float32)
        r = O.gptq(W, X, 3, 2, True, damp=0.0)
        H = 2.0 * X.T @ X
        scale = float(r.scale[0, 0])
        w = W[0].astype(np.float64)
        errs = []
        for code in range(-4, 4):
            d = np.array([r.w_hat[0, 0], float(np.float32(code * np.float32(scale)))]) - w
            errs.append(d @ H @ d)
        errs = np.array(errs)
        best = int(np.argmin(errs)) - 4
        # the kept code is the best one, unless two codes are within rounding of a tie
        assert r.q[0, 1] == best or errs[int(r.q[0, 1]) + 4] <= errs.min() * (1 + 1e-9), trial


def test_gptq_fits_each_group_on_the_corrected_weights():
    # "fit on already-corrected weights" ("AWQ vs GPTQ ...", "GPTQ: compensate
    # the error you just made").  Choose the factor first:
    #       U = [[1, 0, 2, -1], [0, 1, 6, -8], [0, 0, 1, 1], [0, 0, 0, 1]]
    # and X = U^-T (4 tokens), so H = 2 X^T X = 2 U^-1 U^-T, H^-1 = U^T U / 2
    # and the oracle's factor is U / sqrt(2) (damp 0).  The update of column j
    # by column i uses U[i, j] / U[i, i], in which sqrt(2) cancels.
    # One row w = [-3, 1.25, 1, 0.25], 3-bit symmetric (L = 3), group 2:
    #   group 0 at column 0: step max(3, 1.25) / 3 = 1
    #   column 0: -3 -> code -3, error 0 (nothing passed on)
    #   column 1: 1.25 -> code 1, error 0.25: column 2 -= 0.25 * 6 -> -0.5,
    #             column 3 -= 0.25 * (-8) -> 2.25
    #   group 1 at column 2, fitted on [-0.5, 2.25]: step 2.25 / 3 = 0.75
    #             (fitted on the original [1, 0.25] it would be 1/3)
    #   column 2: -0.5 / 0.75 = -0.667 -> code -1, w_hat -0.75, error 0.25:
    #             column 3 -= 0.25 * 1 -> 2.0
    #   column 3: 2.0 / 0.75 = 2.667 -> code 3, w_hat 2.25
    U = np.array([[1, 0, 2, -1], [0, 1, 6, -8], [0, 0, 1, 1], [0, 0, 0, 1]], np.float64)
    X = np.linalg.inv(U).T
    W = np.array([[-3.0, 1.25, 1.0, 0.25]], np.float32)
    r = O.gptq(W, X, 3, 2, True, damp=0.0)
    assert r.scale.tolist() == [[1.0, 0.75]]
    assert r.q.tolist() == [[-3.0, 1.0, -1.0, 3.0]]
    assert r.w_hat.tolist() == [[-3.0, 1.0, -0.75, 2.25]]
    assert np.allclose(O.inverse_hessian_factor(X, 0.0) * np.sqrt(2.0), U, rtol=0, atol=1e-12)


def test_error_splits_into_row_slices():
    # err is a mean over every (token, output row) entry and s depends on X
    # alone, so the search over slices of the output rows sums back to the
    # whole layer's search: N out err = sum over slices of N rows_p err_p
    rng = np.random.default_rng(15)
    W = rng.normal(0, 0.02, size=(10, 64)).astype(np.float32)
    X = rng.normal(size=(7, 64))
    X[:, 5] *= 20.0
    full = O.awq_search(W, X, bits=3, group=32, grid=8, sym=False)
    parts = [O.awq_search(W[a:b], X, bits=3, group=32, grid=8, sym=False)
             for a, b in ((0, 3), (3, 4), (4, 10))]
    total = sum(p.errs * (b - a) for p, (a, b) in zip(parts, ((0, 3), (3, 4), (4, 10))))
    assert np.allclose(total / 10, full.errs, rtol=1e-12, atol=0)
    for p in parts:
        assert np.array_equal(p.s32, full.s32)


# --------------------------------------------------------------------------
# Degenerate layers
# --------------------------------------------------------------------------

@pytest.mark.parametrize("sym", [True, False])
def test_zero_weights_give_zero_error_and_alpha_zero(sym):
    # every group's range is 0: the step is the 1e-8 floor, every code is the
    # zero point, the quantized weights are exactly 0 = W
    X = np.random.default_rng(13).normal(size=(9, 64))
    r = O.awq_search(np.zeros((4, 64), np.float32), X, bits=4, group=32, grid=6, sym=sym)
    assert np.all(r.errs == 0.0) and r.best == 0
    qw, sc, z = O.quantize_pack(np.zeros((4, 64), np.float32), r.s32[0], 4, 32, sym)
    assert np.all(sc == np.float32(1e-8))
    u = O.unpack_bits(qw, 4, 64)
    assert np.all(u == (8 if sym else 0)) and np.all(z == (8 if sym else 0))


def test_zero_activations_are_flat_salience():
    # s_X = 1e-8 for every channel: flat, so every alpha is RTN and alpha 0 wins
    W = np.random.default_rng(14).normal(0, 0.02, size=(4, 64)).astype(np.float32)
    r = O.awq_search(W, np.zeros((5, 64)), bits=4, group=32, grid=6, sym=True)
    assert np.all(r.sx == 1e-8) and r.best == 0
    assert np.all(r.s32 == np.float32(1.0))
