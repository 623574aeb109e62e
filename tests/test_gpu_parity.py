"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Acceptance (per alpha error, chosen alpha, final codes):
  * per-alpha errors within 2e-3 relative (fp16 tensor-core operands,
    fp32 accumulation, float64 sums);
  * the same alpha unless the two grid errors are within 1e-3 relative;
  * given the oracle's scale vector, codes, group scales and zero points
    bit-exact;
  * s_X equal to the oracle's float64 statistic (exactly for 16-bit X).
"""
import numpy as np
import pytest
import torch

from oracle import awq_oracle as O
from synthetic import make_random_layer

pytestmark = pytest.mark.gpu

ERR_RTOL = 2e-3
TIE_RTOL = 1e-3


@pytest.fixture(scope="module")
def awq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import post_weight_quantization_32_b300 as m
    return m


def _np_w(W):
    return W.float().numpy()


def _np_x(X):
    return X.double().numpy()


def _dev(*ts):
    return [t.cuda() for t in ts]


def check_search(awq, W, X, bits, group, sym, grid, label=""):
    Wd, Xd = _dev(W, X)
    diag = torch.zeros(4, dtype=torch.int32, device="cuda")
    opts = awq.SearchOpts()
    opts.diag = diag.data_ptr()
    st = awq.new_status()
    err, best, s_best = awq.awq_search(Wd, Xd, bits=bits, group=group, sym=sym, grid=grid,
                                       dev_status=st, opts=opts, check=False)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, "%s status %d, wait diagnostics %s" % (label, int(st.item()),
                                                                      diag.cpu().tolist())
    res = O.awq_search(_np_w(W), _np_x(X), bits=bits, group=group, grid=grid, sym=sym)
    e = err.cpu().numpy()
    b = int(best.item())
    rel = np.abs(e - res.errs) / np.maximum(res.errs, 1e-300)
    assert rel.max() <= ERR_RTOL, "%s per-alpha rel err %g (alpha %d)" % (label, rel.max(), rel.argmax())
    if b != res.best:
        assert abs(res.errs[b] - res.errs[res.best]) <= TIE_RTOL * res.errs[res.best], (label, b, res.best)
    sb = s_best.cpu().numpy()
    ref = res.s32[b]
    ulps = np.abs(sb.view(np.int32).astype(np.int64) - ref.view(np.int32).astype(np.int64))
    assert ulps.max() <= 1 and (ulps > 0).sum() <= max(2, sb.size // 1000), label
    return e, b, res


def check_pack(awq, W, s32, bits, group, sym, rows=None):
    Wd = W.cuda()
    sd = torch.from_numpy(np.ascontiguousarray(s32, dtype=np.float32)).cuda()
    qw, sc, z = awq.awq_quantize_pack(Wd, sd, bits=bits, group=group, sym=sym)
    Wn = _np_w(W)
    if rows is not None:
        Wn = Wn[rows]
        qw, sc, z = qw[rows], sc[rows], z[rows]
    qo, so, zo = O.quantize_pack(Wn, s32, bits, group, sym)
    assert np.array_equal(qw.cpu().numpy().view(np.uint32), qo)
    assert np.array_equal(sc.cpu().numpy(), so)
    assert np.array_equal(z.cpu().numpy(), zo)


# ---------------------------------------------------------------- statistics

@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("shape", [(64, 256), (1, 8), (300, 4104), (7, 3), (33, 77)])
def test_channel_stats(awq, dtype, shape):
    N, n_in = shape
    _, X = make_random_layer(4, n_in, N, dtype=dtype, seed=N + n_in)
    sx = awq.awq_channel_stats(X.cuda()).cpu().numpy()
    ref = O.channel_salience(_np_x(X))
    if dtype == "f32":
        assert np.allclose(sx, ref, rtol=1e-14, atol=0)
    else:
        assert np.array_equal(sx, ref)   # float64 sums of 16-bit values are exact


# ---------------------------------------------------------------- packing

PACK_CASES = [
    (4, 128, True), (4, 128, False), (3, 128, True), (3, 128, False), (2, 64, False),
    (8, 32, True), (5, 16, False), (4, 8, True), (4, 256, False),
    (4, 96, True), (3, 96, False), (4, 384, False), (4, None, True), (3, 24, True),
]


@pytest.mark.parametrize("bits,group,sym", PACK_CASES)
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_quantize_pack_bit_exact(awq, bits, group, sym, dtype):
    W, X = make_random_layer(37, 768, 16, dtype=dtype, seed=bits * 100 + (group or 0))
    g = 768 if group is None else group
    rng = np.random.default_rng(5)
    s32 = rng.uniform(0.05, 20.0, size=768).astype(np.float32)
    check_pack(awq, W, s32, bits, g, sym)


def test_quantize_pack_special_groups(awq):
    W, _ = make_random_layer(8, 256, 4, dtype="bf16", seed=3)
    W = W.clone()
    W[0, :128] = W[0, :128].abs()        # all-positive group
    W[1, :128] = -W[1, :128].abs()       # all-negative group
    W[2, :128] = 0                       # all-zero group
    W[3, 128:] = 1e-30                   # tiny: the 1e-8 floor of the step applies
    s32 = np.ones(256, dtype=np.float32)
    for sym in (True, False):
        check_pack(awq, W, s32, 4, 128, sym)


def test_quantize_pack_ragged_shapes(awq):
    for out, n_in, g in ((1, 8, 8), (5, 40, 8), (3, 2, 2), (1, 2, 2), (9, 264, 8)):
        W, _ = make_random_layer(out, n_in, 2, dtype="bf16", seed=out * n_in)
        s32 = np.random.default_rng(out).uniform(0.5, 2.0, size=n_in).astype(np.float32)
        for bits in (3, 4):
            for sym in (True, False):
                check_pack(awq, W, s32, bits, g, sym)


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), -float("inf")])
@pytest.mark.parametrize("bits,group,sym", [(4, 128, True), (4, 128, False), (3, 64, True),
                                            (8, 32, False), (4, 8, True)])
def test_quantize_pack_nonfinite_reports(awq, bad, bits, group, sym):
    W, _ = make_random_layer(4, 128, 2, dtype="bf16", seed=9)
    W = W.clone()
    W[2, 5] = bad
    st = awq.new_status()
    qw, _, _ = awq.awq_quantize_pack(W.cuda(), torch.ones(128, device="cuda"), bits, group, sym,
                                     dev_status=st, check=False)
    assert int(st.item()) == 3
    # the other rows are unaffected: bit-exact against the oracle
    Wn = _np_w(W)
    ref, _, _ = O.quantize_pack(np.concatenate([Wn[:2], Wn[3:]]), np.ones(128, np.float32), bits,
                                group, sym)
    got = qw.cpu().numpy().view(np.uint32)
    np.testing.assert_array_equal(np.concatenate([got[:2], got[3:]]), ref)


@pytest.mark.parametrize("bits,group,sym,n_in", [(8, 512, True, 2560), (2, 512, False, 2560),
                                                 (4, 256, True, 2560), (4, 32, False, 2560),
                                                 (2, 32, True, 2560), (4, 1024, True, 3072),
                                                 (8, 1024, False, 2048)])
def test_quantize_pack_wide_groups(awq, bits, group, sym, n_in):
    # 2560 columns: two full 1024-column segments and a half one; 70 rows: a
    # partial block of rows
    W, _ = make_random_layer(70, n_in, 2, dtype="f16", seed=bits + group)
    s32 = np.random.default_rng(group).uniform(0.1, 10.0, size=n_in).astype(np.float32)
    check_pack(awq, W, s32, bits, group, sym)


# ---------------------------------------------------------------- search

SEARCH_CASES = [
    # (out, in, N, dtype, bits, group, sym, grid)
    (128, 256, 64, "f32", 4, 128, True, 20),       # the tiny configuration's shape
    (300, 384, 100, "bf16", 4, 128, False, 20),    # ragged rows, 3 row tiles, odd K groups
    (256, 512, 300, "f16", 4, 128, True, 10),      # two token tiles
    (200, 256, 32, "bf16", 3, 64, True, 8),        # 3 bits, group 64, 8 alphas per unit
    (130, 96, 17, "bf16", 4, 32, False, 5),        # group 32, partial K block
    (64, 1024, 513, "bf16", 4, 128, False, 4),     # three token tiles, 16 K blocks
    (1, 128, 1, "bf16", 4, 128, True, 20),         # one row, one token
    (384, 640, 256, "f16", 2, 64, False, 20),
    (128, 256, 16, "bf16", 4, 128, True, 20),      # 8 alphas per unit, both producer banks
    (96, 1024, 20, "bf16", 4, 128, False, 20),     # 8 alphas per unit over 8 K groups
    (256, 384, 48, "bf16", 4, 128, True, 20),      # odd number of K groups
    (160, 512, 40, "f32", 4, 64, False, 12),
    # narrow groups inside a 64-column job: eight or four per job
    (130, 768, 40, "f16", 3, 8, True, 6),
    (200, 768, 64, "bf16", 4, 16, False, 8),       # the AWQ guide's "a scale per 16"
    (96, 256, 300, "f16", 3, 16, True, 20),        # two token tiles, X pre-divided by s
    # groups the 64-column jobs do not align with: ranges from a pass over W,
    # each 8-column chunk takes its group's step
    (256, 768, 300, "bf16", 4, 96, False, 10),     # two token tiles
    (96, 768, 50, "f16", 4, 48, True, 12),
    (70, 1536, 20, "bf16", 4, 24, False, 8),       # up to four groups in one job
    (33, 240, 9, "f32", 3, 40, True, 5),           # ragged K block
    # the same with more than 128 tokens and 16-bit: X pre-divided by s, the
    # stored ranges scaled by the same power of two as t
    (160, 480, 200, "f16", 4, 96, True, 10),
    (96, 384, 150, "bf16", 3, 24, False, 8),
]


@pytest.mark.parametrize("case", SEARCH_CASES, ids=lambda c: "%dx%d_n%d_%s_b%d_g%d_%s_G%d" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "sym" if c[6] else "asym", c[7]))
def test_search_matches_oracle(awq, case):
    out, n_in, N, dtype, bits, group, sym, grid = case
    W, X = make_random_layer(out, n_in, N, dtype=dtype, seed=out + n_in + N,
                             n_outlier=max(1, n_in // 64))
    e, b, res = check_search(awq, W, X, bits, group, sym, grid, label=str(case))
    # the kept scales reproduce the oracle's codes exactly
    check_pack(awq, W, res.s32[b], bits, group, sym)


WIDE_GROUP_CASES = [
    # (out, in, N, dtype, bits, group, sym, grid); group None = one group per row.
    # Groups wider than a 128-column producer job take their ranges from the
    # pass over W ahead of the search.
    (256, 512, 64, "bf16", 4, 256, True, 10),
    (200, 768, 40, "f16", 3, None, False, 8),
    (130, 1024, 33, "f32", 2, 512, True, 5),
    (64, 96, 16, "bf16", 4, None, False, 6),       # one row group narrower than one job
    (300, 2056, 20, "bf16", 8, None, False, 4),    # ragged last K block
    (128, 1024, 300, "f16", 4, 1024, True, 20),    # two token tiles
    (100, 1536, 24, "bf16", 4, 768, False, 20),    # three 256-column multiples per group
    # more than 128 tokens and 16-bit: the pre-divided kernel with the stored
    # ranges scaled by its power of two
    (256, 1024, 256, "bf16", 4, 256, False, 20),
    (192, 2048, 200, "f16", 3, None, True, 10),
    (96, 2056, 160, "bf16", 4, None, False, 6),    # ragged last K block
]


@pytest.mark.parametrize("case", WIDE_GROUP_CASES, ids=lambda c: "%dx%d_n%d_%s_b%d_g%s_%s_G%d" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "sym" if c[6] else "asym", c[7]))
def test_search_wide_groups_match_oracle(awq, case):
    out, n_in, N, dtype, bits, group, sym, grid = case
    W, X = make_random_layer(out, n_in, N, dtype=dtype, seed=out + n_in + N + 7,
                             n_outlier=max(1, n_in // 64))
    e, b, res = check_search(awq, W, X, bits, group, sym, grid, label=str(case))
    check_pack(awq, W, res.s32[b], bits, n_in if group is None else group, sym)


# 16-bit layers take a tensor-core kernel.  Layers with few 128-row x
# 128-token tiles split each tile's K range over a cluster of CTAs: four a
# tile for (300, 1032, 300) (ragged rows, tokens and K: 1032 = 16 blocks of
# 64 + 8) and (384, 1024, 100), two a tile for (4096, 512, 256).  The others
# take the persistent kernel (token tiles of 32, 64, 128 or 256, two K
# blocks a ring stage below 256): (256, 512, 64) 64-token tiles; (2048,
# 2048, 1024) 256 units, more than one a CTA, so both accumulators
# alternate; (9600, 136, 250) 128-token tiles; (9600, 512, 600) 225 units;
# (19000, 64, 256) 256-token tiles, one K block; (130, 264, 17) a 32-token
# tile for 17 tokens; (1, 64, 1) one row and one token.  float32 takes the
# GEMM route.
@pytest.mark.parametrize("dtype,shape", [("f16", (256, 512, 64)), ("bf16", (300, 1032, 300)),
                                         ("f16", (2048, 2048, 1024)), ("bf16", (384, 1024, 100)),
                                         ("f16", (4096, 512, 256)),
                                         ("f16", (9600, 136, 250)), ("bf16", (9600, 512, 600)),
                                         ("bf16", (19000, 64, 256)), ("bf16", (130, 264, 17)),
                                         ("f32", (96, 256, 17)), ("bf16", (1, 64, 1))])
def test_output_power_matches_oracle(awq, dtype, shape):
    out, n_in, N = shape
    W, X = make_random_layer(out, n_in, N, dtype=dtype, seed=out * 3 + N,
                             n_outlier=max(1, n_in // 64))
    Wd, Xd = _dev(W, X)
    p = awq.awq_output_power(Wd, Xd)
    ref = O.output_power(_np_w(W), _np_x(X))
    assert abs(float(p.item()) - ref) <= ERR_RTOL * ref, (float(p.item()), ref)
    # a fixed summation order: a second call gives the same bits
    assert torch.equal(awq.awq_output_power(Wd, Xd).view(torch.int64), p.view(torch.int64))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_output_power_routes_agree(awq, dtype):
    """X two bytes off a 16-byte boundary cannot be read by TMA: the call
    takes the GEMM route instead, and the two routes agree."""
    W, X = make_random_layer(384, 1024, 200, dtype=dtype, seed=5, n_outlier=16)
    Wd, Xd = _dev(W, X)
    buf = torch.empty(Xd.numel() + 1, dtype=Xd.dtype, device=Xd.device)
    Xm = buf[1:].view(Xd.shape)
    Xm.copy_(Xd)
    assert Xm.data_ptr() % 16 != 0
    p_tc = float(awq.awq_output_power(Wd, Xd).item())
    p_gemm = float(awq.awq_output_power(Wd, Xm).item())
    ref = O.output_power(_np_w(W), _np_x(X))
    assert abs(p_tc - ref) <= ERR_RTOL * ref and abs(p_gemm - ref) <= ERR_RTOL * ref
    assert abs(p_tc - p_gemm) <= 1e-4 * ref, (p_tc, p_gemm)


def test_sweep_matches_oracle(awq):
    """Bit widths and group sizes of the pages' sweeps, RTN beside AWQ."""
    W, X = make_random_layer(192, 1024, 64, dtype="bf16", seed=11, n_outlier=16)
    settings = [(8, 128), (4, 128), (3, 128), (2, 128), (4, 32), (4, 64), (4, 256), (4, None)]
    got = awq.awq_sweep(*_dev(W, X), settings, sym=True, grid=10)
    ref = O.sweep(_np_w(W), _np_x(X), settings, sym=True, grid=10)
    for g, r in zip(got, ref):
        label = (g["bits"], g["group"])
        if g["best"] != r["best"]:
            assert abs(r["errs"][g["best"]] - r["err_awq"]) <= TIE_RTOL * r["err_awq"], label
        else:
            assert g["alpha"] == r["alpha"], label
        for key in ("err_rtn", "rel_rtn"):
            assert abs(g[key] - r[key]) <= ERR_RTOL * r[key], (label, key, g[key], r[key])
        assert abs(g["rel_awq"] - r["rel_awq"]) <= (ERR_RTOL + TIE_RTOL) * r["rel_awq"], label
        assert g["err_awq"] <= g["err_rtn"], label


@pytest.mark.parametrize("bits,group,sym,dtype", [(4, 128, False, "bf16"), (4, 128, True, "f16"),
                                                  (2, 64, False, "bf16"), (8, 32, True, "f32"),
                                                  (4, 256, False, "bf16")])
def test_export_checkpoint_matches_oracle(awq, bits, group, sym, dtype):
    out, n_in = 72, 512   # 72 outputs: a partial 32-wide tile and, at 4 bits, 9 zero words
    W, _ = make_random_layer(out, n_in, 2, dtype=dtype, seed=bits * group)
    s32 = np.random.default_rng(group).uniform(0.2, 5.0, size=n_in).astype(np.float32)
    qw, sc, z = awq.awq_quantize_pack(W.cuda(), torch.from_numpy(s32).cuda(), bits, group, sym)
    qw_t, sc_h, qz = awq.awq_export_checkpoint(qw, sc, z, n_in, bits, group)
    ref = O.export_checkpoint(*O.quantize_pack(_np_w(W), s32, bits, group, sym), n_in, bits)
    assert np.array_equal(qw_t.cpu().numpy().view(np.uint32), ref.qweight)
    assert np.array_equal(sc_h.cpu().numpy().view(np.uint16), ref.scales.view(np.uint16))
    assert np.array_equal(qz.cpu().numpy().view(np.uint32), ref.qzeros)


def test_export_checkpoint_reports_fp16_overflow(awq):
    W, _ = make_random_layer(8, 128, 2, dtype="f32", seed=2)
    W = W.clone()
    W[3, 7] = 1.0e6   # its group's step, 1e6 / 7, is beyond the binary16 range
    qw, sc, z = awq.awq_quantize_pack(W.cuda(), torch.ones(128, device="cuda"), 4, 128, True)
    st = awq.new_status()
    awq.awq_export_checkpoint(qw, sc, z, 128, 4, 128, dev_status=st, check=False)
    assert int(st.item()) == 3


CLIP_CASES = [
    # (out, in, N, dtype, bits, group, sym, n_grid, max_shrink_steps)
    (64, 256, 40, "bf16", 3, 128, True, 20, 10),
    (37, 192, 17, "f16", 4, 64, False, 20, 10),
    (50, 96, 300, "f32", 2, 32, True, 10, 5),
    (130, 512, 64, "bf16", 4, 128, False, 20, 11),
    (9, 128, 1, "bf16", 3, 128, False, 20, 0),      # one factor: nothing to choose
]


@pytest.mark.parametrize("case", CLIP_CASES, ids=lambda c: "%dx%d_n%d_%s_b%d_g%d_%s_%d_%d" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "sym" if c[6] else "asym", c[7], c[8]))
def test_clip_search_matches_oracle(awq, case):
    out, n_in, N, dtype, bits, group, sym, n_grid, steps = case
    W, X = make_random_layer(out, n_in, N, dtype=dtype, seed=out + n_in + 3,
                             n_outlier=max(1, n_in // 64))
    s32 = np.random.default_rng(n_in).uniform(0.5, 2.0, size=n_in).astype(np.float32)
    Wd, Xd = _dev(W, X)
    clip, errs = awq.awq_clip_search(Wd, Xd, torch.from_numpy(s32).cuda(), bits, group, sym,
                                     n_grid, steps, want_errs=True)
    ref = O.clip_search(_np_w(W), _np_x(X), s32, bits, group, sym, n_grid, steps / n_grid)
    e = errs.cpu().numpy().astype(np.float64)
    floor = 1e-6 * ref.errs.max(axis=-1, keepdims=True)
    assert np.all(np.abs(e - ref.errs) <= ERR_RTOL * ref.errs + floor)
    got = clip.cpu().numpy()
    idx = np.argmax(got[..., None] == ref.factors[None, None, :], axis=-1)
    assert np.all(got == ref.factors[idx])
    chosen = np.take_along_axis(ref.errs, idx[..., None], -1)[..., 0]
    best = np.take_along_axis(ref.errs, ref.best[..., None], -1)[..., 0]
    assert np.all(chosen <= best * (1 + TIE_RTOL) + floor[..., 0])
    # the kept factors give the oracle's codes exactly
    qw, sc, z = awq.awq_quantize_pack_clipped(Wd, torch.from_numpy(s32).cuda(), clip, bits, group,
                                              sym)
    qo, so, zo = O.quantize_pack_clipped(_np_w(W), s32, bits, group, sym, got)
    assert np.array_equal(qw.cpu().numpy().view(np.uint32), qo)
    assert np.array_equal(sc.cpu().numpy(), so)
    assert np.array_equal(z.cpu().numpy(), zo)


GPTQ_CASES = [
    # (out, in, N, dtype, bits, group, sym, with AWQ scales).  A power-of-two
    # count of 64-column blocks (in = 256, 512, 1024) takes the doubling
    # inverse; 384 and 160 the block-row loop
    (64, 256, 512, "bf16", 4, 128, True, True),
    (48, 384, 300, "f16", 3, 64, False, True),
    (37, 160, 50, "f32", 4, 32, True, False),      # fewer tokens than inputs; partial blocks
    (96, 512, 2048, "bf16", 2, 128, False, True),
    (64, 1024, 256, "f16", 4, 128, True, True),    # four doubling levels
]


@pytest.mark.parametrize("case", GPTQ_CASES, ids=lambda c: "%dx%d_n%d_%s_b%d_g%d_%s_%s" % (
    c[0], c[1], c[2], c[3], c[4], c[5], "sym" if c[6] else "asym", "awq" if c[7] else "plain"))
def test_gptq_matches_oracle(awq, case):
    out, n_in, N, dtype, bits, group, sym, with_s = case
    W, X = make_random_layer(out, n_in, N, dtype=dtype, seed=out * 7 + n_in,
                             n_outlier=max(1, n_in // 64))
    s32 = (np.random.default_rng(n_in).uniform(0.5, 2.0, size=n_in).astype(np.float32)
           if with_s else None)
    Wd, Xd = _dev(W, X)
    qw, sc, z = awq.awq_gptq(Wd, Xd, None if s32 is None else torch.from_numpy(s32).cuda(), bits,
                             group, sym)
    r = O.gptq(_np_w(W), _np_x(X), bits, group, sym, s32)
    u_ref = O.stored_codes(r.q, bits, sym)
    u = O.unpack_bits(qw.cpu().numpy().view(np.uint32), bits, n_in)
    # fp32 against float64 running weights: a code may differ where a corrected
    # weight lies within rounding of a decision boundary
    assert (u != u_ref).mean() <= 1e-3
    z_ref = (np.full(r.zero.shape, 1 << (bits - 1)) if sym else r.zero).astype(np.uint8)
    assert (z.cpu().numpy() != z_ref).mean() <= 1e-3
    assert np.allclose(sc.cpu().numpy(), r.scale, rtol=1e-4, atol=0)
    # the layer's output error matches the oracle's
    g = np.arange(n_in) // group
    zz = z.cpu().numpy().astype(np.float64)[:, g]
    w_hat = sc.cpu().numpy().astype(np.float64)[:, g] * (u.astype(np.float64) - zz)
    s64 = np.ones(n_in) if s32 is None else s32.astype(np.float64)
    Xn = _np_x(X)
    ref = Xn @ _np_w(W).astype(np.float64).T
    e_gpu = O.output_mse(Xn, w_hat / s64[None, :], ref)
    e_ref = O.output_mse(Xn, r.Wq, ref)
    assert abs(e_gpu - e_ref) <= ERR_RTOL * e_ref, (e_gpu, e_ref)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_search_degenerate_layers(awq, dtype):
    """All-zero weights: every error is 0 and alpha 0 is kept; all-zero
    inputs: flat salience, every alpha is RTN, alpha 0 is kept."""
    W, X = make_random_layer(128, 256, 32, dtype=dtype, seed=21)
    zw = torch.zeros_like(W)
    err, best, _ = awq.awq_search(*_dev(zw, X), 4, 128, False, 8)
    assert int(best.item()) == 0 and torch.all(err == 0)
    qw, sc, z = awq.awq_quantize_pack(zw.cuda(), torch.ones(256, device="cuda"), 4, 128, True)
    assert torch.all(sc == torch.tensor(1e-8, dtype=torch.float32, device="cuda"))
    assert np.all(O.unpack_bits(qw.cpu().numpy().view(np.uint32), 4, 256) == 8)
    zx = torch.zeros_like(X)
    err, best, s_best = awq.awq_search(*_dev(W, zx), 4, 128, True, 8)
    res = O.awq_search(_np_w(W), _np_x(zx), bits=4, group=128, grid=8, sym=True)
    assert int(best.item()) == 0 and torch.all(s_best == 1.0)
    assert np.all(err.cpu().numpy() == 0) and np.all(res.errs == 0)


def test_search_shared_input_group(awq):
    """q/k/v share X and one s: the concatenated rows are searched at once."""
    ws, X = [], None
    for i in range(3):
        w, x = make_random_layer(128, 256, 96, dtype="bf16", seed=40 + i, n_outlier=3)
        ws.append(w)
        X = x if X is None else X
    W = torch.cat(ws, 0).contiguous()
    check_search(awq, W, X, 4, 128, False, 20, "qkv")


def test_search_flat_salience_keeps_alpha_zero(awq):
    """Equal mean |X| per channel: every alpha has s = 1, the errors tie, the
    first alpha is kept, and the errors still match the oracle."""
    W, _ = make_random_layer(256, 256, 8, dtype="bf16", seed=1)
    sign = torch.where(torch.rand(64, 256, generator=torch.Generator().manual_seed(2)) < 0.5, -1.0, 1.0)
    X = (sign * 0.375).to(torch.bfloat16)
    e, b, res = check_search(awq, W, X, 4, 128, True, 20, "flat")
    assert b == 0 and res.best == 0
    assert np.all(e == e[0])


def test_search_is_deterministic(awq):
    W, X = make_random_layer(512, 1024, 256, dtype="bf16", seed=77, n_outlier=10)
    Wd, Xd = _dev(W, X)
    r1 = [t.clone() for t in awq.awq_search(Wd, Xd, 4, 128, False, 20)]
    r2 = awq.awq_search(Wd, Xd, 4, 128, False, 20)
    for a, b in zip(r1, r2):
        assert torch.equal(a, b)


def test_search_given_sx(awq):
    W, X = make_random_layer(256, 512, 64, dtype="bf16", seed=5, n_outlier=4)
    Wd, Xd = _dev(W, X)
    sx = awq.awq_channel_stats(Xd)
    a = awq.awq_search(Wd, Xd, 4, 128, True, 20)
    b = awq.awq_search(Wd, Xd, 4, 128, True, 20, sx=sx)
    for u, v in zip(a, b):
        assert torch.equal(u, v)


def test_search_nonfinite_input(awq):
    W, X = make_random_layer(128, 256, 16, dtype="bf16", seed=6)
    X = X.clone()
    X[3, 7] = float("nan")
    st = awq.new_status()
    err, best, _ = awq.awq_search(W.cuda(), X.cuda(), 4, 128, True, 20, dev_status=st, check=False)
    torch.cuda.synchronize()
    assert int(st.item()) == 3
    assert int(best.item()) == -1
    # alpha = 0 has s = 1 in every column, so the NaN channel still reaches
    # the error only through X; every alpha's error is NaN
    assert torch.isnan(err).all()


def test_search_wait_timeout_reports_and_recovers(awq):
    """A wait on a barrier nothing arrives at runs out (50 ms); the kernel
    returns with AWQ_ERR_TIMEOUT, records a wait site, and the context stays
    usable.  The unset barrier stalls the whole pipeline, so whichever
    bounded wait runs out first (the MMA issuer's, or a producer's or
    loader's waiting behind it) is the one recorded."""
    W, X = make_random_layer(256, 512, 64, dtype="bf16", seed=8)
    Wd, Xd = _dev(W, X)
    diag = torch.zeros(4, dtype=torch.int32, device="cuda")
    opts = awq.SearchOpts()
    opts.wait_limit_ns = 50_000_000
    opts.test_timeout = 1
    opts.diag = diag.data_ptr()
    st = awq.new_status()
    awq.awq_search(Wd, Xd, 4, 128, True, 20, dev_status=st, opts=opts, check=False)
    torch.cuda.synchronize()
    assert int(st.item()) == 4
    assert diag[0].item() in (1, 3, 5, 6, 7, 8, 10, 11, 12, 13)   # a known wait site
    check_search(awq, W, X, 4, 128, True, 20, "after timeout")


def test_search_rejects_unsupported_group(awq):
    # groups of 4 columns divide in but are not a multiple of 8: the method
    # allows them, the search kernels do not (the pack does)
    W, X = make_random_layer(64, 256, 16, dtype="bf16", seed=1)
    with pytest.raises(awq.AWQError) as ei:
        awq.awq_search(W.cuda(), X.cuda(), 4, 4, True, 20)
    assert ei.value.code == 2


# ---------------------------------------------------------------- row split

@pytest.mark.parametrize("cuts", [(128,), (64, 200), (1, 299)])
def test_row_split_matches_whole_search(awq, cuts):
    """The search run slice by slice over the output rows, then finished from
    the slices' sums, gives the whole layer's errors, alpha and scales."""
    out, n_in, N = 300, 512, 96
    W, X = make_random_layer(out, n_in, N, dtype="bf16", seed=77, n_outlier=8)
    Wd, Xd = _dev(W, X)
    e_full, b_full, s_full = awq.awq_search(Wd, Xd, 4, 128, False, 20)
    bounds = (0,) + tuple(cuts) + (out,)
    parts, tables = [], []
    for r0, r1 in zip(bounds[:-1], bounds[1:]):
        sums, tab = awq.awq_search_rows(Wd[r0:r1].contiguous(), Xd, 4, 128, False, 20)
        parts.append(sums)
        tables.append(tab)
    for tab in tables[1:]:
        assert torch.equal(tab, tables[0])     # s depends on X alone
    e, b, sb = awq.awq_search_finish(torch.stack(parts, 0), N, out, tables[0])
    torch.cuda.synchronize()
    e, e_full = e.cpu().numpy(), e_full.cpu().numpy()
    # each slice scales its weight changes into fp16 by a power of two from
    # its own max|W|, which moves the fp16 rounding of the smallest entries:
    # the sums agree to about 1e-8, far inside the search's 2e-3
    assert (np.abs(e - e_full) / e_full).max() <= 1e-6
    b, bf = int(b.item()), int(b_full.item())
    if b != bf:
        assert abs(e_full[b] - e_full[bf]) <= TIE_RTOL * e_full[bf]
    else:
        assert torch.equal(sb, s_full)
