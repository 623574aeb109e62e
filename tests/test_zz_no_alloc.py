"""awq_search_noalloc: the search for callers that cannot allocate device
memory (for example a plug-in whose host application owns all device
memory, or real-time code where cudaMalloc is forbidden because it can
stall the device).  Its scratch is a fixed array inside the library.

The test calls the entry point through the C ABI twice in a row, on two
different layers, and compares each result with the ordinary awq_search
(caller-provided workspace) within the tolerances of the other parity
tests.  The second layer's inputs are a million times smaller than the
first's (its weights a thousand times), so scratch left over from the
first call (the operand scaling is derived from max|X| and max|W|) would
show up as a mismatch.

This file is named to be collected last: if it fails, a run that stops at
the first failure has already run every other test.
"""
import numpy as np
import pytest
import torch

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


def _compare(awq, W, X, bits, group, sym, grid):
    Wd, Xd = W.cuda(), X.cuda()
    e_ref, b_ref, s_ref = awq.awq_search(Wd, Xd, bits, group, sym, grid)
    e_na, b_na, s_na = awq.awq_search_noalloc(Wd, Xd, bits, group, sym, grid)
    torch.cuda.synchronize()
    e_ref, e_na = e_ref.cpu().numpy(), e_na.cpu().numpy()
    assert np.isfinite(e_ref).all() and np.isfinite(e_na).all()
    rel = np.abs(e_na - e_ref) / e_ref
    assert rel.max() <= ERR_RTOL, rel.max()
    br, bn = int(b_ref.item()), int(b_na.item())
    if bn != br:
        assert abs(e_ref[bn] - e_ref[br]) <= TIE_RTOL * e_ref[br]
    else:
        assert torch.equal(s_na, s_ref)


def test_noalloc_matches_workspace_search_twice(awq):
    W1, X1 = make_random_layer(512, 1024, 300, dtype="bf16", seed=901, n_outlier=12)
    W2, X2 = make_random_layer(256, 512, 64, dtype="bf16", seed=902, n_outlier=5)
    X2 = (X2.float() * 1e-6).to(torch.bfloat16)
    W2 = (W2.float() * 1e-3).to(torch.bfloat16)
    _compare(awq, W1, X1, 4, 128, False, 20)
    _compare(awq, W2, X2, 4, 128, True, 20)


def test_noalloc_at_the_edge_of_its_scratch(awq):
    # 256 x 4096 bf16 with the largest N whose workspace still fits the fixed
    # array's 32 MiB (the fp16 copy of X dominates it; about 4000 tokens):
    # it runs and matches the workspace search; one token more is refused
    # before anything is enqueued.
    out, n_in, grid = 256, 4096, 20

    def need(N):
        return awq.awq_search_workspace_min_bytes(torch.bfloat16, out, n_in, N, 128, grid)

    lo, hi = 1, 1 << 16
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if need(mid) <= awq.NOALLOC_SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid - 1
    n_edge = lo
    assert awq.NOALLOC_SCRATCH_BYTES - 16384 < need(n_edge) <= awq.NOALLOC_SCRATCH_BYTES
    assert need(n_edge + 1) > awq.NOALLOC_SCRATCH_BYTES
    W, X = make_random_layer(out, n_in, n_edge + 1, dtype="bf16", seed=903, n_outlier=40)
    _compare(awq, W, X[:n_edge].contiguous(), 4, 128, False, grid)
    with pytest.raises(awq.AWQError) as ei:
        awq.awq_search_noalloc(W.cuda(), X.cuda(), 4, 128, False, grid)
    assert ei.value.code == 2   # AWQ_ERR_UNSUPPORTED


def test_noalloc_rejects_problems_beyond_its_scratch(awq):
    # 8192 x 28672 bf16 with N = 1024 needs far more than the fixed array;
    # the size check returns before anything is enqueued, so the tensors
    # passed here are never read.
    out, n_in, N, grid = 8192, 28672, 1024, 40
    need = awq.awq_search_workspace_min_bytes(torch.bfloat16, out, n_in, N, 128, grid)
    assert need > awq.NOALLOC_SCRATCH_BYTES
    dummy = torch.empty(64, dtype=torch.uint8, device="cuda")
    p = dummy.data_ptr()
    code = awq.lib.awq_search_noalloc(p, p, 2, out, n_in, N, None, 4, 128, 0, grid, p, p, p, p,
                                      torch.cuda.current_stream().cuda_stream)
    assert code == 2   # AWQ_ERR_UNSUPPORTED
