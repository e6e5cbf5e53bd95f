"""eagle3_fuse_noalloc: the feature fusion for callers that cannot allocate device memory.

Some callers of this library must not allocate on the GPU where they run the
fusion: a serving loop that may never block on or fragment the allocator, an
embedder with no device allocator of its own, or code under a policy that forbids
allocation at that point.  They cannot hand eagle3_fuse the workspace it needs for
its split-K partial sums, so this entry point keeps that scratch in a fixed 4 MiB
array inside the library.

The tests call it through the C ABI twice in a row -- first a larger shape, which
leaves non-zero partial sums over more of the shared array, then a smaller one of
another shape and tile width -- and check each result against eagle3_fuse on the
same inputs and against the oracle's fp64 fusion, within the bf16 tolerance of
the other tests.  They also check the documented row limit (25 rows at
d = d_out = 4096 fit, 26 are refused) and that a successful call clears the
error message of an earlier failed one.  This file is collected last, so a
failure here leaves every other result in.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_round_gb300 import synth
from gpu_util import assert_close, bf16_dev, host

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3

E3_ERR_CAPACITY = 4


def fused_inputs(seed, M, d, dout):
    hs = [bf16_dev(synth.normal(seed, f"na_h{i}", (M, d), 0.02)) for i in range(3)]
    W = bf16_dev(synth.normal(seed, "na_W", (dout, 3 * d), 0.02))
    bias = synth.normal(seed, "na_b", (dout,), 0.02)
    return hs, W, bias


def run_both(seed, M, d, dout):
    """eagle3_fuse (caller workspace) and eagle3_fuse_noalloc on the same inputs;
    returns (noalloc result, eagle3_fuse result, oracle) as host arrays."""
    hs, (W, W32), bias = fused_inputs(seed, M, d, dout)
    bias_t = torch.from_numpy(bias).cuda()
    need = e3.eagle3_fuse_workspace_bytes(M, d, dout, e3.E3_BF16)
    assert 0 < need <= e3.eagle3_fuse_noalloc_max_scratch_bytes()
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ref = torch.empty((M, dout), dtype=torch.bfloat16, device="cuda")
    e3.eagle3_fuse(*[h for h, _ in hs], W, bias_t, ref, M, d, dout, e3.E3_BF16, ws, need)
    got = torch.full((M, dout), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    e3.eagle3_fuse_noalloc(*[h for h, _ in hs], W, bias_t, got, M, d, dout, e3.E3_BF16, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle.fuse(*[h32 for _, h32 in hs], W32, bias)
    return host(got), host(ref), want


def test_fuse_noalloc_matches_fuse_and_oracle_on_two_calls_in_a_row():
    # 25 rows at 4096 -> 4096 fill almost all of the fixed scratch; the second call
    # (7 rows, 2048 -> 3072: another tile width and split count) reads a region the
    # first call left full of its own partial sums
    for seed, (M, d, dout) in ((11, (25, 4096, 4096)), (12, (7, 2048, 3072))):
        got, ref, want = run_both(seed, M, d, dout)
        assert_close(got, ref, 2e-2, f"noalloc vs eagle3_fuse, M={M}")
        assert_close(got, want, 2e-2, f"noalloc vs oracle, M={M}")


def test_fuse_noalloc_row_limit_at_4096():
    d = dout = 4096
    cap = e3.eagle3_fuse_noalloc_max_scratch_bytes()
    assert e3.eagle3_fuse_workspace_bytes(25, d, dout, e3.E3_BF16) <= cap
    assert e3.eagle3_fuse_workspace_bytes(26, d, dout, e3.E3_BF16) > cap
    x = torch.zeros((26, d), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((dout, 3 * d), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((26, dout), dtype=torch.bfloat16, device="cuda")
    e3.eagle3_fuse_noalloc(x, x, x, W, None, g, 25, d, dout, e3.E3_BF16)  # fits
    with pytest.raises(e3.E3Error) as ei:
        e3.eagle3_fuse_noalloc(x, x, x, W, None, g, 26, d, dout, e3.E3_BF16)
    assert ei.value.status == E3_ERR_CAPACITY  # refused on the host, before any launch
    torch.cuda.synchronize()


def test_fuse_noalloc_clears_the_error_of_an_earlier_call():
    M, d, dout = 4096, 4096, 4096
    assert e3.eagle3_fuse_workspace_bytes(M, d, dout, e3.E3_BF16) > e3.eagle3_fuse_noalloc_max_scratch_bytes()
    x = torch.zeros((M, d), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((dout, 3 * d), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((M, dout), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(e3.E3Error) as ei:
        e3.eagle3_fuse_noalloc(x, x, x, W, None, g, M, d, dout, e3.E3_BF16)
    assert ei.value.status == E3_ERR_CAPACITY
    assert e3.last_error() != ""
    e3.eagle3_fuse_noalloc(x, x, x, W, None, g, 7, d, dout, e3.E3_BF16)
    torch.cuda.synchronize()
    assert e3.last_error() == ""
    assert np.all(host(g[:7]) == 0.0)
