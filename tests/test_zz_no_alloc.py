"""eagle3_fuse_noalloc: fusion for callers that cannot allocate device memory.

Such callers (an allocator-free serving loop, an embedder without a device
allocator) cannot hand eagle3_fuse a workspace; this entry point keeps its
split-K scratch in a fixed array inside the library.  The test calls it through
the C ABI twice in a row, with different inputs, and checks each result against
eagle3_fuse on the same inputs, within the bf16 tolerance of the other tests.
This file is collected last so that a failure here leaves every other result in.
"""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_round_gb300 import synth
from gpu_util import assert_close, bf16_dev, host

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3


def fused_inputs(seed, M, d, dout):
    hs = [bf16_dev(synth.normal(seed, f"na_h{i}", (M, d), 0.02))[0] for i in range(3)]
    W = bf16_dev(synth.normal(seed, "na_W", (dout, 3 * d), 0.02))[0]
    bias = torch.from_numpy(synth.normal(seed, "na_b", (dout,), 0.02)).cuda()
    return hs, W, bias


def test_fuse_noalloc_matches_fuse_on_two_calls_in_a_row():
    M, d, dout = 7, 4096, 4096  # 8B-shaped fusion, 7 committed tokens
    need = e3.eagle3_fuse_workspace_bytes(M, d, dout, e3.E3_BF16)
    assert 0 < need <= e3.eagle3_fuse_noalloc_max_scratch_bytes()
    for seed in (11, 12):
        hs, W, bias = fused_inputs(seed, M, d, dout)
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        ref = torch.empty((M, dout), dtype=torch.bfloat16, device="cuda")
        e3.eagle3_fuse(*hs, W, bias, ref, M, d, dout, e3.E3_BF16, ws, need)
        got = torch.full((M, dout), float("nan"), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        e3.eagle3_fuse_noalloc(*hs, W, bias, got, M, d, dout, e3.E3_BF16, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_close(host(got), host(ref), 2e-2, f"noalloc fuse, call with seed {seed}")


def test_fuse_noalloc_rejects_shapes_beyond_its_scratch():
    M, d, dout = 4096, 4096, 4096
    assert e3.eagle3_fuse_workspace_bytes(M, d, dout, e3.E3_BF16) > e3.eagle3_fuse_noalloc_max_scratch_bytes()
    x = torch.zeros((M, d), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((dout, 3 * d), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((M, dout), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(e3.E3Error) as ei:
        e3.eagle3_fuse_noalloc(x, x, x, W, None, g, M, d, dout, e3.E3_BF16)
    assert ei.value.status == 4  # E3_ERR_CAPACITY, raised before any launch
