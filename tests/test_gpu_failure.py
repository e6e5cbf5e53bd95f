"""Failure detection on the GPU without a fault: a bounded wait that runs out.

With the self-test bit E3_KV_SELFTEST_STALL, tree_verify_attn's tensor-core kernel
makes its MMA thread wait on an mbarrier that nothing arrives on.  The wait is
bounded (about a second of %globaltimer); when it runs out the kernel raises its
abort flag, the other warps leave their loops, every copy it issued is waited for,
its tensor memory is freed, and E3_DEV_ERR_TIMEOUT is OR-ed into dev_err, which the
host reads.  The context must stay usable: the same call without the bit, on the
same buffers, right after, is exact against the oracle (a leaked tensor-memory
allocation or a lost copy would show up there).  Covers the cluster-merge split
(8B shape, 2048-key prefix) and the one-wave split with the merge kernel (12000 keys).
"""
import math
import time

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_round_gb300 import synth
from gpu_util import assert_close, kv_paged, random_tree

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3
    from test_gpu_steps import mask_from_parent, run_gpu_verify


@pytest.mark.parametrize("lens", [[2048], [12000]])
def test_verify_wait_runs_out_and_the_context_survives(lens):
    R, H, KVH, hd, ps, D = 61, 32, 8, 128, 64, 6
    seed = 4242 + lens[0]
    pt, npages, K, Vc = kv_paged(seed, lens, R, KVH, hd, ps, 1.0, "bf16")
    Q = synth.to_bf16_f32(synth.normal(seed, "Q", (1, R, H, hd), 1.0))
    par = random_tree(np.random.default_rng(seed), R, D)[0][None]
    mask = np.stack([mask_from_parent(p) for p in par])
    t0 = time.perf_counter()
    _, _, err = run_gpu_verify(Q, K, Vc, pt, npages, lens, mask, H, KVH, hd, ps, "bf16",
                               flags=e3.E3_KV_SELFTEST_STALL | e3.E3_KV_PREFIX_STABLE)
    took = time.perf_counter() - t0
    assert err & e3.E3_DEV_ERR_TIMEOUT, f"dev_err {err:#x}: the stalled wait did not report a timeout"
    assert took >= 0.5, f"the stalled call returned after {took:.3f} s: the wait did not run its bound"
    # the same call, same buffers, no stall: exact, so nothing leaked and the context is sound
    O, lse, err = run_gpu_verify(Q, K, Vc, pt, npages, lens, mask, H, KVH, hd, ps, "bf16",
                                 flags=e3.E3_KV_PREFIX_STABLE)
    assert err == 0
    Oref, lref = oracle.tree_verify_attn_dense(Q, K, Vc, pt, np.array(lens), mask, 1.0 / math.sqrt(hd))
    assert_close(O, Oref, 2e-2, "O after a timeout")
    assert_close(lse, lref, 2e-2, "lse after a timeout")
    torch.cuda.synchronize()
