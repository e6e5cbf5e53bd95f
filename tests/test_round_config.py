"""Host-side checks of the round driver's configuration (CPU, no launch): tree
sizes, the sampled-draft invariant (every candidate kept), buffer sizes, and that
every benchmarked configuration respects the library's limits."""
import os
import sys

import pytest
import torch

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
sys.path.insert(0, ROOT)


@pytest.fixture(scope="module")
def rnd():
    from eagle_speculative_decoding_round_gb300 import build
    build.build()
    from eagle_speculative_decoding_round_gb300 import round as rnd
    return rnd


def small(rnd, **kw):
    base = dict(B=2, N=6, D=2, k=2, W=2, H=4, KVH=2, hd=64, d=256, V=512, L=1, max_kv_len=64, dtype="f32")
    base.update(kw)
    return rnd.RoundConfig(**base)


def test_frontier_sizes(rnd):
    c = small(rnd, D=4, k=3, W=5)
    sizes, n = c.frontier_sizes()
    assert sizes == [(1, 0), (3, 3), (5, 12), (5, 27)] and n == 42
    c = small(rnd, D=3, k=1, W=1)
    assert c.frontier_sizes() == ([(1, 0), (1, 1), (1, 2)], 3)


def test_sampled_rounds_keep_every_candidate(rnd):
    pt = torch.zeros((2, 2), dtype=torch.int32)
    with pytest.raises(ValueError, match="keep every candidate"):
        rnd.RoundBuffers(small(rnd, sampled=True, N=5), pt, 4, device="cpu")
    b = rnd.RoundBuffers(small(rnd, sampled=True, N=6), pt, 4, device="cpu")
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3
    assert b.q_stats.numel() == 2 * (6 + 1) * e3.QSTAT_BYTES
    assert tuple(b.node_cand.shape) == (2, 7)


def test_benchmarked_configurations_fit_the_library(rnd):
    import bench
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3
    for name, c in bench.CONFIGS.items():
        cfg = small(rnd, B=c["B"], N=c["N"], D=c["D"], k=c["k"], W=c["W"], V=c["V"])
        sizes, n_cand = cfg.frontier_sizes()
        assert 1 <= c["N"] <= min(n_cand, 255), name
        assert c["D"] <= 16 and c["k"] <= 32, name
        assert all(F * c["k"] <= 2048 for F, _ in sizes), name
        assert n_cand <= 4096, name
        if c.get("sampled"):
            assert c["N"] == n_cand, name  # drawn children are never dropped
        assert c["workload"], name
        assert c["temps"] == "mixed" or len(c["temps"]) in (1, c["B"]), name
    assert e3.E3_ACCEPT_SAMPLED == 1
