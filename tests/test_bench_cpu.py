"""The benchmark's CPU-baseline leg (the oracle timed on a sample of a round)
runs end to end on a tiny workload held in CPU tensors, for top-k and for
sampled drafts (no GPU: the sample only reads the workload's buffers)."""
import os
import sys
import types

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_round_gb300 import synth

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
sys.path.insert(0, ROOT)


def fake_workload(sampled: bool):
    import bench
    from eagle_speculative_decoding_round_gb300 import build
    build.build()
    from eagle_speculative_decoding_round_gb300.round import RoundConfig
    B, k, W, D, V, H, KVH, hd, L, P, ps = 2, 2, 2, 2, 64, 2, 1, 32, 2, 40, 16
    cfg = RoundConfig(B=B, N=6 if sampled else 4, D=D, k=k, W=W, H=H, KVH=KVH, hd=hd, d=H * hd, V=V, L=L,
                      max_kv_len=P, dtype="f32", page_size=ps, sampled=sampled, draw_seed=5)
    R = cfg.R
    sizes, n_cand = cfg.frontier_sizes()
    rng = np.random.default_rng(1)
    pt, npages = synth.page_table(3, [P + R] * B, ps)
    t = lambda *shape: torch.from_numpy(rng.standard_normal(shape).astype(np.float32))  # noqa: E731
    drafts = [t(B, F, V) for F, _ in sizes]
    tok = np.zeros((B, R), np.int32)
    par = np.zeros((B, R), np.int32)
    for b in range(B):  # the tree the round would build from these drafts
        c = oracle.new_cands(n_cand)
        fid, fsc = np.array([-1], np.int32), np.zeros(1, np.float32)
        for di, (F, off) in enumerate(sizes):
            z = drafts[di][b].numpy()
            if sampled:
                fid, fsc, _, _ = oracle.expand_sampled(z, k, W, fsc, fid, di + 1, off, c, cfg.draw_seed, b)
            else:
                fid, fsc = oracle.expand(z, k, W, fsc, fid, di + 1, off, c)
        tr = oracle.build_tree(c, n_cand, cfg.N, 3, P)
        tok[b], par[b] = tr["tok"], tr["parent"]
    bufs = types.SimpleNamespace(
        h=[t(cfg.M, cfg.d) for _ in range(3)], W_f=t(cfg.d, 3 * cfg.d), draft_logits=drafts,
        root_tok=torch.full((B,), 3, dtype=torch.int32), K=[t(npages, KVH, ps, hd) for _ in range(L)],
        Vc=[t(npages, KVH, ps, hd) for _ in range(L)], Q=[t(B, R, H, hd) for _ in range(L)],
        O=[t(B, R, H, hd) for _ in range(L)], W_lm=t(V, H * hd), logits=t(B * R, V),
        tok=torch.from_numpy(tok), parent=torch.from_numpy(par),
        u_acc=torch.from_numpy(synth.uniforms(1, synth.PURPOSE_ACCEPT, B, R).view(np.int32)),
        u_bonus=torch.from_numpy(synth.uniforms(1, synth.PURPOSE_BONUS, B, R).view(np.int32)))
    w = types.SimpleNamespace(bufs=bufs, cfg=cfg, c={"P": [P] * B, "temps": [1.0]}, pt=pt,
                              kv_len0=torch.full((B,), P, dtype=torch.int32))
    return bench, w


@pytest.mark.parametrize("sampled", [False, True])
def test_oracle_sample_runs_on_a_tiny_workload(sampled):
    bench, w = fake_workload(sampled)
    o = bench.oracle_sample(w, budget_s=0.5)
    assert o["round_s"] > 0 and o["verify_layers"] >= 1 and o["cores"] >= 1
    assert set(o["times"]) == {"fuse", "expand_build", "verify", "lmhead", "accept"}
