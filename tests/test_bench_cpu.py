"""The benchmark's CPU-baseline leg (the oracle timed over a whole round, or on a
sample of one) runs end to end on a tiny workload held in CPU tensors, for top-k
and for sampled drafts (no GPU: the oracle only reads the workload's buffers)."""
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
    Kall = t(L, npages, KVH, ps, hd)
    Vall = t(L, npages, KVH, ps, hd)
    pages = torch.tensor(sorted({int(pt[b, q]) for b in range(B) for q in range(P // ps, (P + R - 1) // ps + 1)}))
    bufs = types.SimpleNamespace(
        h=[t(cfg.M, cfg.d) for _ in range(3)], W_f=t(cfg.d, 3 * cfg.d), K_all=Kall, V_all=Vall,
        O=[t(B, R, H, hd) for _ in range(L)], W_lm=t(V, H * hd), logits=t(B * R, V),
        tok=torch.from_numpy(tok), parent=torch.from_numpy(par), temp=torch.ones(B))
    st = bench.InputSet(drafts, [t(B, R, H, hd) for _ in range(L)], torch.full((B,), 3, dtype=torch.int32))
    st.pages, st.snapK, st.snapV = pages, Kall.index_select(1, pages), Vall.index_select(1, pages)
    uni = [(torch.from_numpy(synth.uniforms(1, synth.PURPOSE_ACCEPT, B, R).view(np.int32)),
            torch.from_numpy(synth.uniforms(1, synth.PURPOSE_BONUS, B, R).view(np.int32)))]

    class W:
        pass
    w = W()
    w.bufs, w.cfg, w.c, w.pt, w.sets, w.uni = bufs, cfg, {"P": [P] * B, "temps": [1.0]}, pt, [st], uni
    w.kv_len0 = torch.full((B,), P, dtype=torch.int32)

    def use(k):
        s_ = w.sets[k % len(w.sets)]
        bufs.draft_logits, bufs.Q, bufs.root_tok = s_.drafts, s_.Q, s_.root_tok
        bufs.u_acc, bufs.u_bonus = w.uni[k % len(w.uni)]
    w.use = use
    return bench, w


@pytest.mark.parametrize("sampled", [False, True])
def test_oracle_sample_runs_on_a_tiny_workload(sampled):
    bench, w = fake_workload(sampled)
    times, n_layers = bench.oracle_sample(w, budget_s=0.5)
    assert n_layers >= 1 and all(v >= 0 for v in times.values())
    assert set(times) == {"fuse", "expand_build", "verify", "lmhead", "accept"}


@pytest.mark.parametrize("sampled", [False, True])
def test_oracle_whole_round_runs_on_a_tiny_workload(sampled):
    bench, w = fake_workload(sampled)
    times = bench.oracle_round(w, 0)
    assert set(times) == {"fuse", "expand_build", "verify", "lmhead", "accept", "compact"}
    assert all(v >= 0 for v in times.values())
    assert bench.whole_round_feasible(w)
    out = bench.cpu_baseline(w, budget_s=60.0)
    assert out["value"] > 0 and out["kind"] == "oracle" and out["threads_all"]["threads"] >= 1
    assert "estimate" not in out


def test_blas_thread_control_round_trips():
    import bench
    bt = BlasThreads = bench.BlasThreads()
    n = bt.threads()
    if n is None:
        pytest.skip("numpy's BLAS exports no thread setter here")
    assert BlasThreads.use(1) == 1
    assert bt.use(n) == n
