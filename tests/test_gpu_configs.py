"""Every benchmarked configuration, one whole round on the GPU in the benchmark's
own launch configuration (its workload, buffers and round function), checked
against the oracle.  The round's inputs are built without the library under test
(tests/oracle_workload.py: draft logits = the oracle's fp64 target logits of each
frontier node + seeded noise; trees from the oracle's expansion):

  fusion        every output element, within the dtype tolerance
  expansion     every candidate of every request and depth, bit-exact (drawn
                children for the sampled configurations)
  tree          tokens, parents, depths, positions and mask rows, bit-exact
  verify        the whole O and lse tensors of the last layer (every request,
                node and head; the 65536-key prefix and the 70B batch included)
                against the oracle's dense masked form, and sampled rows of the
                first layer, within the dtype tolerance (norm-wise over the tensor)
  LM head       whole vocabulary rows (every row up to 64, else 64 sampled rows)
                within tolerance; the softmax statistics of every row bit-exact
                from the GPU logits
  accept        accepted length, path and emitted tokens, bit-exact (the
                min(1, p/q) rule for the sampled configurations)
  compaction    slots P + j of sampled layers hold what slot P + path[j] held
"""
import math
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from gpu_util import assert_close
from oracle_workload import oracle_workload

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
sys.path.insert(0, ROOT)

pytestmark = pytest.mark.gpu


def host(t):
    return t.cpu().numpy()


def f32(t):
    return t.float().cpu().numpy()


@pytest.mark.parametrize("name", ["tiny", "8b", "8b_d8", "8b_chain3", "8b_sampled", "8b_chain3_sampled", "batched",
                                  "long", "70b"])
def test_round_matches_oracle(name):
    w = oracle_workload(name, seed=11)
    b, c = w.bufs, w.cfg
    B, R, L = c.B, c.R, c.L
    rng = np.random.default_rng(7)
    tol = 2e-2 if c.dtype == "bf16" else 1e-5

    # what the round reads, before it runs
    hs = [f32(t) for t in b.h]
    drafts = [host(x) for x in b.draft_logits]
    P = host(w.kv_len0)
    layers = sorted({0, L - 1})
    Kpre = {l: f32(b.K[l]) for l in layers}
    Vpre = {l: f32(b.Vc[l]) for l in layers}
    Qs = {l: f32(b.Q[l]) for l in layers}

    w.round()
    torch.cuda.synchronize()
    assert int(b.dev_err.item()) == 0

    # fusion: every output element
    assert_close(f32(b.g), oracle.fuse(hs[0], hs[1], hs[2], f32(b.W_f)), tol, "fusion")

    # expansion and tree, per request
    sizes, n_cand = c.frontier_sizes()
    ctok, cpar, cdep, csc = host(b.c_tok), host(b.c_parent), host(b.c_depth), host(b.c_score)
    roots = host(b.root_tok)
    tok, par, dep, pos, mask = host(b.tok), host(b.parent), host(b.depth), host(b.pos), host(b.mask)
    qrows = []  # sampled drafts: candidate (root -1) -> the draft row it was expanded with
    for bb in range(B):
        cands = oracle.new_cands(n_cand)
        fid, fsc = np.array([-1], np.int32), np.zeros(1, np.float32)
        rows = {}
        for di, (F, off) in enumerate(sizes):
            if c.sampled:
                for f in range(F):
                    rows[int(fid[f])] = drafts[di][bb][f]
                fid, fsc, _, _ = oracle.expand_sampled(drafts[di][bb][:F], c.k, c.W, fsc, fid, di + 1, off, cands,
                                                       c.draw_seed, bb)
            else:
                fid, fsc = oracle.expand(drafts[di][bb][:F], c.k, c.W, fsc, fid, di + 1, off, cands)
        qrows.append(rows)
        assert np.array_equal(ctok[bb], cands["tok"]), (name, bb)
        assert np.array_equal(cpar[bb], cands["parent"]), (name, bb)
        assert np.array_equal(cdep[bb], cands["depth"]), (name, bb)
        assert np.array_equal(csc[bb].view(np.uint32), cands["score"].view(np.uint32)), (name, bb)
        tree = oracle.build_tree(cands, n_cand, c.N, int(roots[bb]), int(P[bb]))
        for key, got in (("tok", tok), ("parent", par), ("depth", dep), ("pos", pos)):
            assert np.array_equal(got[bb], tree[key]), (name, key, bb)
        if c.sampled:
            assert np.array_equal(host(b.node_cand)[bb], tree["node_cand"]), (name, bb)
        assert np.array_equal(mask[bb].view(np.uint64), tree["mask"]), (name, bb)

    # verify: the whole last layer (dense masked form), sampled rows of the first
    sm = 1.0 / math.sqrt(c.hd)
    Oref, lref = oracle.tree_verify_attn_dense(Qs[L - 1], Kpre[L - 1], Vpre[L - 1], w.pt, P, mask.view(np.uint64), sm)
    assert_close(f32(b.O[L - 1]), Oref, tol, f"O layer {L - 1} (whole tensor)")
    assert_close(host(b.lse[L - 1]), lref, tol, f"lse layer {L - 1} (whole tensor)")
    if L > 1:
        rows = [(int(rng.integers(B)), int(rng.integers(R)), int(rng.integers(c.H))) for _ in range(12)]
        Orow, lrow = oracle.tree_verify_attn_rows(Qs[0], Kpre[0], Vpre[0], w.pt, P, par, sm, rows)
        Og, lg = f32(b.O[0]), host(b.lse[0])
        assert_close(np.stack([Og[bb, i, h] for bb, i, h in rows]), Orow, tol, "O layer 0")
        assert_close(np.array([lg[bb, i, h] for bb, i, h in rows]), lrow, tol, "lse layer 0")

    # LM head: whole vocabulary rows; statistics of every row
    z = host(b.logits)
    hrow = f32(b.O[L - 1]).reshape(B * R, c.H * c.hd)
    sel = np.arange(B * R) if B * R <= 64 else np.sort(rng.choice(B * R, 64, replace=False))
    assert_close(z[sel], oracle.lmhead_logits(hrow[sel], f32(b.W_lm)), tol, "logits")
    m, Q, am, bad = oracle.row_stats(z, host(b.temp_rows))
    assert not bad.any()
    assert np.array_equal(host(b.row_max).view(np.uint32), m.view(np.uint32))
    assert np.array_equal(host(b.row_Q).view(np.uint64), Q)
    assert np.array_equal(host(b.row_argmax), am)

    # accept, per request
    temps, ua, ub = host(b.temp), host(b.u_acc).view(np.uint32), host(b.u_bonus).view(np.uint32)
    acc, path, out = host(b.acc_len), host(b.path), host(b.out_tok)
    nc = host(b.node_cand)
    for bb in range(B):
        tree_b = {"tok": tok[bb], "parent": par[bb]}
        if c.sampled:
            qlog = np.zeros((R, c.V), np.float32)
            for u in range(R):
                key = -1 if u == 0 else int(nc[bb, u])
                if key in qrows[bb]:
                    qlog[u] = qrows[bb][key]
            a, p, o = oracle.accept_sampled(tree_b, z[bb * R:(bb + 1) * R], temps[bb], qlog, 1.0, ua[bb], ub[bb], c.D)
        else:
            a, p, o = oracle.accept(tree_b, z[bb * R:(bb + 1) * R], temps[bb], ua[bb], ub[bb], c.D)
        assert acc[bb] == a and np.array_equal(path[bb], p) and np.array_equal(out[bb], o), (name, bb)
    assert np.array_equal(host(b.kv_len), P + 1 + acc)

    # compaction: logical slot P + j now holds what P + path[j] held (K and V)
    for l in layers:
        for pre, cache in ((Kpre[l], b.K[l]), (Vpre[l], b.Vc[l])):
            post = f32(cache)
            for bb in range(B):
                a = int(acc[bb])
                before = oracle.gather_tokens(pre, w.pt[bb], int(P[bb]), int(P[bb]) + R)
                after = oracle.gather_tokens(post, w.pt[bb], int(P[bb]), int(P[bb]) + a + 1)
                assert np.array_equal(after, before[path[bb][:a + 1]]), (name, l, bb)

    del w, b
    torch.cuda.empty_cache()
