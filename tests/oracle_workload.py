"""Whole-round inputs for the GPU parity tests, built without the library under test.

The benchmark's own workload (``bench.Workload``: buffers, seeded random K/V,
weights, token-keyed tree Q/K/V tables, launch configuration) is created with
``drafts=None``; then this module fills in what the benchmark's draft stand-in
would compute on the GPU, using only the oracle, numpy and torch copies:

* W_lm is scaled so that the roots' target logits have std ~ 4 (the logits are
  the oracle's fp64 LM head of the oracle's fp64 last-layer attention);
* at each depth, the draft logits of a frontier node are the oracle's fp64 target
  logits of that node (its mini-tree: the frontier and its ancestors, ancestor-only
  attention over the prefix) plus seeded N(0, noise^2);
* the frontier, the candidates and the final tree come from the oracle's
  expansion and tree build on those rows;
* the final tree's Q (every layer) and K/V (slots P .. P+R-1) are the token-keyed
  table rows, written with torch indexing.

So no input of the parity test has passed through libeagle3.
"""
import math
import os
import sys

import numpy as np
import torch

import oracle
from eagle_speculative_decoding_round_gb300 import synth

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
import bench  # noqa: E402


def f32(t):
    return t.float().cpu().numpy()


def _ancestor_masks(par):
    B, Rm = par.shape
    mask = np.zeros((B, Rm, (Rm + 63) // 64), np.uint64)
    for bb in range(B):
        for i in range(Rm):
            j = i
            while j >= 0:
                mask[bb, i, j >> 6] |= np.uint64(1 << (j & 63))
                j = int(par[bb, j])
    return mask


def oracle_workload(name, seed=11):
    w = bench.Workload(name, seed=seed, drafts=None)
    b, c = w.bufs, w.cfg
    st = w.add_set(0)
    B, V, ps = c.B, c.V, c.page_size
    P = np.asarray(w.c["P"], np.int64)
    pt = w.pt
    Kl, Vl = f32(b.K[c.L - 1]), f32(b.Vc[c.L - 1])
    Qtab, Ktab, Vtab = f32(w.Qtab), f32(w.Ktab), f32(w.Vtab)
    roots = st.root_tok.cpu().numpy().astype(np.int64)
    sm = 1.0 / math.sqrt(c.hd)

    def target_rows(tok, par, rows, W64):
        """fp64 target logits of the (b, i) rows of per-request mini-trees (tok/par
        [B, R']): the mini-tree's K/V at slots P .. P+R'-1 of the last layer."""
        Rm = tok.shape[1]
        key = tok % bench.TAB_ROWS
        for bb in range(B):
            for i in range(Rm):
                slot = int(P[bb]) + i
                Kl[pt[bb, slot // ps], :, slot % ps] = Ktab[key[bb, i]]
                Vl[pt[bb, slot // ps], :, slot % ps] = Vtab[key[bb, i]]
        O, _ = oracle.tree_verify_attn_dense(Qtab[key], Kl, Vl, pt, P, _ancestor_masks(par), sm)
        h = np.stack([O[bb, i].reshape(-1) for bb, i in rows])
        return oracle.lmhead_logits(h, W64)

    # calibration: target logits of the roots with std ~ 4
    W64 = f32(b.W_lm).astype(np.float64)
    z = target_rows(roots[:, None], np.full((B, 1), -1), [(bb, 0) for bb in range(B)], W64)
    scale = 4.0 / float(z.std())
    b.W_lm.copy_((b.W_lm.float() * scale).to(c.tdtype))
    W64 = f32(b.W_lm).astype(np.float64)

    sizes, n_cand = c.frontier_sizes()
    cands = [oracle.new_cands(n_cand) for _ in range(B)]
    fid = [np.array([-1], np.int32) for _ in range(B)]
    fsc = [np.zeros(1, np.float32) for _ in range(B)]
    paths = [{-1: [int(roots[bb])]} for bb in range(B)]
    for di, (F, off) in enumerate(sizes):
        tok, par, rows = bench.mini_trees(paths, np.stack(fid), roots)
        zt = target_rows(tok, par, rows, W64).reshape(B, F, V)
        noise = synth.normal(seed, f"oracle_draft_noise{di}", (B, F, V), float(w.c["noise"]))
        d = (zt + noise).astype(np.float32)
        st.drafts[di].copy_(torch.from_numpy(d))
        for bb in range(B):
            if c.sampled:
                fid[bb], fsc[bb], _, _ = oracle.expand_sampled(d[bb], c.k, c.W, fsc[bb], fid[bb], di + 1, off,
                                                               cands[bb], c.draw_seed, bb)
            else:
                fid[bb], fsc[bb] = oracle.expand(d[bb], c.k, c.W, fsc[bb], fid[bb], di + 1, off, cands[bb])
            for i in range(off, off + F * c.k):
                paths[bb][i] = paths[bb][int(cands[bb]["parent"][i])] + [int(cands[bb]["tok"][i])]
    trees = [oracle.build_tree(cands[bb], n_cand, c.N, int(roots[bb]), int(P[bb])) for bb in range(B)]
    toks = torch.from_numpy(np.stack([t["tok"] for t in trees]).astype(np.int64)).to(w.device)
    w.finish_set(st, toks)
    w.use(0)
    torch.cuda.synchronize()
    return w
