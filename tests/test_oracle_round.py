"""Round-level pins for the oracle (CPU): greedy acceptance equals sequential
decoding, sampling is lossless (chi-square), the pages' acceptance example,
and KV compaction semantics."""
import json
import os

import numpy as np
import pytest
from scipy.special import softmax
from scipy.stats import chi2

import oracle
from eagle_speculative_decoding_round_gb300 import synth
from roundlib import TinySetup

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def oracle_round(ts: TinySetup, T: float):
    """Draft (expand per depth), build, verify, logits, accept, compact -- all oracle."""
    c = oracle.new_cands(ts.n_cand)
    fid = np.array([-1], np.int32)
    fsc = np.zeros(1, np.float32)
    fpath = {-1: [ts.root_tok]}
    off = 0
    for d in range(1, ts.D + 1):
        z = np.stack([ts.draft_logits(fpath[int(f)], int(f)) for f in fid])
        nid, nsc = oracle.expand(z, ts.k, ts.W, fsc, fid, d, off, c)
        for i in range(off, off + len(fid) * ts.k):
            fpath[i] = fpath[int(c["parent"][i])] + [int(c["tok"][i])]
        off += len(fid) * ts.k
        fid, fsc = nid, nsc
    tree = oracle.build_tree(c, off, off, ts.root_tok, ts.P)
    R = off + 1
    pt, Kc, Vc = ts.make_cache(R)
    ts.write_tree_kv(Kc, Vc, pt, tree)
    Q = ts.tree_q(tree)
    O, _ = oracle.tree_verify_attn(Q, Kc, Vc, pt, np.array([ts.P], np.int32), tree["parent"][None], ts.scale)
    logits = oracle.lmhead_logits(O.reshape(R, -1), ts.tt.W_lm).astype(np.float32)
    ua = synth.uniforms(ts.seed, synth.PURPOSE_ACCEPT, 1, R)[0]
    ub = synth.uniforms(ts.seed, synth.PURPOSE_BONUS, 1, R)[0]
    acc, path, out = oracle.accept(tree, logits, T, ua, ub, ts.D)
    (K2, V2), kv2 = oracle.kv_compact([Kc, Vc], pt, np.array([ts.P], np.int32), path[None], np.array([acc]))
    return dict(tree=tree, logits=logits, acc=acc, path=path, out=out, K=K2, V=V2, kv_len=kv2, pt=pt)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_greedy_round_equals_sequential_decoding(seed):
    ts = TinySetup(seed, noise=0.02 if seed % 2 == 0 else 3.0)
    r = oracle_round(ts, T=0.0)
    acc = r["acc"]
    seq = ts.sequential_greedy(acc + 1)
    assert list(r["out"][:acc + 1]) == seq[1:acc + 2]
    assert r["kv_len"][0] == ts.P + 1 + acc
    # committed KV rows P..P+acc equal the sequential run's rows
    ps = ts.page_size
    for j in range(acc + 1):
        pos = ts.P + j
        assert np.array_equal(r["K"][r["pt"][0, pos // ps], :, pos % ps], ts.tt.k(seq[j], pos))
        assert np.array_equal(r["V"][r["pt"][0, pos // ps], :, pos % ps], ts.tt.v(seq[j], pos))
    if seed == 0:
        assert acc == ts.D  # low draft noise: the whole chain of argmaxes is in the tree


def chi_square(counts, probs, min_expected=5.0):
    n = counts.sum()
    exp = probs * n
    keep = exp >= min_expected
    c = np.append(counts[keep], counts[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    if e[-1] == 0:
        c, e = c[:-1], e[:-1]
    stat = ((c - e) ** 2 / e).sum()
    return stat, len(c) - 1


def full_binary_tree(D):
    parent = [-1]
    for d in range(1, D + 1):
        start = len(parent) - 2 ** (d - 1)
        for p in range(start, start + 2 ** (d - 1)):
            parent += [p, p]
    return np.array(parent, np.int32)


def test_sampling_is_lossless_chi_square():
    """[SpecForge] the output distribution equals the target's: first emitted token
    ~ p_root, and the second token given the first is an accepted child c ~ p_c."""
    V, D, n, T = 16, 3, 200_000, 1.0
    parent = full_binary_tree(D)
    R = len(parent)
    rng = np.random.default_rng(123)
    logits = (rng.standard_normal((R, V)) * 1.0).astype(np.float32)
    tok = np.zeros(R, np.int32)
    for u in range(R):  # children of u carry the two highest-logit tokens of row u
        kids = [c for c in range(R) if parent[c] == u]
        top = np.argsort(-logits[u], kind="stable")[:len(kids)]
        for c, t in zip(kids, top):
            tok[c] = t
    tok[0] = 0
    ua = synth.uniforms(77, synth.PURPOSE_ACCEPT, n, R)
    ub = synth.uniforms(77, synth.PURPOSE_BONUS, n, R)
    acc, path, out = oracle.accept_many(tok, parent, D, logits, T, ua, ub)
    p = softmax(logits.astype(np.float64) / T, axis=1)
    crit = chi2.ppf(1 - 1e-3, V - 1)
    stat, dof = chi_square(np.bincount(out[:, 0], minlength=V).astype(float), p[0])
    assert stat < chi2.ppf(1 - 1e-3, dof), (stat, dof)
    for c in [1, 2]:
        sel = out[:, 0] == tok[c]
        assert (path[sel, 1] == c).all()  # a child token can only be emitted by acceptance
        stat, dof = chi_square(np.bincount(out[sel, 1], minlength=V).astype(float), p[c])
        assert stat < chi2.ppf(1 - 1e-3, dof), (c, stat, dof)
    assert crit > 37.6 and crit < 37.8


def test_sampling_test_detects_a_planted_mistake():
    """Power check: drawing the bonus from the full row instead of the residual
    (a plausible bug) must fail the same chi-square test."""
    V, T, n = 16, 1.0, 200_000
    rng = np.random.default_rng(123)
    z = (rng.standard_normal(V)).astype(np.float64)
    p = softmax(z)
    top2 = np.argsort(-z)[:2]
    u = np.random.default_rng(5).random((n, 3))
    out = np.zeros(n, np.int64)
    for i in range(n):
        if u[i, 0] < p[top2[0]]:
            out[i] = top2[0]
        elif u[i, 1] < p[top2[1]] / (1 - p[top2[0]]):
            out[i] = top2[1]
        else:  # planted bug: sample from p, not from the residual
            out[i] = np.searchsorted(np.cumsum(p), u[i, 2] * p.sum())
    stat, dof = chi_square(np.bincount(out, minlength=V).astype(float), p)
    assert stat > chi2.ppf(1 - 1e-3, dof)


def test_pages_acceptance_example():
    fx = json.load(open(os.path.join(GOLD, "dflash_accept_example.json")))
    pE, pF, pG = fx["accept_prob"]
    V = 8
    E, F_, G, altF, altG = 1, 2, 3, 4, 5
    tok = np.array([0, E, F_, G], np.int32)
    parent = np.array([-1, 0, 1, 2], np.int32)
    z = np.full((4, V), -100.0, np.float32)
    z[0, E] = 0.0                      # p(E) = 1.0
    z[1, F_], z[1, altF] = np.log(pF), np.log(1 - pF)
    z[2, G], z[2, altG] = np.log(pG), np.log(1 - pG)
    z[3, 6] = 0.0
    names = {E: "E", F_: "F", G: "G"}
    for case in ("a", "b"):
        u = fx[f"uniforms_case_{case}"]
        ua = np.zeros(4, np.uint32)
        ua[1:] = [int(x * 2 ** 32) for x in u]
        ub = np.zeros(4, np.uint32)
        acc, path, out = oracle.accept({"tok": tok, "parent": parent}, z, 1.0, ua, ub, 3)
        assert [names[int(t)] for t in out[:acc]] == fx[f"accepted_case_{case}"]
        if case == "a":
            assert out[acc] == altG  # correction drawn from the residual at F
        else:
            assert out[acc] == 6


def test_compaction_overlap_and_untouched_rows():
    """Path [0, 3, 4, 5]: slot P+1 takes old P+3, P+2 old P+4, P+3 old P+5 (a
    source slot that is also another element's destination)."""
    ps, KVH, hd, P, R = 4, 2, 3, 10, 8
    pt, npages = synth.page_table(1, [P + R, P + R], ps)
    cache = np.zeros((npages, KVH, ps, hd), np.float32)
    for b in range(2):
        for t in range(P + R):
            cache[pt[b, t // ps], :, t % ps, :] = 1000 * b + t
    path = np.array([[0, 3, 4, 5], [0, 1, -1, -1]], np.int32)
    acc = np.array([3, 0])
    (new,), kv = oracle.kv_compact([cache], pt, np.array([P, P], np.int32), path, acc)
    def val(b, t):
        return new[pt[b, t // ps], 0, t % ps, 0]
    assert [val(0, P + j) for j in range(4)] == [P, P + 3, P + 4, P + 5]
    assert all(val(0, t) == t for t in list(range(P)) + list(range(P + 4, P + R)))
    assert all(val(1, t) == 1000 + t for t in range(P + R))
    assert list(kv) == [P + 4, P + 1]
