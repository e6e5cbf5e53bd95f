"""Pins for the oracle's sampled-draft mode (CPU): the random stream, the draw of
children without replacement, the acceptance rule min(1, p_res / q_res) with
its residual, and losslessness of whole rounds.

"EAGLE 系列与 DFlash", §四 DFlash: each draft token is accepted with probability
min(1, p_target / p_draft), the dice rolled left to right.  "SpecForge…",
先看 checkpoint 最终要参与什么计算: the correction at the rejection point keeps the
output distribution equal to the target's.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax
from scipy.stats import chi2

import oracle
from eagle_speculative_decoding_round_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")
GAMMA = 0x9E3779B97F4A7C15
M64 = 2 ** 64 - 1


def chi_square(counts, probs, min_expected=5.0):
    n = counts.sum()
    exp = probs * n
    keep = exp >= min_expected
    c = np.append(counts[keep], counts[~keep].sum())
    e = np.append(exp[keep], exp[~keep].sum())
    if e[-1] == 0:
        c, e = c[:-1], e[:-1]
    return ((c - e) ** 2 / e).sum(), len(c) - 1


def qprobs(z, inv_T=1.0):
    """The fixed-point draft distribution of one row: Q_j / sum Q (from the recipe)."""
    z = np.asarray(z, np.float32)
    s = (z * np.float32(inv_T)).astype(np.float32)
    m = s.max()
    Q = np.array([oracle.qmass(float(x), float(m)) for x in s], np.float64)
    return Q / Q.sum()


# ------------------------------------------------------------------ stream ----

def test_splitmix64_reference_vectors():
    """The published reference outputs of SplitMix64 (Vigna's splitmix64.c):
    seed 0 starts 0xe220a8397b1dcdaf, 0x6e789e6aa1b965f4; seed 1234567 starts
    6457827717110365317, 3203168211198807973, 9817491932198370423,
    4593380528125082431, 16408922859458223821."""
    assert oracle.splitmix64_at(0, 1) == 0xE220A8397B1DCDAF
    assert oracle.splitmix64_at(0, 2) == 0x6E789E6AA1B965F4
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
            16408922859458223821]
    assert [oracle.splitmix64_at(1234567, i) for i in range(1, 6)] == want
    # the input generators' finaliser is the same mix, applied to x + gamma
    for seed, i in [(3, 1), (2 ** 63 + 5, 77), (M64, 1 << 40)]:
        x = np.array([(seed + (i - 1) * GAMMA) & M64], np.uint64)
        assert int(synth.splitmix64(x)[0]) == oracle.splitmix64_at(seed, i)


def test_exp_variate_is_minus_log_of_the_stream_uniform():
    rng = np.random.default_rng(0)
    for _ in range(300):
        seed = int(rng.integers(0, 2 ** 63))
        b, d, f, j = (int(rng.integers(0, 64)), int(rng.integers(1, 9)), int(rng.integers(0, 64)),
                      int(rng.integers(0, 128256)))
        n = (b << 44) | (d << 36) | (f << 24) | j
        U = ((oracle.splitmix64_at(seed, n + 1) >> 40) + 1) / 2 ** 24
        E = oracle.exp_variate(seed, b, d, f, j)
        assert E >= 0.0
        assert abs(E - (-math.log(U))) <= 4e-7 * max(1.0, -math.log(U)) + 1e-7
    # the variates have the Exp(1) mean and variance
    E = np.array([oracle.exp_variate(11, 0, 1, 0, j) for j in range(20000)])
    assert abs(E.mean() - 1.0) < 0.03 and abs(E.var() - 1.0) < 0.08


# ------------------------------------------------------- sampled children ----

def draw_children(z, k, n, seed0=1000, inv_T=1.0):
    out = np.zeros((n, k), np.int64)
    for i in range(n):
        c = oracle.new_cands(k)
        oracle.expand_sampled(z[None], k, k, np.zeros(1, np.float32), np.array([-1], np.int32), 1, 0, c,
                              seed0 + i, 0, inv_T)
        out[i] = c["tok"]
    return out


def test_sampled_children_are_draws_without_replacement():
    """First child ~ q; second child given the first ~ q without the first;
    children distinct; a token of zero fixed-point mass is never drawn."""
    V, k, n = 8, 3, 40000
    z = np.array([2.0, 1.5, 1.0, 0.5, 0.0, -0.5, -1.0, -100.0], np.float32)
    q = qprobs(z)
    assert q[7] == 0.0
    ch = draw_children(z, k, n)
    assert all(len(set(r)) == k for r in ch[:2000])
    assert not (ch == 7).any()
    stat, dof = chi_square(np.bincount(ch[:, 0], minlength=V).astype(float), q)
    assert stat < chi2.ppf(1 - 1e-3, dof)
    sel = ch[:, 0] == 0
    q2 = q.copy()
    q2[0] = 0
    q2 /= q2.sum()
    stat, dof = chi_square(np.bincount(ch[sel, 1], minlength=V).astype(float), q2)
    assert stat < chi2.ppf(1 - 1e-3, dof)
    # power: the same draws do not fit the distribution without the removal
    stat, dof = chi_square(np.bincount(ch[sel, 1], minlength=V).astype(float), q)
    assert stat > chi2.ppf(1 - 1e-3, dof)


def test_ordered_pairs_of_draws_follow_the_without_replacement_law():
    """P(first = a, second = b) = q_a q_b / (1 - q_a) for a != b: chi-square over
    all 20 ordered pairs of a 5-token row."""
    V, n = 5, 30000
    z = np.array([1.2, 0.4, 0.0, -0.6, -1.5], np.float32)
    q = qprobs(z)
    ch = draw_children(z, 2, n, seed0=31)
    pairs = [(a, b) for a in range(V) for b in range(V) if a != b]
    p = np.array([q[a] * q[b] / (1 - q[a]) for a, b in pairs])
    assert abs(p.sum() - 1.0) < 1e-12
    idx = {pr: i for i, pr in enumerate(pairs)}
    counts = np.bincount([idx[(int(a), int(b))] for a, b in ch], minlength=len(pairs)).astype(float)
    stat, dof = chi_square(counts, p)
    assert stat < chi2.ppf(1 - 1e-3, dof)
    # power: the law that forgets the removal (pairs weighted q_a q_b, renormalised
    # over a != b) is rejected by the same draws
    p_wrong = np.array([q[a] * q[b] for a, b in pairs])
    p_wrong /= p_wrong.sum()
    stat, dof = chi_square(counts, p_wrong)
    assert stat > chi2.ppf(1 - 1e-3, dof)


def test_sampled_children_at_temperature_and_k_equal_V():
    V = 6
    z = np.array([1.0, 0.3, -0.2, 0.8, 0.0, -1.0], np.float32)
    ch = draw_children(z, 2, 20000, seed0=5, inv_T=0.5)
    stat, dof = chi_square(np.bincount(ch[:, 0], minlength=V).astype(float), qprobs(z, 0.5))
    assert stat < chi2.ppf(1 - 1e-3, dof)
    full = draw_children(z, V, 50, seed0=9)
    assert all(sorted(r) == list(range(V)) for r in full)


def test_expand_sampled_scores_frontier_and_stats():
    """Child scores are the path's draft log-probabilities; the next frontier is
    the W best children by score; the row statistics are the row's max and mass."""
    rng = np.random.default_rng(3)
    F, V, k, W = 3, 50, 4, 5
    z = (rng.standard_normal((F, V)) * 2).astype(np.float32)
    ps = np.array([-0.5, -1.25, -2.0], np.float32)
    pid = np.array([4, 7, 9], np.int32)
    c = oracle.new_cands(20 + F * k)
    nid, nsc, rm, rq = oracle.expand_sampled(z, k, W, ps, pid, 3, 20, c, 77, 2)
    for f in range(F):
        lp = z[f].astype(np.float64) - logsumexp(z[f].astype(np.float64))
        for r in range(k):
            ci = 20 + f * k + r
            t = c["tok"][ci]
            assert c["parent"][ci] == pid[f] and c["depth"][ci] == 3
            assert abs(c["score"][ci] - (ps[f] + lp[t])) < 1e-5
        assert rm[f] == z[f].max()
        assert abs(float(rq[f]) / 2 ** 40 - np.exp(z[f].astype(np.float64) - z[f].max()).sum()) < 1e-5 * V
    order = sorted(range(20, 20 + F * k), key=lambda i: (-c["score"][i], i))[:W]
    assert list(nid) == order and np.array_equal(nsc, c["score"][order])
    # another request index or seed gives other draws
    c2 = oracle.new_cands(20 + F * k)
    oracle.expand_sampled(z, k, W, ps, pid, 3, 20, c2, 77, 3)
    assert not np.array_equal(c["tok"], c2["tok"])


def test_tree_node_cand_maps_flat_nodes_to_candidates():
    rng = np.random.default_rng(4)
    V, k, W, D = 40, 3, 4, 3
    c = oracle.new_cands(3 + 12 + 12)
    fid, fsc, off = np.array([-1], np.int32), np.zeros(1, np.float32), 0
    for d in range(1, D + 1):
        z = (rng.standard_normal((len(fid), V)) * 2).astype(np.float32)
        fid, fsc = oracle.expand(z, k, W, fsc, fid, d, off, c)
        off += len(z) * k
    t = oracle.build_tree(c, off, 14, 5, 100)
    nc = t["node_cand"]
    assert nc[0] == -1 and len(set(nc[1:])) == 14
    for u in range(1, 15):
        assert c["tok"][nc[u]] == t["tok"][u] and c["depth"][nc[u]] == t["depth"][u]
        p = t["parent"][u]
        assert c["parent"][nc[u]] == (nc[p] if p > 0 else -1)


# -------------------------------------------------------------- acceptance ----

def chain(tokens):
    R = len(tokens) + 1
    return {"tok": np.array([0] + list(tokens), np.int32), "parent": np.arange(-1, R - 1, dtype=np.int32)}


def test_one_hot_draft_rows_reduce_to_the_point_mass_rule():
    """A draft that puts all its mass on the proposed token is the point-mass
    proposal of the deterministic mode: the two accept rules agree bit for bit."""
    rng = np.random.default_rng(8)
    V, D = 64, 4
    for trial in range(200):
        toks = rng.integers(0, V, D)
        tree = chain(toks)
        z = (rng.standard_normal((D + 1, V)) * 2).astype(np.float32)
        zq = np.full((D + 1, V), -200.0, np.float32)
        for u in range(D):
            zq[u, toks[u]] = 0.0
        ua = rng.integers(0, 2 ** 32, D + 1, dtype=np.uint64).astype(np.uint32)
        ub = rng.integers(0, 2 ** 32, D + 1, dtype=np.uint64).astype(np.uint32)
        T = [1.0, 0.7, 1.3][trial % 3]
        a1, p1, o1 = oracle.accept(tree, z, T, ua, ub, D)
        a2, p2, o2 = oracle.accept_sampled(tree, z, T, zq, 1.0, ua, ub, D)
        assert a1 == a2 and np.array_equal(p1, p2) and np.array_equal(o1, o2)


def test_draft_equal_to_target_accepts_every_draw():
    """q = p: the ratio is 1 for every drawn token."""
    rng = np.random.default_rng(9)
    V, D = 100, 5
    for trial in range(50):
        z = (rng.standard_normal((D + 1, V)) * 2).astype(np.float32)
        toks = rng.integers(0, V, D)
        ua = np.full(D + 1, 2 ** 32 - 1, np.uint32)
        ub = rng.integers(0, 2 ** 32, D + 1, dtype=np.uint64).astype(np.uint32)
        a, _, out = oracle.accept_sampled(chain(toks), z, 1.0, z, 1.0, ua, ub, D)
        assert a == D and list(out[:D]) == list(toks)


def test_greedy_target_is_the_argmax_walk():
    rng = np.random.default_rng(10)
    V, D = 30, 3
    z = (rng.standard_normal((D + 1, V)) * 2).astype(np.float32)
    toks = [int(np.argmax(z[0])), int(np.argmax(z[1])), (int(np.argmax(z[2])) + 1) % V]
    zq = (rng.standard_normal((D + 1, V))).astype(np.float32)
    a, _, out = oracle.accept_sampled(chain(toks), z, 0.0, zq, 1.0, np.zeros(D + 1, np.uint32),
                                      np.zeros(D + 1, np.uint32), D)
    assert a == 2 and list(out[:3]) == [toks[0], toks[1], int(np.argmax(z[2]))]


def test_pages_acceptance_example_sampled_chain():
    """The DFlash worked example with drafts sampled from q: per-position ratios
    p/q = 1.0, 0.89, 0.20 (p(E) >= q(E)); uniforms 0.5, 0.5, 0.5 accept E, F and
    reject G; with 0.1 at G it is accepted too.  The correction after G's
    rejection comes from max(0, p - q) at F."""
    fx = json.load(open(os.path.join(GOLD, "dflash_accept_example.json")))
    rE, rF, rG = fx["accept_prob"]
    V = 8
    E, F_, G, alt = 1, 2, 3, 4
    qv = 0.5
    pv = {E: min(1.0, 0.6), F_: rF * qv, G: rG * qv}
    assert rE == 1.0
    z = np.full((4, V), -100.0, np.float32)
    zq = np.full((4, V), -100.0, np.float32)
    for row, t in ((0, E), (1, F_), (2, G)):
        z[row, t], z[row, alt] = np.log(pv[t]), np.log(1 - pv[t])
        zq[row, t], zq[row, 5] = np.log(qv), np.log(1 - qv)
    z[3, 6] = 0.0
    names = {E: "E", F_: "F", G: "G"}
    tree = chain([E, F_, G])
    for case in ("a", "b"):
        u = fx[f"uniforms_case_{case}"]
        ua = np.zeros(4, np.uint32)
        ua[1:] = [int(x * 2 ** 32) for x in u]
        a, _, out = oracle.accept_sampled(tree, z, 1.0, zq, 1.0, ua, np.zeros(4, np.uint32), 3)
        assert [names[int(t)] for t in out[:a]] == fx[f"accepted_case_{case}"]
        if case == "a":
            assert out[a] == alt  # the only token with p > q at F's row
    # the ratio, not p alone, decides: at F, u = 0.6 > p(F) = 0.445 but < 0.89 accepts
    ua = np.array([0, 0, int(0.6 * 2 ** 32), int(0.99 * 2 ** 32)], np.uint32)
    a, _, out = oracle.accept_sampled(tree, z, 1.0, zq, 1.0, ua, np.zeros(4, np.uint32), 3)
    assert a == 2


def test_rejection_leaves_the_residual_max_p_minus_q():
    """One node, one drawn child that is rejected: the bonus follows
    norm(max(0, p - q)) (chi-square over the bonus uniforms)."""
    rng = np.random.default_rng(12)
    V = 10
    zp = (rng.standard_normal(V) * 1.2).astype(np.float32)
    zq = (rng.standard_normal(V) * 1.2).astype(np.float32)
    p, q = qprobs(zp), qprobs(zq)
    t = int(np.argmax(q / p))  # the token with the smallest acceptance ratio
    tree = {"tok": np.array([0, t], np.int32), "parent": np.array([-1, 0], np.int32)}
    z = np.stack([zp, np.zeros(V, np.float32)])
    zqq = np.stack([zq, np.zeros(V, np.float32)])
    n = 30000
    ua = np.full((n, 2), 2 ** 32 - 1, np.uint32)  # always reject (p/q < 1 at t)
    ub = synth.uniforms(4, synth.PURPOSE_BONUS, n, 2)
    counts = np.zeros(V)
    for i in range(n):
        a, _, out = oracle.accept_sampled(tree, z, 1.0, zqq, 1.0, ua[i], ub[i], 1)
        assert a == 0
        counts[out[0]] += 1
    res = np.maximum(p - q, 0)
    res /= res.sum()
    stat, dof = chi_square(counts, res)
    assert stat < chi2.ppf(1 - 1e-3, dof)


# ------------------------------------------------------------ losslessness ----

def small_model(seed, V=16, D=3, Fmax=4, sharp=1.5):
    rng = np.random.default_rng(seed)
    qtab = (rng.standard_normal((D, Fmax, V)) * sharp).astype(np.float32)
    ptab = (rng.standard_normal((V + 1, V)) * sharp).astype(np.float32)
    return qtab, ptab


@pytest.mark.parametrize("k,W,T,inv_Tq", [(2, 2, 1.0, 1.0), (1, 1, 1.0, 1.0), (3, 2, 0.6, 1.25)])
def test_sampled_rounds_are_lossless(k, W, T, inv_Tq):
    """2*10^5 rounds with fresh draws and uniforms: the first emitted token
    follows p_root, and the second, given that the first was an accepted draft,
    follows the target row after that token (chi-square, alpha = 1e-3)."""
    V, D, n = 16, 3, 200000
    qtab, ptab = small_model(k * 10 + W)
    Rcap = 64
    ua = synth.uniforms(21, synth.PURPOSE_ACCEPT, n, Rcap)
    ub = synth.uniforms(21, synth.PURPOSE_BONUS, n, Rcap)
    acc, out = oracle.sampled_trials(n, k, W, D, qtab, inv_Tq, ptab, T, 555, ua, ub)
    p_root = qprobs(ptab[0], 1.0 / T)
    stat, dof = chi_square(np.bincount(out[:, 0], minlength=V).astype(float), p_root)
    assert stat < chi2.ppf(1 - 1e-3, dof)
    assert 0.2 < (acc > 0).mean() < 0.95  # a non-degenerate mix of accepts and rejects
    x = np.bincount(out[acc > 0, 0], minlength=V).argmax()
    sel = (acc > 0) & (out[:, 0] == x)
    stat, dof = chi_square(np.bincount(out[sel, 1], minlength=V).astype(float), qprobs(ptab[1 + x], 1.0 / T))
    assert stat < chi2.ppf(1 - 1e-3, dof)


def test_chi_square_detects_a_missing_residual():
    """Power check: one drawn token accepted with min(1, p/q) but, on rejection,
    the correction drawn from p instead of max(0, p - q) is detected."""
    V, n = 16, 200000
    qtab, ptab = small_model(7)
    p, q = softmax(ptab[0].astype(np.float64)), softmax(qtab[0, 0].astype(np.float64))
    rng = np.random.default_rng(6)
    x = rng.choice(V, n, p=q)
    acc = rng.random(n) < np.minimum(1.0, p[x] / q[x])
    out = np.where(acc, x, rng.choice(V, n, p=p))  # planted mistake: no residual
    stat, dof = chi_square(np.bincount(out, minlength=V).astype(float), p)
    assert stat > chi2.ppf(1 - 1e-3, dof)
