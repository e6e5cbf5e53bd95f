"""Pins for dynamic-tree expansion, rerank, flattening and the tree mask (CPU)."""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import log_softmax

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def tree_from_fixture(name, decoys=True):
    """Candidate list for a fixture tree: fixture nodes get scores that decrease
    with depth; every fixture node also gets a decoy child with a much lower
    score that the rerank must drop."""
    fx = json.load(open(os.path.join(GOLD, "tree_examples.json")))[name]
    names = [n for n, _ in fx["nodes"]]
    idx = {}
    tok, par, sc, dep = [], [], [], []
    depth_of = {}
    for n, p in fx["nodes"]:
        d = 1 if p is None else depth_of[p] + 1
        depth_of[n] = d
    # depth-major candidate order (the fixture lists nodes depth by depth)
    order = sorted(range(len(names)), key=lambda i: (depth_of[names[i]], i))
    for i in order:
        n, p = fx["nodes"][i]
        idx[n] = len(tok)
        tok.append(100 + i)
        par.append(-1 if p is None else idx[p])
        sc.append(-1.0 * depth_of[n] - 0.001 * i)
        dep.append(depth_of[n])
    if decoys:
        for i in order:
            n = names[i]
            tok.append(500 + i)
            par.append(idx[n])
            sc.append(sc[idx[n]] - 50.0)
            dep.append(depth_of[n] + 1)
    C = len(tok)
    c = {"tok": np.array(tok, np.int32), "parent": np.array(par, np.int32),
         "score": np.array(sc, np.float32), "depth": np.array(dep, np.int32)}
    return fx, names, c, C


@pytest.mark.parametrize("name", ["p2_eagle2_k3", "p3_eight_nodes", "p5_a_to_f"])
def test_page_trees_flatten_and_mask(name):
    fx, names, cands, C = tree_from_fixture(name)
    N = len(names)
    tree = oracle.build_tree(cands, C, N, root_tok=7, kv_len=1000)
    name_of_tok = {100 + i: n for i, n in enumerate(names)}
    flat_names = ["root"] + [name_of_tok[int(t)] for t in tree["tok"][1:]]
    assert flat_names == fx["flat"]
    pos_of = {n: i for i, n in enumerate(flat_names)}
    dense = oracle.mask_to_dense(tree["mask"], N + 1)
    for n, seen in fx["sees"].items():
        row = set(np.flatnonzero(dense[pos_of[n]]))
        assert row == {pos_of[s] for s in seen}, (n, row)
    for n, unseen in fx["not_sees"].items():
        for s in unseen:
            assert not dense[pos_of[n], pos_of[s]]
    # positions follow depth; the root is at kv_len
    assert tree["pos"][0] == 1000 and tree["parent"][0] == -1
    for i in range(1, N + 1):
        assert tree["pos"][i] == 1000 + tree["depth"][i]
        assert tree["depth"][i] == tree["depth"][tree["parent"][i]] + 1


def test_chain_tree_mask_is_causal():
    # top-k = 1: the tree is a chain and the mask is lower triangular
    D = 9
    c = oracle.new_cands(D)
    for d in range(D):
        c["tok"][d] = d + 3
        c["parent"][d] = d - 1 if d else -1
        c["score"][d] = -0.5 * (d + 1)
        c["depth"][d] = d + 1
    tree = oracle.build_tree(c, D, D, root_tok=1, kv_len=0)
    dense = oracle.mask_to_dense(tree["mask"], D + 1)
    assert (dense == np.tril(np.ones((D + 1, D + 1), bool))).all()


def test_mask_words_beyond_64_nodes():
    # a 99-deep chain crosses two uint64 words
    D = 99
    c = oracle.new_cands(D)
    for d in range(D):
        c["tok"][d], c["parent"][d], c["score"][d], c["depth"][d] = d, d - 1 if d else -1, -d, d + 1
    tree = oracle.build_tree(c, D, D, root_tok=0, kv_len=5)
    dense = oracle.mask_to_dense(tree["mask"], D + 1)
    assert tree["mask"].shape == (D + 1, 2)
    assert (dense == np.tril(np.ones((D + 1, D + 1), bool))).all()


def run_expansion(logit_fn, V, k, W, D, root_score=0.0):
    """Drive the oracle's expansion depth by depth; logit_fn(cand_id) gives the
    draft logits of a frontier node (cand_id -1 = root)."""
    n_cand = k + (D - 1) * W * k
    c = oracle.new_cands(n_cand)
    fid = np.array([-1], np.int32)
    fsc = np.array([root_score], np.float32)
    off = 0
    for d in range(1, D + 1):
        z = np.stack([logit_fn(int(f)) for f in fid]).astype(np.float32)
        nid, nsc = oracle.expand(z, k, W, fsc, fid, d, off, c)
        off += len(fid) * k
        fid, fsc = nid, nsc
    return c, off


def test_expansion_against_fp64_path_probabilities():
    """Children are the top-k tokens of their row and the score of a node equals
    the fp64 log-probability of its whole path (product of draft softmaxes)."""
    V, k, W, D = 16, 3, 3, 4
    rng = np.random.default_rng(5)
    table = {}

    def logits(cid):
        if cid not in table:
            table[cid] = (rng.standard_normal(V) * 2.0).astype(np.float32)
        return table[cid]

    c, C = run_expansion(logits, V, k, W, D)
    for i in range(C):
        p = int(c["parent"][i])
        row = logits(p)
        lp = log_softmax(row.astype(np.float64))
        # token is among the top-k of the parent's row (ties to lower id)
        order = sorted(range(V), key=lambda j: (-float(row[j]), j))
        sibs = [j for j in range(C) if c["parent"][j] == p]
        assert [int(c["tok"][j]) for j in sibs] == order[:k]
        # cumulative path log-probability
        ref = 0.0
        j = i
        while j >= 0:
            pj = int(c["parent"][j])
            ref += log_softmax(logits(pj).astype(np.float64))[c["tok"][j]]
            j = pj
        assert abs(float(c["score"][i]) - ref) <= 2e-5 * (1 + abs(ref)), (i, c["score"][i], ref)
        if p >= 0:
            assert c["score"][i] <= c["score"][p]


def test_frontier_is_top_w_by_confidence():
    V, k, W = 16, 4, 3
    rng = np.random.default_rng(9)
    z = (rng.standard_normal((5, V)) * 2).astype(np.float32)
    c = oracle.new_cands(5 * k)
    ps = np.array([-0.1, -0.5, -0.2, -3.0, -0.05], np.float32)
    nid, nsc = oracle.expand(z, k, W, ps, np.arange(5, dtype=np.int32) + 100, 2, 0, c)
    exact = []
    for f in range(5):
        lp = log_softmax(z[f].astype(np.float64))
        for r, t in enumerate(sorted(range(V), key=lambda j: (-float(z[f][j]), j))[:k]):
            exact.append((ps[f] + lp[t], f * k + r))
    best = [i for _, i in sorted(exact, key=lambda x: (-x[0], x[1]))[:W]]
    assert list(nid) == best
    assert (nsc == c["score"][nid]).all()


def test_ties_break_to_lower_token_and_candidate_index():
    V, k = 8, 3
    z = np.zeros((1, V), np.float32)
    z[0, [6, 2, 4]] = 5.0  # three-way tie at the top
    c = oracle.new_cands(k)
    nid, _ = oracle.expand(z, k, 2, np.zeros(1, np.float32), np.array([-1], np.int32), 1, 0, c)
    assert list(c["tok"][:3]) == [2, 4, 6]
    assert c["score"][0] == c["score"][1] == c["score"][2]
    assert list(nid) == [0, 1]


def test_rerank_keeps_most_probable_nodes_and_is_closed():
    """Keeping N of the expanded candidates keeps the N most probable paths
    (fp64 path probability), and the kept set is closed under parents."""
    V, k, W, D, N = 32, 4, 4, 5, 17
    rng = np.random.default_rng(21)
    table = {}

    def logits(cid):
        if cid not in table:
            table[cid] = (rng.standard_normal(V) * 3.0).astype(np.float32)
        return table[cid]

    c, C = run_expansion(logits, V, k, W, D)
    tree = oracle.build_tree(c, C, N, root_tok=0, kv_len=0)
    # fp64 path log-probabilities of all candidates
    lp = np.zeros(C)
    for i in range(C):
        j, acc = i, 0.0
        while j >= 0:
            pj = int(c["parent"][j])
            acc += log_softmax(logits(pj).astype(np.float64))[c["tok"][j]]
            j = pj
        lp[i] = acc
    order = np.argsort(-lp, kind="stable")
    gap = lp[order[N - 1]] - lp[order[N]]
    assert gap > 1e-4  # seed chosen without a near tie at the cut
    kept_paths = set()
    for i in range(1, N + 1):
        path = []
        j = i
        while j > 0:
            path.append(int(tree["tok"][j]))
            j = int(tree["parent"][j])
        kept_paths.add(tuple(reversed(path)))
    want = set()
    for i in order[:N]:
        path = []
        j = int(i)
        while j >= 0:
            path.append(int(c["tok"][j]))
            j = int(c["parent"][j])
        want.add(tuple(reversed(path)))
    assert kept_paths == want
