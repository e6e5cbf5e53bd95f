"""Pins for the drafter oracle (CPU): rotary embedding, RMSNorm and SiLU against
independent forms; the input wiring ([e(x); h], g at the first step, the parent
step's output a afterwards); and the tree/chain bookkeeping against a plain
sequential causal decoder recomputed from scratch with a dense mask.

"论文专题讲解：EAGLE-3", 推理流程：多层特征融合 + 单层 draft decoder; "SpecForge…",
第二步为什么没有"正确隐藏状态"可用 and 从序列到动态草稿树 (ancestor-only attention).
"""
import numpy as np
from scipy.special import expit

import oracle
from oracle import draft as dr


def small(seed=0, V=40, d=32, H=4, KVH=2, hd=8, f=48):
    rng = np.random.default_rng(seed)
    return rng, dr.random_weights(rng, V, d, H, KVH, hd, f, std=0.2)


# ------------------------------------------------------------ building blocks ----

def test_rope_is_a_complex_rotation_per_pair():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((5, 3, 16))
    pos = np.array([0, 1, 7, 100, 4095])
    got = dr.rope(x, pos)
    half = 8
    theta = 10000.0 ** (-np.arange(half) / half)
    z = (x[..., :half] + 1j * x[..., half:]) * np.exp(1j * pos[:, None, None] * theta)
    assert np.allclose(got[..., :half], z.real, atol=1e-12) and np.allclose(got[..., half:], z.imag, atol=1e-12)
    assert np.allclose(dr.rope(x, np.zeros(5)), x)  # position 0 is the identity


def test_rope_scores_depend_on_relative_position_only():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(16), rng.standard_normal(16)
    for m, n, s in [(5, 2, 10), (0, 9, 300), (17, 17, 1)]:
        a = dr.rope(q, np.array(m)) @ dr.rope(k, np.array(n))
        b = dr.rope(q, np.array(m + s)) @ dr.rope(k, np.array(n + s))
        assert abs(a - b) < 1e-10


def test_rmsnorm_and_silu():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 64)) * 3
    y = dr.rmsnorm(x, np.ones(64))
    assert np.allclose(np.sqrt(np.mean(y * y, axis=1)), 1.0, atol=1e-6)
    assert np.allclose(dr.rmsnorm(7.5 * x, np.ones(64)), y, atol=1e-6)  # scale invariant
    w = rng.standard_normal(64)
    assert np.allclose(dr.rmsnorm(x, w), y * w)
    t = np.linspace(-20, 20, 101)
    assert np.allclose(dr.silu(t), t * expit(t))


# ------------------------------------------------------------------- wiring ----

def test_input_wiring_embedding_then_feature():
    """With the attention and MLP outputs switched off, a is the input projection:
    W_in = [I, 0] selects e(x), W_in = [0, I] selects the feature h."""
    rng, W = small(4)
    d = W["W_in"].shape[0]
    W["Wo"][:] = 0.0
    W["Wd"][:] = 0.0
    h = rng.standard_normal((3, d))
    tok = [5, 0, 39]
    ctx = [(np.zeros((0, 2, 8)), np.zeros((0, 2, 8)))] * 3
    W["W_in"] = np.concatenate([np.eye(d), np.zeros((d, d))], axis=1)
    a, _, _, logits = dr.draft_step(W, h, tok, [0, 1, 2], ctx)
    assert np.allclose(a, W["emb"][tok])
    assert np.allclose(logits, dr.rmsnorm(a, W["normf"]) @ W["lm"].T)
    W["W_in"] = np.concatenate([np.zeros((d, d)), np.eye(d)], axis=1)
    a, _, _, _ = dr.draft_step(W, h, tok, [0, 1, 2], ctx)
    assert np.allclose(a, h)


def test_lone_key_attention_returns_its_value():
    """A row with an empty context attends only to itself: the attention output
    of head h is v of its KV head, so a - x0 = Wo [v repeated per group] (MLP off)."""
    rng, W = small(5)
    d = W["W_in"].shape[0]
    W["Wd"][:] = 0.0
    h = rng.standard_normal((2, d))
    ctx = [(np.zeros((0, 2, 8)), np.zeros((0, 2, 8)))] * 2
    a, k, v, _ = dr.draft_step(W, h, [3, 4], [6, 6], ctx)
    x0 = np.concatenate([W["emb"][[3, 4]], h], axis=1) @ W["W_in"].T
    o = np.repeat(v, 2, axis=1).reshape(2, -1)  # H = 4 query heads over KVH = 2
    assert np.allclose(a - x0, o @ W["Wo"].T, atol=1e-12)


# ------------------------------------------------- chains and trees vs scratch ----

def forced_expand(children_tokens):
    """An expansion that gives each frontier row (in order) the listed children."""
    state = {"off": 0}

    def expand(logits, depth, fid, fsc):
        kids, ids = {}, []
        toks = children_tokens[depth - 1]
        for i, par in enumerate(fid):
            for t in toks[i]:
                ci = state["off"]
                state["off"] += 1
                kids[ci] = (t, int(par))
                ids.append(ci)
        return np.array(ids, np.int32), np.zeros(len(ids), np.float32), kids
    return expand


def sequential_decoder(W, g, tokens, K_pre, V_pre):
    """From scratch: positions P..P+n-1 carry tokens[0..n-1]; position P's feature
    is g, position P+i's is the output of position P+i-1.  Every position is
    recomputed with one dense causal attention over [prefix; positions so far]."""
    P = K_pre.shape[0]
    H, KVH, hd = W["H"], W["KVH"], W["hd"]
    outs, logits_all = [], []
    for n in range(1, len(tokens) + 1):
        feats = [np.asarray(g, np.float64)] + outs[:n - 1]
        x = np.concatenate([W["emb"][tokens[:n]], np.stack(feats)], axis=1) @ W["W_in"].T
        y = dr.rmsnorm(x, W["norm1"])
        pos = P + np.arange(n)
        q = dr.rope((y @ W["Wq"].T).reshape(n, H, hd), pos)
        k = np.concatenate([K_pre, dr.rope((y @ W["Wk"].T).reshape(n, KVH, hd), pos)], 0)
        v = np.concatenate([V_pre, (y @ W["Wv"].T).reshape(n, KVH, hd)], 0)
        mask = np.arange(P + n)[None, :] <= (P + np.arange(n))[:, None]  # [n, P+n] causal
        o = np.zeros((n, H, hd))
        for h in range(H):
            S = q[:, h, :] @ k[:, h // (H // KVH), :].T / np.sqrt(hd)
            S = np.where(mask, S, -np.inf)
            Pm = np.exp(S - S.max(axis=1, keepdims=True))
            o[:, h, :] = (Pm / Pm.sum(axis=1, keepdims=True)) @ v[:, h // (H // KVH), :]
        x = x + o.reshape(n, -1) @ W["Wo"].T
        y2 = dr.rmsnorm(x, W["norm2"])
        a = x + (dr.silu(y2 @ W["Wg"].T) * (y2 @ W["Wu"].T)) @ W["Wd"].T
        outs = [a[i] for i in range(n)]
        logits_all = dr.rmsnorm(a, W["normf"]) @ W["lm"].T
    return np.stack(outs), logits_all


def test_chain_draft_equals_sequential_decoding():
    rng, W = small(6)
    d = W["W_in"].shape[0]
    P = 9
    K_pre, V_pre = rng.standard_normal((P, 2, 8)), rng.standard_normal((P, 2, 8))
    g = rng.standard_normal(d)
    root, chain = 7, [12, 3, 30]
    logits, a_of, _ = dr.draft_tree(W, g, root, K_pre, V_pre, 4, forced_expand([[[t]] for t in chain] + [[[1]]]))
    outs, ref_logits = sequential_decoder(W, g, [root] + chain, K_pre, V_pre)
    assert np.allclose(np.concatenate(logits), ref_logits, atol=1e-9)
    assert np.allclose(a_of[-1], outs[0]) and np.allclose(a_of[2], outs[3])


def test_tree_node_sees_only_its_ancestors():
    """Each node's draft logits equal those of the chain along its own path; the
    cousins drafted beside it change nothing."""
    rng, W = small(7)
    d = W["W_in"].shape[0]
    P = 5
    K_pre, V_pre = rng.standard_normal((P, 2, 8)), rng.standard_normal((P, 2, 8))
    g = rng.standard_normal(d)
    root = 2
    # depth 1: root -> [10, 11, 12]; depth 2: 10 -> [20, 21], 11 -> [22], 12 -> [23, 24]
    kids = [[[10, 11, 12]], [[20, 21], [22], [23, 24]], [[0]] * 5]
    logits, _, fronts = dr.draft_tree(W, g, root, K_pre, V_pre, 3, forced_expand(kids))
    paths = {0: [10], 1: [11], 2: [12], 3: [10, 20], 4: [10, 21], 5: [11, 22], 6: [12, 23], 7: [12, 24]}
    rows = {1: [0, 1, 2], 2: [3, 4, 5, 6, 7]}  # candidate index of each frontier row at depths 2 and 3
    for depth, cands in rows.items():
        for i, ci in enumerate(cands):
            _, ref = sequential_decoder(W, g, [root] + paths[ci], K_pre, V_pre)
            assert np.allclose(logits[depth][i], ref[-1], atol=1e-9), (depth, ci)


def test_drafted_tree_drives_the_top_k_expansion():
    """End to end with the oracle's own top-k expansion: the first depth's
    children are the top-k of the root's draft logits."""
    rng, W = small(8, V=64)
    d = W["W_in"].shape[0]
    P, k, D = 6, 3, 3
    K_pre, V_pre = rng.standard_normal((P, 2, 8)), rng.standard_normal((P, 2, 8))
    g = rng.standard_normal(d)
    cands = oracle.new_cands(k + k * k + k * k)
    state = {"off": 0}

    def expand(logits, depth, fid, fsc):
        off = state["off"]
        nid, nsc = oracle.expand(logits, k, k, fsc, fid, depth, off, cands)
        state["off"] += len(fid) * k
        kids = {ci: (int(cands["tok"][ci]), int(cands["parent"][ci])) for ci in range(off, state["off"])}
        return nid, nsc, kids

    logits, _, fronts = dr.draft_tree(W, g, 11, K_pre, V_pre, D, expand)
    top = np.argsort(-logits[0][0].astype(np.float32), kind="stable")[:k]
    assert list(cands["tok"][:k]) == list(top)
    assert [len(x) for x in logits] == [1, k, k]
