"""Draft decoder step of EAGLE-3 -- TEST INFRASTRUCTURE ONLY (like the rest of
``oracle``: only tests/, smoke() and the benchmark's CPU baseline may use it).

Plain fp64 numpy.  What the pages fix:
  "论文专题讲解：EAGLE-3", 推理流程：多层特征融合 + 单层 draft decoder: the drafter is a
  single Transformer decoder layer; its first step reads the fused feature g and
  the previous token's embedding, later steps (tokens the target has not seen)
  read the drafter's own previous output a and the embedding of the token just
  proposed ("方法主线：为什么叫 Training-time Test": a1 + token embedding -> step 2
  -> a2 ...).  "SpecForge…", 第二步为什么没有"正确隐藏状态"可用: a_{t+1} = D(g_t or a_t,
  e(x_t)), and the output through an LM head gives the next token's draft
  distribution; "从序列到动态草稿树": in a tree every node attends only to its
  ancestor path.

Readings where the pages leave the step open (listed in the design notes):
  * the two inputs are concatenated as [e(x); h] (2d values) and projected to d by
    one fully connected layer W_in [d][2d], as the fusion does with three features;
  * the layer is a pre-norm decoder block of the target family: RMSNorm ->
    grouped-query attention with rotary positions -> residual -> RMSNorm -> SwiGLU
    MLP -> residual; its output is a; the draft logits are W_lm RMSNorm(a);
  * the attention context of a node is the drafter's own KV cache of the committed
    prefix (positions 0..P-1, an input here), the K/V its ancestors produced at
    earlier depths, and its own; a node at tree depth t (root 0) has position P + t.

Parity pins: ``tests/test_oracle_draft.py``.
"""
from __future__ import annotations

import numpy as np

EPS = 1e-6
ROPE_BASE = 10000.0


def rmsnorm(x, w):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + EPS) * np.asarray(w, np.float64)


def rope(x, pos):
    """Rotary embedding of the last axis (hd even) at integer positions ``pos``
    (broadcast over the leading axes but the head axis): dimension i is paired
    with i + hd/2 and rotated by pos * base^(-2i/hd)."""
    x = np.asarray(x, np.float64)
    hd = x.shape[-1]
    half = hd // 2
    inv = ROPE_BASE ** (-np.arange(half, dtype=np.float64) * 2.0 / hd)
    ang = np.asarray(pos, np.float64)[..., None] * inv  # [..., half]
    while ang.ndim < x.ndim:
        ang = ang[..., None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def silu(x):
    return x / (1.0 + np.exp(-x))


def random_weights(rng, V, d, H, KVH, hd, f, std=0.02):
    """A drafter with random weights (the shapes of one decoder layer): projections
    N(0, std^2), norm weights 1 + N(0, std^2), embedding and LM head N(0, 1)."""
    n = lambda *s: rng.standard_normal(s) * std  # noqa: E731
    return {"emb": rng.standard_normal((V, d)), "W_in": n(d, 2 * d), "norm1": 1.0 + n(d), "Wq": n(H * hd, d),
            "Wk": n(KVH * hd, d), "Wv": n(KVH * hd, d), "Wo": n(d, H * hd), "norm2": 1.0 + n(d),
            "Wg": n(f, d), "Wu": n(f, d), "Wd": n(d, f), "normf": 1.0 + n(d), "lm": rng.standard_normal((V, d)),
            "H": H, "KVH": KVH, "hd": hd}


def draft_step(Wt, h_in, tok, pos, ctx):
    """One drafter step for F rows.

    h_in [F, d]: g (first step) or the output a of the step that proposed the
    row's token; tok [F]: the row's token; pos [F]: its position; ctx: per row a
    pair (K [n, KVH, hd], V [n, KVH, hd]) of the keys it attends to besides its
    own (prefix + ancestors).  Returns a [F, d], the row's own k and v
    [F, KVH, hd] (rotary applied to k) and the draft logits [F, V].
    """
    H, KVH, hd = Wt["H"], Wt["KVH"], Wt["hd"]
    grp = H // KVH
    h_in = np.asarray(h_in, np.float64)
    F = h_in.shape[0]
    x = np.concatenate([Wt["emb"][np.asarray(tok)], h_in], axis=1) @ Wt["W_in"].T  # [F, d]
    y = rmsnorm(x, Wt["norm1"])
    q = rope((y @ Wt["Wq"].T).reshape(F, H, hd), pos)
    k = rope((y @ Wt["Wk"].T).reshape(F, KVH, hd), pos)
    v = (y @ Wt["Wv"].T).reshape(F, KVH, hd)
    o = np.zeros((F, H, hd))
    for r in range(F):
        Kc, Vc = ctx[r]
        Kr = np.concatenate([np.asarray(Kc, np.float64).reshape(-1, KVH, hd), k[r:r + 1]], axis=0)
        Vr = np.concatenate([np.asarray(Vc, np.float64).reshape(-1, KVH, hd), v[r:r + 1]], axis=0)
        for h in range(H):
            s = Kr[:, h // grp, :] @ q[r, h] / np.sqrt(hd)
            w = np.exp(s - s.max())
            o[r, h] = (w @ Vr[:, h // grp, :]) / w.sum()
    x = x + o.reshape(F, H * hd) @ Wt["Wo"].T
    y2 = rmsnorm(x, Wt["norm2"])
    a = x + (silu(y2 @ Wt["Wg"].T) * (y2 @ Wt["Wu"].T)) @ Wt["Wd"].T
    logits = rmsnorm(a, Wt["normf"]) @ Wt["lm"].T
    return a, k, v, logits


def draft_tree(Wt, g, root_tok, K_pre, V_pre, D, expand):
    """Draft a whole tree: D steps, each over the current frontier.

    g [d]: fused feature of the root; K_pre / V_pre [P, KVH, hd]: the drafter's KV
    cache of the committed prefix.  ``expand(logits, depth, frontier_ids,
    frontier_scores)`` (logits [F, V] float32 of the frontier rows) performs one
    depth of the expansion (top-k or sampled) and returns (next_ids, next_scores,
    children) with children = {candidate index: (token, parent candidate index)}.
    Returns the draft logits of every depth ([F_t, V] fp64), the step output a of
    every expanded node (keyed by candidate index, root -1) and the frontiers.
    """
    P = K_pre.shape[0]
    a_of, kv_of = {}, {}  # expanded node -> its output a, and the (k, v) it produced
    parent, tok_of, depth_of = {}, {-1: int(root_tok)}, {-1: 0}
    fid, fsc = np.array([-1], np.int32), np.zeros(1, np.float32)
    all_logits, fronts = [], []
    for t in range(D):
        rows = [int(x) for x in fid]
        h_in = np.stack([np.asarray(g, np.float64) if u == -1 else a_of[parent[u]] for u in rows])
        ctx = []
        for u in rows:  # prefix, then the ancestors root first (the node itself is added by the step)
            anc, x = [], u
            while x != -1:
                x = parent[x]
                anc.append(x)
            anc = anc[::-1]
            ctx.append((np.concatenate([K_pre] + [kv_of[x][0][None] for x in anc], 0),
                        np.concatenate([V_pre] + [kv_of[x][1][None] for x in anc], 0)))
        a, kk, vv, logits = draft_step(Wt, h_in, [tok_of[u] for u in rows], [P + depth_of[u] for u in rows], ctx)
        for i, u in enumerate(rows):
            a_of[u] = a[i]
            kv_of[u] = (kk[i], vv[i])
        all_logits.append(logits)
        nid, nsc, children = expand(logits.astype(np.float32), t + 1, fid, fsc)
        for ci, (tk, par) in children.items():
            tok_of[ci] = int(tk)
            parent[ci] = int(par)
            depth_of[ci] = t + 1
        fronts.append((nid, nsc))
        fid, fsc = nid, nsc
    return all_logits, a_of, fronts
