"""CPU oracle for one EAGLE-3 draft-and-verify round -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline``
leg (and its ``--impl reference`` arm) may import this package.  It shares no
code with the CUDA path (``eagle_speculative_decoding_round_gb300``): neither
imports the other.  Inputs come from ``eagle_speculative_decoding_round_gb300.synth``
(seeded generators only) or from the tests.

Float math is fp64 (numpy), computed from the same bf16/fp32 values the GPU
reads.  The integer decisions (top-k, rerank, accept/reject, bonus sampling)
live in ``eagle3_oracle.c`` and use the fp32 fixed-point recipe written out
there, so that they can be compared bit for bit.

Sources (web pages on EAGLE-3, cited by title and section):
  [EAGLE-3 deep dive] "论文专题讲解：EAGLE-3：Training-time Test 的投机推理加速",
      "推理流程：多层特征融合 + 单层 draft decoder" and the "训练细节" table
      (concatenate l, m, h into 3k and project to k with one FC layer).
  [SpecForge] "SpecForge：把 EAGLE3 从训练样本交付到 SGLang",
      "多层特征融合到底融合了什么" (g_t = W_f [h_low; h_mid; h_high]),
      "从序列到动态草稿树" (each node attends only to its ancestor path).
  [EAGLE系列] "EAGLE 系列与 DFlash" (pzsr.cn), §二 EAGLE-2 阶段二/三.
  [USP] "EAGLE-3 投机解码与 USP 长序列训练优化", "USP 核心设计：三步走"
      (main segment and branch segment merged by their LSE).
  [TB] "Thinking Budget 与 EAGLE-3", "一棵候选树怎样被验证" (commit only the
      accepted path's KV).

Parity pins: every function here is pinned by tests in ``tests/test_oracle_*.py``
against values or identities that do not come from this file.  ``oracle.draft``
holds the drafter's decoder step (pinned in ``tests/test_oracle_draft.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "eagle3_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C part with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, f32, u64 = ctypes.c_int, ctypes.c_float, ctypes.c_uint64
            lib.e3o_exp.restype = f32
            lib.e3o_exp.argtypes = [f32]
            lib.e3o_qmass.restype = u64
            lib.e3o_qmass.argtypes = [f32, f32]
            lib.e3o_ell.restype = f32
            lib.e3o_ell.argtypes = [u64]
            lib.e3o_row_stats_batch.restype = None
            lib.e3o_row_stats_batch.argtypes = [P, i32, i32, P, P, P, P, P]
            lib.e3o_expand.restype = i32
            lib.e3o_expand.argtypes = [P, i32, i32, i32, i32, f32, P, P, i32, i32, P, P, P, P, P, P]
            lib.e3o_build_tree.restype = i32
            lib.e3o_build_tree.argtypes = [i32, P, P, P, P, i32, i32, i32, P, P, P, P, P, i32]
            lib.e3o_accept.restype = i32
            lib.e3o_accept.argtypes = [P, P, i32, i32, P, i32, f32, P, P, P, P, P]
            lib.e3o_accept_many.restype = None
            lib.e3o_accept_many.argtypes = [i32, P, P, i32, i32, P, i32, f32, P, P, P, P, P]
            lib.e3o_splitmix64_at.restype = u64
            lib.e3o_splitmix64_at.argtypes = [u64, u64]
            lib.e3o_exp_variate.restype = f32
            lib.e3o_exp_variate.argtypes = [u64, i32, i32, i32, i32]
            lib.e3o_expand_sampled.restype = i32
            lib.e3o_expand_sampled.argtypes = [P, i32, i32, i32, i32, f32, P, P, i32, i32, u64, i32, P, P, P,
                                               P, P, P, P, P]
            lib.e3o_build_tree_cand.restype = i32
            lib.e3o_build_tree_cand.argtypes = [i32, P, P, P, P, i32, i32, i32, P, P, P, P, P, i32, P]
            lib.e3o_accept_sampled.restype = i32
            lib.e3o_accept_sampled.argtypes = [P, P, i32, i32, P, i32, f32, P, f32, P, P, P, P, P]
            lib.e3o_sampled_trials.restype = i32
            lib.e3o_sampled_trials.argtypes = [i32, i32, i32, i32, i32, P, i32, f32, P, f32, u64, P, P, i32,
                                               P, P]
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------
# fp32 decision arithmetic (thin wrappers over the C recipe)
# ---------------------------------------------------------------------------

def exp_recipe(x: float) -> float:
    """E(x) of the fixed-point recipe (fp32), x <= 0."""
    return float(_load().e3o_exp(float(x)))


def qmass(s: float, m: float) -> int:
    """floor(2^40 * E(s - m)) for fp32 s <= m."""
    return int(_load().e3o_qmass(float(s), float(m)))


def ell(Q: int) -> float:
    """ln(Q * 2^-40) by the recipe (fp32)."""
    return float(_load().e3o_ell(int(Q)))


def row_stats(logits: np.ndarray, temp) -> tuple:
    """Per-row softmax statistics of fp32 logits [M, V]: (row_max, row_Q, argmax, nonfinite).

    row_max/argmax are over s = z * (1/T) (s = z when T <= 0); row_Q is the
    fixed-point total mass.  This is the "softmax" part of the LM-head step.
    """
    z = np.ascontiguousarray(logits, dtype=np.float32)
    M, V = z.shape
    T = np.ascontiguousarray(np.broadcast_to(np.asarray(temp, np.float32), (M,)))
    m = np.zeros(M, np.float32)
    Q = np.zeros(M, np.uint64)
    am = np.zeros(M, np.int32)
    bad = np.zeros(M, np.int32)
    _load().e3o_row_stats_batch(_p(z), M, V, _p(T), _p(m), _p(Q), _p(am), _p(bad))
    return m, Q, am, bad


# ---------------------------------------------------------------------------
# a1: feature fusion  g = W_f [h_low; h_mid; h_high]
# ---------------------------------------------------------------------------

def fuse(h_low, h_mid, h_high, W_f, bias=None) -> np.ndarray:
    """g[m, o] = sum_j W_f[o, j] x[m, j], x = [h_low | h_mid | h_high] (fp64).

    [SpecForge] "多层特征融合到底融合了什么": concatenate the three d-dim vectors
    of the same token and project with one fully connected layer.
    """
    x = np.concatenate([np.asarray(h, np.float64) for h in (h_low, h_mid, h_high)], axis=1)
    g = x @ np.asarray(W_f, np.float64).T
    if bias is not None:
        g = g + np.asarray(bias, np.float64)[None, :]
    return g


# ---------------------------------------------------------------------------
# a2 / a3: expansion and tree construction (C)
# ---------------------------------------------------------------------------

def expand(logits, k, W, parent_score, parent_id, depth, cand_offset, cands, inv_T=1.0):
    """One depth of dynamic-tree expansion for one request.

    logits: [F, V] fp32 draft logits of the frontier rows.  ``cands`` is a dict of
    numpy arrays tok/parent/score/depth (capacity C) updated in place.  Returns
    (next_id, next_score) of the next frontier.
    """
    z = np.ascontiguousarray(logits, dtype=np.float32)
    F, V = z.shape
    ps = np.ascontiguousarray(parent_score, np.float32)
    pid = np.ascontiguousarray(parent_id, np.int32)
    nf_cap = min(W, F * k)
    nid = np.zeros(nf_cap, np.int32)
    nsc = np.zeros(nf_cap, np.float32)
    rc = _load().e3o_expand(_p(z), F, V, k, W, float(np.float32(inv_T)), _p(ps), _p(pid), depth,
                            cand_offset, _p(cands["tok"]), _p(cands["parent"]), _p(cands["score"]),
                            _p(cands["depth"]), _p(nid), _p(nsc))
    if rc < 0:
        raise FloatingPointError("non-finite draft logit")
    return nid, nsc


def splitmix64_at(seed: int, i: int) -> int:
    """Output number i >= 1 of the SplitMix64 stream started at ``seed``."""
    return int(_load().e3o_splitmix64_at(seed & (2 ** 64 - 1), i & (2 ** 64 - 1)))


def exp_variate(seed: int, b: int, depth: int, f: int, j: int) -> float:
    """E = -ln U of the draw for token j of frontier row f at ``depth`` of request b (fp32)."""
    return float(_load().e3o_exp_variate(seed & (2 ** 64 - 1), b, depth, f, j))


def expand_sampled(logits, k, W, parent_score, parent_id, depth, cand_offset, cands, seed, b, inv_T=1.0):
    """One depth of expansion with sampled children, one request (request index b
    keys the draws).  Each row's k children are drawn without replacement from
    the draft distribution (exponential race on E_j / e_j), in draw order; scores
    and the next frontier are as in ``expand``.  Returns (next_id, next_score,
    row_m, row_Q): the next frontier and each row's draft statistics.

    "EAGLE 系列与 DFlash", §四 DFlash: drafts proposed by the drafter and checked
    with min(1, p_target / p_draft); drawing them from the draft distribution is
    what makes that rule exact.
    """
    z = np.ascontiguousarray(logits, dtype=np.float32)
    F, V = z.shape
    ps = np.ascontiguousarray(parent_score, np.float32)
    pid = np.ascontiguousarray(parent_id, np.int32)
    nf_cap = min(W, F * k)
    nid = np.zeros(nf_cap, np.int32)
    nsc = np.zeros(nf_cap, np.float32)
    rm = np.zeros(F, np.float32)
    rq = np.zeros(F, np.uint64)
    rc = _load().e3o_expand_sampled(_p(z), F, V, k, W, float(np.float32(inv_T)), _p(ps), _p(pid), depth,
                                    cand_offset, seed & (2 ** 64 - 1), b, _p(cands["tok"]),
                                    _p(cands["parent"]), _p(cands["score"]), _p(cands["depth"]), _p(nid),
                                    _p(nsc), _p(rm), _p(rq))
    if rc < 0:
        raise FloatingPointError("non-finite draft logit")
    return nid, nsc, rm, rq


def new_cands(C: int) -> dict:
    return {"tok": np.full(C, -1, np.int32), "parent": np.full(C, -1, np.int32),
            "score": np.zeros(C, np.float32), "depth": np.zeros(C, np.int32)}


def build_tree(cands: dict, n_cand: int, N: int, root_tok: int, kv_len: int):
    """Rerank to the N best candidates, flatten, positions and ancestor mask."""
    R = N + 1
    words = (R + 63) // 64
    tok = np.zeros(R, np.int32)
    parent = np.zeros(R, np.int32)
    depth = np.zeros(R, np.int32)
    pos = np.zeros(R, np.int32)
    mask = np.zeros((R, words), np.uint64)
    node_cand = np.zeros(R, np.int32)
    c = {k: np.ascontiguousarray(v[:n_cand]) for k, v in cands.items()}
    rc = _load().e3o_build_tree_cand(n_cand, _p(c["tok"]), _p(c["parent"]), _p(c["score"]), _p(c["depth"]),
                                     N, int(root_tok), int(kv_len), _p(tok), _p(parent), _p(depth), _p(pos),
                                     _p(mask), words, _p(node_cand))
    if rc != 0:
        raise AssertionError("kept candidate set is not closed under parents")
    return {"tok": tok, "parent": parent, "depth": depth, "pos": pos, "mask": mask, "node_cand": node_cand}


def mask_to_dense(mask: np.ndarray, R: int) -> np.ndarray:
    """uint64 bit rows [R, words] -> bool [R, R] (bit j of row i = node i sees node j)."""
    out = np.zeros((R, R), bool)
    for i in range(R):
        for j in range(R):
            out[i, j] = (int(mask[i, j >> 6]) >> (j & 63)) & 1
    return out


# ---------------------------------------------------------------------------
# paged KV helpers
# ---------------------------------------------------------------------------

def gather_tokens(cache: np.ndarray, page_table_row: np.ndarray, t0: int, t1: int) -> np.ndarray:
    """Logical tokens [t0, t1) of one request from a paged cache [pages, KVH, page, hd]
    -> [t1 - t0, KVH, hd] fp64."""
    ps = cache.shape[2]
    out = []
    for t in range(t0, t1):
        out.append(cache[page_table_row[t // ps], :, t % ps, :])
    if not out:
        return np.zeros((0, cache.shape[1], cache.shape[3]), np.float64)
    return np.stack(out).astype(np.float64)


# ---------------------------------------------------------------------------
# a4: tree-masked verify attention
# ---------------------------------------------------------------------------

def tree_verify_attn(Q, Kc, Vc, page_table, kv_len, parent, sm_scale):
    """(i) Per node over its explicit key list: prefix [0, P) plus the tree slots
    P + j for j on the node's ancestor path (walked through ``parent``), itself
    included.

    Q [B, R, H, hd]; Kc/Vc paged [pages, KVH, page, hd]; parent [B, R].
    Returns O [B, R, H, hd] and lse [B, R, H] (natural log of the sum of
    exp(score)), both fp64.  Query head h reads KV head h // (H / KVH).
    """
    Q = np.asarray(Q, np.float64)
    B, R, H, hd = Q.shape
    KVH = Kc.shape[1]
    grp = H // KVH
    O = np.zeros((B, R, H, hd))
    lse = np.zeros((B, R, H))
    for b in range(B):
        P = int(kv_len[b])
        Kb = gather_tokens(Kc, page_table[b], 0, P + R)
        Vb = gather_tokens(Vc, page_table[b], 0, P + R)
        for i in range(R):
            keys = _node_keys(P, parent[b], i)
            for h in range(H):
                O[b, i, h], lse[b, i, h] = _attend(Kb, Vb, keys, Q[b, i, h], h // grp, sm_scale)
    return O, lse


def _node_keys(P, parent_row, i):
    """Key slots node i attends to: the prefix [0, P) and P + j for the nodes j on
    its ancestor path (itself included)."""
    anc = []
    j = i
    while j >= 0:
        anc.append(j)
        j = int(parent_row[j])
    return list(range(P)) + [P + j for j in sorted(anc)]


def _attend(Kb, Vb, keys, q, kh, sm_scale):
    """One query row over its key list: softmax(q . K / sqrt) V and the lse (fp64)."""
    s = (Kb[keys, kh, :] @ np.asarray(q, np.float64)) * sm_scale
    mx = s.max()
    w = np.exp(s - mx)
    den = w.sum()
    return (w @ Vb[keys, kh, :]) / den, mx + np.log(den)


def tree_verify_attn_rows(Q, Kc, Vc, page_table, kv_len, parent, sm_scale, rows):
    """tree_verify_attn for the listed (b, i, h) query rows only (the same key lists
    and the same per-row arithmetic); returns O [n, hd] and lse [n] in fp64."""
    Q = np.asarray(Q, np.float64)
    B, R, H, hd = Q.shape
    grp = H // Kc.shape[1]
    O = np.zeros((len(rows), hd))
    lse = np.zeros(len(rows))
    cache = {}
    for n, (b, i, h) in enumerate(rows):
        if b not in cache:
            P = int(kv_len[b])
            cache[b] = (P, gather_tokens(Kc, page_table[b], 0, P + R), gather_tokens(Vc, page_table[b], 0, P + R))
        P, Kb, Vb = cache[b]
        O[n], lse[n] = _attend(Kb, Vb, _node_keys(P, parent[b], i), Q[b, i, h], h // grp, sm_scale)
    return O, lse


def tree_verify_attn_dense(Q, Kc, Vc, page_table, kv_len, mask, sm_scale):
    """(ii) Dense form: one (P+R)-column masked softmax per query row, with the
    tree part of the 0/1 mask materialised from the uint64 ancestor bit rows."""
    Q = np.asarray(Q, np.float64)
    B, R, H, hd = Q.shape
    KVH = Kc.shape[1]
    grp = H // KVH
    O = np.zeros((B, R, H, hd))
    lse = np.zeros((B, R, H))
    for b in range(B):
        P = int(kv_len[b])
        Kb = gather_tokens(Kc, page_table[b], 0, P + R)
        Vb = gather_tokens(Vc, page_table[b], 0, P + R)
        allowed = np.ones((R, P + R), bool)
        allowed[:, P:] = mask_to_dense(mask[b], R)
        for h in range(H):
            kh = h // grp
            S = (Q[b, :, h, :] @ Kb[:, kh, :].T) * sm_scale  # [R, P+R]
            S = np.where(allowed, S, -np.inf)
            mx = S.max(axis=1, keepdims=True)
            W_ = np.exp(S - mx)
            den = W_.sum(axis=1, keepdims=True)
            O[b, :, h, :] = (W_ @ Vb[:, kh, :]) / den
            lse[b, :, h] = (mx + np.log(den))[:, 0]
    return O, lse


# ---------------------------------------------------------------------------
# a5: LM-head logits and softmax statistics
# ---------------------------------------------------------------------------

def lmhead_logits(h, W_lm) -> np.ndarray:
    """logits[m, v] = sum_j h[m, j] W_lm[v, j] in fp64."""
    return np.asarray(h, np.float64) @ np.asarray(W_lm, np.float64).T


# ---------------------------------------------------------------------------
# a6: accept / reject
# ---------------------------------------------------------------------------

def accept(tree: dict, logits, T, u_acc, u_bonus, D):
    """Accept/reject on one request's flattened tree, given fp32 logits [R, V]."""
    z = np.ascontiguousarray(logits, dtype=np.float32)
    R, V = z.shape
    ua = np.ascontiguousarray(u_acc, np.uint32)
    ub = np.ascontiguousarray(u_bonus, np.uint32)
    acc = np.zeros(1, np.int32)
    path = np.zeros(D + 1, np.int32)
    out = np.zeros(D + 1, np.int32)
    rc = _load().e3o_accept(_p(np.ascontiguousarray(tree["tok"], np.int32)),
                            _p(np.ascontiguousarray(tree["parent"], np.int32)), R, D, _p(z), V,
                            float(np.float32(T)), _p(ua), _p(ub), _p(acc), _p(path), _p(out))
    if rc != 0:
        raise FloatingPointError("non-finite target logit")
    return int(acc[0]), path, out


def accept_many(tok, parent, D, logits, T, u_acc, u_bonus):
    """Same tree and logits, n independent uniform draws: u_acc/u_bonus [n, R]."""
    z = np.ascontiguousarray(logits, dtype=np.float32)
    R, V = z.shape
    n = u_acc.shape[0]
    ua = np.ascontiguousarray(u_acc, np.uint32)
    ub = np.ascontiguousarray(u_bonus, np.uint32)
    acc = np.zeros(n, np.int32)
    path = np.zeros((n, D + 1), np.int32)
    out = np.zeros((n, D + 1), np.int32)
    _load().e3o_accept_many(n, _p(np.ascontiguousarray(tok, np.int32)),
                            _p(np.ascontiguousarray(parent, np.int32)), R, D, _p(z), V,
                            float(np.float32(T)), _p(ua), _p(ub), _p(acc), _p(path), _p(out))
    return acc, path, out


def accept_sampled(tree: dict, logits, T, qlogits, inv_Tq, u_acc, u_bonus, D):
    """Accept/reject for children drawn from the draft distribution.

    logits: [R, V] fp32 target logits of the flattened nodes; qlogits: [R, V]
    fp32, row u = the draft row from which node u's children were drawn (any
    values for nodes without children), at inverse temperature ``inv_Tq``.
    Child c is accepted with probability min(1, p_res(c) / q_res(c)); a
    rejection replaces p_res by norm(max(0, p_res - q_res)) and removes c from
    q_res ("EAGLE 系列与 DFlash", §四 DFlash; "SpecForge…", 先看 checkpoint 最终要参与
    什么计算: correct at the rejection point).  Integer recipe: see
    ``e3o_accept_sampled`` in eagle3_oracle.c.
    """
    z = np.ascontiguousarray(logits, dtype=np.float32)
    zq = np.ascontiguousarray(qlogits, dtype=np.float32)
    R, V = z.shape
    assert zq.shape == (R, V)
    ua = np.ascontiguousarray(u_acc, np.uint32)
    ub = np.ascontiguousarray(u_bonus, np.uint32)
    acc = np.zeros(1, np.int32)
    path = np.zeros(D + 1, np.int32)
    out = np.zeros(D + 1, np.int32)
    rc = _load().e3o_accept_sampled(_p(np.ascontiguousarray(tree["tok"], np.int32)),
                                    _p(np.ascontiguousarray(tree["parent"], np.int32)), R, D, _p(z), V,
                                    float(np.float32(T)), _p(zq), float(np.float32(inv_Tq)), _p(ua), _p(ub),
                                    _p(acc), _p(path), _p(out))
    if rc != 0:
        raise FloatingPointError("non-finite logit")
    return int(acc[0]), path, out


def sampled_trials(n, k, W, D, qtab, inv_Tq, ptab, T, seed0, u_acc, u_bonus):
    """n rounds of a small synthetic model with sampled drafts (see
    ``e3o_sampled_trials``): qtab [D, Fmax, V] draft logits per (depth, frontier
    row), ptab [V + 1, V] target logits (row 0 the root, row 1 + t after token t).
    u_acc / u_bonus: [n, Rcap] uint32.  Returns (acc_len [n], out_tok [n, D+1])."""
    qt = np.ascontiguousarray(qtab, np.float32)
    pt = np.ascontiguousarray(ptab, np.float32)
    Dq, Fmax, V = qt.shape
    assert Dq >= D and pt.shape == (V + 1, V)
    ua = np.ascontiguousarray(u_acc, np.uint32)
    ub = np.ascontiguousarray(u_bonus, np.uint32)
    acc = np.zeros(n, np.int32)
    out = np.zeros((n, D + 1), np.int32)
    R = _load().e3o_sampled_trials(n, V, k, W, D, _p(qt), Fmax, float(np.float32(inv_Tq)), _p(pt),
                                   float(np.float32(T)), seed0 & (2 ** 64 - 1), _p(ua), _p(ub), ua.shape[1],
                                   _p(acc), _p(out))
    if R < 0:
        raise ValueError("tree larger than the uniform arrays")
    return acc, out


# ---------------------------------------------------------------------------
# a7: KV compaction onto the accepted path
# ---------------------------------------------------------------------------

def kv_compact(caches, page_table, kv_len, path, acc_len):
    """Copy semantics, into fresh arrays: for every layer cache (K and V alike),
    request b and j = 1..acc_len[b], logical slot P+j receives what slot
    P+path[b][j] held before the call (P = kv_len[b]).  New kv_len = P + 1 + acc.

    [TB] "一棵候选树怎样被验证" step 5: only the accepted path's KV is committed.
    """
    out = []
    for cache in caches:
        old = np.array(cache, copy=True)
        new = np.array(cache, copy=True)
        ps = cache.shape[2]
        for b in range(len(kv_len)):
            P = int(kv_len[b])
            for j in range(1, int(acc_len[b]) + 1):
                src = P + int(path[b][j])
                dst = P + j
                new[page_table[b][dst // ps], :, dst % ps, :] = old[page_table[b][src // ps], :, src % ps, :]
        out.append(new)
    new_len = np.asarray(kv_len, np.int64) + 1 + np.asarray(acc_len, np.int64)
    return out, new_len.astype(np.int32)
