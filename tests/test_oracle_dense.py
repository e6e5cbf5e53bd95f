"""Pins for the oracle's float steps: fusion, tree-masked attention, LM head (CPU)."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from eagle_speculative_decoding_round_gb300 import synth


# ---------------------------------------------------------------- fusion ----

def test_fuse_block_identity_closed_form():
    d, M = 24, 5
    hl, hm, hh = (synth.normal(1, n, (M, d), 1.0) for n in ("l", "m", "h"))
    I = np.eye(d)
    W = np.concatenate([I, 2 * I, 4 * I], axis=1)  # [d, 3d]
    g = oracle.fuse(hl, hm, hh, W)
    assert np.array_equal(g, hl.astype(np.float64) + 2 * hm.astype(np.float64) + 4 * hh.astype(np.float64))


def test_fuse_one_hot_picks_weight_columns_and_bias():
    d, dout = 8, 6
    W = synth.normal(2, "W", (dout, 3 * d), 1.0)
    bias = synth.normal(2, "b", (dout,), 1.0)
    for j in range(3 * d):
        x = np.zeros((1, 3 * d), np.float32)
        x[0, j] = 1.0
        g = oracle.fuse(x[:, :d], x[:, d:2 * d], x[:, 2 * d:], W, bias)
        assert np.allclose(g[0], W[:, j].astype(np.float64) + bias, atol=0, rtol=0)


# -------------------------------------------------------------- LM head ----

def test_lmhead_one_hot_rows():
    V, d = 50, 12
    W = synth.normal(3, "lm", (V, d), 1.0)
    h = np.eye(d, dtype=np.float32)[[3, 0, 11]]
    z = oracle.lmhead_logits(h, W)
    assert np.array_equal(z, W[:, [3, 0, 11]].T.astype(np.float64))


# ------------------------------------------------------------ attention ----

def make_kv(seed, B, lens, R, KVH, hd, page_size, std=0.5):
    pt, npages = synth.page_table(seed, [n + R for n in lens], page_size)
    K = synth.normal(seed, "K", (npages, KVH, page_size, hd), std)
    Vc = synth.normal(seed, "V", (npages, KVH, page_size, hd), std)
    return pt, K, Vc


def tree_parent(seed, R):
    rng = np.random.default_rng(seed)
    par = np.full(R, -1, np.int32)
    for i in range(1, R):
        par[i] = rng.integers(0, i)  # any earlier node: a valid BFS-ordered tree
    return par


def ancestors(par, i):
    out = []
    while i >= 0:
        out.append(i)
        i = int(par[i])
    return out


def mask_from_parent(par):
    R = len(par)
    words = (R + 63) // 64
    m = np.zeros((R, words), np.uint64)
    for i in range(R):
        for j in ancestors(par, i):
            m[i, j >> 6] |= np.uint64(1 << (j & 63))
    return m


def sdpa_reference(Q, K, Vc, pt, lens, par, scale):
    """torch scaled_dot_product_attention (fp64) with a boolean mask built from the
    ancestor lists of the test's own tree."""
    B, R, H, hd = Q.shape
    KVH = K.shape[1]
    out = np.zeros((B, R, H, hd))
    for b in range(B):
        P = lens[b]
        kb = torch.from_numpy(oracle.gather_tokens(K, pt[b], 0, P + R))
        vb = torch.from_numpy(oracle.gather_tokens(Vc, pt[b], 0, P + R))
        allow = torch.zeros(R, P + R, dtype=torch.bool)
        allow[:, :P] = True
        for i in range(R):
            for j in ancestors(par[b], i):
                allow[i, P + j] = True
        kb = kb.repeat_interleave(H // KVH, dim=1).permute(1, 0, 2)  # [H, T, hd]
        vb = vb.repeat_interleave(H // KVH, dim=1).permute(1, 0, 2)
        q = torch.from_numpy(Q[b].astype(np.float64)).permute(1, 0, 2)  # [H, R, hd]
        o = F.scaled_dot_product_attention(q, kb, vb, attn_mask=allow, scale=scale)
        out[b] = o.permute(1, 0, 2).numpy()
    return out


@pytest.mark.parametrize("case", [
    dict(B=2, lens=[37, 70], R=9, H=4, KVH=2, hd=16, ps=16),
    dict(B=1, lens=[128], R=15, H=4, KVH=4, hd=64, ps=64),
    dict(B=1, lens=[5], R=1, H=8, KVH=2, hd=32, ps=4),      # N = 0: plain decode
    dict(B=1, lens=[0], R=6, H=2, KVH=1, hd=8, ps=8),       # empty prefix
])
def test_tree_attention_equals_dense_and_sdpa(case):
    B, lens, R, H, KVH, hd, ps = (case[k] for k in ("B", "lens", "R", "H", "KVH", "hd", "ps"))
    pt, K, Vc = make_kv(4, B, lens, R, KVH, hd, ps)
    Q = synth.normal(4, "Q", (B, R, H, hd), 0.5)
    par = np.stack([tree_parent(10 + b, R) for b in range(B)])
    mask = np.stack([mask_from_parent(par[b]) for b in range(B)])
    kv_len = np.array(lens, np.int32)
    scale = 1.0 / math.sqrt(hd)
    O1, l1 = oracle.tree_verify_attn(Q, K, Vc, pt, kv_len, par, scale)
    O2, l2 = oracle.tree_verify_attn_dense(Q, K, Vc, pt, kv_len, mask, scale)
    assert np.abs(O1 - O2).max() <= 1e-12
    assert np.abs(l1 - l2).max() <= 1e-12
    ref = sdpa_reference(Q, K, Vc, pt, lens, par, scale)
    assert np.abs(O1 - ref).max() <= 1e-12


def test_chain_tree_equals_causal_attention():
    # a chain of R nodes behind a P-token prefix is ordinary causal attention
    P, R, H, hd = 20, 7, 2, 16
    pt, K, Vc = make_kv(6, 1, [P], R, H, hd, 8)
    Q = synth.normal(6, "Q", (1, R, H, hd), 0.5)
    par = np.arange(-1, R - 1, dtype=np.int32)[None]
    O, _ = oracle.tree_verify_attn(Q, K, Vc, pt, np.array([P], np.int32), par, 0.25)
    kb = torch.from_numpy(oracle.gather_tokens(K, pt[0], 0, P + R)).permute(1, 0, 2)
    vb = torch.from_numpy(oracle.gather_tokens(Vc, pt[0], 0, P + R)).permute(1, 0, 2)
    q = torch.from_numpy(Q[0].astype(np.float64)).permute(1, 0, 2)
    causal = torch.ones(P + R, P + R, dtype=torch.bool).tril()[P:]
    ref = F.scaled_dot_product_attention(q, kb, vb, attn_mask=causal, scale=0.25)
    assert np.abs(O[0] - ref.permute(1, 0, 2).numpy()).max() <= 1e-12


def test_lse_closed_form_with_identical_keys():
    # all keys equal: softmax is uniform over prefix + ancestors + self, so
    # lse = q.k * scale + ln(P + depth + 1) and O = mean of the visible values.
    P, R, H, hd, ps = 13, 8, 2, 8, 4
    pt, K, Vc = make_kv(8, 1, [P], R, H, hd, ps)
    K[:] = K[0, 0, 0]
    Q = synth.normal(8, "Q", (1, R, H, hd), 0.5)
    par = tree_parent(3, R)[None]
    O, lse = oracle.tree_verify_attn(Q, K, Vc, pt, np.array([P], np.int32), par, 0.3)
    kvec = K[0, 0, 0].astype(np.float64)
    vals = oracle.gather_tokens(Vc, pt[0], 0, P + R)
    for i in range(R):
        anc = ancestors(par[0], i)
        n = P + len(anc)
        keys = list(range(P)) + [P + j for j in anc]
        for h in range(H):
            assert abs(lse[0, i, h] - (0.3 * float(Q[0, i, h].astype(np.float64) @ kvec) + math.log(n))) < 1e-12
            assert np.abs(O[0, i, h] - vals[keys, h, :].mean(axis=0)).max() < 1e-12


def test_lse_merge_of_prefix_and_tree_segments():
    """[USP] the main (prefix) segment and the branch (tree) segment merged by
    their log-sum-exp equal one softmax over both: checked on the oracle's
    (O, lse) by splitting its own inputs."""
    P, R, H, hd = 40, 6, 2, 16
    pt, K, Vc = make_kv(12, 1, [P], R, H, hd, 8)
    Q = synth.normal(12, "Q", (1, R, H, hd), 0.5)
    par = tree_parent(4, R)[None]
    O, lse = oracle.tree_verify_attn(Q, K, Vc, pt, np.array([P], np.int32), par, 0.25)
    kb = oracle.gather_tokens(K, pt[0], 0, P + R)
    vb = oracle.gather_tokens(Vc, pt[0], 0, P + R)
    for i in range(R):
        anc = ancestors(par[0], i)
        for h in range(H):
            q = Q[0, i, h].astype(np.float64)
            s1 = kb[:P, h] @ q * 0.25
            s2 = kb[[P + j for j in anc], h] @ q * 0.25
            l1, l2 = np.logaddexp.reduce(s1), np.logaddexp.reduce(s2)
            o1 = np.exp(s1 - l1) @ vb[:P, h]
            o2 = np.exp(s2 - l2) @ vb[[P + j for j in anc], h]
            lm = np.logaddexp(l1, l2)
            om = math.exp(l1 - lm) * o1 + math.exp(l2 - lm) * o2
            assert abs(lse[0, i, h] - lm) < 1e-12
            assert np.abs(O[0, i, h] - om).max() < 1e-12


def test_verify_rows_equal_full_oracle():
    """The sampled-row form runs the same per-row step as the full form."""
    rng = np.random.default_rng(5)
    B, R, H, KVH, hd, ps = 2, 7, 4, 2, 16, 4
    lens = [9, 3]
    npages = sum((p + R + ps - 1) // ps for p in lens)
    pt = np.full((B, 8), -1, np.int32)
    nxt = 0
    for b, p in enumerate(lens):
        for j in range((p + R + ps - 1) // ps):
            pt[b, j] = nxt
            nxt += 1
    K = rng.standard_normal((npages, KVH, ps, hd))
    V = rng.standard_normal((npages, KVH, ps, hd))
    Q = rng.standard_normal((B, R, H, hd))
    par = np.array([[-1, 0, 0, 1, 1, 2, 5], [-1, 0, 1, 2, 3, 4, 5]])
    O, lse = oracle.tree_verify_attn(Q, K, V, pt, np.array(lens), par, 0.25)
    rows = [(0, 6, 3), (1, 0, 0), (1, 5, 2), (0, 3, 1)]
    Or, lr = oracle.tree_verify_attn_rows(Q, K, V, pt, np.array(lens), par, 0.25, rows)
    for n, (b, i, h) in enumerate(rows):
        assert np.array_equal(Or[n], O[b, i, h]) and lr[n] == lse[b, i, h]
