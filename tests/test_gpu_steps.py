"""GPU parity of each step of the round, through the C ABI, against the oracle.

Floats: 1e-5 relative (fp32) and 2e-2 relative (bf16), norm-wise.  Integer
results (candidates, tree, mask, accepted paths, compaction) are bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_round_gb300 import synth
from gpu_util import assert_close, bf16_dev, host, kv_paged, random_tree, to_dev, tree_tokens

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3


def i32(n, fill=0):
    return torch.full((n,) if isinstance(n, int) else n, fill, dtype=torch.int32, device="cuda")


# ------------------------------------------------------------------ fusion ----

@pytest.mark.parametrize("M,d,dout,dt", [(3, 256, 256, "f32"), (1, 256, 256, "f32"), (7, 4096, 4096, "bf16"),
                                         (13, 256, 384, "bf16"), (130, 512, 256, "bf16"), (1, 64, 128, "bf16"),
                                         (300, 128, 200, "bf16"), (5, 96, 256, "bf16"),
                                         # fp32 with more than 16 rows: the tiled SIMT GEMM
                                         (20, 128, 192, "f32"), (70, 96, 130, "f32")])
def test_fuse(M, d, dout, dt):
    hs = [synth.normal(M * d + dout, f"h{i}", (M, d), 0.02) for i in range(3)]
    W = synth.normal(M * d + dout, "Wf", (dout, 3 * d), 0.02)
    bias = synth.normal(1, "bias", (dout,), 0.02) if d == 256 else None
    if dt == "bf16":
        tens = [bf16_dev(h) for h in hs]
        hd_ = [t for t, _ in tens]
        hs = [r for _, r in tens]
        Wt, W = bf16_dev(W)
        g = torch.empty((M, dout), dtype=torch.bfloat16, device="cuda")
        code, tol = e3.E3_BF16, 2e-2
    else:
        hd_ = [to_dev(h) for h in hs]
        Wt = to_dev(W)
        g = torch.empty((M, dout), dtype=torch.float32, device="cuda")
        code, tol = e3.E3_F32, 1e-5
    ws_b = e3.eagle3_fuse_workspace_bytes(M, d, dout, code)
    ws = torch.empty(max(ws_b, 16), dtype=torch.uint8, device="cuda")
    bt = to_dev(bias) if bias is not None else None
    err = i32(1)
    e3.eagle3_fuse(hd_[0], hd_[1], hd_[2], Wt, bt, g, M, d, dout, code, ws, ws_b, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle.fuse(hs[0], hs[1], hs[2], W, bias)
    assert_close(host(g), ref, tol, "fuse")


# ----------------------------------------------------------------- LM head ----

@pytest.mark.parametrize("M,d,V,dt", [(15, 256, 1024, "f32"), (61, 4096, 128256, "bf16"), (3, 128, 1000, "bf16"),
                                      (200, 256, 4096, "bf16"), (300, 192, 2048, "bf16"), (1, 64, 256, "bf16"),
                                      (20, 256, 1000, "bf16"), (40, 100, 512, "bf16"),
                                      # fp32 with more than 16 rows: the tiled SIMT GEMM
                                      (20, 256, 1000, "f32"), (67, 100, 515, "f32")])
def test_lmhead_logits_and_stats(M, d, V, dt):
    h = synth.normal(V + M, "h", (M, d), 1.0)
    W = synth.normal(V + M, "Wlm", (V, d), 4.0 / math.sqrt(d))
    temps = np.array([[1.0, 0.7, 0.0, 1.0, 2.0][i % 5] for i in range(M)], np.float32)
    if dt == "bf16":
        ht, h = bf16_dev(h)
        Wt, W = bf16_dev(W)
        code, tol = e3.E3_BF16, 2e-2
    else:
        ht, Wt = to_dev(h), to_dev(W)
        code, tol = e3.E3_F32, 1e-5
    logits = torch.empty((M, V), dtype=torch.float32, device="cuda")
    rmax = torch.empty(M, dtype=torch.float32, device="cuda")
    rQ = torch.empty(M, dtype=torch.int64, device="cuda")
    ram = i32(M)
    err = i32(1)
    e3.lmhead_logits(ht, Wt, M, d, V, to_dev(temps), logits, rmax, rQ, ram, err, code)
    torch.cuda.synchronize()
    z = host(logits)
    ref = oracle.lmhead_logits(h, W)
    assert_close(z, ref, tol, "logits")
    # softmax statistics: bit-exact against the oracle on the same fp32 logits
    m, Q, am, bad = oracle.row_stats(z, temps)
    assert not bad.any() and int(err.item()) == 0
    assert np.array_equal(host(rmax).view(np.uint32), m.view(np.uint32))
    assert np.array_equal(host(rQ).view(np.uint64), Q)
    assert np.array_equal(host(ram), am)


def test_lmhead_stats_extreme_temperatures():
    """Temperatures whose inverse is 0, denormal or huge: the statistics pass sums the
    masses of the row's tokens only (every CTA chunk of the full vocabulary ends in a
    partial group of loads), bit-exact against the oracle."""
    M, d, V = 6, 64, 128256
    h = synth.normal(11, "h", (M, d), 1.0)
    W = synth.normal(11, "W", (V, d), 0.125)
    temps = np.array([np.inf, 1e30, 3e38, 1e-30, 0.5, 1.0], np.float32)
    ht, h = bf16_dev(h)
    Wt, W = bf16_dev(W)
    logits = torch.empty((M, V), dtype=torch.float32, device="cuda")
    rmax = torch.empty(M, dtype=torch.float32, device="cuda")
    rQ = torch.empty(M, dtype=torch.int64, device="cuda")
    ram = i32(M)
    err = i32(1)
    e3.lmhead_logits(ht, Wt, M, d, V, to_dev(temps), logits, rmax, rQ, ram, err, e3.E3_BF16)
    torch.cuda.synchronize()
    m, Q, am, bad = oracle.row_stats(host(logits), temps)
    assert not bad.any() and int(err.item()) == 0
    assert np.array_equal(host(rmax).view(np.uint32), m.view(np.uint32))
    assert np.array_equal(host(rQ).view(np.uint64), Q)
    assert np.array_equal(host(ram), am)
    assert int(Q[0]) == V << 40  # 1/T = 0: every token has mass 2^40


def test_lmhead_flags_nonfinite():
    M, d, V = 4, 64, 256
    h = synth.normal(3, "h", (M, d), 1.0)
    h[2, 5] = np.inf
    W = synth.normal(3, "W", (V, d), 1.0)
    logits = torch.empty((M, V), dtype=torch.float32, device="cuda")
    err = i32(1)
    e3.lmhead_logits(to_dev(h), to_dev(W), M, d, V, to_dev(np.ones(M, np.float32)), logits,
                     torch.empty(M, device="cuda"), torch.empty(M, dtype=torch.int64, device="cuda"), i32(M), err,
                     e3.E3_F32)
    torch.cuda.synchronize()
    assert int(err.item()) & e3.E3_DEV_ERR_NONFINITE


# ---------------------------------------------------------------- expansion ----

def run_gpu_expansion(logits_per_depth, B, k, W, D):
    """logits_per_depth[d]: [B, F_d, V] fp32 numpy.  Returns candidate arrays and frontiers."""
    sizes, off = [], 0
    F = 1
    for _ in range(D):
        sizes.append((F, off))
        off += F * k
        F = min(W, F * k)
    C = off
    ct, cp, cs, cd = i32((B, C), -7), i32((B, C), -7), torch.zeros((B, C), device="cuda"), i32((B, C), -7)
    cand = e3.make_cand(ct, cp, cs, cd, C)
    fid = i32((B, 1), -1)
    fsc = torch.zeros((B, 1), device="cuda")
    err = i32(1)
    fronts = []
    for di, (F, o) in enumerate(sizes):
        Wn = min(W, F * k)
        nid, nsc = i32((B, Wn)), torch.zeros((B, Wn), device="cuda")
        z = to_dev(logits_per_depth[di])
        e3.eagle3_expand(z, B, F, z.shape[2], k, W, 1.0, fsc, fid, di + 1, o, cand, nid, nsc, err)
        fronts.append((nid, nsc))
        fid, fsc = nid, nsc
    torch.cuda.synchronize()
    return dict(tok=host(ct), parent=host(cp), score=host(cs), depth=host(cd)), fronts, sizes, C, int(err.item())


@pytest.mark.parametrize("V,k,W,D,B,ties", [(1024, 2, 1 << 20, 3, 1, False), (128256, 10, 10, 3, 1, False),
                                            (4096, 10, 10, 6, 3, False), (512, 4, 4, 4, 2, True),
                                            (300, 7, 9, 3, 2, False),
                                            # 320 rows x 8 CTAs: several waves, SMs reused
                                            (128256, 10, 10, 2, 32, False),
                                            # k above 16: the 32-wide per-thread lists
                                            (4096, 20, 20, 3, 2, False), (1000, 32, 64, 3, 1, True),
                                            (999, 24, 40, 3, 2, True)])
def test_expand_bitexact(V, k, W, D, B, ties):
    rng = np.random.default_rng(V + k + D)
    sizes, F = [], 1
    for _ in range(D):
        sizes.append(F)
        F = min(W, F * k)
    logits = []
    for F in sizes:
        z = (rng.standard_normal((B, F, V)) * 3).astype(np.float32)
        if ties:
            z = np.round(z).astype(np.float32)  # many equal values
        logits.append(z)
    got, fronts, gsizes, C, err = run_gpu_expansion(logits, B, k, W, D)
    assert err == 0
    for b in range(B):
        c = oracle.new_cands(C)
        fid = np.array([-1], np.int32)
        fsc = np.zeros(1, np.float32)
        for di, (F, off) in enumerate(gsizes):
            nid, nsc = oracle.expand(logits[di][b], k, W, fsc, fid, di + 1, off, c)
            assert np.array_equal(host(fronts[di][0])[b], nid), ("frontier ids", b, di)
            assert np.array_equal(host(fronts[di][1])[b].view(np.uint32), nsc.view(np.uint32))
            fid, fsc = nid, nsc
        for key in ("tok", "parent", "depth"):
            assert np.array_equal(got[key][b], c[key]), (key, b)
        assert np.array_equal(got["score"][b].view(np.uint32), c["score"].view(np.uint32)), ("score", b)


def test_expand_flags_nonfinite():
    z = np.zeros((1, 1, 64), np.float32)
    z[0, 0, 9] = np.nan
    _, _, _, _, err = run_gpu_expansion([z], 1, 2, 2, 1)
    assert err & e3.E3_DEV_ERR_NONFINITE


# ---------------------------------------------------------------- tree build ----

@pytest.mark.parametrize("V,k,W,D,N,B", [(1024, 2, 1 << 20, 3, 14, 1), (4096, 10, 10, 6, 60, 3),
                                         (2048, 4, 4, 7, 32, 2), (512, 8, 16, 8, 255, 1), (512, 3, 3, 2, 1, 2),
                                         # 1296 candidates: the shared-memory sort over 1024 threads
                                         (4096, 16, 16, 6, 60, 2)])
def test_tree_build_bitexact(V, k, W, D, N, B):
    rng = np.random.default_rng(N + D)
    sizes, F = [], 1
    for _ in range(D):
        sizes.append(F)
        F = min(W, F * k)
    logits = [(rng.standard_normal((B, F, V)) * 2).astype(np.float32) for F in sizes]
    cands, _, _, C, err = run_gpu_expansion(logits, B, k, W, D)
    assert err == 0 and C >= N
    # feed the GPU candidates back on the device and build the tree there
    ct, cp, cs, cd = (to_dev(cands[x]) for x in ("tok", "parent", "score", "depth"))
    cand = e3.make_cand(ct, cp, cs, cd, C)
    R = N + 1
    kvl = rng.integers(0, 5000, B).astype(np.int32)
    root = rng.integers(0, V, B).astype(np.int32)
    out = {x: i32((B, R), -9) for x in ("tok", "parent", "depth", "pos", "node_cand")}
    mask = torch.zeros((B, R, (R + 63) // 64), dtype=torch.int64, device="cuda")
    e3.tree_build_mask(cand, B, C, N, to_dev(root), to_dev(kvl), out["tok"], out["parent"], out["depth"],
                       out["pos"], mask, node_cand=out["node_cand"])
    torch.cuda.synchronize()
    for b in range(B):
        cb = {x: np.ascontiguousarray(cands[x][b]) for x in ("tok", "parent", "score", "depth")}
        ref = oracle.build_tree(cb, C, N, int(root[b]), int(kvl[b]))
        for x in ("tok", "parent", "depth", "pos", "node_cand"):
            assert np.array_equal(host(out[x])[b], ref[x]), (x, b)
        assert np.array_equal(host(mask)[b].view(np.uint64), ref["mask"]), ("mask", b)


def test_tree_build_page_example():
    """The pages' K=3 example through the GPU: flatten order and x_1a's mask row."""
    import json, os
    fx = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "tree_examples.json")))["p2_eagle2_k3"]
    names = [n for n, _ in fx["nodes"]]
    idx = {}
    tok, par, sc, dep = [], [], [], []
    dmap = {}
    for i, (n, p) in enumerate(fx["nodes"]):
        dmap[n] = 1 if p is None else dmap[p] + 1
        idx[n] = i
        tok.append(100 + i)
        par.append(-1 if p is None else idx[p])
        sc.append(-1.0 * dmap[n] - 0.001 * i)
        dep.append(dmap[n])
    C = len(tok)
    keep = [to_dev(np.array(a, t)) for a, t in ((tok, np.int32), (par, np.int32), (sc, np.float32), (dep, np.int32))]
    cand = e3.make_cand(*keep, C)  # make_cand keeps raw addresses: `keep` holds the tensors alive
    R = C + 1
    out = {x: i32((1, R)) for x in ("tok", "parent", "depth", "pos")}
    mask = torch.zeros((1, R, 1), dtype=torch.int64, device="cuda")
    e3.tree_build_mask(cand, 1, C, C, to_dev(np.array([7], np.int32)), to_dev(np.array([50], np.int32)),
                       out["tok"], out["parent"], out["depth"], out["pos"], mask)
    torch.cuda.synchronize()
    flat = ["root"] + [names[int(t) - 100] for t in host(out["tok"])[0][1:]]
    assert flat == fx["flat"]
    row = int(host(mask)[0, flat.index("x_1a"), 0].view(np.uint64))
    assert row == sum(1 << flat.index(n) for n in fx["sees"]["x_1a"])
    assert not (row >> flat.index("x_2")) & 1


@pytest.mark.parametrize("n_cand,N,B,levels", [(510, 60, 2, 3), (1000, 255, 1, 2), (300, 100, 3, 40),
                                               (2000, 200, 1, 4)])
def test_tree_build_score_ties(n_cand, N, B, levels):
    """Candidate sets whose scores take only a few values: the rank of a key among
    equal scores is settled by the candidate index (score descending, index
    ascending), bit-exact against the oracle."""
    rng = np.random.default_rng(n_cand + N)
    C = n_cand
    cands = {x: np.zeros((B, C), t) for x, t in (("tok", np.int32), ("parent", np.int32), ("score", np.float32),
                                                 ("depth", np.int32))}
    for b in range(B):
        for i in range(C):
            # a parent earlier in the list, scores that never rise along a path and
            # repeat across the set
            p = -1 if i < 8 or rng.random() < 0.1 else int(rng.integers(0, i))
            d = 1 if p < 0 else min(cands["depth"][b, p] + 1, 16)
            if d > 1 and cands["depth"][b, p] >= 16:
                p, d = -1, 1
            ps = 0.0 if p < 0 else float(cands["score"][b, p])
            cands["parent"][b, i] = p
            cands["depth"][b, i] = d
            cands["score"][b, i] = ps - float(rng.integers(0, levels))
            cands["tok"][b, i] = int(rng.integers(0, 1 << 20))
    ct, cp, cs, cd = (to_dev(cands[x]) for x in ("tok", "parent", "score", "depth"))
    cand = e3.make_cand(ct, cp, cs, cd, C)
    R = N + 1
    kvl = rng.integers(0, 5000, B).astype(np.int32)
    root = rng.integers(0, 1000, B).astype(np.int32)
    out = {x: i32((B, R), -9) for x in ("tok", "parent", "depth", "pos", "node_cand")}
    mask = torch.zeros((B, R, (R + 63) // 64), dtype=torch.int64, device="cuda")
    e3.tree_build_mask(cand, B, C, N, to_dev(root), to_dev(kvl), out["tok"], out["parent"], out["depth"],
                       out["pos"], mask, node_cand=out["node_cand"])
    torch.cuda.synchronize()
    for b in range(B):
        cb = {x: np.ascontiguousarray(cands[x][b]) for x in ("tok", "parent", "score", "depth")}
        ref = oracle.build_tree(cb, C, N, int(root[b]), int(kvl[b]))
        for x in ("tok", "parent", "depth", "pos", "node_cand"):
            assert np.array_equal(host(out[x])[b], ref[x]), (x, b)
        assert np.array_equal(host(mask)[b].view(np.uint64), ref["mask"]), ("mask", b)


# ---------------------------------------------------------------- attention ----

def run_gpu_verify(Q, K, Vc, pt, npages, kv_len, mask, H, KVH, hd, page_size, dt, max_kv_len=None, scale=None,
                   flags=0):
    B, R = Q.shape[0], Q.shape[1]
    max_kv_len = int(max(kv_len)) if max_kv_len is None else max_kv_len
    scale = scale or 1.0 / math.sqrt(hd)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    code = e3.E3_BF16 if dt == "bf16" else e3.E3_F32
    Qt = to_dev(Q).to(tdt)
    Kt, Vt = to_dev(K).to(tdt), to_dev(Vc).to(tdt)
    ptt = to_dev(pt)
    kv = e3.make_kv_layer(Kt, Vt, ptt, npages, page_size, pt.shape[1], KVH, hd, code, flags)
    O = torch.full((B, R, H, hd), float("nan"), dtype=tdt, device="cuda")
    lse = torch.full((B, R, H), float("nan"), device="cuda")
    wsb = e3.eagle3_verify_workspace_bytes(B, R, H, KVH, hd, max_kv_len, code)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    err = i32(1)
    e3.tree_verify_attn(Qt, kv, to_dev(np.asarray(kv_len, np.int32)), to_dev(mask.view(np.int64)), B, R, H,
                        max_kv_len, scale, O, lse, err, ws, wsb)
    torch.cuda.synchronize()
    return host(O), host(lse), int(err.item())


def mask_from_parent(par):
    R = len(par)
    m = np.zeros((R, (R + 63) // 64), np.uint64)
    for i in range(R):
        j = i
        while j >= 0:
            m[i, j >> 6] |= np.uint64(1 << (j & 63))
            j = int(par[j])
    return m


@pytest.mark.parametrize("case", [
    dict(dt="f32", lens=[128], R=15, H=4, KVH=4, hd=64, ps=64, D=3),            # tiny config
    dict(dt="bf16", lens=[2048], R=61, H=32, KVH=8, hd=128, ps=64, D=6),        # 8B shape
    dict(dt="bf16", lens=[517, 64, 1500, 9], R=61, H=32, KVH=8, hd=128, ps=64, D=6),  # ragged batch
    dict(dt="bf16", lens=[300, 1000], R=61, H=64, KVH=8, hd=128, ps=64, D=6),   # 70B heads (G = 8)
    dict(dt="bf16", lens=[700], R=33, H=32, KVH=8, hd=128, ps=64, D=7),         # long-context tree shape
    dict(dt="bf16", lens=[0, 33], R=9, H=8, KVH=2, hd=64, ps=16, D=4),          # empty prefix, hd 64
    dict(dt="bf16", lens=[77], R=1, H=8, KVH=8, hd=128, ps=32, D=0),            # N = 0: plain decode
    dict(dt="f32", lens=[200, 3], R=130, H=2, KVH=1, hd=32, ps=16, D=9),        # > 64 nodes: 3 mask words
    dict(dt="bf16", lens=[100], R=256, H=4, KVH=2, hd=128, ps=64, D=16),        # maximum tree
    dict(dt="bf16", lens=[0, 128, 64, 65], R=20, H=8, KVH=2, hd=128, ps=64, D=5),  # empty / page-aligned prefixes
    dict(dt="bf16", lens=[300, 1], R=61, H=16, KVH=16, hd=128, ps=128, D=6),    # 128-token pages, MHA (G = 1)
    dict(dt="bf16", lens=[12000], R=61, H=32, KVH=8, hd=128, ps=64, D=6),       # long prefix: one wave + merge kernel
    dict(dt="bf16", lens=[12000, 5, 1000], R=61, H=32, KVH=8, hd=128, ps=64, D=6),  # ragged long: empty segments
    dict(dt="bf16", lens=[30000], R=61, H=16, KVH=4, hd=128, ps=64, D=6),       # long: one wave without clusters
])
@pytest.mark.parametrize("flags", [0, 1])  # 1: E3_KV_PREFIX_STABLE (prefix loads before the grid-dependency wait)
def test_verify_attention(case, flags):
    dt, lens, R, H, KVH, hd, ps, D = (case[x] for x in ("dt", "lens", "R", "H", "KVH", "hd", "ps", "D"))
    B = len(lens)
    seed = sum(lens) + R
    pt, npages, K, Vc = kv_paged(seed, lens, R, KVH, hd, ps, 1.0, dt)
    Q = synth.normal(seed, "Q", (B, R, H, hd), 1.0)
    if dt == "bf16":
        Q = synth.to_bf16_f32(Q)
    rng = np.random.default_rng(seed)
    par = np.stack([random_tree(rng, R, max(D, 1))[0] for _ in range(B)])
    mask = np.stack([mask_from_parent(p) for p in par])
    O, lse, err = run_gpu_verify(Q, K, Vc, pt, npages, lens, mask, H, KVH, hd, ps, dt, flags=flags)
    assert err == 0
    Oref, lref = oracle.tree_verify_attn(Q, K, Vc, pt, np.array(lens), par, 1.0 / math.sqrt(hd))
    tol = 2e-2 if dt == "bf16" else 1e-5
    assert_close(O, Oref, tol, "O")
    assert_close(lse, lref, tol, "lse")


def test_verify_capacity_is_flagged_not_faulted():
    lens, R, H, KVH, hd, ps = [64], 5, 4, 4, 64, 16
    pt, npages, K, Vc = kv_paged(1, lens, R, KVH, hd, ps)
    Q = synth.to_bf16_f32(synth.normal(1, "Q", (1, R, H, hd), 1.0))
    mask = mask_from_parent(np.arange(-1, R - 1))[None]
    # kv_len beyond max_kv_len: the request is skipped and flagged
    O, lse, err = run_gpu_verify(Q, K, Vc, pt, npages, [70], mask, H, KVH, hd, ps, "bf16", max_kv_len=64)
    assert err & e3.E3_DEV_ERR_CAPACITY


# ------------------------------------------------------------------- accept ----

def accept_case(seed, B, R, D, V, temps, zstd=2.0):
    rng = np.random.default_rng(seed)
    trees = [random_tree(rng, R, D) for _ in range(B)]
    # logits from the GPU LM head (exact fp32 products of one-hot rows)
    z = (rng.standard_normal((B * R, V)) * zstd).astype(np.float32)
    toks = np.stack([tree_tokens(rng, trees[b][0], z[b * R:(b + 1) * R]) for b in range(B)])
    par = np.stack([t[0] for t in trees])
    return z, toks, par


def gpu_stats(table, row_index, temps_rows):
    """Logits row m = table[row_index[m]], produced by the GPU LM head as an exact
    fp32 product of one-hot rows with W_lm = table^T; returns the GPU logits and
    the GPU softmax statistics."""
    n_tab, V = table.shape
    M = len(row_index)
    h = np.zeros((M, n_tab), np.float32)
    h[np.arange(M), row_index] = 1.0
    W = np.ascontiguousarray(table.T)
    rmax = torch.empty(M, device="cuda")
    rQ = torch.empty(M, dtype=torch.int64, device="cuda")
    ram = i32(M)
    err = i32(1)
    logits = torch.empty((M, V), device="cuda")
    e3.lmhead_logits(to_dev(h), to_dev(W), M, n_tab, V, to_dev(np.asarray(temps_rows, np.float32)), logits, rmax,
                     rQ, ram, err, e3.E3_F32)
    return logits, rmax, rQ, ram, err


@pytest.mark.parametrize("B,R,D,V", [(64, 15, 3, 1000), (8, 61, 6, 128256), (32, 33, 7, 4096), (4, 256, 16, 300)])
def test_accept_bitexact(B, R, D, V):
    temps = np.array([[1.0, 0.0, 0.7, 1.5][b % 4] for b in range(B)], np.float32)
    z, toks, par = accept_case(B * R + V, B, R, D, V, temps)
    logits, rmax, rQ, ram, err = gpu_stats(z, np.arange(B * R), np.repeat(temps, R))
    ua = synth.uniforms(B + R, synth.PURPOSE_ACCEPT, B, R)
    ub = synth.uniforms(B + R, synth.PURPOSE_BONUS, B, R)
    acc, path, out, st = i32(B), i32((B, D + 1)), i32((B, D + 1)), i32(B)
    e3.spec_accept(to_dev(toks), to_dev(par), B, R, D, logits, rmax, rQ, ram, V, to_dev(temps),
                   to_dev(ua.view(np.int32)), to_dev(ub.view(np.int32)), e3.E3_ACCEPT_TREE_DET, acc, path, out, st)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    zl = host(logits)
    assert np.array_equal(zl, z)
    for b in range(B):
        a, p, o = oracle.accept({"tok": toks[b], "parent": par[b]}, zl[b * R:(b + 1) * R], temps[b], ua[b], ub[b], D)
        assert host(acc)[b] == a, b
        assert np.array_equal(host(path)[b], p), b
        assert np.array_equal(host(out)[b], o), b
        assert host(st)[b] == 0


def test_accept_wide_nodes():
    """Nodes with more children than a warp has lanes (the walk tests a node's children 32
    at a time): the root has 40 children (the first the most likely token, the rest from
    the least to the most likely of the next 39), its first child 33 children (from the
    least to the most likely, so the greedy match is the 33rd, beyond the first 32).
    Bit-exact against the oracle."""
    R, D, V = 1 + 40 + 33 + 3, 3, 2000
    parent = np.full(R, -1, np.int32)
    parent[1:41] = 0
    parent[41:74] = 1
    parent[74:77] = 41
    B = 16
    temps = np.array([[0.0, 1.0, 0.7, 1.5][b % 4] for b in range(B)], np.float32)
    rng = np.random.default_rng(31)
    z = (rng.standard_normal((B * R, V)) * 2.0).astype(np.float32)
    toks = np.zeros((B, R), np.int32)
    for b in range(B):
        zb = z[b * R:(b + 1) * R]
        for u in range(R):
            kids = [c for c in range(R) if parent[c] == u]
            if kids:
                top = np.argsort(-zb[u], kind="stable")[:len(kids)]
                order = np.concatenate([top[:1], top[1:][::-1]]) if u == 0 else top[::-1]
                for c, t in zip(kids, order):
                    toks[b, c] = t
    par = np.tile(parent, (B, 1))
    logits, rmax, rQ, ram, err = gpu_stats(z, np.arange(B * R), np.repeat(temps, R))
    ua = synth.uniforms(B + R + 1, synth.PURPOSE_ACCEPT, B, R)
    ub = synth.uniforms(B + R + 1, synth.PURPOSE_BONUS, B, R)
    acc, path, out, st = i32(B), i32((B, D + 1)), i32((B, D + 1)), i32(B)
    e3.spec_accept(to_dev(toks), to_dev(par), B, R, D, logits, rmax, rQ, ram, V, to_dev(temps),
                   to_dev(ua.view(np.int32)), to_dev(ub.view(np.int32)), e3.E3_ACCEPT_TREE_DET, acc, path, out, st)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    zl = host(logits)
    deep = 0
    for b in range(B):
        a, pth, o = oracle.accept({"tok": toks[b], "parent": par[b]}, zl[b * R:(b + 1) * R], temps[b], ua[b], ub[b], D)
        assert host(acc)[b] == a, b
        assert np.array_equal(host(path)[b], pth), b
        assert np.array_equal(host(out)[b], o), b
        assert host(st)[b] == 0
        deep += a >= 2
    assert deep > 0  # the greedy walks accept node 1's 33rd child


def test_accept_sampling_lossless_on_gpu():
    """Chi-square losslessness run on the GPU: 200k independent requests with the
    same tree and logits, fresh uniforms each."""
    from scipy.special import softmax
    from scipy.stats import chi2
    from test_oracle_round import chi_square, full_binary_tree
    V, D, n = 16, 3, 200_000
    parent = full_binary_tree(D)
    R = len(parent)
    rng = np.random.default_rng(123)
    zr = (rng.standard_normal((R, V))).astype(np.float32)
    tok = np.zeros(R, np.int32)
    for u in range(R):
        kids = [c for c in range(R) if parent[c] == u]
        for c, t in zip(kids, np.argsort(-zr[u], kind="stable")[:len(kids)]):
            tok[c] = t
    logits, rmax, rQ, ram, err = gpu_stats(zr, np.tile(np.arange(R), n), np.ones(n * R, np.float32))
    ua = synth.uniforms(77, synth.PURPOSE_ACCEPT, n, R)
    ub = synth.uniforms(77, synth.PURPOSE_BONUS, n, R)
    acc, path, out, st = i32(n), i32((n, D + 1)), i32((n, D + 1)), i32(n)
    e3.spec_accept(to_dev(np.tile(tok, (n, 1))), to_dev(np.tile(parent, (n, 1))), n, R, D, logits, rmax, rQ, ram, V,
                   to_dev(np.ones(n, np.float32)), to_dev(ua.view(np.int32)), to_dev(ub.view(np.int32)),
                   e3.E3_ACCEPT_TREE_DET, acc, path, out, st)
    torch.cuda.synchronize()
    out = host(out)
    p = softmax(zr.astype(np.float64), axis=1)
    stat, dof = chi_square(np.bincount(out[:, 0], minlength=V).astype(float), p[0])
    assert stat < chi2.ppf(1 - 1e-3, dof)
    for c in (1, 2):
        sel = out[:, 0] == tok[c]
        stat, dof = chi_square(np.bincount(out[sel, 1], minlength=V).astype(float), p[c])
        assert stat < chi2.ppf(1 - 1e-3, dof)
    # and identical to the oracle on the same uniforms
    a2, p2, o2 = oracle.accept_many(tok, parent, D, zr, 1.0, ua, ub)
    assert np.array_equal(out, o2)


# ---------------------------------------------------------------- compaction ----

@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_kv_compact_bitexact(dt):
    L, B, KVH, hd, ps, R, D = 3, 4, 2, 64, 16, 12, 5
    lens = [40, 17, 0, 63]
    rng = np.random.default_rng(3)
    pt, npages, _, _ = kv_paged(5, lens, R, KVH, hd, ps, 1.0, dt)
    caches = []
    for l in range(2 * L):
        a = synth.normal(l, "c", (npages, KVH, ps, hd), 1.0)
        caches.append(synth.to_bf16_f32(a) if dt == "bf16" else a)
    paths = np.full((B, D + 1), -1, np.int32)
    acc = np.array([3, 0, 5, 1], np.int32)
    paths[0, :4] = [0, 3, 4, 5]          # overlap: slot 3 is a source and a destination
    paths[1, :1] = [0]
    paths[2, :6] = [0, 2, 5, 7, 9, 11]
    paths[3, :2] = [0, 8]
    tdt = torch.bfloat16 if dt == "bf16" else torch.float32
    code = e3.E3_BF16 if dt == "bf16" else e3.E3_F32
    tens = [to_dev(c).to(tdt) for c in caches]
    ptt = to_dev(pt)
    layers = [e3.make_kv_layer(tens[2 * l], tens[2 * l + 1], ptt, npages, ps, pt.shape[1], KVH, hd, code)
              for l in range(L)]
    kvl = to_dev(np.array(lens, np.int32))
    err = i32(1)
    e3.kv_compact(layers, B, to_dev(paths), to_dev(acc), D, kvl, err)
    torch.cuda.synchronize()
    new, new_len = oracle.kv_compact(caches, pt, np.array(lens), paths, acc)
    for l in range(2 * L):
        assert np.array_equal(host(tens[l]), new[l]), l
    assert np.array_equal(host(kvl), new_len)
    assert int(err.item()) == 0
