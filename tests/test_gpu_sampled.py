"""GPU parity of the sampled-draft mode, through the C ABI, against the oracle:
eagle3_expand_sampled (candidates, frontier and draft statistics bit-exact),
tree_build_mask's node_cand output, spec_accept_sampled (accepted length, path
and emitted tokens bit-exact), and losslessness of whole sampled rounds drawn
and accepted on the GPU (chi-square).

"EAGLE 系列与 DFlash", §四 DFlash: drafts accepted with min(1, p_target / p_draft).
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_round_gb300 import synth
from gpu_util import host, to_dev

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3

QDT = np.dtype([("row", "<u8"), ("Q", "<u8"), ("m", "<f4"), ("it", "<f4")])


def i32(n, fill=0):
    return torch.full((n,) if isinstance(n, int) else n, fill, dtype=torch.int32, device="cuda")


def sizes_of(k, W, D):
    out, F, off = [], 1, 0
    for _ in range(D):
        out.append((F, off))
        off += F * k
        F = min(W, F * k)
    return out, off


def gpu_sampled_expansion(logits, B, k, W, D, seed, inv_T=1.0):
    """logits[d]: [B, F_d, V] fp32 numpy.  Runs eagle3_expand_sampled depth by
    depth; returns host candidates [B, C], the frontiers, the draft statistics
    [B, 1 + C] and the device logits (which the statistics point into)."""
    sizes, C = sizes_of(k, W, D)
    ct, cp, cd = i32((B, C), -7), i32((B, C), -7), i32((B, C), -7)
    cs = torch.zeros((B, C), device="cuda")
    cand = e3.make_cand(ct, cp, cs, cd, C)
    qs = torch.zeros(B * (C + 1) * e3.QSTAT_BYTES, dtype=torch.uint8, device="cuda")
    fid, fsc = i32((B, 1), -1), torch.zeros((B, 1), device="cuda")
    err = i32(1)
    fronts, zdev = [], []
    for di, (F, off) in enumerate(sizes):
        Wn = min(W, F * k)
        nid, nsc = i32((B, Wn)), torch.zeros((B, Wn), device="cuda")
        z = to_dev(logits[di])
        zdev.append(z)
        e3.eagle3_expand_sampled(z, B, F, z.shape[2], k, W, inv_T, fsc, fid, di + 1, off, cand, nid, nsc, seed, qs,
                                 err)
        fronts.append((nid, nsc))
        fid, fsc = nid, nsc
    torch.cuda.synchronize()
    cands = dict(tok=host(ct), parent=host(cp), score=host(cs), depth=host(cd))
    q = host(qs).view(QDT).reshape(B, C + 1)
    return cands, [(host(a), host(b)) for a, b in fronts], q, zdev, C, int(err.item()), cand, (ct, cp, cs, cd)


def draft_logits(rng, B, k, W, D, V, sparse=False, std=2.0):
    sizes, _ = sizes_of(k, W, D)
    out = []
    for F, _ in sizes:
        z = (rng.standard_normal((B, F, V)) * std).astype(np.float32)
        if sparse:  # only 3 tokens per row carry mass: fewer than k can be drawn
            keep = rng.random((B, F, V)) < 3.0 / V
            z = np.where(keep, z, np.float32(-100.0)).astype(np.float32)
        out.append(z)
    return out


@pytest.mark.parametrize("V,k,W,D,B,inv_T,sparse", [
    (128256, 10, 10, 3, 2, 1.0, False), (1000, 4, 4, 3, 3, 1.0, False), (999, 3, 5, 3, 2, 0.8, False),
    (4096, 20, 20, 2, 1, 1.0, False), (128256, 1, 1, 3, 4, 1.25, False), (64, 8, 16, 3, 2, 1.0, False),
    (200, 30, 60, 2, 1, 1.0, False), (64, 5, 5, 2, 2, 1.0, True),
    # 320 frontier rows: several waves of clusters
    (128256, 10, 10, 2, 32, 1.0, False)])
def test_expand_sampled_bitexact(V, k, W, D, B, inv_T, sparse):
    rng = np.random.default_rng(V + k + D)
    logits = draft_logits(rng, B, k, W, D, V, sparse)
    seed = int(rng.integers(0, 2 ** 63))
    got, fronts, q, zdev, C, err, _, _ = gpu_sampled_expansion(logits, B, k, W, D, seed, inv_T)
    assert err == 0
    sizes, _ = sizes_of(k, W, D)
    for b in range(B):
        c = oracle.new_cands(C)
        fid, fsc = np.array([-1], np.int32), np.zeros(1, np.float32)
        for di, (F, off) in enumerate(sizes):
            nid, nsc, rm, rq = oracle.expand_sampled(logits[di][b], k, W, fsc, fid, di + 1, off, c, seed, b, inv_T)
            assert np.array_equal(fronts[di][0][b], nid), ("frontier", b, di)
            assert np.array_equal(fronts[di][1][b].view(np.uint32), nsc.view(np.uint32))
            for f in range(F):  # the draft statistics of the node row f expanded
                e = q[b, int(fid[f]) + 1]
                assert int(e["row"]) == zdev[di].data_ptr() + ((b * F + f) * V) * 4, (b, di, f)
                assert int(e["Q"]) == int(rq[f]) and e["m"].view(np.uint32) == rm[f].view(np.uint32)
                assert e["it"] == np.float32(inv_T)
            fid, fsc = nid, nsc
        for key in ("tok", "parent", "depth"):
            assert np.array_equal(got[key][b], c[key]), (key, b)
        assert np.array_equal(got["score"][b].view(np.uint32), c["score"].view(np.uint32)), ("score", b)
        for i in range(C):  # siblings are distinct tokens
            sib = got["tok"][b][(i // k) * k:(i // k + 1) * k]
            assert len(set(sib.tolist())) == k


def test_expand_sampled_draws_depend_on_seed_and_request():
    V, k, B = 4096, 6, 2
    rng = np.random.default_rng(1)
    z = np.repeat((rng.standard_normal((1, 1, V)) * 0.5).astype(np.float32), B, axis=0)
    a = gpu_sampled_expansion([z], B, k, k, 1, 11)[0]["tok"]
    b = gpu_sampled_expansion([z], B, k, k, 1, 12)[0]["tok"]
    assert not np.array_equal(a[0], a[1])  # same row, another request: other draws
    assert not np.array_equal(a[0], b[0])  # another seed: other draws


def target_stats(z, temps_rows):
    """GPU LM head on one-hot rows (exact fp32 copies of z) and its statistics."""
    M, V = z.shape
    h = np.eye(M, dtype=np.float32)
    rmax = torch.empty(M, device="cuda")
    rQ = torch.empty(M, dtype=torch.int64, device="cuda")
    ram = i32(M)
    err = i32(1)
    logits = torch.empty((M, V), device="cuda")
    e3.lmhead_logits(to_dev(h), to_dev(np.ascontiguousarray(z.T)), M, M, V, to_dev(np.asarray(temps_rows, np.float32)),
                     logits, rmax, rQ, ram, err, e3.E3_F32)
    return logits, rmax, rQ, ram, err


def qrow_table(logits, fronts, sizes, k, b):
    """Candidate index -> draft logit row (numpy) it was expanded with, from the
    frontiers (independent of the GPU's statistics); the root is key -1."""
    table = {}
    fid = np.array([-1], np.int32)
    for di, (F, _) in enumerate(sizes):
        for f in range(F):
            table[int(fid[f])] = logits[di][b][f]
        fid = fronts[di][0][b]
    return table


@pytest.mark.parametrize("B,V,k,W,D,noise", [(8, 1000, 3, 3, 3, 1.0), (4, 128256, 4, 4, 4, 1.0),
                                             (16, 4096, 1, 1, 3, 1.5), (2, 64, 8, 8, 2, 3.0),
                                             (6, 300, 2, 4, 5, 0.5), (3, 2000, 6, 6, 3, 4.0)])
def test_accept_sampled_bitexact(B, V, k, W, D, noise):
    rng = np.random.default_rng(B * 7 + V + k)
    logits = draft_logits(rng, B, k, W, D, V)
    seed = int(rng.integers(0, 2 ** 63))
    inv_Tq = 1.0
    cands, fronts, q, zdev, C, err, cand, keep = gpu_sampled_expansion(logits, B, k, W, D, seed, inv_Tq)
    assert err == 0
    N, R = C, C + 1
    kvl = np.zeros(B, np.int32)
    root = rng.integers(0, V, B).astype(np.int32)
    out = {x: i32((B, R), -9) for x in ("tok", "parent", "depth", "pos", "nc")}
    mask = torch.zeros((B, R, (R + 63) // 64), dtype=torch.int64, device="cuda")
    e3.tree_build_mask(cand, B, C, N, to_dev(root), to_dev(kvl), out["tok"], out["parent"], out["depth"], out["pos"],
                       mask, node_cand=out["nc"])
    tok, par, nc = host(out["tok"]), host(out["parent"]), host(out["nc"])
    sizes, _ = sizes_of(k, W, D)
    # target rows: near the draft row of the node where it has one (a mix of
    # accepts and rejects), else random
    z = np.zeros((B * R, V), np.float32)
    qlog = np.zeros((B, R, V), np.float32)
    has_kids = np.zeros((B, R), bool)
    for b in range(B):
        tab = qrow_table(logits, fronts, sizes, k, b)
        for u in range(R):
            has_kids[b, u] = (par[b] == u).any()
            key = -1 if u == 0 else int(nc[b, u])
            if has_kids[b, u]:
                qlog[b, u] = tab[key]
                z[b * R + u] = (tab[key] + rng.standard_normal(V) * noise).astype(np.float32)
            else:
                z[b * R + u] = (rng.standard_normal(V) * 2).astype(np.float32)
    temps = np.array([[1.0, 0.7, 0.0, 1.3][b % 4] for b in range(B)], np.float32)
    zl, rmax, rQ, ram, e_stats = target_stats(z, np.repeat(temps, R))
    ua = synth.uniforms(B + V, synth.PURPOSE_ACCEPT, B, R)
    ub = synth.uniforms(B + V, synth.PURPOSE_BONUS, B, R)
    qs = to_dev(q.reshape(-1).view(np.uint8))
    acc, path, outt, st = i32(B), i32((B, D + 1)), i32((B, D + 1)), i32(B)
    e3.spec_accept_sampled(out["tok"], out["parent"], out["nc"], B, R, D, zl, rmax, rQ, ram, V, to_dev(temps), qs,
                           C + 1, to_dev(ua.view(np.int32)), to_dev(ub.view(np.int32)), acc, path, outt, st)
    torch.cuda.synchronize()
    assert int(e_stats.item()) == 0
    zh = host(zl)
    assert np.array_equal(zh, z)
    n_acc = 0
    for b in range(B):
        ref = oracle.build_tree({x: np.ascontiguousarray(cands[x][b]) for x in ("tok", "parent", "score", "depth")},
                                C, N, int(root[b]), 0)
        assert np.array_equal(nc[b], ref["node_cand"]), b
        a, p, o = oracle.accept_sampled({"tok": tok[b], "parent": par[b]}, zh[b * R:(b + 1) * R], temps[b], qlog[b],
                                        inv_Tq, ua[b], ub[b], D)
        assert host(st)[b] == 0, b
        assert host(acc)[b] == a, (b, host(acc)[b], a)
        assert np.array_equal(host(path)[b], p), b
        assert np.array_equal(host(outt)[b], o), b
        n_acc += a
    del zdev, keep


def test_accept_sampled_flags_missing_draft_statistics():
    """A node with children whose statistics entry was never written (row NULL)
    is reported, not faulted."""
    B, V, R, D = 1, 32, 3, 2
    tok = to_dev(np.array([[0, 5, 7]], np.int32))
    par = to_dev(np.array([[-1, 0, 1]], np.int32))
    nc = to_dev(np.array([[-1, 0, 1]], np.int32))
    z = np.zeros((R, V), np.float32)
    zl, rmax, rQ, ram, _ = target_stats(z, np.ones(R, np.float32))
    qs = torch.zeros(3 * e3.QSTAT_BYTES, dtype=torch.uint8, device="cuda")
    acc, path, outt, st = i32(B), i32((B, D + 1)), i32((B, D + 1)), i32(B)
    u = to_dev(np.zeros((B, R), np.int32))
    e3.spec_accept_sampled(tok, par, nc, B, R, D, zl, rmax, rQ, ram, V, to_dev(np.ones(B, np.float32)), qs, 3, u, u,
                           acc, path, outt, st)
    torch.cuda.synchronize()
    assert host(st)[0] == e3.E3_DEV_ERR_NONFINITE and host(acc)[0] == 0
    assert list(host(path)[0]) == [0, -1, -1] and list(host(outt)[0]) == [-1, -1, -1]


def test_sampled_rounds_lossless_on_gpu():
    """200k requests, each with its own tree drawn on the GPU (k = 2, W = 2,
    D = 3, V = 16) and accepted there: the first emitted token follows p_root and
    the second, after an accepted draft x, follows the target row after x."""
    from scipy.stats import chi2
    from test_oracle_sampled import chi_square, qprobs, small_model
    n, V, k, W, D = 200_000, 16, 2, 2, 3
    qtab, ptab = small_model(3, V=V, D=D, Fmax=4)
    sizes, C = sizes_of(k, W, D)
    R = C + 1
    logits = [np.ascontiguousarray(np.broadcast_to(qtab[di][:F], (n, F, V))) for di, (F, _) in enumerate(sizes)]
    cands, fronts, q, zdev, C2, err, cand, keep = gpu_sampled_expansion(logits, n, k, W, D, 2024)
    assert err == 0 and C2 == C
    out = {x: i32((n, R), -9) for x in ("tok", "parent", "depth", "pos", "nc")}
    mask = torch.zeros((n, R, 1), dtype=torch.int64, device="cuda")
    e3.tree_build_mask(cand, n, C, C, to_dev(np.zeros(n, np.int32)), to_dev(np.zeros(n, np.int32)), out["tok"],
                       out["parent"], out["depth"], out["pos"], mask, node_cand=out["nc"])
    tok = host(out["tok"])
    rows = np.where(np.arange(R)[None, :] == 0, 0, tok + 1).reshape(-1)  # target row of every node
    zl = torch.from_numpy(ptab).cuda()[torch.from_numpy(rows).cuda()].contiguous()
    M = n * R
    rmax = torch.empty(M, device="cuda")
    rQ = torch.empty(M, dtype=torch.int64, device="cuda")
    ram = i32(M)
    # statistics of the V + 1 distinct rows from the LM head, gathered per node
    tl, tm, tq, ta, e_st = target_stats(ptab, np.ones(V + 1, np.float32))
    idx = torch.from_numpy(rows).cuda()
    rmax.copy_(tm[idx])
    rQ.copy_(tq[idx])
    ram.copy_(ta[idx])
    ua = synth.uniforms(5, synth.PURPOSE_ACCEPT, n, R)
    ub = synth.uniforms(5, synth.PURPOSE_BONUS, n, R)
    qs = to_dev(q.reshape(-1).view(np.uint8))
    acc, path, outt, st = i32(n), i32((n, D + 1)), i32((n, D + 1)), i32(n)
    e3.spec_accept_sampled(out["tok"], out["parent"], out["nc"], n, R, D, zl, rmax, rQ, ram, V,
                           to_dev(np.ones(n, np.float32)), qs, C + 1, to_dev(ua.view(np.int32)),
                           to_dev(ub.view(np.int32)), acc, path, outt, st)
    torch.cuda.synchronize()
    assert int(e_st.item()) == 0 and not host(st).any()
    acc, outt = host(acc), host(outt)
    stat, dof = chi_square(np.bincount(outt[:, 0], minlength=V).astype(float), qprobs(ptab[0]))
    assert stat < chi2.ppf(1 - 1e-3, dof)
    assert 0.2 < (acc > 0).mean() < 0.95
    x = np.bincount(outt[acc > 0, 0], minlength=V).argmax()
    sel = (acc > 0) & (outt[:, 0] == x)
    stat, dof = chi_square(np.bincount(outt[sel, 1], minlength=V).astype(float), qprobs(ptab[1 + x]))
    assert stat < chi2.ppf(1 - 1e-3, dof)
    # a sample of the requests against the oracle, bit for bit
    zh = ptab[rows].reshape(n, R, V)
    nc, par = host(out["nc"]), host(out["parent"])
    for b in range(0, n, n // 50):
        tab = qrow_table(logits, fronts, sizes, k, b)
        qlog = np.zeros((R, V), np.float32)
        for u in range(R):
            key = -1 if u == 0 else int(nc[b, u])
            if key in tab:
                qlog[u] = tab[key]
        a, p, o = oracle.accept_sampled({"tok": tok[b], "parent": par[b]}, zh[b], 1.0, qlog, 1.0, ua[b], ub[b], D)
        assert acc[b] == a and np.array_equal(outt[b], o), b
    del zdev, keep
