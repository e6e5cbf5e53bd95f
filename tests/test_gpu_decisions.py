"""Decision bit-exactness over 10^4 seeded rounds per benchmarked configuration.

For every configuration's decision shape (vocabulary, top-k, frontier width,
depth, node budget, temperatures, top-k or sampled drafts) this runs 64 seeded
trees (two calls of 32 requests) and 160 seeded uniform sets per tree, i.e.
10240 (tree, uniforms) rounds, through the library's expansion, tree build,
accept/reject and KV compaction, and checks every decision against the oracle:
candidates (tokens, parents, depths, score bits), the flattened tree and mask,
the accepted length, path and emitted tokens, and the compaction indices (the
slots a compaction actually moved).  Losslessness of the acceptance rests on
exactly these decisions ("SpecForge…", 先看 checkpoint 最终要参与什么计算;
"EAGLE 系列与 DFlash", §二 阶段三 and §四).

The logits are GPU-produced: a table of 512 target rows from the library's LM
head (lmhead_logits on seeded hidden states, with its fixed-point softmax
statistics, themselves checked bit for bit against the oracle's), and the draft
rows are target rows plus rows of a seeded noise table (a plain fp32 add, the
same on both sides).  A node's target row is the table row of its token, a
frontier node's draft row the table row of its token plus noise: drafts track
the target, so acceptance walks deep into the trees.  The oracle side runs in a
spawn process pool over the host cores.
"""
import math
import multiprocessing as mp
import os
import sys

import numpy as np
import pytest
import torch

import oracle
from decision_oracle import noise_index, run_request
from eagle_speculative_decoding_round_gb300 import synth

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

pytestmark = pytest.mark.gpu

N_TAB, N_NOISE = 512, 512
B_CALL, N_CALLS, N_UNI = 32, 2, 160  # 64 trees x 160 uniform sets = 10240 rounds per configuration
NAMES = ["tiny", "8b", "8b_d8", "8b_chain3", "8b_sampled", "8b_chain3_sampled", "batched", "long", "70b"]


@pytest.fixture(scope="module")
def pool():
    p = mp.get_context("spawn").Pool(max(2, min(16, os.cpu_count() or 2)))
    yield p
    p.close()
    p.join()


def request_temps(name, c, n):
    if name == "tiny":
        return [0.0 if b % 2 == 0 else 1.0 for b in range(n)]  # greedy and temperature 1
    if c["temps"] == "mixed":
        return [0.0 if b % 2 == 0 else 1.0 for b in range(n)]
    return [float(c["temps"][0])] * n


@pytest.mark.parametrize("name", NAMES)
def test_decisions_bitexact_over_10k_rounds(name, pool, tmp_path):
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3
    from eagle_speculative_decoding_round_gb300.round import RoundBuffers, RoundConfig, build_tree, expand_depth

    c = dict(bench.CONFIGS[name])
    seed = 5000 + NAMES.index(name)
    V, k, W, D, N = c["V"], c["k"], c["W"], c["D"], c["N"]
    R, d, sampled = N + 1, c["H"] * c["hd"], bool(c.get("sampled", False))
    dt = e3.E3_BF16 if c["dtype"] == "bf16" else e3.E3_F32
    td = torch.bfloat16 if c["dtype"] == "bf16" else torch.float32
    temps = request_temps(name, c, B_CALL)
    Tset = sorted(set(temps))
    dev = "cuda"

    # -- GPU-produced target table and its statistics at every temperature used
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    h_tab = torch.randn((N_TAB, d), generator=g, device=dev).to(td)
    W_lm = (torch.randn((V, d), generator=g, device=dev) * (4.0 / math.sqrt(d))).to(td)
    tgt = torch.empty((N_TAB, V), device=dev)
    smax = torch.empty((len(Tset), N_TAB), device=dev)
    sQ = torch.empty((len(Tset), N_TAB), dtype=torch.int64, device=dev)
    sam = torch.empty((len(Tset), N_TAB), dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for ti, T in enumerate(Tset):
        e3.lmhead_logits(h_tab, W_lm, N_TAB, d, V, torch.full((N_TAB,), T, device=dev), tgt, smax[ti], sQ[ti],
                         sam[ti], err, dt)
    del W_lm
    noise_h = synth.normal(seed, "decision_noise", (N_NOISE, V), float(c["noise"]))
    noise = torch.from_numpy(noise_h).to(dev)
    tgt_h = tgt.cpu().numpy()
    tgt_path, noise_path = str(tmp_path / "tgt.npy"), str(tmp_path / "noise.npy")
    np.save(tgt_path, tgt_h)
    np.save(noise_path, noise_h)

    # -- the oracle's jobs go to the pool first (they only need the tables)
    rng = np.random.default_rng(seed)
    roots = [rng.integers(0, V, B_CALL).astype(np.int32) for _ in range(N_CALLS)]
    Ps = np.array([100 + 37 * b for b in range(B_CALL)], np.int32)
    uni_seeds = [[seed * 100003 + ci * N_UNI + u for u in range(N_UNI)] for ci in range(N_CALLS)]
    draw_seeds = [seed * 7 + ci for ci in range(N_CALLS)]
    jobs = [dict(tgt_path=tgt_path, noise_path=noise_path, k=k, W=W, D=D, N=N, sampled=sampled,
                 root=int(roots[ci][b]), P=int(Ps[b]), T=temps[b], b_global=ci * B_CALL + b, b=b,
                 draw_seed=draw_seeds[ci], uni_seeds=uni_seeds[ci])
            for ci in range(N_CALLS) for b in range(B_CALL)]
    pending = pool.map_async(run_request, jobs, chunksize=1)

    # the statistics tables, bit-exact against the oracle's
    for ti, T in enumerate(Tset):
        m, Q, am, bad = oracle.row_stats(tgt_h, np.full(N_TAB, T, np.float32))
        assert not bad.any()
        assert np.array_equal(smax[ti].cpu().numpy().view(np.uint32), m.view(np.uint32)), (name, T)
        assert np.array_equal(sQ[ti].cpu().numpy().view(np.uint64), Q), (name, T)
        assert np.array_equal(sam[ti].cpu().numpy(), am), (name, T)

    # -- the GPU side: two calls of 32 requests
    cfg = RoundConfig(B=B_CALL, N=N, D=D, k=k, W=W, H=c["H"], KVH=c["KVH"], hd=c["hd"], d=d, V=V, L=1,
                      max_kv_len=int(Ps.max()), dtype=c["dtype"], sampled=sampled)
    pt, npages = synth.page_table(seed, [int(p) + R for p in Ps], 64)
    bufs = RoundBuffers(cfg, torch.from_numpy(pt), npages)
    sizes, n_cand = cfg.frontier_sizes()
    tix = torch.tensor([Tset.index(t) for t in temps], device=dev)[:, None]
    # small paged cache whose K rows hold their own logical slot number (compaction check)
    Kh = np.zeros((npages, 1, 64, 32), np.float32)
    for b in range(B_CALL):
        t = np.arange(int(Ps[b]) + R)
        Kh[pt[b, t // 64], 0, t % 64, :] = t[:, None].astype(np.float32)
    Kc = torch.from_numpy(Kh).to(dev)
    K0 = Kc.clone()
    Vc = -Kc
    ptt = torch.from_numpy(pt).to(dev)
    kvl = e3.make_kv_layer(Kc, Vc, ptt, npages, 64, pt.shape[1], 1, 32, e3.E3_F32)
    slot = torch.from_numpy(Ps).long().to(dev)[:, None] + torch.arange(D + 1, device=dev)[None]
    slot_page = torch.gather(ptt.long(), 1, slot // 64)
    P_dev = torch.from_numpy(Ps).to(dev)
    gpu = []
    for ci in range(N_CALLS):
        cfg.draw_seed = draw_seeds[ci]
        bufs.set_temperature(torch.tensor(temps, dtype=torch.float32))
        bufs.root_tok.copy_(torch.from_numpy(roots[ci]))
        bg = torch.arange(ci * B_CALL, (ci + 1) * B_CALL, device=dev)[:, None]
        for di, (F, off) in enumerate(sizes):
            if di == 0:
                ftok = bufs.root_tok.long()[:, None]
            else:
                ftok = torch.gather(bufs.c_tok.long(), 1, bufs.f_id[di][:, :F].long())
            j = (bg * 64 + di * 16 + torch.arange(F, device=dev)[None]) % N_NOISE
            assert int(j[0, 0]) == noise_index(ci * B_CALL, di, 0, N_NOISE)
            bufs.draft_logits[di].copy_(tgt[ftok % N_TAB] + noise[j])
            expand_depth(bufs, di)
        bufs.kv_len.copy_(P_dev)
        build_tree(bufs)
        idx = bufs.tok.long() % N_TAB
        bufs.logits.copy_(tgt[idx].reshape(B_CALL * R, V))
        bufs.row_max.copy_(smax[tix, idx].reshape(-1))
        bufs.row_Q.copy_(sQ[tix, idx].reshape(-1))
        bufs.row_argmax.copy_(sam[tix, idx].reshape(-1))
        ua = torch.from_numpy(np.stack([synth.uniforms(s, synth.PURPOSE_ACCEPT, B_CALL, R) for s in uni_seeds[ci]])
                              .view(np.int32)).to(dev)
        ub = torch.from_numpy(np.stack([synth.uniforms(s, synth.PURPOSE_BONUS, B_CALL, R) for s in uni_seeds[ci]])
                              .view(np.int32)).to(dev)
        acc = torch.empty((N_UNI, B_CALL), dtype=torch.int32, device=dev)
        path = torch.empty((N_UNI, B_CALL, D + 1), dtype=torch.int32, device=dev)
        out = torch.empty((N_UNI, B_CALL, D + 1), dtype=torch.int32, device=dev)
        status = torch.empty(B_CALL, dtype=torch.int32, device=dev)
        moved = torch.empty((N_UNI, B_CALL, D + 1), device=dev)
        kv_after = torch.empty((N_UNI, B_CALL), dtype=torch.int32, device=dev)
        kv_len = torch.empty(B_CALL, dtype=torch.int32, device=dev)
        for u in range(N_UNI):
            if sampled:
                e3.spec_accept_sampled(bufs.tok, bufs.parent, bufs.node_cand, B_CALL, R, D, bufs.logits,
                                       bufs.row_max, bufs.row_Q, bufs.row_argmax, V, bufs.temp, bufs.q_stats,
                                       n_cand + 1, ua[u], ub[u], acc[u], path[u], out[u], status)
            else:
                e3.spec_accept(bufs.tok, bufs.parent, B_CALL, R, D, bufs.logits, bufs.row_max, bufs.row_Q,
                               bufs.row_argmax, V, bufs.temp, ua[u], ub[u], e3.E3_ACCEPT_TREE_DET, acc[u], path[u],
                               out[u], status)
            Kc.copy_(K0)
            kv_len.copy_(P_dev)
            e3.kv_compact([kvl], B_CALL, path[u], acc[u], D, kv_len, err)
            moved[u] = Kc[slot_page, 0, slot % 64, 0]
            kv_after[u] = kv_len
        torch.cuda.synchronize()
        assert int(err.item()) == 0 and int(bufs.dev_err.item()) == 0
        gpu.append(dict(c_tok=bufs.c_tok.cpu().numpy(), c_parent=bufs.c_parent.cpu().numpy(),
                        c_depth=bufs.c_depth.cpu().numpy(), c_score=bufs.c_score.cpu().numpy(),
                        tok=bufs.tok.cpu().numpy(), parent=bufs.parent.cpu().numpy(),
                        depth=bufs.depth.cpu().numpy(), pos=bufs.pos.cpu().numpy(), mask=bufs.mask.cpu().numpy(),
                        node_cand=bufs.node_cand.cpu().numpy(), acc=acc.cpu().numpy(), path=path.cpu().numpy(),
                        out=out.cpu().numpy(), moved=moved.cpu().numpy(), kv_after=kv_after.cpu().numpy()))

    # -- compare every decision
    results = pending.get(timeout=1800)
    deep = 0
    for n_job, res in enumerate(results):
        ci, b = divmod(n_job, B_CALL)
        gp = gpu[ci]
        cd, tr = res["cands"], res["tree"]
        assert np.array_equal(gp["c_tok"][b], cd["tok"]), (name, ci, b, "candidate tokens")
        assert np.array_equal(gp["c_parent"][b], cd["parent"]), (name, ci, b, "candidate parents")
        assert np.array_equal(gp["c_depth"][b], cd["depth"]), (name, ci, b, "candidate depths")
        assert np.array_equal(gp["c_score"][b].view(np.uint32), cd["score"].view(np.uint32)), (name, ci, b, "scores")
        for key in ("tok", "parent", "depth", "pos"):
            assert np.array_equal(gp[key][b], tr[key]), (name, ci, b, key)
        assert np.array_equal(gp["mask"][b].view(np.uint64), tr["mask"]), (name, ci, b, "mask")
        if sampled:
            assert np.array_equal(gp["node_cand"][b], tr["node_cand"]), (name, ci, b, "node_cand")
        assert np.array_equal(gp["acc"][:, b], res["acc"]), (name, ci, b, "acc_len")
        assert np.array_equal(gp["path"][:, b], res["path"]), (name, ci, b, "path")
        assert np.array_equal(gp["out"][:, b], res["out"]), (name, ci, b, "out_tok")
        # compaction: slot P + j holds (the slot number of) P + path[j] for j <= a
        for u in range(N_UNI):
            a = int(res["acc"][u])
            assert np.array_equal(gp["moved"][u, b, :a + 1], Ps[b] + res["path"][u, :a + 1].astype(np.float32)), \
                (name, ci, b, u, "compaction")
            assert gp["kv_after"][u, b] == Ps[b] + 1 + a
        deep = max(deep, int(res["acc"].max()))
    n_rounds = len(results) * N_UNI
    assert n_rounds >= 10000
    # the sweep is not trivial: some rounds accept drafted nodes, and except for the
    # deliberately low-acceptance long-context setting some walk two levels or more
    assert deep >= (1 if name == "long" else 2), (name, deep)

