"""Benchmark of one EAGLE-3 draft-and-verify round on synthetic data.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config 8b|tiny|batched|long|70b] [--impl ours|reference]

A step is one whole round: fuse -> expand x D -> tree_build_mask -> tree_verify_attn
x L -> lmhead_logits -> spec_accept -> kv_compact (all L layers), over one batch of
synthetic input that is resident in HBM.  The K timed steps are one CUDA graph of K
rounds (each round first resets kv_len, so every step does the same work).  Inputs
exceed L2: the per-layer KV (276 MB at 8B) and the 1.05 GB LM head stream from HBM
in every step.  --impl reference times the CPU oracle on a bounded sample instead.
Multi-GPU: replicas only (independent requests per GPU, no collective on the path).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

CONFIGS = {
    "tiny": dict(B=1, P=[128], N=14, D=3, k=2, W=1 << 20, H=4, KVH=4, hd=64, d=256, V=1024, L=1, dtype="f32",
                 temps=[1.0], noise=1.0,
                 workload="tiny fp32 single-layer target: d=256, 4x64 heads, vocab 1024, batch 1, prefix 128, "
                          "depth 3, top-k 2 (14 nodes)"),
    "8b": dict(B=1, P=[2048], N=60, D=6, k=10, W=10, H=32, KVH=8, hd=128, d=4096, V=128256, L=32, dtype="bf16",
               temps=[1.0], noise=1.0,
               workload="Llama-3.1-8B-shaped verify round, bf16: d=4096, 32/8 heads x 128, vocab 128256, batch 1, "
                        "prefix 2048, 60-node depth-6 tree, top-k 10, 32 layers, fusion 12288->4096, temp 1"),
    "8b_d8": dict(B=1, P=[2048], N=60, D=8, k=10, W=10, H=32, KVH=8, hd=128, d=4096, V=128256, L=32, dtype="bf16",
                  temps=[1.0], noise=1.0,
                  workload="Llama-3.1-8B-shaped verify round with an EAGLE-3 depth-8 tree at the same node count: "
                           "d=4096, 32/8 heads x 128, vocab 128256, batch 1, prefix 2048, 60-node depth-8 tree, "
                           "top-k 10, 32 layers, fusion 12288->4096, temp 1"),
    "8b_chain3": dict(B=1, P=[2048], N=3, D=3, k=1, W=1, H=32, KVH=8, hd=128, d=4096, V=128256, L=32, dtype="bf16",
                      temps=[1.0], noise=1.0,
                      workload="Llama-3.1-8B-shaped verify round with a chain draft (top-1, three tokens): d=4096, "
                               "32/8 heads x 128, vocab 128256, batch 1, prefix 2048, 32 layers, "
                               "fusion 12288->4096, temp 1"),
    "8b_sampled": dict(B=1, P=[2048], N=52, D=4, k=4, W=4, H=32, KVH=8, hd=128, d=4096, V=128256, L=32,
                       dtype="bf16", temps=[1.0], noise=1.0, sampled=True,
                       workload="Llama-3.1-8B-shaped verify round with drafts sampled from the draft distribution "
                                "and accepted with min(1, p/q): d=4096, 32/8 heads x 128, vocab 128256, batch 1, "
                                "prefix 2048, 4 draws per node, frontier 4, depth 4 (52 nodes), 32 layers, "
                                "fusion 12288->4096, temp 1"),
    "8b_chain3_sampled": dict(B=1, P=[2048], N=3, D=3, k=1, W=1, H=32, KVH=8, hd=128, d=4096, V=128256, L=32,
                              dtype="bf16", temps=[1.0], noise=1.0, sampled=True,
                              workload="Llama-3.1-8B-shaped verify round with a sampled chain draft (three tokens "
                                       "drawn from the draft distribution, accepted with min(1, p/q)): d=4096, "
                                       "32/8 heads x 128, vocab 128256, batch 1, prefix 2048, 32 layers, "
                                       "fusion 12288->4096, temp 1"),
    "batched": dict(B=32, P="uniform:512:8192", N=60, D=6, k=10, W=10, H=32, KVH=8, hd=128, d=4096, V=128256,
                    L=32, dtype="bf16", temps="mixed", noise=1.0,
                    workload="batched serving, 8B shape, bf16: 32 requests, prefix U[512,8192], 60-node depth-6 "
                             "trees, mixed greedy/temp-1, ragged 64-token pages"),
    "long": dict(B=1, P=[65536], N=32, D=7, k=4, W=4, H=32, KVH=8, hd=128, d=4096, V=128256, L=32, dtype="bf16",
                 temps=[0.7], noise=2.0,
                 workload="long-context agent shape, 8B dims, bf16: batch 1, prefix 65536, 32-node depth-7 tree, "
                          "top-k 4, draft noise N(0,2), temp 0.7"),
    "70b": dict(B=8, P=[4096] * 8, N=60, D=6, k=10, W=10, H=64, KVH=8, hd=128, d=8192, V=128256, L=80,
                dtype="bf16", temps=[1.0], noise=1.0,
                workload="Llama-3-70B-shaped verify round, bf16: d=8192, 64/8 heads x 128, vocab 128256, batch 8, "
                         "prefix 4096, fusion 24576->8192, 60-node depth-6 tree, temp 1, 80 layers"),
}
METRIC = "tree-verify rounds/s & nodes/s (8B-shape, 60-node tree); % HBM/tensor roofline"
# dram__bytes_read.sum + dram__bytes_write.sum per launch, from one ncu capture of the
# kernel on this workload (None until the current kernel has been captured)
TRAFFIC = {
    "8b": {"verify": 9231616, "lmhead": 1082488832},
    "long": {"verify": 272763392, "lmhead": None},
}
TAB_ROWS = 4096  # token-keyed Q/K/V tables of the synthetic target (token id modulo this)


def cfg_values(name, seed, layers=None):
    c = dict(CONFIGS[name])
    if layers:
        c["L"] = int(layers)
    rng = np.random.default_rng(seed)
    if isinstance(c["P"], str):
        lo, hi = (int(x) for x in c["P"].split(":")[1:])
        c["P"] = [int(x) for x in rng.integers(lo, hi + 1, c["B"])]
    if c["temps"] == "mixed":
        c["temps"] = [0.0 if b % 2 == 0 else 1.0 for b in range(c["B"])]
    return c


# ---------------------------------------------------------------------------
# synthetic workload on the GPU
# ---------------------------------------------------------------------------

class Workload:
    def __init__(self, name, seed=0, device="cuda", layers=None):
        import torch

        from eagle_speculative_decoding_round_gb300 import eagle3 as e3
        from eagle_speculative_decoding_round_gb300 import synth
        from eagle_speculative_decoding_round_gb300.round import RoundBuffers, RoundConfig

        self.torch, self.e3, self.synth = torch, e3, synth
        c = cfg_values(name, seed, layers)
        self.name, self.c, self.seed = name, c, seed
        R = c["N"] + 1
        self.cfg = RoundConfig(B=c["B"], N=c["N"], D=c["D"], k=c["k"], W=c["W"], H=c["H"], KVH=c["KVH"],
                               hd=c["hd"], d=c["d"], V=c["V"], L=c["L"], max_kv_len=max(c["P"]), dtype=c["dtype"],
                               sampled=bool(c.get("sampled", False)), draw_seed=seed * 7919 + 17)
        pt, npages = synth.page_table(seed, [p + R for p in c["P"]], self.cfg.page_size)
        self.pt = pt
        self.bufs = b = RoundBuffers(self.cfg, torch.from_numpy(pt), npages, device)
        g = torch.Generator(device=device)
        g.manual_seed(seed)
        self.gen = g
        td = self.cfg.tdtype

        def randn(shape, std):
            return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(td)

        for l in range(c["L"]):
            b.K[l].copy_(randn(b.K[l].shape, 1.0))
            b.Vc[l].copy_(randn(b.Vc[l].shape, 1.0))
        for t in b.h:
            t.copy_(randn(t.shape, 0.02))
        b.W_f.copy_(randn(b.W_f.shape, 0.02))
        b.W_lm.copy_(randn(b.W_lm.shape, 1.0 / math.sqrt(self.cfg.H * self.cfg.hd)))
        self.Qtab = randn((TAB_ROWS, c["H"], c["hd"]), 1.0)
        self.Ktab = randn((TAB_ROWS, c["KVH"], c["hd"]), 1.0)
        self.Vtab = randn((TAB_ROWS, c["KVH"], c["hd"]), 1.0)
        self.kv_len0 = torch.tensor(c["P"], dtype=torch.int32, device=device)
        b.kv_len.copy_(self.kv_len0)
        rt = np.random.default_rng(seed + 1).integers(0, c["V"], c["B"]).astype(np.int32)
        b.root_tok.copy_(torch.from_numpy(rt))
        b.set_temperature(torch.tensor(c["temps"], dtype=torch.float32))
        b.u_acc.copy_(torch.from_numpy(synth.uniforms(seed, synth.PURPOSE_ACCEPT, c["B"], R).view(np.int32)))
        b.u_bonus.copy_(torch.from_numpy(synth.uniforms(seed, synth.PURPOSE_BONUS, c["B"], R).view(np.int32)))
        self.calibrate_and_draft()

    # -- token-keyed tree Q/K/V of the synthetic target -----------------------
    def write_nodes(self, toks, layers, R):
        """toks [B, R] int64 (device): write Q (given layers) and K/V at slots P..P+R-1."""
        torch, b, c = self.torch, self.bufs, self.cfg
        key = toks % TAB_ROWS
        q = self.Qtab[key]                      # [B, R, H, hd]
        kk, vv = self.Ktab[key], self.Vtab[key]  # [B, R, KVH, hd]
        P = self.kv_len0.long()[:, None] + torch.arange(R, device=toks.device)[None]
        page = torch.gather(b.page_table.long(), 1, P // c.page_size)
        slot = P % c.page_size
        for l in layers:
            if l < len(b.Q) and b.Q[l].shape[1] == R:
                b.Q[l].copy_(q)
            b.K[l][page, :, slot, :] = kk
            b.Vc[l][page, :, slot, :] = vv
        return q

    def target_logits_of(self, node_tok, node_par, rows):
        """Target logits of selected nodes of per-request mini-trees, by the library's
        own verify (last layer) + LM head.  node_tok/node_par: numpy [B, R'];
        rows: list of (b, i) in output order."""
        torch, e3, b, c = self.torch, self.e3, self.bufs, self.cfg
        B, Rm = node_tok.shape
        q = self.write_nodes(torch.from_numpy(node_tok).long().cuda(), [c.L - 1], Rm)
        mask = np.zeros((B, Rm, (Rm + 63) // 64), np.uint64)
        for bb in range(B):
            for i in range(Rm):
                j = i
                while j >= 0:
                    mask[bb, i, j >> 6] |= np.uint64(1 << (j & 63))
                    j = int(node_par[bb, j])
        maskt = torch.from_numpy(mask.view(np.int64)).cuda()
        O = torch.empty((B, Rm, c.H, c.hd), dtype=c.tdtype, device="cuda")
        lse = torch.empty((B, Rm, c.H), device="cuda")
        wsb = e3.eagle3_verify_workspace_bytes(B, Rm, c.H, c.KVH, c.hd, c.max_kv_len, c.dt)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        e3.tree_verify_attn(q.contiguous(), b.kv[c.L - 1], b.kv_len, maskt, B, Rm, c.H, c.max_kv_len,
                            1.0 / math.sqrt(c.hd), O, lse, b.dev_err, ws, wsb)
        sel = torch.tensor([bb * Rm + i for bb, i in rows], device="cuda")
        h = O.view(B * Rm, c.H * c.hd)[sel].contiguous()
        M = h.shape[0]
        z = torch.empty((M, c.V), device="cuda")
        e3.lmhead_logits(h, b.W_lm, M, c.H * c.hd, c.V, torch.ones(M, device="cuda"), z,
                         torch.empty(M, device="cuda"), torch.empty(M, dtype=torch.int64, device="cuda"),
                         torch.empty(M, dtype=torch.int32, device="cuda"), b.dev_err, c.dt)
        return z

    def calibrate_and_draft(self):
        """Draft stand-in: at each depth the frontier nodes' target logits (verify +
        LM head on the frontier's own mini-tree) plus N(0, noise^2) are the draft
        logits.  W_lm is first scaled so that target logits have std ~ 4."""
        from eagle_speculative_decoding_round_gb300.round import build_tree, expand_depth
        torch, e3, b, c = self.torch, self.e3, self.bufs, self.cfg
        B = c.B
        roots = b.root_tok.cpu().numpy()
        z = self.target_logits_of(roots[:, None].astype(np.int64), np.full((B, 1), -1), [(bb, 0) for bb in range(B)])
        scale = 4.0 / float(z.float().std())
        b.W_lm.copy_((b.W_lm.float() * scale).to(c.tdtype))
        sizes, n_cand = c.frontier_sizes()
        paths = [{-1: [int(roots[bb])]} for bb in range(B)]
        for di, (F, off) in enumerate(sizes):
            fid = b.f_id[di].cpu().numpy()[:, :F]
            # per request: mini-tree = root + frontier nodes' ancestors + frontier nodes
            node_lists = []
            for bb in range(B):
                nodes = {(): -1}
                order = [()]
                for f in fid[bb]:
                    p = paths[bb][int(f)][1:]
                    for depth in range(1, len(p) + 1):
                        key = tuple(p[:depth])
                        if key not in nodes:
                            nodes[key] = len(order)
                            order.append(key)
                order.sort(key=lambda t: (len(t), t))
                node_lists.append(order)
            Rm = max(len(o) for o in node_lists)
            tok = np.zeros((B, Rm), np.int64)
            par = np.full((B, Rm), -1, np.int64)
            rows = []
            for bb, order in enumerate(node_lists):
                index = {key: i for i, key in enumerate(order)}
                for i, key in enumerate(order):
                    tok[bb, i] = key[-1] if key else roots[bb]
                    par[bb, i] = index[key[:-1]] if key else -1
                for i in range(len(order), Rm):  # padding nodes hang off the root
                    par[bb, i] = 0
                for f in fid[bb]:
                    rows.append((bb, index[tuple(paths[bb][int(f)][1:])]))
            zt = self.target_logits_of(tok, par, rows).view(B, F, c.V)
            noise = torch.randn(zt.shape, generator=self.gen, device="cuda") * self.c["noise"]
            b.draft_logits[di].copy_(zt + noise)
            expand_depth(b, di)
            ct, cp = b.c_tok.cpu().numpy(), b.c_parent.cpu().numpy()
            for bb in range(B):
                for i in range(off, off + F * c.k):
                    paths[bb][i] = paths[bb][int(cp[bb, i])] + [int(ct[bb, i])]
        # the final tree (same every step) and its Q/K/V in every layer
        build_tree(b)
        self.write_nodes(b.tok.long(), range(c.L), c.R)
        torch.cuda.synchronize()
        assert int(b.dev_err.item()) == 0, "device error during setup"

    def round(self, stream=None):
        from eagle_speculative_decoding_round_gb300.round import run_round
        self.bufs.kv_len.copy_(self.kv_len0)
        run_round(self.bufs, stream=stream)


# ---------------------------------------------------------------------------
# algorithmic work per round (the units of the roofline)
# ---------------------------------------------------------------------------

def work_model(w):
    c, cfg = w.c, w.cfg
    esz = 2 if cfg.dtype == "bf16" else 4
    B, R, H, KVH, hd, d, V, L = cfg.B, cfg.R, cfg.H, cfg.KVH, cfg.hd, cfg.d, cfg.V, cfg.L
    P = c["P"]
    par = w.bufs.parent.cpu().numpy()
    anc = 0
    for bb in range(B):
        for i in range(R):
            j = i
            while j >= 0:
                anc += 1
                j = int(par[bb, j])
    verify_bytes = sum(2 * KVH * hd * esz * (p + R) for p in P) + 2 * B * R * H * hd * esz + B * R * H * 4
    verify_flops = 4 * H * hd * (sum(R * p for p in P) + anc)
    M = B * R
    lm_bytes = V * d * esz + M * d * esz + M * V * 4
    lm_flops = 2 * M * d * V
    fuse_bytes = 3 * d * d * esz + 4 * cfg.M * d * esz
    return dict(verify_bytes=verify_bytes, verify_flops=verify_flops, lm_bytes=lm_bytes, lm_flops=lm_flops,
                fuse_bytes=fuse_bytes, fuse_flops=2 * cfg.M * 3 * d * d)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        out_dir = os.environ.get("E3_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample)
# ---------------------------------------------------------------------------

def oracle_sample(w, budget_s=20.0):
    """Time the oracle on a bounded sample of one round of the same workload and
    scale to a whole round.  Sample: fusion, all expansion depths, tree build and
    accept in full; verify attention of request 0 on as many layers as fit about
    60% of budget_s (at least one; scaled by L over the layers done and by the
    requests' keys); LM head on a 1/4 slice of the vocabulary (scaled by 4)."""
    import torch

    import oracle
    try:
        from threadpoolctl import threadpool_info
        blas_threads = max([x.get("num_threads", 1) for x in threadpool_info()] or [1])
    except Exception:
        blas_threads = os.cpu_count()
    b, cfg = w.bufs, w.cfg
    f = lambda t: t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()  # noqa: E731
    B, R, V = cfg.B, cfg.R, cfg.V
    times = {}
    t0 = time.perf_counter()
    hs = [f(t) for t in b.h]
    Wf = f(b.W_f)
    t = time.perf_counter()
    oracle.fuse(*hs, Wf)
    times["fuse"] = time.perf_counter() - t
    sizes, n_cand = cfg.frontier_sizes()
    drafts = [f(x) for x in b.draft_logits]
    t = time.perf_counter()
    trees, qrows = [], []
    for bb in range(B if B <= 2 else 1):
        c = oracle.new_cands(n_cand)
        fid, fsc = np.array([-1], np.int32), np.zeros(1, np.float32)
        rows = {}  # candidate (root -1) -> the draft row it was expanded with
        for di, (F, off) in enumerate(sizes):
            if cfg.sampled:
                for fr in range(F):
                    rows[int(fid[fr])] = drafts[di][bb][fr]
                fid, fsc, _, _ = oracle.expand_sampled(drafts[di][bb], cfg.k, cfg.W, fsc, fid, di + 1, off, c,
                                                       cfg.draw_seed, bb)
            else:
                fid, fsc = oracle.expand(drafts[di][bb], cfg.k, cfg.W, fsc, fid, di + 1, off, c)
        trees.append(oracle.build_tree(c, n_cand, cfg.N, int(b.root_tok[bb]), int(w.kv_len0[bb])))
        qrows.append(rows)
    times["expand_build"] = (time.perf_counter() - t) * (B / len(trees))
    p0 = int(w.c["P"][0])
    scale_b = sum(p + R for p in w.c["P"]) / (p0 + R)
    spent, n_layers = 0.0, 0
    for l in range(cfg.L - 1, -1, -1):
        K, Vc = f(b.K[l]), f(b.Vc[l])
        Q = f(b.Q[l])[:1]
        t = time.perf_counter()
        oracle.tree_verify_attn(Q, K, Vc, w.pt[:1], w.kv_len0.cpu().numpy()[:1], trees[0]["parent"][None],
                                1.0 / math.sqrt(cfg.hd))
        spent += time.perf_counter() - t
        n_layers += 1
        if spent >= 0.6 * budget_s:
            break
    times["verify"] = spent / n_layers * cfg.L * scale_b
    Wl = f(b.W_lm)
    h = f(b.O[cfg.L - 1]).reshape(B * R, -1)
    sl = slice(0, V // 4)
    t = time.perf_counter()
    z = oracle.lmhead_logits(h, Wl[sl])
    oracle.row_stats(z.astype(np.float32), 1.0)
    times["lmhead"] = (time.perf_counter() - t) * 4
    zl = f(b.logits)
    t = time.perf_counter()
    tt = {"tok": b.tok.cpu().numpy()[0], "parent": b.parent.cpu().numpy()[0]}
    ua, ub = b.u_acc.cpu().numpy()[0].view(np.uint32), b.u_bonus.cpu().numpy()[0].view(np.uint32)
    if cfg.sampled:
        qlog = np.zeros((R, V), np.float32)
        for u in range(R):
            key = -1 if u == 0 else int(trees[0]["node_cand"][u])
            if key in qrows[0]:
                qlog[u] = qrows[0][key]
        oracle.accept_sampled(tt, zl[:R], float(w.c["temps"][0]), qlog, 1.0, ua, ub, cfg.D)
    else:
        oracle.accept(tt, zl[:R], float(w.c["temps"][0]), ua, ub, cfg.D)
    times["accept"] = (time.perf_counter() - t) * B
    total = sum(times.values())
    wall = time.perf_counter() - t0
    return {"round_s": total, "times": times, "cores": blas_threads, "wall_s": wall, "verify_layers": n_layers}


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="8b", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling only: fewer target layers than the configuration (small ncu captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        return reference_arm(args, rank, world)
    torch.cuda.set_device(local)
    w = Workload(args.config, seed=args.seed + 1000 * rank, layers=args.layers)
    cfg = w.cfg
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for _ in range(args.warmup):
            w.bufs.kv_len.copy_(w.kv_len0)  # every round starts from the same request lengths
            w.round()
    s.synchronize()
    accepted = w.bufs.acc_len.cpu().numpy().copy()

    # The timed region: one graph of K rounds (nothing but the rounds: each round first
    # resets kv_len).  A second graph of the same rounds with events at the phase
    # boundaries gives the phase split; it is replayed separately, because an event
    # between two kernels also cuts the programmatic launch edge between them.
    K = args.steps
    phases = ["fuse", "expand", "tree", "verify", "lmhead", "accept", "compact"]
    ev = [[graph_event() for _ in range(len(phases) + 1)] for _ in range(K)]
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3
    graph = torch.cuda.CUDAGraph()
    counts = []  # library launch counter at each phase boundary of the first captured round
    n0 = e3.launch_count()
    with torch.cuda.graph(graph, stream=s):
        for k in range(K):
            w.bufs.kv_len.copy_(w.kv_len0)
            run_round_phased(w, None, e3, counts if k == 0 else None)
    launches_timed = e3.launch_count() - n0  # libeagle3 kernels in the K captured rounds
    phase_launches = {p: counts[i + 1] - counts[i] for i, p in enumerate(phases)}
    graph_phased = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_phased, stream=s):
        for k in range(K):
            w.bufs.kv_len.copy_(w.kv_len0)
            run_round_phased(w, ev[k], e3)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        graph.replay()  # one untimed replay of the captured work
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(s):
        t0.record(s)
        graph.replay()
        t1.record(s)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    # keep the GPU busy a little longer so the clock sampler sees load
    extra = 0
    while extra < 3 and ms * (extra + 1) < 1500:
        with torch.cuda.stream(s):
            graph.replay()
        extra += 1
    torch.cuda.synchronize()
    clk = clocks.stop()
    with torch.cuda.stream(s):
        graph_phased.replay()  # the phase split (not timed as a whole)
    torch.cuda.synchronize()
    check_dev_err(w, "timed rounds")
    ms = ranks_max(ms, world)
    ms_step = ms / K
    phase_ms = {p: statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K))
                for i, p in enumerate(phases)}
    rounds_s = job_rounds_per_s(ms_step, world)
    nodes_s = rounds_s * cfg.B * cfg.N

    wm = work_model(w)
    peaks = load_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    tflops = peaks.get("bf16_tflops_sustained", 1700.0)
    src = "of measured" if "hbm_gbs" in peaks else "of fallback"
    traffic = TRAFFIC.get(args.config, {})
    # dominant kernel: verify_tc_kernel, one launch per layer on the single-wave workloads
    # (a second, merge launch per layer where the split spans several waves)
    ver_launches = phase_launches["verify"]
    ver_ms = phase_ms["verify"] / cfg.L  # per layer: its verify_tc launch (+ merge launch, if any)
    ver_gbs = wm["verify_bytes"] / (ver_ms * 1e-3) / 1e9
    roofline = {"kernel": "verify_tc_kernel (tree_verify_attn, one layer)", "bound": "hbm",
                "achieved": round(ver_gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(ver_gbs / hbm, 4),
                "traffic": traffic.get("verify"), "algorithmic_bytes": int(wm["verify_bytes"]),
                "launches_per_layer": ver_launches / cfg.L, "us_per_layer": round(ver_ms * 1e3, 2),
                "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({src})"}
    lm_ms = phase_ms["lmhead"]
    lm_gbs = wm["lm_bytes"] / (lm_ms * 1e-3) / 1e9
    lm_tf = wm["lm_flops"] / (lm_ms * 1e-3) / 1e12
    lm_bound = "hbm" if wm["lm_flops"] / wm["lm_bytes"] < tflops * 1e12 / (hbm * 1e9) else "tensor"
    lm = {"kernel": "lmhead_kernel + row_q_kernel (lmhead_logits)", "bound": lm_bound,
          "traffic": traffic.get("lmhead"), "algorithmic_bytes": int(wm["lm_bytes"]),
          "algorithmic_flops": int(wm["lm_flops"]), "us": round(lm_ms * 1e3, 2)}
    if lm_bound == "hbm":
        lm.update(achieved=round(lm_gbs, 1), peak=hbm, unit="GB/s", frac=round(lm_gbs / hbm, 4),
                  peak_source=f"MEASURED_PEAKS.json hbm_gbs ({src})")
    else:
        lm.update(achieved=round(lm_tf, 1), peak=tflops, unit="TFLOP/s", frac=round(lm_tf / tflops, 4),
                  peak_source="MEASURED_PEAKS.json bf16_tflops_sustained (of measured)")
    lm["tensor_frac"] = round(lm_tf / tflops, 4)
    e2e = None if args.no_e2e else e2e_leg(w, s, K, args.warmup, world)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        o = oracle_sample(w)
        cpu = {"value": round(1.0 / o["round_s"], 6), "unit": "rounds/s", "cores": o["cores"], "kind": "oracle",
               "sample": "one round of the same workload: fusion, expansion, tree build, accept in full; verify "
                         f"of request 0 on {o['verify_layers']} of the L layers, scaled by L and by the batch's keys; "
                         f"LM head on 1/4 of the vocabulary scaled by 4 (wall {o['wall_s']:.1f} s)",
               "seconds_per_round": round(o["round_s"], 3),
               "breakdown_s": {k: round(v, 3) for k, v in o["times"].items()}}
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(rounds_s, 3), "unit": "rounds/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (seeded; random-init weights)",
            "config": {"workload": w.c["workload"], "global_batch": cfg.B * world, "prefix_lens": summarize(w.c["P"]),
                       "nodes": cfg.N, "depth": cfg.D, "topk": cfg.k, "layers": cfg.L,
                       "l2": "inputs larger than L2 per step (L distinct per-layer KV caches + 1 LM head)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "nodes_per_s": round(nodes_s, 1),
            "accepted_mean": float(np.mean(accepted)),
            "accepted_hist": np.bincount(accepted.astype(np.int64), minlength=cfg.D + 1).tolist(),
            "phase_ms": {k: round(v, 4) for k, v in phase_ms.items()},
            "roofline": roofline,
            "roofline_lmhead": lm,
            "gpu_launches": launches_timed,
            "launches_per_round": phase_launches,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def graph_event():
    """A timing event that becomes an event-record node when captured in a graph."""
    import torch
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:  # older torch without graph event-record nodes
        return torch.cuda.Event(enable_timing=True)


def summarize(P):
    return P if len(P) <= 4 else {"n": len(P), "min": min(P), "max": max(P), "mean": float(np.mean(P))}


def run_round_phased(w, evs, e3, counts=None):
    """One round (the same calls as Workload.round, through run_round) with a timing
    event recorded at each of its 8 phase boundaries (none when ``evs`` is None).
    With ``counts`` (a list), also append the library's launch counter there."""
    import torch

    from eagle_speculative_decoding_round_gb300.round import run_round
    s = torch.cuda.current_stream()

    def mark(i):
        if evs is not None:
            evs[i].record(s)
        if counts is not None:
            counts.append(e3.launch_count())

    run_round(w.bufs, stream=s, mark=mark)


def e2e_leg(w, s, K, warmup, world=1):
    """Same rounds through the C ABI, from pinned HOST buffers: each step copies the
    round's inputs host->device (fusion inputs, draft logits, per-layer Q, uniforms,
    temperatures, root tokens, request lengths), runs the round, and copies the
    result (emitted tokens, path, accepted length) back."""
    import torch
    b = w.bufs
    ins = [*b.h, *b.draft_logits, *b.Q, b.u_acc, b.u_bonus, b.temp, b.temp_rows, b.root_tok, b.kv_len]
    outs = [b.out_tok, b.path, b.acc_len]
    h_in = [t.detach().cpu().pin_memory() for t in ins[:-1]] + [w.kv_len0.detach().cpu().pin_memory()]
    h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs]
    bi = sum(t.numel() * t.element_size() for t in ins)
    bo = sum(t.numel() * t.element_size() for t in outs)
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=s):
        w.round()
    torch.cuda.synchronize()

    def step():
        with torch.cuda.stream(s):
            for d, h in zip(ins, h_in):
                d.copy_(h, non_blocking=True)
            g1.replay()
            for h, d in zip(h_out, outs):
                h.copy_(d, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record(s)
    for _ in range(K):
        step()
    z.record(s)
    torch.cuda.synchronize()
    check_dev_err(w, "e2e")
    ms = ranks_max(a.elapsed_time(z) / K, world)
    return {"value": round(job_rounds_per_s(ms, world), 3), "unit": "rounds/s", "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": round(ms, 4)}


def check_dev_err(w, where):
    """A round that flagged a device error (capacity, non-finite, timeout) took an
    early-exit path: its timing is not a measurement of the round."""
    err = int(w.bufs.dev_err.item())
    if err != 0:
        raise RuntimeError(f"{where}: device error flags {err:#x} set during the timed rounds")


def job_rounds_per_s(ms_per_step, world):
    """Whole-job throughput: each of the `world` replicas completes one round per
    step, and a step lasts as long as the slowest rank's (ms_per_step is that max)."""
    return world * 1000.0 / ms_per_step


def ranks_max(x, world):
    """Largest value of x over the ranks (x itself for one process).  NCCL reduces
    GPU tensors, gloo CPU tensors."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        return json.load(open(p))
    except Exception:
        return {}


def reference_arm(args, rank, world):
    """The oracle, as it stands, timed on the host cores: each step is a bounded
    sample of one round of the same workload (see oracle_sample), scaled to a round."""
    if rank != 0:
        return 0
    import torch
    w = Workload(args.config, seed=args.seed)
    # each step's sample is sized so that the whole run stays near two minutes
    budget = max(2.0, 120.0 / (args.steps + 1))
    for _ in range(max(0, min(args.warmup, 1))):
        oracle_sample(w, budget)
    per = []
    cores = 1
    layers = 1
    for _ in range(args.steps):
        o = oracle_sample(w, budget)
        per.append(o["round_s"])
        cores = o["cores"]
        layers = o["verify_layers"]
    sec = float(np.mean(per))
    v = 1.0 / sec
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "rounds/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1000, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; random-init weights)",
            "config": {"workload": w.c["workload"], "global_batch": w.cfg.B},
            "cpu_baseline": {"value": round(v, 6), "unit": "rounds/s", "cores": cores, "kind": "oracle",
                             "sample": f"per step: one round with verify on {layers} of the L layers (scaled by L) "
                                       "and LM head on 1/4 of the vocabulary (scaled by 4)"},
            "e2e": {"value": round(v, 6), "unit": "rounds/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    main()
