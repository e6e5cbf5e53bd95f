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
    "8b": {"verify": 9240064, "lmhead": 1082488832},
    "long": {"verify": None, "lmhead": None},  # the verify kernel changed since its capture
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

class InputSet:
    """What differs between the rounds of one configuration: the draft logits of
    each depth, the root tokens, the per-layer tree Q, and the tree pages of every
    layer's K/V cache as they are before the round (the round's own tree K/V
    written at slots P .. P+R-1; compaction changes them, so they are restored
    before each round)."""

    def __init__(self, drafts, Q, root_tok):
        self.drafts, self.Q, self.root_tok = drafts, Q, root_tok
        self.pages = self.snapK = self.snapV = None


class Workload:
    """Device buffers and synthetic inputs of one configuration.

    ``n_sets`` distinct input sets (trees, roots, draft logits, tree Q/K/V) and
    ``n_uniform`` uniform sets; round k uses input set k % n_sets and uniform set
    k % n_uniform.  ``drafts="gpu"`` builds the draft logits with the stand-in
    below (the library's own verify + LM head on each frontier's mini-tree, plus
    noise); ``drafts=None`` leaves drafts, trees and tree Q/K/V unset for the
    caller to fill (``add_set`` / ``finish_set``)."""

    def __init__(self, name, seed=0, device="cuda", layers=None, n_sets=1, n_uniform=1, drafts="gpu"):
        import torch

        from eagle_speculative_decoding_round_gb300 import eagle3 as e3
        from eagle_speculative_decoding_round_gb300 import synth
        from eagle_speculative_decoding_round_gb300.round import RoundBuffers, RoundConfig

        self.torch, self.e3, self.synth = torch, e3, synth
        c = cfg_values(name, seed, layers)
        self.name, self.c, self.seed, self.device = name, c, seed, device
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
        b.set_temperature(torch.tensor(c["temps"], dtype=torch.float32))
        # pages holding each request's tree slots [P, P + R): restored before every round
        ps = self.cfg.page_size
        pg = sorted({int(pt[bb, t // ps]) for bb, P in enumerate(c["P"]) for t in (P, P + R - 1)} |
                    {int(pt[bb, q]) for bb, P in enumerate(c["P"]) for q in range(P // ps, (P + R - 1) // ps + 1)})
        self.tree_pages = torch.tensor(pg, dtype=torch.long, device=device)
        self.uni = []
        for u in range(max(1, n_uniform)):
            su = seed if u == 0 else seed * 1000003 + 7919 * u
            self.uni.append((torch.from_numpy(synth.uniforms(su, synth.PURPOSE_ACCEPT, c["B"], R).view(np.int32))
                             .to(device),
                             torch.from_numpy(synth.uniforms(su, synth.PURPOSE_BONUS, c["B"], R).view(np.int32))
                             .to(device)))
        self.sets = []
        if drafts == "gpu":
            for si in range(max(1, n_sets)):
                st = self.add_set(si)
                if si == 0:
                    self.calibrate()
                self.draft_on_gpu()
                from eagle_speculative_decoding_round_gb300.round import build_tree
                build_tree(b)
                self.finish_set(st, b.tok.long())
            self.use(0)
            torch.cuda.synchronize()
            assert int(b.dev_err.item()) == 0, "device error during setup"

    # -- input sets --------------------------------------------------------------
    def root_tokens(self, si):
        rs = self.seed + 1 if si == 0 else self.seed * 104729 + 31 * si + 1
        return np.random.default_rng(rs).integers(0, self.c["V"], self.c["B"]).astype(np.int32)

    def add_set(self, si):
        """Allocate input set si (its draft-logit and Q buffers, root tokens) and make
        it the current one."""
        torch, b, c = self.torch, self.bufs, self.cfg
        drafts = [torch.empty_like(x) for x in b.draft_logits] if self.sets else b.draft_logits
        Q = [torch.empty_like(x) for x in b.Q] if self.sets else b.Q
        st = InputSet(drafts, Q, torch.from_numpy(self.root_tokens(si)).to(self.device))
        self.sets.append(st)
        self._bind(st)
        return st

    def finish_set(self, st, toks):
        """Write the set's tree (toks [B, R]: Q in every layer, K/V at slots P..P+R-1)
        and snapshot the tree pages of every layer."""
        b = self.bufs
        self._bind(st)
        self.write_nodes(toks, range(self.cfg.L), self.cfg.R)
        st.pages = self.tree_pages
        st.snapK = b.K_all.index_select(1, st.pages)
        st.snapV = b.V_all.index_select(1, st.pages)

    def _bind(self, st):
        b = self.bufs
        b.draft_logits, b.Q, b.root_tok = st.drafts, st.Q, st.root_tok

    def use(self, k):
        """Point the round's buffers at the inputs of round k (no copies)."""
        self._bind(self.sets[k % len(self.sets)])
        self.bufs.u_acc, self.bufs.u_bonus = self.uni[k % len(self.uni)]

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

    def calibrate(self):
        """Scale W_lm so that the target logits of the roots have std ~ 4."""
        b, c = self.bufs, self.cfg
        roots = b.root_tok.cpu().numpy()
        z = self.target_logits_of(roots[:, None].astype(np.int64), np.full((c.B, 1), -1),
                                  [(bb, 0) for bb in range(c.B)])
        scale = 4.0 / float(z.float().std())
        b.W_lm.copy_((b.W_lm.float() * scale).to(c.tdtype))

    def draft_on_gpu(self):
        """Draft stand-in: at each depth the frontier nodes' target logits (verify +
        LM head on the frontier's own mini-tree) plus N(0, noise^2) are the draft
        logits of the current input set."""
        from eagle_speculative_decoding_round_gb300.round import expand_depth
        torch, b, c = self.torch, self.bufs, self.cfg
        B = c.B
        roots = b.root_tok.cpu().numpy()
        sizes, n_cand = c.frontier_sizes()
        paths = [{-1: [int(roots[bb])]} for bb in range(B)]
        for di, (F, off) in enumerate(sizes):
            fid = b.f_id[di].cpu().numpy()[:, :F]
            tok, par, rows = mini_trees(paths, fid, roots)
            zt = self.target_logits_of(tok, par, rows).view(B, F, c.V)
            noise = torch.randn(zt.shape, generator=self.gen, device="cuda") * self.c["noise"]
            b.draft_logits[di].copy_(zt + noise)
            expand_depth(b, di)
            ct, cp = b.c_tok.cpu().numpy(), b.c_parent.cpu().numpy()
            for bb in range(B):
                for i in range(off, off + F * c.k):
                    paths[bb][i] = paths[bb][int(cp[bb, i])] + [int(ct[bb, i])]

    def round(self, k=0, stream=None, mark=None):
        """Round k: its inputs bound, request lengths reset, tree pages restored, then
        the seven steps."""
        from eagle_speculative_decoding_round_gb300.round import run_round
        b = self.bufs
        self.use(k)
        st = self.sets[k % len(self.sets)]
        b.kv_len.copy_(self.kv_len0)
        b.K_all.index_copy_(1, st.pages, st.snapK)
        b.V_all.index_copy_(1, st.pages, st.snapV)
        run_round(b, stream=stream, mark=mark)


def mini_trees(paths, fid, roots):
    """Per request, the mini-tree of the frontier rows fid [B, F] (candidate ids, -1
    = root) and their ancestors: tokens [B, R'], parents [B, R'] (flattened by
    depth, then token path; padding nodes hang off the root) and the (b, node)
    row of every frontier entry in order.  paths[b][cand] = token path from the
    root."""
    B = len(paths)
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
        for i in range(len(order), Rm):
            par[bb, i] = 0
        for f in fid[bb]:
            rows.append((bb, index[tuple(paths[bb][int(f)][1:])]))
    return tok, par, rows


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
# CPU oracle baseline: whole rounds of the oracle on the host cores
# ---------------------------------------------------------------------------

class BlasThreads:
    """Sets the thread count of numpy's OpenBLAS (the oracle's fp64 GEMMs) through
    its own exported setter, and reads it back; unknown builds are left alone."""
    NAMES = (("scipy_openblas_set_num_threads64_", "scipy_openblas_get_num_threads64_"),
             ("scipy_openblas_set_num_threads", "scipy_openblas_get_num_threads"),
             ("openblas_set_num_threads64_", "openblas_get_num_threads64_"),
             ("openblas_set_num_threads", "openblas_get_num_threads"))

    def __init__(self):
        import ctypes
        np.dot(np.ones((2, 2)), np.ones((2, 2)))  # the BLAS library is loaded
        self.set = self.get = None
        try:
            paths = {ln.split()[-1] for ln in open("/proc/self/maps") if "blas" in ln.lower() and "/" in ln}
        except OSError:
            paths = set()
        for pth in sorted(paths):
            try:
                lib = ctypes.CDLL(pth)
            except OSError:
                continue
            for sn, gn in self.NAMES:
                if hasattr(lib, sn) and hasattr(lib, gn):
                    self.set, self.get = getattr(lib, sn), getattr(lib, gn)
                    self.set.argtypes = [ctypes.c_int]
                    self.get.restype = ctypes.c_int
                    return

    def threads(self):
        return int(self.get()) if self.get else None

    def use(self, n):
        if self.set:
            self.set(int(n))
        return self.threads()


def whole_round_feasible(w):
    """A whole oracle round fits the CPU sample budget when its fp64 LM head is at
    most ~0.2 TFLOP (8B, long, tiny and the chain/sampled variants; not batched or
    70B)."""
    c = w.cfg
    return c.B * c.R * c.V * c.H * c.hd * 2 <= 2.0e11


def oracle_round(w, k=0):
    """One whole round of the oracle on round k's inputs: fusion, expansion and tree
    build of every request, verify attention of every request on all L layers (the
    oracle's dense masked form), the LM head of the oracle's own last-layer output,
    softmax statistics and accept/reject of every request, and the compaction of
    every layer.  Device data is staged to the host outside the timed parts (one
    layer's cache at a time); returns seconds per phase."""
    import torch

    import oracle
    b, cfg = w.bufs, w.cfg
    B, R, V, L = cfg.B, cfg.R, cfg.V, cfg.L
    f = lambda t: t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()  # noqa: E731
    w.use(k)
    st = w.sets[k % len(w.sets)]
    pages = st.pages.cpu().numpy()
    P = w.kv_len0.cpu().numpy()
    hs = [f(t) for t in b.h]
    Wf = f(b.W_f)
    drafts = [f(x) for x in st.drafts]
    roots = st.root_tok.cpu().numpy()
    temps = b.temp.cpu().numpy()
    ua, ub = b.u_acc.cpu().numpy().view(np.uint32), b.u_bonus.cpu().numpy().view(np.uint32)
    sizes, n_cand = cfg.frontier_sizes()
    times = {}

    def layer_cache(l):
        K, Vc = f(b.K_all[l]), f(b.V_all[l])
        K[pages] = f(st.snapK[l])
        Vc[pages] = f(st.snapV[l])
        return K, Vc

    t = time.perf_counter()
    oracle.fuse(*hs, Wf)
    times["fuse"] = time.perf_counter() - t
    t = time.perf_counter()
    trees, qrows = [], []
    for bb in range(B):
        c = oracle.new_cands(n_cand)
        fid, fsc = np.array([-1], np.int32), np.zeros(1, np.float32)
        rows = {}
        for di, (F, off) in enumerate(sizes):
            if cfg.sampled:
                for fr in range(F):
                    rows[int(fid[fr])] = drafts[di][bb][fr]
                fid, fsc, _, _ = oracle.expand_sampled(drafts[di][bb][:F], cfg.k, cfg.W, fsc, fid, di + 1, off, c,
                                                       cfg.draw_seed, bb)
            else:
                fid, fsc = oracle.expand(drafts[di][bb][:F], cfg.k, cfg.W, fsc, fid, di + 1, off, c)
        trees.append(oracle.build_tree(c, n_cand, cfg.N, int(roots[bb]), int(P[bb])))
        qrows.append(rows)
    times["expand_build"] = time.perf_counter() - t
    mask = np.stack([tr["mask"] for tr in trees])
    sm = 1.0 / math.sqrt(cfg.hd)
    tv = 0.0
    O = None
    for l in range(L):
        K, Vc = layer_cache(l)
        Q = f(st.Q[l])
        t = time.perf_counter()
        O, _ = oracle.tree_verify_attn_dense(Q, K, Vc, w.pt, P, mask, sm)
        tv += time.perf_counter() - t
    times["verify"] = tv
    Wl = f(b.W_lm)
    t = time.perf_counter()
    z = oracle.lmhead_logits(O.reshape(B * R, -1), Wl).astype(np.float32)
    times["lmhead"] = time.perf_counter() - t
    t = time.perf_counter()
    acc, paths = np.zeros(B, np.int32), np.zeros((B, cfg.D + 1), np.int32)
    for bb in range(B):
        zb = z[bb * R:(bb + 1) * R]
        if cfg.sampled:
            qlog = np.zeros((R, V), np.float32)
            for u in range(R):
                key = -1 if u == 0 else int(trees[bb]["node_cand"][u])
                if key in qrows[bb]:
                    qlog[u] = qrows[bb][key]
            a, pth, _ = oracle.accept_sampled(trees[bb], zb, float(temps[bb]), qlog, 1.0, ua[bb], ub[bb], cfg.D)
        else:
            a, pth, _ = oracle.accept(trees[bb], zb, float(temps[bb]), ua[bb], ub[bb], cfg.D)
        acc[bb], paths[bb] = a, pth
    times["accept"] = time.perf_counter() - t
    tc = 0.0
    for l in range(L):
        K, Vc = layer_cache(l)
        t = time.perf_counter()
        oracle.kv_compact([K, Vc], w.pt, P, paths, acc)
        tc += time.perf_counter() - t
    times["compact"] = tc
    return times


def oracle_sample(w, budget_s=20.0):
    """An ESTIMATE of one oracle round for the configurations whose whole round does
    not fit the budget (batched, 70B): fusion, expansion, tree build and accept of
    request 0 scaled by B; verify of request 0 (dense form) on as many layers as fit
    ~60% of budget_s, scaled by L and by the batch's keys; the LM head on 1/4 of the
    vocabulary, scaled by 4."""
    import torch

    import oracle
    b, cfg = w.bufs, w.cfg
    f = lambda t: t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()  # noqa: E731
    B, R, V = cfg.B, cfg.R, cfg.V
    w.use(0)
    st = w.sets[0]
    pages = st.pages.cpu().numpy()
    times = {}
    hs = [f(t) for t in b.h]
    Wf = f(b.W_f)
    t = time.perf_counter()
    oracle.fuse(*hs, Wf)
    times["fuse"] = time.perf_counter() - t
    sizes, n_cand = cfg.frontier_sizes()
    drafts = [f(x) for x in st.drafts]
    t = time.perf_counter()
    c = oracle.new_cands(n_cand)
    fid, fsc = np.array([-1], np.int32), np.zeros(1, np.float32)
    for di, (F, off) in enumerate(sizes):
        if cfg.sampled:
            fid, fsc, _, _ = oracle.expand_sampled(drafts[di][0][:F], cfg.k, cfg.W, fsc, fid, di + 1, off, c,
                                                   cfg.draw_seed, 0)
        else:
            fid, fsc = oracle.expand(drafts[di][0][:F], cfg.k, cfg.W, fsc, fid, di + 1, off, c)
    tree = oracle.build_tree(c, n_cand, cfg.N, int(st.root_tok[0]), int(w.kv_len0[0]))
    times["expand_build"] = (time.perf_counter() - t) * B
    p0 = int(w.c["P"][0])
    scale_b = sum(p + R for p in w.c["P"]) / (p0 + R)
    spent, n_layers = 0.0, 0
    for l in range(cfg.L - 1, -1, -1):
        K, Vc = f(b.K_all[l]), f(b.V_all[l])
        K[pages], Vc[pages] = f(st.snapK[l]), f(st.snapV[l])
        Q = f(st.Q[l])[:1]
        t = time.perf_counter()
        oracle.tree_verify_attn_dense(Q, K, Vc, w.pt[:1], w.kv_len0.cpu().numpy()[:1], tree["mask"][None],
                                      1.0 / math.sqrt(cfg.hd))
        spent += time.perf_counter() - t
        n_layers += 1
        if spent >= 0.6 * budget_s:
            break
    times["verify"] = spent / n_layers * cfg.L * scale_b
    Wl = f(b.W_lm)
    h = f(b.O[cfg.L - 1]).reshape(B * R, -1)
    t = time.perf_counter()
    z = oracle.lmhead_logits(h, Wl[:V // 4])
    times["lmhead"] = (time.perf_counter() - t) * 4
    del z
    zl = f(b.logits)[:R]  # full rows (the GPU's logits of the last round): tokens index the whole vocabulary
    t = time.perf_counter()
    ua, ub = b.u_acc.cpu().numpy()[0].view(np.uint32), b.u_bonus.cpu().numpy()[0].view(np.uint32)
    if cfg.sampled:
        oracle.accept_sampled(tree, zl, float(w.c["temps"][0]), np.ascontiguousarray(zl), 1.0, ua, ub, cfg.D)
    else:
        oracle.accept(tree, zl, float(w.c["temps"][0]), ua, ub, cfg.D)
    times["accept"] = (time.perf_counter() - t) * B
    return times, n_layers


def cpu_baseline(w, budget_s=30.0):
    """The oracle on the host cores: whole rounds at all cores and at one thread
    where a whole round fits the budget, else an estimate from a sample."""
    bt = BlasThreads()
    n_all = bt.threads() or os.cpu_count()
    out = {"kind": "oracle", "unit": "rounds/s"}
    if whole_round_feasible(w):
        t0 = time.perf_counter()
        times = oracle_round(w, 0)
        sec_all = sum(times.values())
        out.update(value=round(1.0 / sec_all, 6), cores=n_all, seconds_per_round=round(sec_all, 3),
                   breakdown_s={k: round(v, 3) for k, v in times.items()},
                   threads_all={"threads": n_all, "rounds_per_s": round(1.0 / sec_all, 6),
                                "seconds_per_round": round(sec_all, 3)},
                   sample="one whole round of the same workload (round 0's inputs): fusion, expansion, tree "
                          "build, verify on all L layers (dense masked form), LM head, statistics and accept "
                          "of every request, compaction of every layer; device data staged to the host "
                          "outside the timed parts")
        if sec_all * 8 <= budget_s and bt.set:
            one = bt.use(1)
            try:
                times1 = oracle_round(w, 0)
            finally:
                bt.use(n_all)
            sec1 = sum(times1.values())
            out["threads_1"] = {"threads": one, "rounds_per_s": round(1.0 / sec1, 6),
                                "seconds_per_round": round(sec1, 3),
                                "breakdown_s": {k: round(v, 3) for k, v in times1.items()}}
        else:
            out["threads_1"] = None
            out["threads_1_note"] = ("BLAS thread control unavailable" if not bt.set else
                                     f"a one-thread round would exceed the {budget_s:.0f} s sample budget")
        out["wall_s"] = round(time.perf_counter() - t0, 1)
    else:
        times, n_layers = oracle_sample(w, budget_s * 0.6)
        sec = sum(times.values())
        out.update(value=round(1.0 / sec, 6), cores=n_all, seconds_per_round=round(sec, 3), estimate=True,
                   breakdown_s={k: round(v, 3) for k, v in times.items()},
                   threads_all={"threads": n_all, "rounds_per_s": round(1.0 / sec, 6)}, threads_1=None,
                   threads_1_note="a whole round does not fit the sample budget at this size",
                   sample=f"ESTIMATE: request 0's fusion, expansion, tree build and accept scaled by B; verify of "
                          f"request 0 on {n_layers} of the L layers scaled by L and by the batch's keys; LM head "
                          f"on 1/4 of the vocabulary scaled by 4")
    return out


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="8b", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--sets", type=int, default=8, help="distinct input sets (trees, roots, drafts) cycled")
    ap.add_argument("--min-time", type=float, default=2.5, help="seconds of timed graph replays")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-draft", action="store_true", help="skip timing the GPU drafter")
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
    K = args.steps
    n_stat = max(K, 32)
    w = Workload(args.config, seed=args.seed + 1000 * rank, layers=args.layers, n_sets=args.sets, n_uniform=n_stat)
    cfg = w.cfg
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3
    with torch.cuda.stream(s):
        for i in range(args.warmup):
            w.round(i)
        # acceptance over n_stat distinct rounds (round k: input set k % sets, uniforms k)
        hist = torch.empty((n_stat, cfg.B), dtype=torch.int32, device="cuda")
        for k in range(n_stat):
            w.round(k)
            hist[k].copy_(w.bufs.acc_len)
    s.synchronize()
    check_dev_err(w, "warm-up rounds")
    accepted = hist.cpu().numpy().reshape(-1)

    # The timed region: one graph of K rounds (round k: its inputs bound, request
    # lengths reset, tree pages restored, the seven steps), replayed for at least
    # --min-time seconds, each replay timed alone; the median replay / K is a step.
    # A second graph of the same rounds with events at the phase boundaries gives
    # the phase split; it is replayed separately, because an event between two
    # kernels also cuts the programmatic launch edge between them.
    phases = ["fuse", "expand", "tree", "verify", "lmhead", "accept", "compact"]
    ev = [[graph_event() for _ in range(len(phases) + 1)] for _ in range(K)]
    graph = torch.cuda.CUDAGraph()
    counts = []  # library launch counter at each phase boundary of the first captured round
    n0 = e3.launch_count()
    with torch.cuda.graph(graph, stream=s):
        for k in range(K):
            run_round_phased(w, k, None, e3, counts if k == 0 else None)
    launches_timed = e3.launch_count() - n0  # libeagle3 kernels in the K captured rounds
    phase_launches = {p: counts[i + 1] - counts[i] for i, p in enumerate(phases)}
    graph_phased = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph_phased, stream=s):
        for k in range(K):
            run_round_phased(w, k, ev[k], e3)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        graph.replay()  # untimed replays of the captured work
        graph.replay()
    torch.cuda.synchronize()
    t = time.perf_counter()
    with torch.cuda.stream(s):
        graph.replay()
    torch.cuda.synchronize()
    est = max(time.perf_counter() - t, 1e-4)
    n_rep = max(3, int(math.ceil(args.min_time / est)))
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_rep)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for a, z in marks:
            a.record(s)
            graph.replay()
            z.record(s)
    torch.cuda.synchronize()
    clk = clocks.stop()
    rep_ms = [a.elapsed_time(z) for a, z in marks]
    check_dev_err(w, "timed rounds")
    ms = ranks_max(statistics.median(rep_ms), world)
    ms_step = ms / K
    phase_ms = {p: 0.0 for p in phases}
    n_ph = 3
    for _ in range(n_ph):
        with torch.cuda.stream(s):
            graph_phased.replay()  # the phase split (not timed as a whole)
        torch.cuda.synchronize()
        for i, p in enumerate(phases):
            phase_ms[p] += statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K)) / n_ph
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
                "tensor_frac": round(wm["verify_flops"] / (ver_ms * 1e-3) / 1e12 / tflops, 4),
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
    draft = None if args.no_draft else draft_leg(w, s)
    if draft is not None:
        # a round whose draft logits come from the drafter on the GPU: drafting + the round
        draft["self_contained_rounds_per_s"] = round(1000.0 / (draft["ms"] + ms_step), 3)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(rounds_s, 3), "unit": "rounds/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (seeded; random-init weights)",
            "config": {"workload": w.c["workload"], "global_batch": cfg.B * world, "prefix_lens": summarize(w.c["P"]),
                       "nodes": cfg.N, "depth": cfg.D, "topk": cfg.k, "layers": cfg.L,
                       "input_sets": len(w.sets), "uniform_sets": len(w.uni),
                       "l2": "inputs larger than L2 per step (L distinct per-layer KV caches + 1 LM head)",
                       "timed": f"median of {n_rep} graph replays of {K} rounds each ({sum(rep_ms) / 1e3:.2f} s); "
                                "each round restores its tree pages (K/V of the tree slots) from its input set",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "nodes_per_s": round(nodes_s, 1),
            "accepted_mean": round(float(np.mean(accepted)), 4),
            "accepted_rounds": int(n_stat),
            "accepted_hist": np.bincount(accepted.astype(np.int64), minlength=cfg.D + 1).tolist(),
            "replay_ms": {"median": round(statistics.median(rep_ms), 4), "min": round(min(rep_ms), 4),
                          "max": round(max(rep_ms), 4), "n": n_rep},
            "phase_ms": {k: round(v, 4) for k, v in phase_ms.items()},
            "roofline": roofline,
            "roofline_lmhead": lm,
            "gpu_launches": launches_timed,
            "launches_per_round": phase_launches,
            "clocks": clk,
            "e2e": e2e,
            "drafter": draft,
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


def run_round_phased(w, k, evs, e3, counts=None):
    """Round k (the same calls as Workload.round) with a timing event recorded at each
    of its 8 phase boundaries (none when ``evs`` is None).  With ``counts`` (a
    list), also append the library's launch counter there."""
    import torch
    s = torch.cuda.current_stream()

    def mark(i):
        if evs is not None:
            evs[i].record(s)
        if counts is not None:
            counts.append(e3.launch_count())

    w.round(k, stream=s, mark=mark)


class Slot:
    """One device copy of everything a round reads that changes per step (e2e)."""

    def __init__(self, w, st):
        b = w.bufs
        self.h = [t.clone() for t in b.h]
        self.drafts = [t.clone() for t in st.drafts]
        self.Q = [t.clone() for t in st.Q]
        self.u_acc, self.u_bonus = b.u_acc.clone(), b.u_bonus.clone()
        self.temp, self.temp_rows = b.temp.clone(), b.temp_rows.clone()
        self.root_tok, self.kv_len0 = st.root_tok.clone(), w.kv_len0.clone()
        self.snapK, self.snapV = st.snapK.clone(), st.snapV.clone()
        self.pages = st.pages

    def tensors(self):
        return [*self.h, *self.drafts, *self.Q, self.u_acc, self.u_bonus, self.temp, self.temp_rows, self.root_tok,
                self.kv_len0, self.snapK, self.snapV]

    def bind(self, b):
        b.h, b.draft_logits, b.Q = self.h, self.drafts, self.Q
        b.u_acc, b.u_bonus, b.temp, b.temp_rows, b.root_tok = (self.u_acc, self.u_bonus, self.temp, self.temp_rows,
                                                               self.root_tok)


def e2e_leg(w, s, K, warmup, world=1):
    """The same rounds through the C ABI, fed from pinned HOST buffers: every step
    copies its round's inputs host -> device (fusion inputs, draft logits, per-layer
    Q, uniforms, temperatures, root tokens, request lengths, the tree pages of every
    layer's K/V), runs the round and reads its result (emitted tokens, path,
    accepted length) back.  Two device slots: step i+1's copies run on a second
    stream while step i computes (events order each slot's reuse)."""
    import torch

    from eagle_speculative_decoding_round_gb300.round import run_round
    b = w.bufs
    saved = (b.h, b.draft_logits, b.Q, b.u_acc, b.u_bonus, b.temp, b.temp_rows, b.root_tok)
    n_host = min(len(w.sets), 4)
    w.use(0)
    slots = [Slot(w, w.sets[0]) for _ in range(2)]
    host_sets = []
    for i in range(n_host):
        w.use(i)
        tmp = Slot(w, w.sets[i])
        host_sets.append([t.detach().cpu().pin_memory() for t in tmp.tensors()])
        del tmp
    outs = [b.out_tok, b.path, b.acc_len]
    h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs] for _ in range(2)]
    bi = sum(t.numel() * t.element_size() for t in slots[0].tensors())
    bo = sum(t.numel() * t.element_size() for t in outs)
    graphs = []
    for sl in slots:
        sl.bind(b)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            b.kv_len.copy_(sl.kv_len0)
            b.K_all.index_copy_(1, sl.pages, sl.snapK)
            b.V_all.index_copy_(1, sl.pages, sl.snapV)
            run_round(b, stream=s)
        graphs.append(g)
    torch.cuda.synchronize()
    cs = torch.cuda.Stream()
    loaded = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        j = i % 2
        cs.wait_event(free[j])  # the round that last used slot j has finished
        with torch.cuda.stream(cs):
            for d, h in zip(slots[j].tensors(), host_sets[i % n_host]):
                d.copy_(h, non_blocking=True)
            loaded[j].record(cs)
        s.wait_event(loaded[j])
        with torch.cuda.stream(s):
            graphs[j].replay()
            for h, d in zip(h_out[j], outs):
                h.copy_(d, non_blocking=True)
            free[j].record(s)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    a.record(cs)
    for i in range(K):
        step(i)
    z.record(s)
    torch.cuda.synchronize()
    check_dev_err(w, "e2e")
    ms = ranks_max(a.elapsed_time(z) / K, world)
    (b.h, b.draft_logits, b.Q, b.u_acc, b.u_bonus, b.temp, b.temp_rows, b.root_tok) = saved
    return {"value": round(job_rounds_per_s(ms, world), 3), "unit": "rounds/s", "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": round(ms, 4),
            "overlap": "double-buffered: step i+1's host-to-device copies on a second stream during step i"}


FFN = {4096: 14336, 8192: 28672}  # MLP width of the target family at each model width


def draft_leg(w, s, reps=20):
    """The drafting phase of a round with the drafter on the GPU: D depths of
    eagle3_draft_step (one decoder layer with random weights of the target's
    shape, the target's vocabulary) each followed by eagle3_expand on its logits,
    for the B requests; captured as one graph and timed by CUDA events.  Reported
    beside the round (whose draft logits are inputs): per depth, and against HBM
    for the weights each depth streams."""
    import torch
    e3, cfg = w.e3, w.cfg
    if cfg.dtype != "bf16" or cfg.sampled:
        return None
    d, H, KVH, hd, V, B = cfg.d, cfg.H, cfg.KVH, cfg.hd, cfg.V, cfg.B
    ffn = FFN.get(d, 4 * d)
    g = torch.Generator(device="cuda")
    g.manual_seed(99)

    def rnd(shape, std, mean=0.0, dt=torch.bfloat16):
        return (torch.randn(shape, generator=g, device="cuda") * std + mean).to(dt)

    Wt = dict(emb=rnd((V, d), 1.0), W_in=rnd((d, 2 * d), 0.02), norm1=rnd((d,), 0.02, 1.0, torch.float32),
              W_qkv=rnd(((H + 2 * KVH) * hd, d), 0.02), W_o=rnd((d, H * hd), 0.02),
              norm2=rnd((d,), 0.02, 1.0, torch.float32), W_gu=rnd((2 * ffn, d), 0.02), W_down=rnd((d, ffn), 0.02),
              norm_f=rnd((d,), 0.02, 1.0, torch.float32), W_lm=rnd((V, d), 4.0 / math.sqrt(d)))
    dr = e3.make_drafter(Wt["emb"], Wt["W_in"], Wt["norm1"], Wt["W_qkv"], Wt["W_o"], Wt["norm2"], Wt["W_gu"],
                         Wt["W_down"], Wt["norm_f"], Wt["W_lm"], d, H, KVH, hd, ffn, V)
    sizes, n_cand = cfg.frontier_sizes()
    bases = [0]
    for F, _ in sizes:
        bases.append(bases[-1] + F)
    R_slots = bases[-1]
    P = w.c["P"]
    pt, npages = w.synth.page_table(7, [p + R_slots for p in P], cfg.page_size)
    Kc, Vc = rnd((npages, KVH, cfg.page_size, hd), 1.0), rnd((npages, KVH, cfg.page_size, hd), 1.0)
    ptt = torch.from_numpy(pt).cuda()
    kv = e3.make_kv_layer(Kc, Vc, ptt, npages, cfg.page_size, pt.shape[1], KVH, hd, e3.E3_BF16,
                          e3.E3_KV_PREFIX_STABLE)
    kv_len = torch.tensor(P, dtype=torch.int32, device="cuda")
    gfeat = rnd((B, d), 1.0)
    roots = torch.randint(0, V, (B,), generator=g, device="cuda", dtype=torch.int32)
    i32 = dict(dtype=torch.int32, device="cuda")
    c_tok, c_par = torch.zeros((B, n_cand), **i32), torch.zeros((B, n_cand), **i32)
    c_sc, c_dep = torch.zeros((B, n_cand), device="cuda"), torch.zeros((B, n_cand), **i32)
    cands = e3.make_cand(c_tok, c_par, c_sc, c_dep, n_cand)
    f_id = [torch.full((B, 1), -1, **i32)] + [torch.zeros((B, min(cfg.W, F * cfg.k)), **i32) for F, _ in sizes]
    f_sc = [torch.zeros((B, 1), device="cuda")] + [torch.zeros((B, min(cfg.W, F * cfg.k)), device="cuda")
                                                   for F, _ in sizes]
    a_slots = torch.zeros((B, R_slots, d), device="cuda")
    mask = torch.zeros((B, R_slots, (R_slots + 63) // 64), dtype=torch.int64, device="cuda")
    Fmax = max(F for F, _ in sizes)
    logits = [torch.empty((B, F, V), device="cuda") for F, _ in sizes]
    rmax, rQ = torch.empty(B * Fmax, device="cuda"), torch.empty(B * Fmax, dtype=torch.int64, device="cuda")
    ram = torch.empty(B * Fmax, **i32)
    wsb = e3.eagle3_draft_workspace_bytes(dr, B, Fmax, R_slots, max(P))
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, **i32)
    ev = [graph_event() for _ in range(len(sizes) + 1)]

    def drafting(marks):
        for di, (F, off) in enumerate(sizes):
            if marks:
                ev[di].record(s)
            prev = f_id[di - 1] if di else f_id[0]
            e3.eagle3_draft_step(dr, kv, kv_len, max(P), B, di + 1, F, f_id[di], bases[di], prev.shape[1] if di else 0,
                                 prev if di else None, bases[di - 1] if di else 0, R_slots, cands, roots, gfeat, a_slots,
                                 mask, logits[di], rmax, rQ, ram, ws, wsb, err, stream=s)
            e3.eagle3_expand(logits[di], B, F, V, cfg.k, cfg.W, 1.0, f_sc[di], f_id[di], di + 1, off, cands,
                             f_id[di + 1], f_sc[di + 1], err, stream=s)
        if marks:
            ev[-1].record(s)

    with torch.cuda.stream(s):
        drafting(False)
    torch.cuda.synchronize()
    n0 = e3.launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        drafting(False)
    launches = e3.launch_count() - n0
    gph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gph, stream=s):
        drafting(True)
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        graph.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(reps):
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            a.record(s)
            graph.replay()
            z.record(s)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(z))
    with torch.cuda.stream(s):
        gph.replay()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"drafting: device error flags {int(err.item()):#x}")
    per_depth = [ev[i].elapsed_time(ev[i + 1]) for i in range(len(sizes))]
    # weights each depth streams (the embedding table only by the rows it gathers)
    wbytes = 2 * (2 * d * d + (H + 2 * KVH) * hd * d + d * H * hd + 3 * ffn * d + V * d)
    ms = statistics.median(times)
    peaks = load_peaks()
    hbm = peaks.get("hbm_gbs", 6800.0)
    gbs = wbytes * len(sizes) / (ms * 1e-3) / 1e9
    return {"what": "drafter on the GPU: D x (eagle3_draft_step + eagle3_expand), random weights of the target's "
                    f"shape (d={d}, {H}/{KVH} heads x {hd}, MLP {ffn}, vocabulary {V})",
            "ms": round(ms, 4), "per_depth_ms": [round(x, 4) for x in per_depth], "launches": launches,
            "weight_bytes_per_depth": wbytes, "achieved_gbs": round(gbs, 1),
            "hbm_frac": round(gbs / hbm, 4), "self_contained_rounds_per_s": None}


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
    """The oracle, as it stands, on the host cores: every step is one whole oracle
    round of the same workload (round k's inputs, all BLAS threads), where a whole
    round fits; otherwise an estimate from a bounded sample, said so in the line."""
    if rank != 0:
        return 0
    w = Workload(args.config, seed=args.seed, n_sets=min(args.sets, 2), n_uniform=max(args.steps, 1))
    bt = BlasThreads()
    cores = bt.threads() or os.cpu_count()
    whole = whole_round_feasible(w)
    per = []
    if whole:
        for i in range(max(0, min(args.warmup, 1))):
            oracle_round(w, i)
        for k in range(args.steps):
            per.append(sum(oracle_round(w, k).values()))
        sample = "per step: one whole oracle round (round k's inputs) -- fusion, expansion, tree build, verify on " \
                 "all L layers, LM head, statistics, accept, compaction"
    else:
        budget = max(2.0, 120.0 / (args.steps + 1))
        for _ in range(args.steps):
            times, n_layers = oracle_sample(w, budget)
            per.append(sum(times.values()))
        sample = "ESTIMATE per step: a bounded sample of one round scaled to a whole round (the whole round " \
                 "does not fit the run's time at this size)"
    sec = float(np.mean(per))
    v = 1.0 / sec
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": "rounds/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1000, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; random-init weights)",
            "config": {"workload": w.c["workload"], "global_batch": w.cfg.B},
            "cpu_baseline": {"value": round(v, 6), "unit": "rounds/s", "cores": cores, "kind": "oracle",
                             "sample": sample, "estimate": not whole},
            "e2e": {"value": round(v, 6), "unit": "rounds/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    main()
