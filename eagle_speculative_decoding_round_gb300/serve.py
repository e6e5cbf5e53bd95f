"""Multi-round speculative decoding with an adaptive draft-tree budget, over libeagle3.

One round per budget level and step: the requests whose controller level is l run
together as one round of that level's tree shape (node budget N, depth D, top-k,
frontier width), in buffers of their own that share one paged KV cache per layer
with the other levels.  After a round every request's bonus token becomes its next
root, its committed length advances by 1 + accepted ("Thinking Budget 与 EAGLE-3",
一棵候选树怎样被验证: commit only the accepted path, the correction token opens
the next round; "EAGLE 系列与 DFlash", §二 阶段三), and the library's host-side
controller (eagle3_budget_update) picks its next level from its accepted lengths
("Thinking Budget 与 EAGLE-3", 服务端应怎样联合控制: the execution controller changes
only the speculative budget, so the emitted tokens are those of the target's own
decoding at every level).

The model around the path is the caller's: ``drafter(bufs, rows, di)`` writes the
draft logits of depth di + 1 for the requests in ``rows`` (the frontier of the
previous depth is in ``bufs.f_id[di]``), ``target(bufs, rows)`` writes the tree
nodes' Q (every layer) and K/V (slots kv_len .. kv_len + R - 1) once the tree is
built.  Nothing here computes: every step is a library call.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

from . import eagle3 as e3
from . import synth
from .round import RoundBuffers, RoundConfig, run_round


@dataclasses.dataclass
class Request:
    rid: int
    root_tok: int            # the newest token: its K/V is not in the cache yet
    kv_len: int              # tokens with K/V in the cache
    temp: float = 0.0        # 0: greedy
    emitted: list = dataclasses.field(default_factory=list)  # tokens committed so far, in order
    accepted: list = dataclasses.field(default_factory=list)  # accepted drafted tokens per round
    levels: list = dataclasses.field(default_factory=list)    # budget level of each round


@dataclasses.dataclass
class Level:
    N: int   # drafted nodes
    D: int   # depth
    k: int   # top-k per expanded node
    W: int   # frontier width


class ServingLoop:
    """Rounds for ``len(requests)`` requests sharing ``kv_cache`` (K_all, V_all:
    [L][pages][KVH][page][hd]) through ``page_table`` [B][max_pages]."""

    def __init__(self, shape: dict, levels: list, kv_cache, page_table: torch.Tensor, n_pages: int,
                 W_lm: torch.Tensor, requests: list, policy: dict | None = None, seed: int = 0, device="cuda"):
        self.shape, self.levels = shape, [Level(*lv) for lv in levels]
        self.kv_cache, self.page_table, self.n_pages = kv_cache, page_table, n_pages
        self.W_lm, self.requests, self.seed, self.device = W_lm, requests, seed, device
        self.B = len(requests)
        self.policy = e3.budget_policy([(lv.N, lv.D) for lv in self.levels], **(policy or {}))
        self.state = e3.eagle3_budget_init(self.policy, self.B)
        self.level = [int(s.level) for s in self.state]
        self.bufs = {}
        self.rounds = 0
        self.max_kv_len = int(page_table.shape[1]) * shape["page_size"]

    def buffers(self, li: int) -> RoundBuffers:
        """The round buffers of level li (created on first use, for every request)."""
        if li not in self.bufs:
            lv, sh = self.levels[li], self.shape
            cfg = RoundConfig(B=self.B, N=lv.N, D=lv.D, k=lv.k, W=lv.W, H=sh["H"], KVH=sh["KVH"], hd=sh["hd"],
                              d=sh["d"], V=sh["V"], L=sh["L"], max_kv_len=self.max_kv_len - lv.N - 1,
                              dtype=sh["dtype"], page_size=sh["page_size"], M_fuse=self.B)
            # a page table of its own: its first rows are overwritten with the rows of each round's requests
            b = RoundBuffers(cfg, self.page_table.clone(), self.n_pages, self.device, kv_cache=self.kv_cache,
                             W_lm=self.W_lm)
            for t in b.h:
                t.zero_()
            b.W_f.zero_()
            self.bufs[li] = b
        return self.bufs[li]

    def step(self, drafter, target, spare: float = 1.0, draft_cost: float = 0.0, stream=None):
        """One round for every request (one library round per budget level in use)."""
        acc_all = np.zeros(self.B, np.int32)
        for li in sorted(set(self.level)):
            rows = [i for i in range(self.B) if self.level[i] == li]
            b = self.buffers(li)
            n = len(rows)
            reqs = [self.requests[i] for i in rows]
            idx = torch.tensor(rows, dtype=torch.long, device=self.device)
            b.page_table[:n].copy_(self.page_table.index_select(0, idx))
            b.kv_len[:n].copy_(torch.tensor([r.kv_len for r in reqs], dtype=torch.int32))
            b.root_tok[:n].copy_(torch.tensor([r.root_tok for r in reqs], dtype=torch.int32))
            temps = torch.tensor([r.temp for r in reqs], dtype=torch.float32)
            b.temp[:n].copy_(temps)
            b.temp_rows[:n * b.cfg.R].copy_(temps.repeat_interleave(b.cfg.R))
            R = b.cfg.R
            us = self.seed * 1000003 + self.rounds
            ua = np.stack([synth.uniforms(us, synth.PURPOSE_ACCEPT, 1, R, req0=r.rid)[0] for r in reqs])
            ub = np.stack([synth.uniforms(us, synth.PURPOSE_BONUS, 1, R, req0=r.rid)[0] for r in reqs])
            b.u_acc[:n].copy_(torch.from_numpy(ua.view(np.int32)))
            b.u_bonus[:n].copy_(torch.from_numpy(ub.view(np.int32)))
            run_round(b, stream=stream, B=n, draft=lambda bb, di: drafter(bb, rows, di),
                      write_tree_qkv=lambda bb: target(bb, rows))
            acc = b.acc_len[:n].cpu().numpy()
            out = b.out_tok[:n].cpu().numpy()
            kv_new = b.kv_len[:n].cpu().numpy()
            if int(b.dev_err.item()) != 0:
                raise RuntimeError(f"device error flags {int(b.dev_err.item()):#x} in a level-{li} round")
            for j, r in enumerate(reqs):
                a = int(acc[j])
                r.emitted.extend(int(t) for t in out[j, :a + 1])
                r.accepted.append(a)
                r.levels.append(li)
                r.root_tok = int(out[j, a])
                r.kv_len = int(kv_new[j])
                acc_all[rows[j]] = a
        self.level = e3.eagle3_budget_update(self.policy, self.state, acc_all, spare, draft_cost)
        self.rounds += 1
        return acc_all
