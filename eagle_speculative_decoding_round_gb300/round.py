"""One EAGLE-3 draft-and-verify round driven through libeagle3's C ABI.

``RoundBuffers`` owns the device buffers of one configuration (torch is only
the allocator); ``run_round`` enqueues the seven steps on one stream:

  fuse -> expand x D -> tree_build_mask -> [caller writes tree Q/K/V]
       -> tree_verify_attn x L -> lmhead_logits -> spec_accept -> kv_compact

Nothing here computes: every step is a library kernel.  The draft model that
turns the fused feature into draft logits needs trained weights and is not
part of the round; its logits (one [B, F_d, V] block per depth) are inputs.

With ``RoundConfig.sampled`` the children are drawn from the draft
distribution (eagle3_expand_sampled, keyed by ``draw_seed``), every candidate
is kept (N = number of candidates) and the accept step is spec_accept_sampled:
"EAGLE 系列与 DFlash", §四 DFlash, acceptance min(1, p_target / p_draft).
"""
from __future__ import annotations

import dataclasses
import math

import torch

from . import eagle3 as e3


@dataclasses.dataclass
class RoundConfig:
    B: int
    N: int            # drafted nodes per request (R = N + 1)
    D: int            # depth
    k: int            # top-k per frontier node
    W: int            # frontier width
    H: int            # query heads
    KVH: int          # KV heads
    hd: int           # head dim
    d: int            # model dim (fusion input dim per source and output dim)
    V: int            # vocabulary
    L: int            # target layers
    max_kv_len: int   # bound on every request's prefix length
    dtype: str = "bf16"
    page_size: int = 64
    M_fuse: int = 0   # rows fused per round (0 -> B * (D + 1))
    sampled: bool = False  # children drawn from the draft distribution
    draw_seed: int = 0     # stream of those draws

    @property
    def R(self) -> int:
        return self.N + 1

    @property
    def dt(self) -> int:
        return e3.E3_BF16 if self.dtype == "bf16" else e3.E3_F32

    @property
    def tdtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def frontier_sizes(self):
        """Rows F_d expanded at depth d = 1..D and the candidate offsets."""
        F, out, off = 1, [], 0
        for _ in range(self.D):
            out.append((F, off))
            off += F * self.k
            F = min(self.W, F * self.k)
        return out, off

    @property
    def n_cand(self) -> int:
        return self.frontier_sizes()[1]

    @property
    def M(self) -> int:
        return self.M_fuse or self.B * (self.D + 1)


class RoundBuffers:
    """Device buffers for one configuration.  KV caches hold every request's pages
    (prefix + room for the R tree slots) for L layers."""

    def __init__(self, cfg: RoundConfig, page_table: torch.Tensor, n_pages: int, device="cuda", kv_cache=None,
                 W_lm=None):
        c = cfg
        dev = torch.device(device)
        self.cfg = c
        td = c.tdtype
        i32 = dict(dtype=torch.int32, device=dev)
        self.page_table = page_table.to(dev, torch.int32).contiguous()
        self.n_pages = n_pages
        self.max_pages = self.page_table.shape[1]
        # one tensor per operand over all layers; layer l's cache is the view [l]
        # (kv_cache: caches shared with other buffers, e.g. one per tree budget of a serving loop)
        if kv_cache is not None:
            self.K_all, self.V_all = kv_cache
        else:
            self.K_all = torch.empty((c.L, n_pages, c.KVH, c.page_size, c.hd), dtype=td, device=dev)
            self.V_all = torch.empty((c.L, n_pages, c.KVH, c.page_size, c.hd), dtype=td, device=dev)
        self.K = list(self.K_all.unbind(0))
        self.Vc = list(self.V_all.unbind(0))
        self.kv_len = torch.zeros(c.B, **i32)
        # fusion
        self.h = [torch.empty((c.M, c.d), dtype=td, device=dev) for _ in range(3)]
        self.W_f = torch.empty((c.d, 3 * c.d), dtype=td, device=dev)
        self.g = torch.empty((c.M, c.d), dtype=td, device=dev)
        self.fuse_ws_bytes = e3.eagle3_fuse_workspace_bytes(c.M, c.d, c.d, c.dt)
        self.fuse_ws = torch.empty(max(self.fuse_ws_bytes, 16), dtype=torch.uint8, device=dev)
        # drafting
        sizes, n_cand = c.frontier_sizes()
        self.draft_logits = [torch.empty((c.B, F, c.V), dtype=torch.float32, device=dev) for F, _ in sizes]
        self.cap = n_cand
        self.c_tok = torch.empty((c.B, n_cand), **i32)
        self.c_parent = torch.empty((c.B, n_cand), **i32)
        self.c_score = torch.empty((c.B, n_cand), dtype=torch.float32, device=dev)
        self.c_depth = torch.empty((c.B, n_cand), **i32)
        self.cand = e3.make_cand(self.c_tok, self.c_parent, self.c_score, self.c_depth, n_cand)
        if c.sampled and c.N != n_cand:
            raise ValueError(f"sampled drafts keep every candidate: N must be {n_cand}, not {c.N}")
        self.q_stats = torch.zeros((c.B * (n_cand + 1) * e3.QSTAT_BYTES if c.sampled else 16,), dtype=torch.uint8,
                                   device=dev)
        Fmax = max(F for F, _ in sizes)
        self.f_id = [torch.empty((c.B, max(F, 1)), **i32) for F, _ in sizes] + [torch.empty((c.B, c.W if c.W < 1 << 20 else Fmax * c.k), **i32)]
        self.f_score = [torch.empty((c.B, max(F, 1)), dtype=torch.float32, device=dev) for F, _ in sizes] + [torch.empty((c.B, c.W if c.W < 1 << 20 else Fmax * c.k), dtype=torch.float32, device=dev)]
        self.f_id[0].fill_(-1)
        self.f_score[0].zero_()
        # tree
        R = c.R
        self.root_tok = torch.zeros(c.B, **i32)
        self.tok = torch.empty((c.B, R), **i32)
        self.parent = torch.empty((c.B, R), **i32)
        self.depth = torch.empty((c.B, R), **i32)
        self.pos = torch.empty((c.B, R), **i32)
        self.mask = torch.empty((c.B, R, (R + 63) // 64), dtype=torch.int64, device=dev)
        self.node_cand = torch.empty((c.B, R), **i32)
        # verify
        self.Q = [torch.empty((c.B, R, c.H, c.hd), dtype=td, device=dev) for _ in range(c.L)]
        self.O = [torch.empty((c.B, R, c.H, c.hd), dtype=td, device=dev) for _ in range(c.L)]
        self.lse = [torch.empty((c.B, R, c.H), dtype=torch.float32, device=dev) for _ in range(c.L)]
        self.ws_bytes = e3.eagle3_verify_workspace_bytes(c.B, R, c.H, c.KVH, c.hd, c.max_kv_len, c.dt)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        # the round's verify calls follow tree_build_mask or the previous layer's verify,
        # neither of which writes the prefix K/V, kv_len or the page table
        self.kv = [e3.make_kv_layer(self.K[l], self.Vc[l], self.page_table, n_pages, c.page_size,
                                    self.max_pages, c.KVH, c.hd, c.dt, e3.E3_KV_PREFIX_STABLE) for l in range(c.L)]
        # logits / accept
        self.W_lm = torch.empty((c.V, c.H * c.hd), dtype=td, device=dev) if W_lm is None else W_lm
        self.temp = torch.ones(c.B, dtype=torch.float32, device=dev)
        self.temp_rows = torch.ones(c.B * R, dtype=torch.float32, device=dev)
        self.logits = torch.empty((c.B * R, c.V), dtype=torch.float32, device=dev)
        self.row_max = torch.empty(c.B * R, dtype=torch.float32, device=dev)
        self.row_Q = torch.empty(c.B * R, dtype=torch.int64, device=dev)
        self.row_argmax = torch.empty(c.B * R, **i32)
        self.u_acc = torch.zeros((c.B, R), **i32)
        self.u_bonus = torch.zeros((c.B, R), **i32)
        self.acc_len = torch.empty(c.B, **i32)
        self.path = torch.empty((c.B, c.D + 1), **i32)
        self.out_tok = torch.empty((c.B, c.D + 1), **i32)
        self.status = torch.empty(c.B, **i32)
        self.dev_err = torch.zeros(1, **i32)

    def set_temperature(self, temp: torch.Tensor):
        self.temp.copy_(temp)
        self.temp_rows.copy_(self.temp.repeat_interleave(self.cfg.R))


def expand_depth(bufs: RoundBuffers, di: int, stream=None, B=None):
    """Depth di + 1 of the draft tree: expand the frontier rows of bufs.draft_logits[di]
    (of the first B requests; all by default)."""
    c = bufs.cfg
    B = c.B if B is None else B
    F, off = c.frontier_sizes()[0][di]
    if c.sampled:
        e3.eagle3_expand_sampled(bufs.draft_logits[di], B, F, c.V, c.k, c.W, 1.0, bufs.f_score[di], bufs.f_id[di],
                                 di + 1, off, bufs.cand, bufs.f_id[di + 1], bufs.f_score[di + 1], c.draw_seed,
                                 bufs.q_stats, bufs.dev_err, stream=stream)
    else:
        e3.eagle3_expand(bufs.draft_logits[di], B, F, c.V, c.k, c.W, 1.0, bufs.f_score[di], bufs.f_id[di],
                         di + 1, off, bufs.cand, bufs.f_id[di + 1], bufs.f_score[di + 1], bufs.dev_err, stream=stream)


def build_tree(bufs: RoundBuffers, stream=None, B=None):
    c = bufs.cfg
    B = c.B if B is None else B
    e3.tree_build_mask(bufs.cand, B, c.n_cand, c.N, bufs.root_tok, bufs.kv_len, bufs.tok, bufs.parent,
                       bufs.depth, bufs.pos, bufs.mask, node_cand=bufs.node_cand if c.sampled else None,
                       stream=stream)


def run_round(bufs: RoundBuffers, stream=None, write_tree_qkv=None, sm_scale=None, mark=None, B=None, draft=None):
    """Enqueue one round for the first B requests of the buffers (all by default).
    ``draft(bufs, di)`` (optional) is called before the expansion of depth di + 1
    to write that depth's draft logits (the frontier of the previous depth is in
    bufs.f_id[di]); without it the caller has written every depth's beforehand.
    ``write_tree_qkv(bufs)`` (optional) is called after tree_build_mask to write
    the tree nodes' Q (all layers) and K/V (slots kv_len .. kv_len+R-1); without
    it the caller has written them beforehand.  ``mark(i)`` (optional) is called
    at the phase boundaries i = 0..7 (before fusion, after fusion, expansion,
    tree, verify, LM head, accept, compaction)."""
    c = bufs.cfg
    B = c.B if B is None else B
    R = c.R
    s = stream
    mark = mark or (lambda i: None)
    sm_scale = sm_scale if sm_scale is not None else 1.0 / math.sqrt(c.hd)
    mark(0)
    M = B * (c.M // c.B)
    e3.eagle3_fuse(bufs.h[0], bufs.h[1], bufs.h[2], bufs.W_f, None, bufs.g, M, c.d, c.d, c.dt,
                   bufs.fuse_ws, bufs.fuse_ws_bytes, bufs.dev_err, stream=s)
    mark(1)
    for di in range(c.D):
        if draft is not None:
            draft(bufs, di)
        expand_depth(bufs, di, stream=s, B=B)
    mark(2)
    build_tree(bufs, stream=s, B=B)
    mark(3)
    if write_tree_qkv is not None:
        write_tree_qkv(bufs)
    for l in range(c.L):
        e3.tree_verify_attn(bufs.Q[l], bufs.kv[l], bufs.kv_len, bufs.mask, B, R, c.H, c.max_kv_len, sm_scale,
                            bufs.O[l], bufs.lse[l], bufs.dev_err, bufs.ws, bufs.ws_bytes, stream=s)
    mark(4)
    e3.lmhead_logits(bufs.O[c.L - 1], bufs.W_lm, B * R, c.H * c.hd, c.V, bufs.temp_rows, bufs.logits,
                     bufs.row_max, bufs.row_Q, bufs.row_argmax, bufs.dev_err, c.dt, stream=s)
    mark(5)
    if c.sampled:
        e3.spec_accept_sampled(bufs.tok, bufs.parent, bufs.node_cand, B, R, c.D, bufs.logits, bufs.row_max,
                               bufs.row_Q, bufs.row_argmax, c.V, bufs.temp, bufs.q_stats, bufs.cap + 1, bufs.u_acc,
                               bufs.u_bonus, bufs.acc_len, bufs.path, bufs.out_tok, bufs.status, stream=s)
    else:
        e3.spec_accept(bufs.tok, bufs.parent, B, R, c.D, bufs.logits, bufs.row_max, bufs.row_Q, bufs.row_argmax,
                       c.V, bufs.temp, bufs.u_acc, bufs.u_bonus, e3.E3_ACCEPT_TREE_DET, bufs.acc_len, bufs.path,
                       bufs.out_tok, bufs.status, stream=s)
    mark(6)
    e3.kv_compact(bufs.kv, B, bufs.path, bufs.acc_len, c.D, bufs.kv_len, bufs.dev_err, stream=s)
    mark(7)
