"""The drafter's decoder step on the GPU (eagle3_draft_step) against the oracle's
fp64 step (oracle/draft.py), depth by depth over a tree the library grows itself
(eagle3_expand on the step's own draft logits): every frontier row's draft logits
and output a within the bf16 tolerance, with the row's context being the drafter's
prefix cache plus the K/V its ancestors produced ("论文专题讲解：EAGLE-3", 推理流程：
多层特征融合 + 单层 draft decoder; "SpecForge…", 第二步为什么没有"正确隐藏状态"可用
and 从序列到动态草稿树).  The oracle follows the GPU's tree (the same tokens and
parents), computing every step from its own fp64 values."""
import math

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_round_gb300 import synth
from gpu_util import assert_close
from oracle import draft as dr

pytestmark = pytest.mark.gpu


def bf16_pair(shape, std, gen, mean=0.0):
    t = (torch.randn(shape, generator=gen, device="cuda") * std + mean).to(torch.bfloat16)
    return t, t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("cfg", [
    dict(B=2, d=256, H=4, KVH=2, hd=64, ffn=512, V=1024, P=[70, 133], k=2, W=3, D=4),       # small, GQA 2
    dict(B=1, d=4096, H=32, KVH=8, hd=128, ffn=14336, V=32768, P=[2048], k=10, W=10, D=3),  # 8B-shaped layer
])
def test_draft_steps_match_the_oracle(cfg):
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3
    B, d, H, KVH, hd, ffn, V = (cfg[x] for x in ("B", "d", "H", "KVH", "hd", "ffn", "V"))
    k, W, D, P = cfg["k"], cfg["W"], cfg["D"], cfg["P"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(17)
    s = 0.02
    wt = {}
    W_ = {}
    for name, shape, std, mean in [("emb", (V, d), 1.0, 0.0), ("W_in", (d, 2 * d), s, 0.0), ("norm1", (d,), s, 1.0),
                                   ("W_qkv", ((H + 2 * KVH) * hd, d), s, 0.0), ("W_o", (d, H * hd), s, 0.0),
                                   ("norm2", (d,), s, 1.0), ("W_gu", (2 * ffn, d), s, 0.0), ("W_down", (d, ffn), s, 0.0),
                                   ("norm_f", (d,), s, 1.0), ("W_lm", (V, d), 1.0, 0.0)]:
        t, h = bf16_pair(shape, std, gen, mean)
        if name.startswith("norm"):
            t = t.float()  # norm weights are fp32 (values on the bf16 grid)
        W_[name], wt[name] = t, h
    drafter = e3.make_drafter(W_["emb"], W_["W_in"], W_["norm1"], W_["W_qkv"], W_["W_o"], W_["norm2"], W_["W_gu"],
                              W_["W_down"], W_["norm_f"], W_["W_lm"], d, H, KVH, hd, ffn, V)
    Wt = {"emb": wt["emb"], "W_in": wt["W_in"], "norm1": wt["norm1"], "Wq": wt["W_qkv"][:H * hd],
          "Wk": wt["W_qkv"][H * hd:(H + KVH) * hd], "Wv": wt["W_qkv"][(H + KVH) * hd:], "Wo": wt["W_o"],
          "norm2": wt["norm2"], "Wg": wt["W_gu"][:ffn], "Wu": wt["W_gu"][ffn:], "Wd": wt["W_down"],
          "normf": wt["norm_f"], "lm": wt["W_lm"], "H": H, "KVH": KVH, "hd": hd}
    # frontier sizes and tree slots per depth
    sizes, off, Fd = [], 0, 1
    for _ in range(D):
        sizes.append((Fd, off))
        off += Fd * k
        Fd = min(W, Fd * k)
    n_cand = off
    bases = np.cumsum([0] + [F for F, _ in sizes])
    R_slots = int(bases[-1])
    # the drafter's paged cache: the committed prefix (random), room for the tree slots
    ps = 64
    pt, npages = synth.page_table(5, [p + R_slots for p in P], ps)
    Kc, Kh = bf16_pair((npages, KVH, ps, hd), 1.0, gen)
    Vc, Vh = bf16_pair((npages, KVH, ps, hd), 1.0, gen)
    ptt = torch.from_numpy(pt).cuda()
    kv = e3.make_kv_layer(Kc, Vc, ptt, npages, ps, pt.shape[1], KVH, hd, e3.E3_BF16)
    kv_len = torch.tensor(P, dtype=torch.int32, device="cuda")
    maxP = max(P)
    g, gh = bf16_pair((B, d), 1.0, gen)
    roots = np.random.default_rng(3).integers(0, V, B).astype(np.int32)
    root_t = torch.from_numpy(roots).cuda()
    i32 = dict(dtype=torch.int32, device="cuda")
    c_tok, c_par = torch.full((B, n_cand), -1, **i32), torch.full((B, n_cand), -1, **i32)
    c_score, c_dep = torch.zeros((B, n_cand), device="cuda"), torch.zeros((B, n_cand), **i32)
    cands = e3.make_cand(c_tok, c_par, c_score, c_dep, n_cand)
    f_id = [torch.full((B, 1), -1, **i32)] + [torch.empty((B, min(W, F * k)), **i32) for F, _ in sizes]
    f_sc = [torch.zeros((B, 1), device="cuda")] + [torch.empty((B, min(W, F * k)), device="cuda") for F, _ in sizes]
    a_slots = torch.zeros((B, R_slots, d), device="cuda")
    mask = torch.zeros((B, R_slots, (R_slots + 63) // 64), dtype=torch.int64, device="cuda")
    Fmax = max(F for F, _ in sizes)
    wsb = e3.eagle3_draft_workspace_bytes(drafter, B, Fmax, R_slots, maxP)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, **i32)

    # oracle state per request: the prefix K/V, and per node (candidate, root -1) its a, k, v, token, parent
    Kpre = [np.stack([Kh[pt[b, t // ps], :, t % ps] for t in range(P[b])]) for b in range(B)]
    Vpre = [np.stack([Vh[pt[b, t // ps], :, t % ps] for t in range(P[b])]) for b in range(B)]
    a_of, kv_of = [dict() for _ in range(B)], [dict() for _ in range(B)]
    for di, (F, off) in enumerate(sizes):
        t = di + 1
        logits = torch.empty((B, F, V), device="cuda")
        rmax, rQ, ram = (torch.empty(B * F, device="cuda"), torch.empty(B * F, dtype=torch.int64, device="cuda"),
                         torch.empty(B * F, **i32))
        prev = f_id[di - 1] if di > 0 else f_id[0]
        e3.eagle3_draft_step(drafter, kv, kv_len, maxP, B, t, F, f_id[di], int(bases[di]),
                             prev.shape[1] if di > 0 else 0, prev if di > 0 else None, int(bases[di - 1]) if di else 0,
                             R_slots, cands, root_t, g, a_slots, mask, logits, rmax, rQ, ram, ws, wsb, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"device error at depth {t}"
        # the oracle's step on the same rows
        fid = f_id[di].cpu().numpy()[:, :F]
        ct, cp = c_tok.cpu().numpy(), c_par.cpu().numpy()
        z_gpu, a_gpu = logits.cpu().numpy(), a_slots.cpu().numpy()
        for b in range(B):
            rows = [int(u) for u in fid[b]]
            toks = [int(roots[b]) if u < 0 else int(ct[b, u]) for u in rows]
            h_in = np.stack([gh[b] if u < 0 else a_of[b][int(cp[b, u])] for u in rows])
            ctx = []
            for u in rows:
                anc, x = [], u
                while x >= 0:
                    x = int(cp[b, x])
                    anc.append(x)
                anc = anc[::-1]  # root first
                ctx.append((np.concatenate([Kpre[b]] + [kv_of[b][x][0][None] for x in anc], 0),
                            np.concatenate([Vpre[b]] + [kv_of[b][x][1][None] for x in anc], 0)))
            a, kk, vv, z = dr.draft_step(Wt, h_in, toks, [P[b] + t - 1] * F, ctx)
            for i, u in enumerate(rows):
                a_of[b][u], kv_of[b][u] = a[i], (kk[i], vv[i])
            assert_close(z_gpu[b], z, 2e-2, f"draft logits, depth {t}, request {b}")
            assert_close(a_gpu[b, bases[di]:bases[di] + F], a, 2e-2, f"a, depth {t}, request {b}")
        # the next frontier: the library's expansion of these draft logits
        e3.eagle3_expand(logits, B, F, V, k, W, 1.0, f_sc[di], f_id[di], t, off, cands, f_id[di + 1], f_sc[di + 1],
                         err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
