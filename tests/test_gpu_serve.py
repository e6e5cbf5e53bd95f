"""The multi-round serving loop with the adaptive draft-tree budget (serve.py), on the
tiny fp32 target: every request's committed tokens over several rounds equal
brute-force sequential greedy decoding of the synthetic target, whatever tree
budgets the controller picked, and the controller moves an accurately drafted
request up the ladder and a badly drafted one down ("Thinking Budget 与 EAGLE-3",
服务端应怎样联合控制: the execution controller changes only the speculative budget,
never the decoded tokens)."""
import numpy as np
import pytest
import torch

from eagle_speculative_decoding_round_gb300 import synth
from roundlib import TinySetup

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rounds", [3, 6])
def test_greedy_serving_loop_equals_sequential_decoding(rounds):
    from eagle_speculative_decoding_round_gb300.serve import Request, ServingLoop
    V, H, KVH, hd, ps = 1024, 4, 4, 64, 64
    base = TinySetup(100)
    # three requests of one model: their own prefixes, drafts of different quality
    setups = []
    for i, (noise, P) in enumerate([(0.02, 128), (4.0, 150), (0.02, 97)]):
        ts = TinySetup(200 + i, P=P, noise=noise)
        ts.tt = base.tt
        ts.prefix = synth.rng(200 + i, "serve_prefix").integers(0, V, P).astype(np.int64)
        setups.append(ts)
    levels = [(2, 1, 2, 2), (6, 2, 2, 1 << 20), (14, 3, 2, 1 << 20)]  # (N, D, k, W), cheapest first
    cap = max(ts.P for ts in setups) + rounds * 4 + 16
    pt, npages = synth.page_table(7, [cap] * len(setups), ps)
    Kc = np.zeros((1, npages, KVH, ps, hd), np.float32)
    Vc = np.zeros_like(Kc)
    for b, ts in enumerate(setups):
        for p, t in enumerate(ts.prefix):
            Kc[0, pt[b, p // ps], :, p % ps] = ts.tt.k(int(t), p)
            Vc[0, pt[b, p // ps], :, p % ps] = ts.tt.v(int(t), p)
    K_all, V_all = torch.from_numpy(Kc).cuda(), torch.from_numpy(Vc).cuda()
    reqs = [Request(rid=b, root_tok=ts.root_tok, kv_len=ts.P, temp=0.0) for b, ts in enumerate(setups)]
    shape = dict(H=H, KVH=KVH, hd=hd, d=H * hd, V=V, L=1, dtype="f32", page_size=ps)
    loop = ServingLoop(shape, levels, (K_all, V_all), torch.from_numpy(pt).cuda(), npages,
                       torch.from_numpy(base.tt.W_lm).cuda(), reqs,
                       policy=dict(base_level=1, alpha=1.0, low=0.3, high=0.9, spread=1.0, cooldown=0, warmup=1),
                       seed=3)
    paths = {}  # (request, candidate id) -> tokens from the request's original root

    def drafter(bufs, rows, di):
        c = bufs.cfg
        F, off = c.frontier_sizes()[0][di]
        fid = bufs.f_id[di][:len(rows), :F].cpu().numpy()
        if di > 0:
            ct, cp = bufs.c_tok.cpu().numpy(), bufs.c_parent.cpu().numpy()
            F0, off0 = c.frontier_sizes()[0][di - 1]
            for j in range(len(rows)):
                for i in range(off0, off0 + F0 * c.k):
                    paths[(rows[j], i)] = paths[(rows[j], int(cp[j, i]))] + [int(ct[j, i])]
        z = np.zeros((len(rows), F, V), np.float32)
        for j, r in enumerate(rows):
            ts, rq = setups[r], reqs[r]
            if di == 0:
                paths[(r, -1)] = [ts.root_tok] + rq.emitted
            for f in range(F):
                z[j, f] = ts.draft_logits(paths[(r, int(fid[j, f]))], int(fid[j, f]) + 1000 * loop.rounds)
        bufs.draft_logits[di][:len(rows)].copy_(torch.from_numpy(z))

    def target(bufs, rows):
        torch.cuda.synchronize()
        tok, pos = bufs.tok.cpu().numpy(), bufs.pos.cpu().numpy()
        K, V_ = K_all[0].cpu().numpy(), V_all[0].cpu().numpy()
        Q = np.zeros((bufs.cfg.B, bufs.cfg.R, H, hd), np.float32)
        for j, r in enumerate(rows):
            ts = setups[r]
            P = reqs[r].kv_len
            for i in range(bufs.cfg.R):
                slot = P + i
                K[pt[r, slot // ps], :, slot % ps] = ts.tt.k(int(tok[j, i]), int(pos[j, i]))
                V_[pt[r, slot // ps], :, slot % ps] = ts.tt.v(int(tok[j, i]), int(pos[j, i]))
                Q[j, i] = ts.tt.q(int(tok[j, i]), int(pos[j, i]))
        K_all[0].copy_(torch.from_numpy(K))
        V_all[0].copy_(torch.from_numpy(V_))
        bufs.Q[0].copy_(torch.from_numpy(Q))

    for _ in range(rounds):
        loop.step(drafter, target)
    for r, (ts, rq) in enumerate(zip(setups, reqs)):
        seq = ts.sequential_greedy(len(rq.emitted))
        assert rq.emitted == seq[1:], (r, rq.levels, rq.accepted)
        assert rq.kv_len == ts.P + len(rq.emitted)
    # the accurate drafters climb, the noisy one stays at the bottom
    assert reqs[0].levels[-1] == 2 and reqs[2].levels[-1] == 2, (reqs[0].levels, reqs[2].levels)
    assert reqs[1].levels[-1] == 0, reqs[1].levels
