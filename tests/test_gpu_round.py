"""A whole round on the tiny fp32 configuration, through the C ABI:
greedy output equals brute-force sequential decoding of the synthetic target,
and every intermediate equals the oracle's round on the same inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_round_gb300 import synth
from gpu_util import assert_close, host, to_dev
from roundlib import TinySetup
from test_oracle_round import oracle_round

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from eagle_speculative_decoding_round_gb300 import eagle3 as e3
    from eagle_speculative_decoding_round_gb300.round import RoundBuffers, RoundConfig, run_round


def gpu_round(ts: TinySetup, T: float):
    cfg = RoundConfig(B=1, N=ts.n_cand, D=ts.D, k=ts.k, W=ts.W, H=ts.H, KVH=ts.KVH, hd=ts.hd, d=ts.H * ts.hd,
                      V=ts.V, L=1, max_kv_len=ts.P, dtype="f32", page_size=ts.page_size, M_fuse=3)
    R = cfg.R
    pt, Kc, Vc = ts.make_cache(R)
    bufs = RoundBuffers(cfg, torch.from_numpy(pt), Kc.shape[0])
    bufs.K[0].copy_(torch.from_numpy(Kc))
    bufs.Vc[0].copy_(torch.from_numpy(Vc))
    bufs.kv_len.fill_(ts.P)
    bufs.root_tok.fill_(ts.root_tok)
    bufs.W_lm.copy_(torch.from_numpy(ts.tt.W_lm))
    bufs.set_temperature(torch.full((1,), T))
    for t in bufs.h:
        t.copy_(torch.from_numpy(synth.normal(ts.seed, "fuse_h", (cfg.M, cfg.d))))
    bufs.W_f.copy_(torch.from_numpy(synth.normal(ts.seed, "fuse_W", (cfg.d, 3 * cfg.d))))
    bufs.u_acc.copy_(torch.from_numpy(synth.uniforms(ts.seed, synth.PURPOSE_ACCEPT, 1, R).view(np.int32)))
    bufs.u_bonus.copy_(torch.from_numpy(synth.uniforms(ts.seed, synth.PURPOSE_BONUS, 1, R).view(np.int32)))
    # draft logits depend on the frontier chosen at the previous depth: expand one
    # depth at a time on the GPU and compute the next depth's draft logits on the host
    sizes, n_cand = cfg.frontier_sizes()
    fpath = {-1: [ts.root_tok]}
    for di, (F, off) in enumerate(sizes):
        fid = host(bufs.f_id[di])[0][:F]
        z = np.stack([ts.draft_logits(fpath[int(f)], int(f)) for f in fid])[None]
        bufs.draft_logits[di].copy_(torch.from_numpy(z))
        e3.eagle3_expand(bufs.draft_logits[di], 1, F, cfg.V, cfg.k, cfg.W, 1.0, bufs.f_score[di], bufs.f_id[di],
                         di + 1, off, bufs.cand, bufs.f_id[di + 1], bufs.f_score[di + 1], bufs.dev_err)
        torch.cuda.synchronize()
        ct, cp = host(bufs.c_tok)[0], host(bufs.c_parent)[0]
        for i in range(off, off + F * cfg.k):
            fpath[i] = fpath[int(cp[i])] + [int(ct[i])]

    # the round proper, with the draft logits now in place
    def write_qkv(b):
        torch.cuda.synchronize()
        tree = {"tok": host(b.tok)[0], "pos": host(b.pos)[0]}
        K2, V2 = host(b.K[0]), host(b.Vc[0])
        ts.write_tree_kv(K2, V2, pt, tree)
        b.K[0].copy_(torch.from_numpy(K2))
        b.Vc[0].copy_(torch.from_numpy(V2))
        b.Q[0].copy_(torch.from_numpy(ts.tree_q(tree)))

    run_round(bufs, write_tree_qkv=write_qkv)
    torch.cuda.synchronize()
    return bufs, pt


@pytest.mark.parametrize("seed,T", [(0, 0.0), (1, 0.0), (2, 0.0), (3, 1.0), (4, 1.0)])
def test_tiny_round_matches_oracle_and_sequential(seed, T):
    ts = TinySetup(seed, noise=0.02 if seed % 2 == 0 else 3.0)
    bufs, pt = gpu_round(ts, T)
    assert int(bufs.dev_err.item()) == 0
    ref = oracle_round(ts, T)
    # tree: bit-exact
    for x in ("tok", "parent", "depth", "pos"):
        assert np.array_equal(host(bufs.__dict__[x])[0], ref["tree"][x]), x
    assert np.array_equal(host(bufs.mask)[0].view(np.uint64), ref["tree"]["mask"])
    # logits within fp32 tolerance
    assert_close(host(bufs.logits), ref["logits"], 1e-5, "logits")
    acc = int(host(bufs.acc_len)[0])
    out = host(bufs.out_tok)[0]
    # decisions: bit-exact given the GPU's own logits
    a2, p2, o2 = oracle.accept(ref["tree"], host(bufs.logits), T, synth.uniforms(seed, 1, 1, ts.n_cand + 1)[0],
                               synth.uniforms(seed, 2, 1, ts.n_cand + 1)[0], ts.D)
    assert acc == a2 and np.array_equal(out, o2) and np.array_equal(host(bufs.path)[0], p2)
    assert int(host(bufs.kv_len)[0]) == ts.P + 1 + acc
    if T == 0.0:
        seq = ts.sequential_greedy(acc + 1)
        assert list(out[:acc + 1]) == seq[1:acc + 2]
        ps = ts.page_size
        K = host(bufs.K[0])
        for j in range(acc + 1):
            pos = ts.P + j
            assert np.array_equal(K[pt[0, pos // ps], :, pos % ps], ts.tt.k(seq[j], pos))
        if seed == 0:
            assert acc == ts.D
    # the fusion ran on the same stream: check it too
    ref_g = oracle.fuse(*(host(t) for t in bufs.h), host(bufs.W_f))
    assert_close(host(bufs.g), ref_g, 1e-5, "fuse")
