"""Oracle side of the decision sweep (tests/test_gpu_decisions.py), run in a spawn
process pool: one request's expansion, tree build and accept/reject under many
uniform sets, from the same tables the GPU side reads.

No torch and no library import here: numpy, the oracle and the seeded uniforms.
"""
import numpy as np

import oracle
from eagle_speculative_decoding_round_gb300 import synth


def frontier_sizes(k, W, D):
    F, out, off = 1, [], 0
    for _ in range(D):
        out.append((F, off))
        off += F * k
        F = min(W, F * k)
    return out, off


def noise_index(b_global, di, f, n_noise):
    """Which noise-table row perturbs frontier row f of request b_global at depth di."""
    return (b_global * 64 + di * 16 + f) % n_noise


def run_request(job):
    """job: dict with the tables' file paths and one request's settings.  Returns the
    candidates, the tree and (acc_len, path, out_tok) under every uniform set."""
    tgt = np.load(job["tgt_path"], mmap_mode="r")
    noise = np.load(job["noise_path"], mmap_mode="r")
    n_tab, n_noise = tgt.shape[0], noise.shape[0]
    k, W, D, N, sampled = job["k"], job["W"], job["D"], job["N"], job["sampled"]
    root, P, T, bg, b = job["root"], job["P"], job["T"], job["b_global"], job["b"]
    sizes, n_cand = frontier_sizes(k, W, D)
    cands = oracle.new_cands(n_cand)
    fid, fsc = np.array([-1], np.int32), np.zeros(1, np.float32)
    qrows = {}
    for di, (F, off) in enumerate(sizes):
        toks = [root if int(f) < 0 else int(cands["tok"][int(f)]) for f in fid[:F]]
        d = np.stack([np.asarray(tgt[t % n_tab]) + np.asarray(noise[noise_index(bg, di, fi, n_noise)])
                      for fi, t in enumerate(toks)]).astype(np.float32)
        if sampled:
            for fi in range(F):
                qrows[int(fid[fi])] = d[fi]
            fid, fsc, _, _ = oracle.expand_sampled(d, k, W, fsc, fid, di + 1, off, cands, job["draw_seed"], b)
        else:
            fid, fsc = oracle.expand(d, k, W, fsc, fid, di + 1, off, cands)
    tree = oracle.build_tree(cands, n_cand, N, root, P)
    R = N + 1
    z = np.ascontiguousarray(np.asarray(tgt)[tree["tok"] % n_tab], np.float32)
    qlog = None
    if sampled:
        qlog = np.zeros_like(z)
        for u in range(R):
            key = -1 if u == 0 else int(tree["node_cand"][u])
            if key in qrows:
                qlog[u] = qrows[key]
    n_u = len(job["uni_seeds"])
    acc = np.zeros(n_u, np.int32)
    path = np.zeros((n_u, D + 1), np.int32)
    out = np.zeros((n_u, D + 1), np.int32)
    for i, us in enumerate(job["uni_seeds"]):
        ua = synth.uniforms(us, synth.PURPOSE_ACCEPT, 1, R, req0=b)[0]
        ub = synth.uniforms(us, synth.PURPOSE_BONUS, 1, R, req0=b)[0]
        if sampled:
            acc[i], path[i], out[i] = oracle.accept_sampled(tree, z, T, qlog, 1.0, ua, ub, D)
        else:
            acc[i], path[i], out[i] = oracle.accept(tree, z, T, ua, ub, D)
    return {"cands": cands, "tree": tree, "acc": acc, "path": path, "out": out}
