"""Helpers shared by the GPU parity tests."""
import numpy as np
import torch

from eagle_speculative_decoding_round_gb300 import synth


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def bf16_dev(a32: np.ndarray):
    """fp32 array -> bf16 CUDA tensor (round to nearest even) and the rounded fp32 values."""
    r = synth.to_bf16_f32(a32)
    return torch.from_numpy(r).to(torch.bfloat16).cuda(), r


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        t = t.float()
    return t.cpu().numpy()


def assert_close(got, ref, tol, what=""):
    """Norm-wise relative error: max|got - ref| <= tol * max|ref|."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), what
    scale = max(np.abs(ref).max(), 1e-30)
    err = np.abs(got - ref).max() / scale
    assert err <= tol, f"{what}: rel err {err:.3e} > {tol:.1e}"
    return err


def random_tree(rng, R, D):
    """A flattened tree with parent[i] < i and depth <= D (node 0 = root)."""
    parent = np.full(R, -1, np.int32)
    depth = np.zeros(R, np.int32)
    for i in range(1, R):
        while True:
            p = int(rng.integers(0, i))
            if depth[p] < D:
                break
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent, depth


def tree_tokens(rng, parent, logits, spread=3):
    """Children carry distinct tokens, mostly among the parent's top logits."""
    R, V = logits.shape
    tok = np.zeros(R, np.int32)
    for u in range(R):
        kids = [c for c in range(R) if parent[c] == u]
        if not kids:
            continue
        order = np.argsort(-logits[u], kind="stable")[:len(kids) + spread]
        pick = rng.permutation(order)[:len(kids)] if rng.random() < 0.5 else order[:len(kids)]
        for c, t in zip(kids, pick):
            tok[c] = t
    return tok


def kv_paged(seed, lens, R, KVH, hd, page_size, std=1.0, dtype="bf16"):
    """Paged caches holding prefix + tree slots for each request (values as fp32 on the
    bf16 grid when dtype is bf16)."""
    pt, npages = synth.page_table(seed, [n + R for n in lens], page_size)
    K = synth.normal(seed, "K", (npages, KVH, page_size, hd), std)
    V = synth.normal(seed, "V", (npages, KVH, page_size, hd), std)
    if dtype == "bf16":
        K = synth.to_bf16_f32(K)
        V = synth.to_bf16_f32(V)
    return pt, npages, K, V
