"""Test helpers: the tiny synthetic target, brute-force sequential decoding and a
whole round driven through the oracle.  Used by the oracle pins and by the GPU
round test (which drives the same round through the C ABI instead)."""
import math

import numpy as np
import torch
import torch.nn.functional as F

from eagle_speculative_decoding_round_gb300 import synth


class TinySetup:
    """Tiny fp32 single-layer target: d = 256 = 4 heads x 64, vocab 1024, batch 1,
    prefix 128 tokens, tree depth 3, top-k 2 (14 nodes)."""

    def __init__(self, seed, V=1024, H=4, KVH=4, hd=64, P=128, D=3, k=2, W=1 << 20,
                 page_size=64, noise=1.0):
        self.seed, self.V, self.H, self.KVH, self.hd, self.P = seed, V, H, KVH, hd, P
        self.D, self.k, self.W, self.noise = D, k, W, noise
        self.tt = synth.TinyTarget(seed, V, H, KVH, hd, std=1.0, lm_std=0.5)
        rng = synth.rng(seed, "prefix")
        self.prefix = rng.integers(0, V, P).astype(np.int64)
        self.root_tok = int(rng.integers(0, V))
        self.scale = 1.0 / math.sqrt(hd)
        n_cand = 0
        F_ = 1
        for d in range(D):
            n_cand += F_ * k
            F_ = min(W, F_ * k)
        self.n_cand = n_cand
        self.N = n_cand if W >= (1 << 20) else None
        self.page_size = page_size

    # ---- brute force: the target decoding one token at a time -------------
    def logits_after(self, toks):
        """fp64 target logits after feeding toks (root first) at positions P, P+1, ..."""
        Ks = [self.tt.k(int(t), p) for p, t in enumerate(self.prefix)]
        Vs = [self.tt.v(int(t), p) for p, t in enumerate(self.prefix)]
        for s, t in enumerate(toks):
            Ks.append(self.tt.k(int(t), self.P + s))
            Vs.append(self.tt.v(int(t), self.P + s))
        p = self.P + len(toks) - 1
        q = torch.from_numpy(self.tt.q(int(toks[-1]), p).astype(np.float64))[:, None, :]  # [H,1,hd]
        k = torch.from_numpy(np.stack(Ks).astype(np.float64)).permute(1, 0, 2)
        v = torch.from_numpy(np.stack(Vs).astype(np.float64)).permute(1, 0, 2)
        g = self.H // self.KVH
        k = k.repeat_interleave(g, dim=0)
        v = v.repeat_interleave(g, dim=0)
        o = F.scaled_dot_product_attention(q, k, v, scale=self.scale)[:, 0, :].reshape(-1).numpy()
        return self.tt.W_lm.astype(np.float64) @ o

    def sequential_greedy(self, n):
        toks = [self.root_tok]
        for _ in range(n):
            z = self.logits_after(toks).astype(np.float32)
            toks.append(int(np.argmax(z)))
        return toks

    # ---- draft logits: target logits along the node's path + noise ----------
    def draft_logits(self, path_toks, cand_id):
        z = self.logits_after(path_toks)
        n = synth.normal(self.seed, f"draftnoise{cand_id}", (self.V,), self.noise)
        return (z + n).astype(np.float32)

    # ---- paged cache with prefix KV (and room for the tree) -----------------
    def make_cache(self, R):
        pt, npages = synth.page_table(self.seed, [self.P + R], self.page_size)
        Kc = np.zeros((npages, self.KVH, self.page_size, self.hd), np.float32)
        Vc = np.zeros_like(Kc)
        for p, t in enumerate(self.prefix):
            Kc[pt[0, p // self.page_size], :, p % self.page_size] = self.tt.k(int(t), p)
            Vc[pt[0, p // self.page_size], :, p % self.page_size] = self.tt.v(int(t), p)
        return pt, Kc, Vc

    def write_tree_kv(self, Kc, Vc, pt, tree):
        """Node i's K/V (rotary position pos[i] = P + depth) go to logical slot P + i."""
        ps = self.page_size
        for i, (t, pos) in enumerate(zip(tree["tok"], tree["pos"])):
            slot = self.P + i
            Kc[pt[0, slot // ps], :, slot % ps] = self.tt.k(int(t), int(pos))
            Vc[pt[0, slot // ps], :, slot % ps] = self.tt.v(int(t), int(pos))

    def tree_q(self, tree):
        return np.stack([self.tt.q(int(t), int(p)) for t, p in zip(tree["tok"], tree["pos"])])[None]
