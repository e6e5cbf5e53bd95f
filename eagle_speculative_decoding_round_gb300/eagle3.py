"""ctypes binding of libeagle3 (include/eagle3.h): same names, argument
marshalling only.  Every step runs in the library's CUDA kernels; there is no
fallback -- importing this module fails if the library is missing.

Arguments that are device buffers accept a torch CUDA tensor (its data_ptr is
passed) or an int address.  ``stream`` defaults to torch's current stream.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libeagle3.so")

E3_OK = 0
E3_F32, E3_BF16 = 0, 1
E3_DEV_ERR_NONFINITE, E3_DEV_ERR_CAPACITY, E3_DEV_ERR_TIMEOUT = 1, 2, 4
E3_ACCEPT_TREE_DET, E3_ACCEPT_SAMPLED = 0, 1
E3_KV_PREFIX_STABLE = 1
E3_KV_SELFTEST_STALL = 0x40000000  # failure-detection self-test only
STATUS_NAMES = {0: "E3_OK", 1: "E3_ERR_INVALID_ARG", 2: "E3_ERR_SHAPE", 3: "E3_ERR_UNSUPPORTED",
                4: "E3_ERR_CAPACITY", 5: "E3_ERR_NONFINITE", 6: "E3_ERR_CUDA", 7: "E3_ERR_TIMEOUT"}
SYMBOLS = ["eagle3_fuse", "eagle3_fuse_workspace_bytes", "eagle3_fuse_noalloc",
           "eagle3_fuse_noalloc_max_scratch_bytes", "eagle3_expand", "eagle3_expand_sampled", "tree_build_mask",
           "tree_verify_attn", "eagle3_verify_workspace_bytes", "lmhead_logits", "spec_accept",
           "spec_accept_sampled", "kv_compact", "eagle3_draft_step", "eagle3_draft_workspace_bytes",
           "eagle3_budget_init", "eagle3_budget_update", "eagle3_last_error",
           "eagle3_abi_version", "eagle3_launch_count"]
MAX_BUDGET_LEVELS = 16


class E3Error(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class e3_cand(ctypes.Structure):
    _fields_ = [("tok", ctypes.c_void_p), ("parent", ctypes.c_void_p), ("score", ctypes.c_void_p),
                ("depth", ctypes.c_void_p), ("cap", ctypes.c_int)]


class e3_qstat(ctypes.Structure):
    _fields_ = [("row", ctypes.c_void_p), ("Q", ctypes.c_uint64), ("m", ctypes.c_float),
                ("inv_temp", ctypes.c_float)]


QSTAT_BYTES = ctypes.sizeof(e3_qstat)  # bytes of one e3_qstat (24)


class e3_kv_layer(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
                ("n_pages", ctypes.c_int), ("page_size", ctypes.c_int), ("max_pages", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("dt", ctypes.c_int),
                ("flags", ctypes.c_int)]


class e3_drafter(ctypes.Structure):
    _fields_ = [("emb", ctypes.c_void_p), ("W_in", ctypes.c_void_p), ("norm1", ctypes.c_void_p),
                ("W_qkv", ctypes.c_void_p), ("W_o", ctypes.c_void_p), ("norm2", ctypes.c_void_p),
                ("W_gu", ctypes.c_void_p), ("W_down", ctypes.c_void_p), ("norm_f", ctypes.c_void_p),
                ("W_lm", ctypes.c_void_p), ("d", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int), ("V", ctypes.c_int),
                ("rope_base", ctypes.c_float), ("eps", ctypes.c_float)]


class e3_budget_policy(ctypes.Structure):
    _fields_ = [("n_levels", ctypes.c_int), ("nodes", ctypes.c_int * MAX_BUDGET_LEVELS),
                ("depth", ctypes.c_int * MAX_BUDGET_LEVELS), ("min_level", ctypes.c_int), ("max_level", ctypes.c_int),
                ("base_level", ctypes.c_int), ("alpha", ctypes.c_float), ("low", ctypes.c_float),
                ("high", ctypes.c_float), ("spread", ctypes.c_float), ("min_spare", ctypes.c_float),
                ("max_draft_cost", ctypes.c_float), ("cooldown", ctypes.c_int), ("warmup", ctypes.c_int)]


class e3_budget_state(ctypes.Structure):
    _fields_ = [("level", ctypes.c_int32), ("hold", ctypes.c_int32), ("rounds", ctypes.c_int32),
                ("mean", ctypes.c_float), ("dev", ctypes.c_float)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libeagle3.so is not built ({LIB_PATH}); run "
                          "eagle_speculative_decoding_round_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    sig = {
        "eagle3_fuse": (I, [P, P, P, P, P, P, I, I, I, I, P, S, P, P]),
        "eagle3_fuse_workspace_bytes": (S, [I, I, I, I]),
        "eagle3_fuse_noalloc": (I, [P, P, P, P, P, P, I, I, I, I, P, P]),
        "eagle3_fuse_noalloc_max_scratch_bytes": (S, []),
        "eagle3_expand": (I, [P, I, I, I, I, I, F, P, P, I, I, ctypes.POINTER(e3_cand), P, P, P, P]),
        "eagle3_expand_sampled": (I, [P, I, I, I, I, I, F, P, P, I, I, ctypes.POINTER(e3_cand), P, P,
                                      ctypes.c_uint64, P, P, P]),
        "tree_build_mask": (I, [ctypes.POINTER(e3_cand), I, I, I, P, P, P, P, P, P, P, P, P]),
        "tree_verify_attn": (I, [P, ctypes.POINTER(e3_kv_layer), P, P, I, I, I, I, F, P, P, P, P, S, P]),
        "eagle3_verify_workspace_bytes": (S, [I, I, I, I, I, I, I]),
        "lmhead_logits": (I, [P, P, I, I, I, P, P, P, P, P, P, I, P]),
        "spec_accept": (I, [P, P, I, I, I, P, P, P, P, I, P, P, P, I, P, P, P, P, P]),
        "spec_accept_sampled": (I, [P, P, P, I, I, I, P, P, P, P, I, P, P, I, P, P, P, P, P, P, P]),
        "kv_compact": (I, [ctypes.POINTER(e3_kv_layer), I, I, P, P, I, P, P, P]),
        "eagle3_draft_step": (I, [ctypes.POINTER(e3_drafter), ctypes.POINTER(e3_kv_layer), P, I, I, I, I, P, I, I,
                                  P, I, I, ctypes.POINTER(e3_cand), P, P, P, P, P, P, P, P, P, S, P, P]),
        "eagle3_draft_workspace_bytes": (S, [ctypes.POINTER(e3_drafter), I, I, I, I]),
        "eagle3_budget_init": (I, [ctypes.POINTER(e3_budget_policy), P, I]),
        "eagle3_budget_update": (I, [ctypes.POINTER(e3_budget_policy), P, I, P, F, F, P]),
        "eagle3_last_error": (ctypes.c_char_p, []),
        "eagle3_abi_version": (I, []),
        "eagle3_launch_count": (ctypes.c_uint64, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def ptr(x) -> int | None:
    """Device address of a torch tensor (or pass an int / None through)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int):
    if st != E3_OK:
        raise E3Error(fn, st, _lib.eagle3_last_error().decode())


def make_cand(tok, parent, score, depth, cap: int) -> e3_cand:
    return e3_cand(ptr(tok), ptr(parent), ptr(score), ptr(depth), cap)


def make_kv_layer(k, v, page_table, n_pages, page_size, max_pages, n_kv_heads, head_dim, dt, flags=0) -> e3_kv_layer:
    return e3_kv_layer(ptr(k), ptr(v), ptr(page_table), n_pages, page_size, max_pages, n_kv_heads, head_dim, dt,
                       flags)


def abi_version() -> int:
    return _lib.eagle3_abi_version()


def last_error() -> str:
    """The calling thread's last error message ("" after a call that succeeded)."""
    return _lib.eagle3_last_error().decode()


def launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(_lib.eagle3_launch_count())


def eagle3_fuse_workspace_bytes(M, d, d_out, dt) -> int:
    return int(_lib.eagle3_fuse_workspace_bytes(M, d, d_out, dt))


def eagle3_fuse(h_low, h_mid, h_high, W_f, bias, g, M, d, d_out, dt, ws=None, ws_bytes=0, dev_err=None,
                stream=None):
    _check("eagle3_fuse", _lib.eagle3_fuse(ptr(h_low), ptr(h_mid), ptr(h_high), ptr(W_f), ptr(bias), ptr(g),
                                           M, d, d_out, dt, ptr(ws), ws_bytes, ptr(dev_err), _stream(stream)))


def eagle3_fuse_noalloc(h_low, h_mid, h_high, W_f, bias, g, M, d, d_out, dt, dev_err=None, stream=None):
    """eagle3_fuse without caller scratch (fixed library array; see include/eagle3.h)."""
    _check("eagle3_fuse_noalloc", _lib.eagle3_fuse_noalloc(ptr(h_low), ptr(h_mid), ptr(h_high), ptr(W_f), ptr(bias),
                                                           ptr(g), M, d, d_out, dt, ptr(dev_err), _stream(stream)))


def eagle3_fuse_noalloc_max_scratch_bytes() -> int:
    return int(_lib.eagle3_fuse_noalloc_max_scratch_bytes())


def eagle3_expand(draft_logits, B, F, V, k, W, inv_temp, parent_score, parent_id, depth, cand_offset,
                  cands: e3_cand, next_id, next_score, dev_err=None, stream=None):
    _check("eagle3_expand", _lib.eagle3_expand(ptr(draft_logits), B, F, V, k, W, inv_temp, ptr(parent_score),
                                               ptr(parent_id), depth, cand_offset, ctypes.byref(cands),
                                               ptr(next_id), ptr(next_score), ptr(dev_err), _stream(stream)))


def eagle3_expand_sampled(draft_logits, B, F, V, k, W, inv_temp, parent_score, parent_id, depth, cand_offset,
                          cands: e3_cand, next_id, next_score, seed, q_stats, dev_err=None, stream=None):
    """q_stats: device buffer of B * (1 + cands.cap) * QSTAT_BYTES bytes."""
    _check("eagle3_expand_sampled",
           _lib.eagle3_expand_sampled(ptr(draft_logits), B, F, V, k, W, inv_temp, ptr(parent_score), ptr(parent_id),
                                      depth, cand_offset, ctypes.byref(cands), ptr(next_id), ptr(next_score),
                                      int(seed) & (2 ** 64 - 1), ptr(q_stats), ptr(dev_err), _stream(stream)))


def tree_build_mask(cands: e3_cand, B, n_cand, N, root_tok, kv_len, tok, parent, depth, pos, mask, node_cand=None,
                    stream=None):
    _check("tree_build_mask", _lib.tree_build_mask(ctypes.byref(cands), B, n_cand, N, ptr(root_tok), ptr(kv_len),
                                                   ptr(tok), ptr(parent), ptr(depth), ptr(pos), ptr(mask),
                                                   ptr(node_cand), _stream(stream)))


def eagle3_verify_workspace_bytes(B, R, n_q_heads, n_kv_heads, head_dim, max_kv_len, dt) -> int:
    return int(_lib.eagle3_verify_workspace_bytes(B, R, n_q_heads, n_kv_heads, head_dim, max_kv_len, dt))


def tree_verify_attn(Q, kv: e3_kv_layer, kv_len, mask, B, R, n_q_heads, max_kv_len, sm_scale, O, lse,
                     dev_err=None, ws=None, ws_bytes=0, stream=None):
    _check("tree_verify_attn", _lib.tree_verify_attn(ptr(Q), ctypes.byref(kv), ptr(kv_len), ptr(mask), B, R,
                                                     n_q_heads, max_kv_len, sm_scale, ptr(O), ptr(lse),
                                                     ptr(dev_err), ptr(ws), ws_bytes, _stream(stream)))


def lmhead_logits(h, W_lm, M, d, V, temp_per_row, logits, row_max, row_Q, row_argmax, dev_err, dt, stream=None):
    _check("lmhead_logits", _lib.lmhead_logits(ptr(h), ptr(W_lm), M, d, V, ptr(temp_per_row), ptr(logits),
                                               ptr(row_max), ptr(row_Q), ptr(row_argmax), ptr(dev_err), dt,
                                               _stream(stream)))


def spec_accept(tok, parent, B, R, D, logits, row_max, row_Q, row_argmax, V, temp, u_acc, u_bonus, mode,
                acc_len, path, out_tok, status, stream=None):
    _check("spec_accept", _lib.spec_accept(ptr(tok), ptr(parent), B, R, D, ptr(logits), ptr(row_max), ptr(row_Q),
                                           ptr(row_argmax), V, ptr(temp), ptr(u_acc), ptr(u_bonus), mode,
                                           ptr(acc_len), ptr(path), ptr(out_tok), ptr(status), _stream(stream)))


def spec_accept_sampled(tok, parent, node_cand, B, R, D, logits, row_max, row_Q, row_argmax, V, temp, q_stats, q_cap,
                        u_acc, u_bonus, acc_len, path, out_tok, status, stream=None):
    _check("spec_accept_sampled",
           _lib.spec_accept_sampled(ptr(tok), ptr(parent), ptr(node_cand), B, R, D, ptr(logits), ptr(row_max),
                                    ptr(row_Q), ptr(row_argmax), V, ptr(temp), ptr(q_stats), q_cap, ptr(u_acc),
                                    ptr(u_bonus), ptr(acc_len), ptr(path), ptr(out_tok), ptr(status),
                                    _stream(stream)))


def kv_compact(layers, B, path, acc_len, D, kv_len, dev_err=None, stream=None):
    arr = (e3_kv_layer * len(layers))(*layers)
    _check("kv_compact", _lib.kv_compact(arr, len(layers), B, ptr(path), ptr(acc_len), D, ptr(kv_len),
                                         ptr(dev_err), _stream(stream)))


def budget_policy(levels, min_level=0, max_level=None, base_level=0, alpha=0.5, low=0.25, high=0.75, spread=0.25,
                  min_spare=0.0, max_draft_cost=1.0, cooldown=2, warmup=2) -> e3_budget_policy:
    """levels: [(N, D), ...] cheapest first."""
    p = e3_budget_policy()
    p.n_levels = len(levels)
    for i, (n, d) in enumerate(levels):
        p.nodes[i], p.depth[i] = n, d
    p.min_level, p.max_level = min_level, len(levels) - 1 if max_level is None else max_level
    p.base_level, p.alpha, p.low, p.high, p.spread = base_level, alpha, low, high, spread
    p.min_spare, p.max_draft_cost, p.cooldown, p.warmup = min_spare, max_draft_cost, cooldown, warmup
    return p


def eagle3_budget_init(pol: e3_budget_policy, B: int):
    """A fresh host state array of B entries at the baseline."""
    st = (e3_budget_state * B)()
    _check("eagle3_budget_init", _lib.eagle3_budget_init(ctypes.byref(pol), ctypes.addressof(st), B))
    return st


def eagle3_budget_update(pol: e3_budget_policy, st, acc_len, spare=1.0, draft_cost=0.0):
    """acc_len: host int sequence of len(st); returns the new levels (list)."""
    import numpy as np
    B = len(st)
    a = np.ascontiguousarray(np.asarray(acc_len, np.int32))
    out = np.zeros(B, np.int32)
    _check("eagle3_budget_update", _lib.eagle3_budget_update(ctypes.byref(pol), ctypes.addressof(st), B,
                                                             a.ctypes.data, float(spare), float(draft_cost),
                                                             out.ctypes.data))
    return out.tolist()


def make_drafter(emb, W_in, norm1, W_qkv, W_o, norm2, W_gu, W_down, norm_f, W_lm, d, n_heads, n_kv_heads, head_dim,
                 ffn, V, rope_base=10000.0, eps=1e-6) -> e3_drafter:
    return e3_drafter(ptr(emb), ptr(W_in), ptr(norm1), ptr(W_qkv), ptr(W_o), ptr(norm2), ptr(W_gu), ptr(W_down),
                      ptr(norm_f), ptr(W_lm), d, n_heads, n_kv_heads, head_dim, ffn, V, rope_base, eps)


def eagle3_draft_workspace_bytes(drafter: e3_drafter, B, F_max, R_slots, max_kv_len) -> int:
    return int(_lib.eagle3_draft_workspace_bytes(ctypes.byref(drafter), B, F_max, R_slots, max_kv_len))


def eagle3_draft_step(drafter: e3_drafter, kv: e3_kv_layer, kv_len, max_kv_len, B, depth, F, frontier, slot_base,
                      F_prev, frontier_prev, slot_base_prev, R_slots, cands: e3_cand, root_tok, g, a_slots, mask,
                      logits, row_max, row_Q, row_argmax, ws, ws_bytes, dev_err=None, stream=None):
    _check("eagle3_draft_step",
           _lib.eagle3_draft_step(ctypes.byref(drafter), ctypes.byref(kv), ptr(kv_len), max_kv_len, B, depth, F,
                                  ptr(frontier), slot_base, F_prev, ptr(frontier_prev), slot_base_prev, R_slots,
                                  ctypes.byref(cands), ptr(root_tok), ptr(g), ptr(a_slots), ptr(mask), ptr(logits),
                                  ptr(row_max), ptr(row_Q), ptr(row_argmax), ptr(ws), ws_bytes, ptr(dev_err),
                                  _stream(stream)))
