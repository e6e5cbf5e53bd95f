"""CPU-side checks of the C ABI: the library loads, exports exactly what
include/eagle3.h declares, and rejects bad arguments on the host (no launch)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "eagle3.h")


@pytest.fixture(scope="module")
def e3():
    from eagle_speculative_decoding_round_gb300 import build
    build.build()
    from eagle_speculative_decoding_round_gb300 import eagle3
    return eagle3


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"E3_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)))


def test_header_declares_the_seven_steps():
    names = declared_functions()
    for n in ["eagle3_fuse", "eagle3_expand", "tree_build_mask", "tree_verify_attn", "lmhead_logits",
              "spec_accept", "kv_compact"]:
        assert n in names


def test_library_exports_every_declared_symbol(e3):
    out = subprocess.run(["nm", "-D", "--defined-only", e3.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, re.M))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(e3.lib(), n)
    assert set(e3.SYMBOLS) == set(declared_functions())
    assert e3.abi_version() == 3
    assert e3.QSTAT_BYTES == 24


def declared_parameter_counts():
    """Function name -> number of parameters, from the declarations in the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"E3_API\s+[\w\s\*]+?\b(\w+)\s*\(([^)]*)\)\s*;", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_lists_match_the_header(e3):
    counts = declared_parameter_counts()
    assert set(counts) == set(declared_functions())
    for name, n in counts.items():
        fn = getattr(e3.lib(), name)
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)


def test_every_entry_point_rejects_null_arguments_without_a_launch(e3):
    """Null pointers (host structs included) and zero sizes: each call returns
    E3_ERR_INVALID_ARG from its host checks and nothing is launched."""
    n0 = e3.launch_count()
    statuses = {}
    for name in e3.SYMBOLS:
        fn = getattr(e3.lib(), name)
        if fn.restype is not ctypes.c_int or not fn.argtypes:  # sizes, messages, counters, version
            continue
        args = []
        for t in fn.argtypes:
            if t is ctypes.c_float:
                args.append(1.0)
            elif t in (ctypes.c_int, ctypes.c_size_t, ctypes.c_uint64):
                args.append(0)
            else:  # device pointers and pointers to host structs
                args.append(None)
        statuses[name] = fn(*args)
    assert statuses and all(v == 1 for v in statuses.values()), statuses
    assert e3.launch_count() == n0


def test_host_validation_rejects_bad_arguments(e3):
    # every call below fails its host checks before touching the device
    with pytest.raises(e3.E3Error) as ei:
        e3.lmhead_logits(0, 0, 1, 1, 1, 0, 0, 0, 0, 0, None, 0, stream=0)
    assert ei.value.status == 1
    with pytest.raises(e3.E3Error) as ei:
        e3.lmhead_logits(8, 8, 0, 1, 1, 8, 8, 8, 8, 8, None, 0, stream=0)  # M = 0
    assert ei.value.status == 2
    cand = e3.make_cand(16, 16, 16, 16, 100)
    with pytest.raises(e3.E3Error) as ei:  # k > E3_MAX_TOPK
        e3.eagle3_expand(16, 1, 1, 1000, 40, 10, 1.0, 16, 16, 1, 0, cand, 16, 16, None, stream=0)
    assert ei.value.status == 2
    with pytest.raises(e3.E3Error) as ei:  # candidates past the capacity
        e3.eagle3_expand(16, 1, 10, 1000, 10, 10, 1.0, 16, 16, 2, 95, cand, 16, 16, None, stream=0)
    assert ei.value.status == 4
    with pytest.raises(e3.E3Error) as ei:  # N > E3_MAX_NODES
        e3.tree_build_mask(e3.make_cand(16, 16, 16, 16, 4000), 1, 4000, 300, 16, 16, 16, 16, 16, 16, 16, stream=0)
    assert ei.value.status == 2
    kv = e3.make_kv_layer(16, 16, 16, 10, 64, 4, 8, 128, e3.E3_BF16)
    with pytest.raises(e3.E3Error) as ei:  # pages cannot hold max_kv_len + R
        e3.tree_verify_attn(16, kv, 16, 16, 1, 61, 32, 250, 0.1, 16, 16, None, 16, 1 << 30, stream=0)
    assert ei.value.status == 4
    bad = e3.make_kv_layer(16, 16, 16, 10, 64, 40, 8, 100, e3.E3_BF16)  # head_dim 100
    with pytest.raises(e3.E3Error) as ei:
        e3.tree_verify_attn(16, bad, 16, 16, 1, 61, 32, 250, 0.1, 16, 16, None, 16, 1 << 30, stream=0)
    assert ei.value.status == 2
    odd = e3.make_kv_layer(16, 16, 16, 10, 64, 40, 8, 128, e3.E3_BF16, 6)  # unknown flag bits
    with pytest.raises(e3.E3Error) as ei:
        e3.tree_verify_attn(16, odd, 16, 16, 1, 61, 32, 250, 0.1, 16, 16, None, 16, 1 << 30, stream=0)
    assert ei.value.status == 1 and "flags" in e3.last_error()
    with pytest.raises(e3.E3Error) as ei:  # unknown accept mode
        e3.spec_accept(*([16] * 2), 1, 15, 3, *([16] * 4), 1000, *([16] * 3), 7, *([16] * 4), stream=0)
    assert ei.value.status == 3
    with pytest.raises(e3.E3Error) as ei:  # sampled mode goes through spec_accept_sampled
        e3.spec_accept(*([16] * 2), 1, 15, 3, *([16] * 4), 1000, *([16] * 3), e3.E3_ACCEPT_SAMPLED, *([16] * 4),
                       stream=0)
    assert ei.value.status == 3 and "spec_accept_sampled" in e3.lib().eagle3_last_error().decode()
    with pytest.raises(e3.E3Error) as ei:  # null q_stats
        e3.eagle3_expand_sampled(16, 1, 1, 1000, 4, 4, 1.0, 16, 16, 1, 0, cand, 16, 16, 5, None, None, stream=0)
    assert ei.value.status == 1
    with pytest.raises(e3.E3Error) as ei:  # vocabulary beyond the draw counter's 24-bit field
        e3.eagle3_expand_sampled(16, 1, 1, 1 << 24, 4, 4, 1.0, 16, 16, 1, 0, cand, 16, 16, 5, 16, None, stream=0)
    assert ei.value.status == 2
    with pytest.raises(e3.E3Error) as ei:  # q_cap out of range
        e3.spec_accept_sampled(16, 16, 16, 1, 15, 3, 16, 16, 16, 16, 1000, 16, 16, 0, 16, 16, 16, 16, 16, 16,
                               stream=0)
    assert ei.value.status == 2
    with pytest.raises(e3.E3Error) as ei:  # too many layers
        e3.kv_compact([kv] * 200, 1, 16, 16, 6, 16, None, stream=0)
    assert ei.value.status == 2
    assert "kv_compact" in e3.lib().eagle3_last_error().decode()


def test_product_path_does_not_reference_the_oracle():
    pkg = os.path.join(ROOT, "eagle_speculative_decoding_round_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "eagle3_oracle" not in text, f


def test_budget_controller_on_the_host(e3):
    """The adaptive tree budget (host code; "Thinking Budget 与 EAGLE-3", 服务端应怎样联合控制):
    raise one level at a time when acceptance is high and stable, not during the
    cool-down, lower on low acceptance or costly drafting, respect the bounds, fall
    back to the baseline on an invalid observation."""
    import numpy as np
    levels = [(6, 2), (14, 3), (30, 4), (60, 6)]
    pol = e3.budget_policy(levels, min_level=0, max_level=2, base_level=1, alpha=0.5, low=0.25, high=0.75,
                           spread=0.25, min_spare=0.2, max_draft_cost=0.5, cooldown=2, warmup=2)
    st = e3.eagle3_budget_init(pol, 3)
    assert [s.level for s in st] == [1, 1, 1]
    hist = []
    for r in range(12):
        acc = [levels[st[0].level][1], 0, levels[st[2].level][1]]  # full, none, full
        hist.append(e3.eagle3_budget_update(pol, st, acc, spare=1.0 if r < 6 else 0.0, draft_cost=0.0))
    lv = np.array(hist)
    assert lv[:, 0].max() == 2 and lv[:, 0].min() >= 1          # capped at max_level
    assert lv[-1, 1] == 0                                        # low acceptance: down to the floor
    assert np.all(np.abs(np.diff(lv, axis=0)) <= 1)              # one level at a time
    for b in range(3):                                           # a change is held through the cool-down
        ch = np.nonzero(np.diff(lv[:, b]))[0]
        assert np.all(np.diff(ch) > pol.cooldown), (b, lv[:, b])
    # no spare verify capacity: no raise (request 2 kept full acceptance after round 6)
    st2 = e3.eagle3_budget_init(pol, 1)
    for r in range(6):
        out = e3.eagle3_budget_update(pol, st2, [levels[st2[0].level][1]], spare=0.0, draft_cost=0.0)
    assert out == [1]
    # costly drafting lowers even a fully accepted request
    for r in range(6):
        out = e3.eagle3_budget_update(pol, st2, [levels[st2[0].level][1]], spare=1.0, draft_cost=0.9)
    assert out == [0]
    # an invalid observation (request finished / failed) resets to the baseline
    out = e3.eagle3_budget_update(pol, st2, [-1], spare=1.0, draft_cost=0.0)
    assert out == [pol.base_level]
    with pytest.raises(e3.E3Error):  # bounds outside the ladder
        e3.eagle3_budget_init(e3.budget_policy(levels, max_level=7), 1)
