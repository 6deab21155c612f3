"""The C-ABI library loads without a GPU, exports every symbol include/moe.h declares, and
its host LRU policy reproduces the oracle's LRU traces bit for bit (CPU only)."""
import os
import re

import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import oracle

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = moe.lib()
    names = declared_functions()
    assert len(names) >= 5
    for n in ["moe_cache_init", "moe_route", "moe_layer_forward", "moe_cache_fill", "moe_stats"]:
        assert n in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert missing == []
    assert sorted(moe.EXPORTS) == names


def test_lru_simulate_matches_oracle_random():
    rng = np.random.default_rng(11)
    for cap in (1, 2, 5, 17, 64):
        n = 4000
        layers = rng.integers(0, 4, n)
        experts = (rng.zipf(1.2, n) - 1) % 40
        kinds = (rng.random(n) < 0.1).astype(np.int32)
        a = moe.lru_simulate(cap, layers, experts, kinds)
        b = oracle.lru_run(cap, layers, experts, kinds)
        assert np.array_equal(a, b), cap


def test_lru_simulate_hand_traces():
    from tests.test_oracle_lru import load_cases
    for case in load_cases():
        acc = np.array(case["acc"], np.int32)
        ev = moe.lru_simulate(case["cap"], acc[:, 1], acc[:, 2], acc[:, 0])
        assert [tuple(r) for r in ev.tolist()] == case["ev"], case["name"]


def test_lru_simulate_rejects_bad_input():
    with pytest.raises(moe.MoeError):
        moe.lru_simulate(0, [0], [0])
    with pytest.raises(moe.MoeError):
        moe.lru_simulate(2, [-1], [0])


def test_init_without_gpu_fails_cleanly():
    """On a machine without a GPU, moe_cache_init returns an error code (no crash)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(moe.MoeError):
        moe.MoeCache(moe.LayerShape(1, 16, 256, 128, 2, 4, 8))


def test_lru_simulate_with_capacity_changes_matches_oracle():
    """The library's host policy and the oracle agree event for event on random sequences
    with capacity changes (kind 2: grow and shrink) mixed into the accesses."""
    rng = np.random.default_rng(21)
    for cap in (1, 3, 8, 30):
        n = 3000
        layers = rng.integers(0, 3, n)
        experts = (rng.zipf(1.3, n) - 1) % 25
        kinds = (rng.random(n) < 0.05).astype(np.int32)
        resize = rng.random(n) < 0.01
        kinds[resize] = 2
        experts[resize] = rng.integers(1, 40, int(resize.sum()))
        a = moe.lru_simulate(cap, layers, experts, kinds)
        b = oracle.lru_run(cap, layers, experts, kinds)
        assert np.array_equal(a, b)
        assert (a[:, 0] == moe.EV_RESIZE_EVICT).any() or cap == 1


def test_lru_simulate_resize_hand_traces():
    from tests.test_oracle_lru import load_cases
    for case in load_cases("lru_resize_traces.txt"):
        acc = np.array(case["acc"], np.int32)
        ev = moe.lru_simulate(case["cap"], acc[:, 1], acc[:, 2], acc[:, 0])
        assert [tuple(r) for r in ev.tolist()] == case["ev"], case["name"]
