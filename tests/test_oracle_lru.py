"""Pins for the oracle's shared LRU over whole (layer, expert) entries (CPU).

Hand-traced sequences (tests/golden/lru_hand_traces.txt), hand-traced capacity changes
(tests/golden/lru_resize_traces.txt), LRU's inclusion property (a stack algorithm: with one
more slot the hit set can only grow), and closed-form counts.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
KIND = {"HIT": 0, "FILL": 1, "PFILL": 2, "PHIT": 3, "REVICT": 4}


def load_cases(name="lru_hand_traces.txt"):
    cases, cur = [], None
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("case"):
            _, name, _, cap = line.split()
            cur = {"name": name, "cap": int(cap), "acc": [], "ev": []}
        elif line == "end":
            cases.append(cur)
        elif line.startswith("C "):
            lhs, rhs = line.split("->")
            cur["acc"].append((2, 0, int(lhs.split()[1])))
            if rhs.strip() != "none":
                for part in rhs.split(";"):
                    kind, l, e, slot = part.split()
                    cur["ev"].append((KIND[kind], int(l), int(e), int(slot), -1, -1))
        else:
            lhs, rhs = line.split("->")
            a, l, e = lhs.split()
            kind, slot, vl, ve = rhs.split()
            cur["acc"].append((0 if a == "R" else 1, int(l), int(e)))
            cur["ev"].append((KIND[kind], int(l), int(e), int(slot), int(vl), int(ve)))
    return cases


@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c["name"])
def test_lru_hand_traces(case):
    acc = np.array(case["acc"], np.int32)
    ev = oracle.lru_run(case["cap"], acc[:, 1], acc[:, 2], acc[:, 0])
    assert [tuple(r) for r in ev.tolist()] == case["ev"]


@pytest.mark.parametrize("case", load_cases("lru_resize_traces.txt"), ids=lambda c: c["name"])
def test_lru_resize_hand_traces(case):
    acc = np.array(case["acc"], np.int32)
    ev = oracle.lru_run(case["cap"], acc[:, 1], acc[:, 2], acc[:, 0])
    assert [tuple(r) for r in ev.tolist()] == case["ev"]


def test_lru_resize_to_the_same_size_changes_nothing():
    """A capacity change to the current capacity with every slot in use evicts nothing and
    renumbers nothing: the run continues exactly as without it."""
    rng = np.random.default_rng(9)
    n, cap = 3000, 7
    e = rng.integers(0, 20, n)
    base = oracle.lru_run(cap, np.zeros(n), e)
    ins = 1500
    assert len(np.unique(e[:ins])) >= cap  # every slot is in use at the change
    l2 = np.concatenate([np.zeros(ins), [0], np.zeros(n - ins)])
    e2 = np.concatenate([e[:ins], [cap], e[ins:]])
    k2 = np.concatenate([np.zeros(ins), [2], np.zeros(n - ins)])
    assert np.array_equal(oracle.lru_run(cap, l2, e2, k2), base)


def test_lru_inclusion_property():
    rng = np.random.default_rng(4)
    n = 3000
    keys = rng.zipf(1.3, n) % 40
    layers = keys // 10
    experts = keys % 10
    prev_hits = None
    for cap in range(1, 45):
        ev = oracle.lru_run(cap, layers, experts)
        hits = ev[:, 0] == 0
        if prev_hits is not None:
            assert np.all(hits[prev_hits])  # every hit at cap-1 is still a hit at cap
        prev_hits = hits
    distinct = len(set(zip(layers.tolist(), experts.tolist())))
    ev = oracle.lru_run(distinct, layers, experts)
    assert np.sum(ev[:, 0] == 1) == distinct  # only cold misses once everything fits
    assert np.all(ev[:, 4] == -1)             # and nothing is ever evicted


def test_lru_slots_never_shared():
    rng = np.random.default_rng(5)
    layers = rng.integers(0, 3, 2000)
    experts = rng.integers(0, 12, 2000)
    cap = 7
    ev = oracle.lru_run(cap, layers, experts)
    resident = {}
    for kind, l, e, slot, vl, ve in ev.tolist():
        assert 0 <= slot < cap
        if kind == 1:
            if vl >= 0:
                assert resident.pop(slot) == (vl, ve)
            else:
                assert slot not in resident
            resident[slot] = (l, e)
        else:
            assert resident[slot] == (l, e)


def test_layer_accesses_ascending_distinct():
    idx = np.array([[5, 2], [2, 9], [0, 5]], np.int32)
    assert oracle.layer_accesses(idx, 16).tolist() == [0, 2, 5, 9]
