"""The unit schedule of the fused decode launch (host only, no GPU). The launch deals the wave's
units round robin over its CTAs (gate/up units first, then down units); the schedule may move the
last down unit of each most-loaded CTA to a less-loaded one. Its correctness conditions, checked
here against a brute-force round robin on the same counts: every unit runs exactly once, every CTA
runs all of its gate/up units before any down unit (down units wait for the h rows that gate/up
units write, so a CTA that took a down unit first could wait on itself), and a schedule is only
returned when it lowers the largest per-CTA load."""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe


def _round_robin_loads(ug, ud, kg, kd, G):
    loads = np.zeros(G, np.int64)
    for g in range(ug + ud):
        loads[g % G] += kg if g < ug else kd
    return loads


def _check(ug, ud, kg, kd, G, cap=1024):
    res = moe.fused_schedule(ug, ud, kg, kd, G, cap)
    rr = _round_robin_loads(ug, ud, kg, kd, G)
    if res is None:
        return None, int(rr.max())
    keep, off, pool = res
    assert off[0] == 0 and np.all(np.diff(off) >= 0) and off[G] == len(pool)
    seen, loads = [], []
    for b in range(G):
        units = [b + i * G for i in range(keep[b])] + pool[off[b]:off[b + 1]].tolist()
        is_gu = [u < ug for u in units]
        assert is_gu == sorted(is_gu, reverse=True), f"CTA {b} runs a down unit before a gate/up unit"
        assert all(u >= ug for u in pool[off[b]:off[b + 1]]), "only down units move"
        seen += units
        loads.append(sum(kg if u < ug else kd for u in units))
    assert sorted(seen) == list(range(ug + ud)), "every unit exactly once"
    assert max(loads) < rr.max(), "a schedule must lower the largest load"
    return max(loads), int(rr.max())


@pytest.mark.parametrize("U,expect", [(6, None), (15, (248, 264)), (30, None)])
def test_decode_layer_waves(U, expect):
    """The decode layer's waves (hidden 4096, intermediate 1536: 24 gate/up and 32 down units per
    expert of 64 and 24 K blocks) at batches 1, 4 and 16 (U = 6, 15 and 30 experts) on 148 CTAs:
    only batch 4 can come down, from 264 to 248 K blocks."""
    ug, ud = 24 * U, 32 * U
    got = _check(ug, ud, 64, 24, min(148, ug + ud))
    if expect is None:
        assert got[0] is None
    else:
        assert got == expect


def test_random_counts():
    rng = np.random.default_rng(11)
    applied = 0
    for _ in range(3000):
        G = int(rng.integers(1, 300))
        ug, ud = int(rng.integers(0, 3000)), int(rng.integers(0, 3000))
        if ug + ud < G:
            continue
        best, _ = _check(ug, ud, int(rng.integers(1, 65)), int(rng.integers(1, 65)), G,
                         int(rng.choice([256, 1024, 4096])))
        applied += best is not None
    assert applied > 100


def test_buffer_bound_and_bad_arguments():
    # a schedule needs up to 4 * grid + 1 ints: a smaller buffer gets the plain round robin
    assert moe.fused_schedule(24 * 15, 32 * 15, 64, 24, 148, cap=4 * 148) is None
    assert moe.fused_schedule(24 * 15, 32 * 15, 64, 24, 148, cap=4 * 148 + 1) is not None
    with pytest.raises(moe.MoeError):
        moe.fused_schedule(10, 10, 0, 24, 4)
    with pytest.raises(moe.MoeError):
        moe.fused_schedule(10, 10, 64, 24, 0)
