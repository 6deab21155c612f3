"""Pins for the oracle's router logits, top-k and gates (CPU only).

Pins come from outside the oracle: hand-worked fp32 cases (tests/golden), exact integer
arithmetic, brute-force enumeration of k-subsets, and closed forms of the softmax.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special

import moe_inputs as mi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ONE_BF16 = 0x3F80


def _golden_router_cases():
    cases = []
    for line in open(os.path.join(GOLDEN, "router_fp32_order.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tok = line.split()
        name, H, bias = tok[0], int(tok[1]), float(tok[2])
        assert tok[3] == "w"
        ws = {}
        i = 4
        while "=" in tok[i]:
            h, v = tok[i].split("=")
            ws[int(h)] = float(v)
            i += 1
        cases.append((name, H, bias, ws, float(tok[i]), float(tok[i + 1])))
    return cases


@pytest.mark.parametrize("case", _golden_router_cases(), ids=lambda c: c[0])
def test_router_fixed_order_golden(case):
    name, H, bias, ws, z32_exp, z64_exp = case
    x = np.full((1, H), ONE_BF16, dtype=np.uint16)
    W = np.zeros((1, H), dtype=np.float32)
    for h, v in ws.items():
        W[0, h] = v
    z32, z64 = oracle.router_logits(x, W, np.array([bias], np.float32))
    assert z32[0, 0] == np.float32(z32_exp), name
    assert z64[0, 0] == z64_exp, name


def test_router_exact_integers():
    """Small-integer weights and activations make every partial sum exact in fp32, so the
    logits must equal the exact integer dot products (pins token/expert indexing)."""
    rng = np.random.default_rng(1)
    T, E, H = 5, 7, 512
    xi = rng.integers(-4, 5, size=(T, H))
    wi = rng.integers(-3, 4, size=(E, H))
    bi = rng.integers(-10, 11, size=E)
    xb = np.array([mi.f32_to_bf16_bits(float(v)) for v in xi.ravel()], dtype=np.uint16).reshape(T, H)
    z32, z64 = oracle.router_logits(xb, wi.astype(np.float32), bi.astype(np.float32))
    exact = np.array([[sum(int(a) * int(b) for a, b in zip(xi[t], wi[e])) + int(bi[e]) for e in range(E)]
                      for t in range(T)])
    assert np.array_equal(z32, exact.astype(np.float32))
    assert np.array_equal(z64, exact.astype(np.float64))


def test_router_fp32_within_error_bound():
    """fp32 logits agree with the double sum within the textbook bound
    |fl(s) - s| <= gamma_n * sum|w x|, n = H/32 + 5 + 1 roundings deep."""
    W = mi.WORKLOADS["decode"]
    x = mi.activations(0, 0, 4, W.H)
    Wr = mi.router_weights(0, 0, W.E, W.H)
    b, _ = mi.router_bias(0, 0, W.E, W.zipf_s)
    z32, z64 = oracle.router_logits(x, Wr, b)
    xf = mi.bf16_bits_to_f32(x).astype(np.float64)
    absdot = np.abs(xf) @ np.abs(Wr.astype(np.float64)).T + np.abs(b)
    n = W.H // 32 + 6
    u = 2.0 ** -24
    assert np.all(np.abs(z32 - z64) <= n * u / (1 - n * u) * absdot)


def _brute_topk(z, k):
    """Enumerate every k-subset; the routed one has every member ranked above every
    non-member (larger logit, or equal logit and lower id)."""
    E = len(z)
    better = lambda a, b: z[a] > z[b] or (z[a] == z[b] and a < b)
    winners = [S for S in itertools.combinations(range(E), k)
               if all(better(a, b) for a in S for b in range(E) if b not in S)]
    assert len(winners) == 1
    S = list(winners[0])
    # order inside the set: each member is ranked above the ones after it
    ordered = []
    while S:
        top = [a for a in S if all(a == b or better(a, b) for b in S)][0]
        ordered.append(top)
        S.remove(top)
    return ordered


def test_topk_brute_force_tiny():
    W = mi.WORKLOADS["tiny"]
    x = mi.activations(0, 3, 8, W.H)
    Wr = mi.router_weights(0, 0, W.E, W.H)
    z32, _ = oracle.router_logits(x, Wr, np.zeros(W.E, np.float32))
    idx, _ = oracle.topk(z32, W.k)
    for t in range(8):
        assert list(idx[t]) == _brute_topk(z32[t], W.k)
    for k in (1, 3, 4):
        idx, _ = oracle.topk(z32[:3], k)
        for t in range(3):
            assert list(idx[t]) == _brute_topk(z32[t], k)


def test_topk_ties_go_to_lower_id():
    z = np.array([[1.0, 3.0, 3.0, 2.0, 3.0, 0.0],
                  [5.0, 5.0, 5.0, 5.0, 5.0, 5.0]], dtype=np.float32)
    idx, w = oracle.topk(z, 3)
    assert idx.tolist() == [[1, 2, 4], [0, 1, 2]]
    for t in range(2):
        assert list(idx[t]) == _brute_topk(z[t], 3)
    assert np.allclose(w, 1.0 / 3.0, rtol=0, atol=1e-15)


def test_gates_closed_forms():
    rng = np.random.default_rng(2)
    z = rng.normal(size=(6, 16)).astype(np.float32)
    # k = E: the plain softmax over all experts (scipy's textbook routine)
    idx, w = oracle.topk(z, 16)
    for t in range(6):
        sm = scipy.special.softmax(z[t].astype(np.float64))
        assert np.allclose(w[t], sm[idx[t]], rtol=1e-12, atol=0)
    # k = 1: the single gate is one
    _, w1 = oracle.topk(z, 1)
    assert np.all(w1 == 1.0)
    # k = 2: w0 = sigmoid(z0 - z1)
    idx2, w2 = oracle.topk(z, 2)
    for t in range(6):
        a, b = float(z[t, idx2[t, 0]]), float(z[t, idx2[t, 1]])
        assert math.isclose(w2[t, 0], 1.0 / (1.0 + math.exp(b - a)), rel_tol=1e-13)


def test_gates_invariants_decode_shape():
    W = mi.WORKLOADS["decode"]
    x = mi.activations(0, 1, 16, W.H)
    Wr = mi.router_weights(0, 0, W.E, W.H)
    b, _ = mi.router_bias(0, 0, W.E, W.zipf_s)
    idx, w, _, _ = oracle.route(x, Wr, b, W.k)
    assert np.allclose(w.sum(1), 1.0, atol=1e-12)
    assert np.all(w > 0) and np.all(w <= 1)
    assert np.all(np.diff(w, axis=1) <= 0)
    for t in range(16):
        assert len(set(idx[t])) == W.k


def test_forced_gates_order_and_softmax():
    z = np.array([[0.5, 2.0, -1.0, 2.0, 0.1]], dtype=np.float32)
    idx, w = oracle.forced_gates(z, np.array([[4, 3, 1]], np.int32))
    assert idx.tolist() == [[1, 3, 4]]  # logits 2.0, 2.0 (tie -> lower id), 0.1
    sm = scipy.special.softmax(np.array([2.0, 2.0, 0.1], np.float64))
    assert np.allclose(w[0], sm, rtol=1e-12)
    with pytest.raises(ValueError):
        oracle.forced_gates(z, np.array([[1, 1, 2]], np.int32))


def test_near_tie_flags():
    z = np.array([[1.0, 0.999999, 0.5], [1.0, 0.5, 0.1]])
    assert oracle.near_ties(z, 1, eps=1e-5).tolist() == [True, False]
