"""Pins for the oracle's expert FFN, sparse layer, dense reference and permutation (CPU).

Closed forms use one-hot (selection) weight matrices, for which the SwiGLU expert reduces
to y[n] = silu(x[a(n)]) * x[b(n)], checked against scipy's logistic function; linearity
pins use experts that are exact power-of-two multiples of one another; the dense
all-experts reference with zero-masked gates is an independent route to the layer output.
"""
import os

import numpy as np
import pytest
import scipy.special

import moe_inputs as mi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ONE = 0x3F80  # bf16 1.0


def _bf16(vals):
    return np.array([mi.f32_to_bf16_bits(float(v)) for v in np.ravel(vals)], dtype=np.uint16).reshape(np.shape(vals))


def _selection_entry(H, I, sel_g, sel_u, sel_d):
    """Entry whose W_gate row i picks x[sel_g[i]], W_up row i picks x[sel_u[i]],
    W_down row n picks h[sel_d[n]]."""
    Wg = np.zeros((I, H), np.uint16)
    Wu = np.zeros((I, H), np.uint16)
    Wd = np.zeros((H, I), np.uint16)
    Wg[np.arange(I), sel_g] = ONE
    Wu[np.arange(I), sel_u] = ONE
    Wd[np.arange(H), sel_d] = ONE
    return np.concatenate([Wg.ravel(), Wu.ravel(), Wd.ravel()])


def _silu(a):
    return a * scipy.special.expit(a)


@pytest.mark.parametrize("H,I", [(16, 16), (32, 8), (8, 24)])
def test_ffn_selection_closed_form(H, I):
    rng = np.random.default_rng(H * 100 + I)
    sel_g = rng.integers(0, H, I)
    sel_u = rng.integers(0, H, I)
    sel_d = rng.integers(0, I, H)
    entry = _selection_entry(H, I, sel_g, sel_u, sel_d)
    x = _bf16(rng.normal(size=H))
    xf = mi.bf16_bits_to_f32(x).astype(np.float64)
    y = oracle.expert_ffn(entry, H, I, x)
    expect = _silu(xf[sel_g[sel_d]]) * xf[sel_u[sel_d]]
    assert np.allclose(y, expect, rtol=1e-14, atol=1e-300)


def test_ffn_zero_down_projection():
    W = mi.WORKLOADS["tiny"]
    e = mi.expert_entry(0, 0, 3, W.H, W.I).copy()
    e[2 * W.H * W.I:] = 0
    y = oracle.expert_ffn(e, W.H, W.I, mi.activations(0, 0, 1, W.H)[0])
    assert np.all(y == 0.0)


def _tiny_setup(step=0):
    W = mi.WORKLOADS["tiny"]
    entries = [mi.expert_entry(0, 0, e, W.H, W.I) for e in range(W.E)]
    x = mi.activations(0, step, 8, W.H)
    resid = mi.bf16_bits_to_f32(x)
    Wr = mi.router_weights(0, 0, W.E, W.H)
    idx, w, _, _ = oracle.route(x, Wr, np.zeros(W.E, np.float32), W.k)
    return W, entries, x, resid, idx, w


def test_sparse_equals_dense_zero_masked():
    W, entries, x, resid, idx, w = _tiny_setup()
    sparse = oracle.moe_layer(entries, W.H, W.I, x, resid, idx, w)
    dense = oracle.moe_dense(entries, W.H, W.I, x, resid, idx, w)
    assert np.max(np.abs(sparse - dense)) <= 1e-12 * np.max(np.abs(dense))


def test_zero_down_projection_passes_residual():
    W, entries, x, resid, idx, w = _tiny_setup()
    zeroed = []
    for e in entries:
        e = e.copy()
        e[2 * W.H * W.I:] = 0
        zeroed.append(e)
    out = oracle.moe_layer(zeroed, W.H, W.I, x, resid, idx, w)
    assert np.array_equal(out, resid.astype(np.float64))


def test_identical_experts_sum_to_one_expert():
    """All experts equal: gates sum to one, so out - resid must be that expert's output."""
    W, entries, x, resid, idx, w = _tiny_setup(step=1)
    same = [entries[0]] * W.E
    out = oracle.moe_layer(same, W.H, W.I, x, resid, idx, w)
    for t in range(8):
        y = oracle.expert_ffn(entries[0], W.H, W.I, x[t])
        assert np.allclose(out[t] - resid[t], y, rtol=0, atol=1e-12)


def test_power_of_two_scaled_experts():
    """Expert e = expert 0 with W_down scaled by 2^s_e (exact in bf16): out - resid must be
    (sum_j w_j 2^s_{e_j}) * y_0 -- pins which expert and which gate meet."""
    W, entries, x, resid, idx, w = _tiny_setup(step=2)
    base = entries[0]
    wd = mi.bf16_bits_to_f32(base[2 * W.H * W.I:])
    scale = [2.0 ** ((e % 5) - 2) for e in range(W.E)]
    scaled = []
    for e in range(W.E):
        s = base.copy()
        s[2 * W.H * W.I:] = _bf16(wd * scale[e])
        scaled.append(s)
    out = oracle.moe_layer(scaled, W.H, W.I, x, resid, idx, w)
    for t in range(8):
        y0 = oracle.expert_ffn(base, W.H, W.I, x[t])
        c = sum(w[t, j] * scale[idx[t, j]] for j in range(W.k))
        assert np.allclose(out[t] - resid[t], c * y0, rtol=0, atol=1e-12)


def _golden_perm():
    for line in open(os.path.join(GOLDEN, "permute_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        head, rows, offs, perm = [s.strip() for s in line.split("|")]
        E, k = map(int, head.split())
        idx = np.array([[int(v) for v in r.split()] for r in rows.split(";")], np.int32)
        yield E, k, idx, [int(v) for v in offs.split()], [int(v) for v in perm.split()]


@pytest.mark.parametrize("case", list(_golden_perm()))
def test_permute_hand_traced(case):
    E, k, idx, offs, perm = case
    o, p = oracle.permute(idx, E)
    assert o.tolist() == offs and p.tolist() == perm


def test_permute_invariants_prefill_shape():
    W = mi.WORKLOADS["prefill"]
    rng = np.random.default_rng(3)
    T = 512
    idx = np.stack([rng.choice(W.E, W.k, replace=False) for _ in range(T)]).astype(np.int32)
    offsets, perm = oracle.permute(idx, W.E)
    P = T * W.k
    assert offsets[0] == 0 and offsets[-1] == P
    assert np.array_equal(np.sort(perm), np.arange(P))                       # bijection
    assert np.array_equal(np.diff(offsets), np.bincount(idx.ravel(), minlength=W.E))  # counts
    flat = idx.ravel()
    for e in range(W.E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)                                      # stable


def test_mxfp4_dequant_hand_worked_blocks():
    """The oracle's MXFP4 reading of the hand-worked blocks (tests/golden/mxfp4_blocks.txt):
    each code's magnitude times 2^(scale - 127), signs from bit 3."""
    from tests.test_inputs import _mxfp4_golden
    expect = {
        "ties": [0, 1, 1, 2, 2, 4, 4, 6, 6, 0.5, 1.5, 3, -0.0, -1, -6, 0.5, 0.5, 1] + [0] * 14,
        "small": [6 * 2 ** -7, -3 * 2 ** -7, 0, 2 ** -7] + [0] * 28,
        "zeros": [-0.0] + [0] * 31,
    }
    for c in _mxfp4_golden():
        got = oracle.mxfp4_dequant(np.array(c["bytes"], np.uint8), np.array([c["scale"]], np.uint8), 32)
        f = mi.bf16_bits_to_f32(got)
        assert f.tolist() == expect[c["name"]], c["name"]
        assert (np.signbit(f) == np.signbit(np.array(expect[c["name"]]))).all()


def test_mxfp4_round_trip_error_is_within_half_a_grid_step():
    """dequant(quant(x)) differs from x by at most half the E2M1 grid step at x's magnitude
    (0.25, 0.5 or 1 times the block scale), or by the clamp for |x| > 6 * scale; values on the
    grid come back exactly."""
    rng = np.random.default_rng(5)
    for trial in range(200):
        x = (rng.standard_normal(32) * 10.0 ** rng.uniform(-4, 1)).astype(np.float32)
        bits = np.array([mi.f32_to_bf16_bits(v) for v in x], np.uint16)
        xb = mi.bf16_bits_to_f32(bits).astype(np.float64)
        q, s = mi.mxfp4_block(bits)
        y = mi.bf16_bits_to_f32(oracle.mxfp4_dequant(q, np.array([s], np.uint8), 32)).astype(np.float64)
        scale = 2.0 ** (s - 127)
        a = np.abs(xb) / scale
        half_step = np.where(a < 2, 0.25, np.where(a < 4, 0.5, 1.0)) * scale
        bound = np.where(a <= 6, half_step, (a - 6) * scale + 1e-30)
        assert (np.abs(y - xb) <= bound * (1 + 1e-12)).all(), trial
        assert np.abs(xb).max() >= 4 * scale  # the scale puts the largest element in [4, 8)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -1.5, -2, -3, -4, -6, 6] * 2) * 2.0 ** -5
    bits = np.array([mi.f32_to_bf16_bits(v) for v in grid], np.uint16)
    q, s = mi.mxfp4_block(bits)
    y = mi.bf16_bits_to_f32(oracle.mxfp4_dequant(q, np.array([s], np.uint8), 32))
    assert np.array_equal(y, grid.astype(np.float32))


def test_mxfp4_entry_reads_back_within_the_block_bounds():
    """The oracle's reading of a whole MXFP4 entry (its scale layout included) gives, for every
    element, a value within the round-trip bound of the seeded bf16 weight it came from, and
    exactly the dequantized value of that element's own block."""
    H, I = 256, 128
    w = mi.bf16_bits_to_f32(mi.expert_entry(0, 1, 2, H, I)).astype(np.float64)
    y = mi.bf16_bits_to_f32(oracle.mxfp4_entry_as_bf16(mi.mxfp4_entry(0, 1, 2, H, I), H, I)).astype(np.float64)
    wb = mi.expert_entry(0, 1, 2, H, I)
    for blk in range(0, w.size // 32, 97):
        q, s = mi.mxfp4_block(wb[32 * blk: 32 * blk + 32])
        ref = mi.bf16_bits_to_f32(oracle.mxfp4_dequant(q, np.array([s], np.uint8), 32))
        assert np.array_equal(y[32 * blk: 32 * blk + 32], ref.astype(np.float64)), blk
    assert np.abs(y - w).max() <= 0.5 * np.abs(w).max()  # coarse: 4-bit weights
    rel = np.linalg.norm(y - w) / np.linalg.norm(w)
    assert 0.05 < rel < 0.2  # MXFP4's relative rms error on Gaussian weights is about 0.1
