"""NVFP4 expert entries, CPU side: the quantizer of the input generator and the oracle's
dequantization, pinned by hand-worked blocks, a brute-force nearest-value search over every
E4M3 code, the format's error bound, and the FFN on float64 weights against the bf16 one.
(The decode kernels read MXFP4 entries; NVFP4 entries are prepared and checked here only.)"""
import os

import numpy as np

import moe_inputs as mi
import oracle


def _golden():
    cases, cur = [], None
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_blocks.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "block":
            cur = {"name": rest[0]}
        elif key == "t":
            cur["t"] = float(rest[0])
        elif key == "x":
            cur["x"] = rest
        elif key == "scale":
            cur["scale"] = int(rest[0])
        elif key == "bytes":
            cur["bytes"] = [int(v) for v in rest]
        elif key == "end":
            cases.append(cur)
    return cases


def _bf16(v: str) -> int:
    return 0x8000 if v.strip() == "-0.0" else mi.f32_to_bf16_bits(float(v))


def test_nvfp4_quantizer_hand_worked_blocks():
    cases = _golden()
    assert len(cases) == 6
    for c in cases:
        x = np.array([_bf16(v) for v in c["x"]], np.uint16)
        assert all(float(mi.bf16_bits_to_f32(np.array([b], np.uint16))[0]) == float(v)
                   for b, v in zip(x, c["x"])), c["name"]  # the listed values are exact in bf16
        q, s = mi.nvfp4_block(x, c["t"])
        assert s == c["scale"], c["name"]
        assert q.tolist() == c["bytes"], c["name"]


def _e4m3_table():
    """Every finite E4M3 value (codes 0 .. 126), from the format's definition."""
    vals = []
    for c in range(127):
        f, m = c >> 3, c & 7
        vals.append(m / 8 * 2.0 ** -6 if f == 0 else (1 + m / 8) * 2.0 ** (f - 7))
    return np.array(vals)


def test_e4m3_codes_round_trip_and_match_the_definition():
    table = _e4m3_table()
    for c in range(127):
        assert mi.e4m3_decode(c) == table[c]
        assert mi.e4m3_encode(table[c]) == c


def test_e4m3_encoder_is_the_nearest_value_ties_to_even():
    """Brute force: the encoder's code is the nearest finite E4M3 value, ties going to the even
    mantissa, values beyond 448 saturating; checked on random values over the whole range and
    on every midpoint between neighbouring codes."""
    table = _e4m3_table()
    rng = np.random.default_rng(5)
    vs = np.concatenate([2.0 ** rng.uniform(-12, 9.5, 4000), (table[:-1] + table[1:]) / 2,
                         np.array([0.0, 448.0, 460.0, 464.0, 470.0, 1e6])]).astype(np.float32)
    for v in vs:
        v = float(v)
        d = np.abs(table - v)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        if v >= 448.0:
            want = 126
        assert mi.e4m3_encode(v) == want, v


def test_oracle_dequant_reads_codes_and_scales_from_their_definitions():
    # one block of codes 0..15 under every valid scale: value = e2m1(code) * e4m3(scale) * t
    e2m1 = [0, 0.5, 1, 1.5, 2, 3, 4, 6]
    q = np.array([lo | (hi << 4) for lo, hi in zip(range(0, 16, 2), range(1, 16, 2))], np.uint8)
    table = _e4m3_table()
    for c in range(127):
        for t in (1.0, 2.0 ** -10, 0.3):
            got = oracle.nvfp4_dequant(q, np.array([c], np.uint8), 16, t)
            t32 = float(np.float32(t))
            want = [(-1 if i & 8 else 1) * e2m1[i & 7] * table[c] * t32 for i in range(16)]
            assert got.tolist() == want, (c, t)


def test_nvfp4_entry_is_the_blocks_of_the_bf16_entry():
    """An NVFP4 entry is the seeded bf16 entry quantized block by block with its matrix's
    tensor scale, each block at the place of the streaming layout, then the three tensor scales."""
    H, I = 256, 128
    w = mi.expert_entry(0, 2, 5, H, I)
    e = mi.nvfp4_entry(0, 2, 5, H, I)
    n = 3 * H * I
    assert e.size == mi.nvfp4_entry_bytes(H, I) == n // 2 + n // 16 + 16
    mats = [w[m * I * H:(m + 1) * I * H] for m in range(3)]
    t = [mi.nvfp4_tensor_scale(float(np.abs(mi.bf16_bits_to_f32(m)).max())) for m in mats]
    assert np.frombuffer(e[-16:-4].tobytes(), np.float32).tolist() == [float(np.float32(v)) for v in t]
    assert e[-4:].tolist() == [0, 0, 0, 0]
    gu = (I // 64) * (H // 64) * 4608
    for mat, row, b in [(0, 0, 0), (0, 3, 5), (1, 127, 15), (1, 64, 6), (2, 0, 0), (2, 255, 7), (2, 130, 1)]:
        K = H if mat < 2 else I
        elem0 = mat * I * H + row * K + 16 * b
        q, s = mi.nvfp4_block(w[elem0: elem0 + 16], t[mat])
        k, j = b // 4, b % 4
        if mat < 2:
            stage = ((row // 64) * (H // 64) + k) * 4608
            co = stage + mat * 2048 + (row % 64) * 32 + j * 8
            so = stage + 4096 + mat * 256 + (row % 64) * 4 + j
        else:
            stage = gu + ((row // 128) * (I // 64) + k) * 4608
            co = stage + (row % 128) * 32 + j * 8
            so = stage + 4096 + (row % 128) * 4 + j
        assert e[co: co + 8].tolist() == q.tolist() and e[so] == s, (mat, row, b)


def test_nvfp4_entry_error_bound():
    """Each dequantized weight is within one block step d = E4M3(s) * t of the bf16 weight: the
    E2M1 grid's widest gap is 2 (between 4 and 6), and a clamped block maximum exceeds 6 d by at
    most 6 d / 16 (the scale's relative rounding of 2^-4). A block whose scale falls below half
    the smallest E4M3 value (max |x| < 6 t 2^-10) is stored as zeros, an error below that."""
    H, I = 512, 256
    w = mi.bf16_bits_to_f32(mi.expert_entry(0, 1, 3, H, I)).astype(np.float64)
    e = mi.nvfp4_entry(0, 1, 3, H, I)
    W = oracle.nvfp4_entry_as_f64(e, H, I)
    t = np.frombuffer(e[-16:-4].tobytes(), np.float32).astype(np.float64)
    err = np.abs(W - w).reshape(-1, 16)
    amax = np.abs(w).reshape(-1, 16).max(axis=1)
    tb = np.repeat(t, I * H // 16)
    d_bound = amax / 6 / (1 - 2.0 ** -4) + 6 * tb * 2.0 ** -10  # a block step, or a flushed block
    assert np.all(err.max(axis=1) <= d_bound * (1 + 1e-6))
    rel = np.abs(W - w).sum() / np.abs(w).sum()
    assert rel < 0.12  # about 9 % mean relative error for N(0, 0.02) weights


def test_ffn_on_float64_weights_is_the_bf16_ffn():
    """The float64-weight FFN restates the bf16 one: on weights that are bf16 values it gives the
    same bits."""
    H, I = 256, 128
    ent = mi.expert_entry(0, 0, 1, H, I)
    x = mi.activations(0, 9, 1, H)[0]
    y16 = oracle.expert_ffn(ent, H, I, x)
    y64 = oracle.expert_ffn_f64(mi.bf16_bits_to_f32(ent).astype(np.float64), H, I, x)
    assert np.array_equal(y16, y64)


def test_layer_on_float64_weights_is_the_bf16_layer():
    """The float64-weight layer restates the bf16 layer (which the dense zero-masked reference
    pins): on weights that are bf16 values, with routing from the oracle's router, it gives the
    same bits -- so a dropped term, a wrong gate or a wrong index in its combine would show."""
    H, I, E, k, T = 256, 128, 16, 2, 6
    ents = [mi.expert_entry(0, 0, e, H, I) for e in range(E)]
    x = mi.activations(0, 11, T, H)
    Wr = mi.router_weights(0, 0, E, H)
    b = np.zeros(E, np.float32)
    idx, w, _, _ = oracle.route(x, Wr, b, k)
    resid = mi.bf16_bits_to_f32(x)
    ref = oracle.moe_layer(ents, H, I, x, resid, idx, w)
    got = oracle.moe_layer_rows_f64(lambda e: mi.bf16_bits_to_f32(ents[e]).astype(np.float64), H, I, x, resid, idx, w)
    assert np.array_equal(ref, got)
    # and it is linear in a power-of-two scaling of W_down (a tensor scale on the down matrix)
    scaled = lambda e: np.concatenate([mi.bf16_bits_to_f32(ents[e][:2 * I * H]).astype(np.float64),
                                       0.25 * mi.bf16_bits_to_f32(ents[e][2 * I * H:]).astype(np.float64)])
    got4 = oracle.moe_layer_rows_f64(scaled, H, I, x, resid, idx, w)
    d = (got4 - resid) - 0.25 * (ref - resid)  # equal up to the rounding of the residual add
    assert np.abs(d).max() <= 1e-12 * np.abs(ref).max()
    assert np.abs(ref - resid).max() > 1e-3  # the experts contribute
