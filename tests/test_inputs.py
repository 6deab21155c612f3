"""The seeded input generator: deterministic, chunk-independent, and drawing what it claims."""
import numpy as np

import moe_inputs as mi


def test_deterministic_and_chunk_independent():
    a = mi.normal_bf16(0, mi.stream_id(mi.KIND_EXPERT, 2, 3), 1001, 0.02)
    b = mi.normal_bf16(0, mi.stream_id(mi.KIND_EXPERT, 2, 3), 1001, 0.02)
    assert np.array_equal(a, b)
    part = mi.normal_bf16(0, mi.stream_id(mi.KIND_EXPERT, 2, 3), 500, 0.02, first=333)
    assert np.array_equal(part, a[333:833])
    c = mi.normal_bf16(0, mi.stream_id(mi.KIND_EXPERT, 2, 4), 1001, 0.02)
    assert not np.array_equal(a, c)


def test_normal_moments():
    z = mi.bf16_bits_to_f32(mi.normal_bf16(7, 11, 2_000_000, 0.02)).astype(np.float64)
    assert abs(z.mean()) < 1e-4 and abs(z.std() - 0.02) < 1e-4
    f = mi.normal_f32(7, 12, 2_000_000, 1.0).astype(np.float64)
    assert abs(f.mean()) < 5e-3 and abs(f.std() - 1.0) < 5e-3
    assert abs(np.mean(f ** 4) - 3.0) < 0.05  # Gaussian kurtosis


def test_bf16_rounding_is_nearest_even():
    assert mi.f32_to_bf16_bits(1.0) == 0x3F80
    # 1 + 2^-8 lies halfway between bf16 neighbours 1.0 and 1 + 2^-7: ties go to even
    assert mi.f32_to_bf16_bits(1.0 + 2 ** -8) == 0x3F80
    assert mi.f32_to_bf16_bits(1.0 + 3 * 2 ** -8) == 0x3F82
    assert mi.f32_to_bf16_bits(-2.0) == 0xC000


def test_zipf_bias_is_log_probabilities():
    b, perm = mi.router_bias(0, 5, 256, 1.1)
    assert sorted(perm.tolist()) == list(range(256))
    assert abs(np.exp(b.astype(np.float64)).sum() - 1.0) < 1e-5
    r = np.arange(1, 257)
    p = r ** -1.1 / np.sum(r ** -1.1)
    assert np.allclose(b[perm], np.log(p).astype(np.float32))


def test_reuse_trace_properties():
    L, steps, B, E, k = 2, 200, 4, 64, 6
    perms = np.stack([mi.router_bias(0, l, E, 1.1)[1] for l in range(L)])
    tr = mi.trace_reuse(0, L, steps, B, E, k, 1.1, 0.7, perms)
    assert tr.shape == (steps, L, B, k)
    assert tr.min() >= 0 and tr.max() < E
    for s in range(steps):
        for l in range(L):
            for b in range(B):
                assert len(set(tr[s, l, b])) == k
    reuse = np.mean([len(set(tr[s, l, b]) & set(tr[s - 1, l, b])) / k
                     for s in range(1, steps) for l in range(L) for b in range(B)])
    assert reuse > 0.7  # at least the forced 70% plus chance repeats of Zipf draws


def test_series_log_matches_the_logarithm():
    """The generator's own logarithm agrees with the exact one within a few ulps over (0, 1],
    including the special points 1 and powers of two."""
    import math
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.random(20000), np.array([2.0 ** -32, 0.5, 0.25, 0.70710678118654752, 0.9999999999])])
    xs = xs[xs > 0]
    for x in xs:
        got, ref = mi.log_unit(float(x)), math.log(float(x))
        assert abs(got - ref) <= 4e-16 * max(1.0, abs(ref)), (x, got, ref)
    assert mi.log_unit(1.0) == 0.0
    assert abs(mi.log_unit(0.5) + math.log(2.0)) <= 2.3e-16


def test_series_sincos_matches_the_circle():
    import math
    rng = np.random.default_rng(4)
    for u in np.concatenate([rng.random(20000), np.array([0.0, 0.125, 0.25, 0.5, 0.75, 0.999999])]):
        s, c = mi.sincos_turn(float(u))
        assert abs(s - math.sin(2 * math.pi * u)) <= 2e-15 and abs(c - math.cos(2 * math.pi * u)) <= 2e-15, u
    assert mi.sincos_turn(0.0) == (0.0, 1.0)
    assert mi.sincos_turn(0.25)[0] == 1.0 and mi.sincos_turn(0.5)[1] == -1.0


def test_cpu_builds_with_and_without_fma_instructions_agree():
    """The generator is built once with libm's fma() and once with the FMA instruction; fused
    multiply-add rounds once in both, so the two builds give the same bits."""
    import ctypes
    mi.build()
    n = 3 * 256 * 128 + 3
    outs = []
    for so in (mi._SO, mi._SO_FMA):
        L = ctypes.CDLL(so)
        L.mi_normal_bf16.argtypes = [ctypes.c_uint64] * 4 + [ctypes.c_double, ctypes.c_void_p]
        b = np.empty(n, np.uint16)
        L.mi_normal_bf16(0, mi.stream_id(mi.KIND_EXPERT, 1, 2), 5, n, 0.02, b.ctypes.data)
        outs.append(b)
    assert np.array_equal(outs[0], outs[1])


def _mxfp4_golden():
    import os
    cases, cur = [], None
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "mxfp4_blocks.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *rest = line.split()
        if key == "block":
            cur = {"name": rest[0]}
        elif key == "x":
            cur["x"] = [float(v) for v in rest]
        elif key == "scale":
            cur["scale"] = int(rest[0])
        elif key == "bytes":
            cur["bytes"] = [int(v) for v in rest]
        elif key == "end":
            cases.append(cur)
    return cases


def test_mxfp4_quantizer_hand_worked_blocks():
    for c in _mxfp4_golden():
        x = np.array([mi.f32_to_bf16_bits(v) for v in c["x"]], np.uint16)
        if c["x"][0] == 0.0 and str(c["x"][0]).startswith("-"):
            x[0] = 0x8000
        q, s = mi.mxfp4_block(x)
        assert s == c["scale"], c["name"]
        assert q.tolist() == c["bytes"], c["name"]


def test_mxfp4_entry_is_the_blocks_of_the_bf16_entry():
    """An MXFP4 entry is the seeded bf16 entry quantized block by block, each block at the place
    the streaming layout gives it: stages of 4096 code bytes + 256 scale bytes, per 64-row tile
    and 64-column slab for gate/up (gate rows, up rows, gate scales, up scales), then per 128-row
    tile and slab for down (rows, scales)."""
    H, I = 256, 128
    w = mi.expert_entry(0, 2, 5, H, I)
    e = mi.mxfp4_entry(0, 2, 5, H, I)
    n = 3 * H * I
    assert e.size == mi.mxfp4_entry_bytes(H, I) == n // 2 + n // 32
    gu = (I // 64) * (H // 64) * 4352
    for mat, row, b in [(0, 0, 0), (0, 3, 5), (1, 127, 7), (1, 64, 6), (2, 0, 0), (2, 255, 3), (2, 130, 1)]:
        K = H if mat < 2 else I
        elem0 = (mat * I * H + row * K if mat < 2 else 2 * I * H + row * K) + 32 * b
        q, s = mi.mxfp4_block(w[elem0: elem0 + 32])
        k, half = b // 2, b % 2
        if mat < 2:
            stage = ((row // 64) * (H // 64) + k) * 4352
            co = stage + mat * 2048 + (row % 64) * 32 + half * 16
            so = stage + 4096 + mat * 128 + (row % 64) * 2 + half
        else:
            stage = gu + ((row // 128) * (I // 64) + k) * 4352
            co = stage + (row % 128) * 32 + half * 16
            so = stage + 4096 + (row % 128) * 2 + half
        assert e[co: co + 16].tolist() == q.tolist() and e[so] == s, (mat, row, b)
