"""The q-star miss split (host only, no GPU): the host expert FFN against the oracle's expert FFN,
the split rule against a brute-force search and its closed-form cases, and the split LRU
simulation against the oracle's LRU on the accesses the split keeps.

The pages give the idea (misses divided between cache fills and host execution from measured
host and PCIe bandwidths: "FreeToken benchmark", "How FreeToken Serves Large MoE Models") but no
formula; the rule checked here is this library's reading, stated in include/moe.h."""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle


@pytest.mark.parametrize("n_tok,threads", [(1, 1), (3, 2), (4, 4), (7, 3)])
def test_host_expert_ffn_matches_the_oracle(n_tok, threads):
    H, I = 256, 128
    ent = mi.expert_entry(0, 0, 3, H, I)
    x = mi.activations(0, 40 + n_tok, n_tok, H)
    y = moe.host_expert_ffn(ent, H, I, x, threads)
    for t in range(n_tok):
        ref = oracle.expert_ffn(ent, H, I, x[t])
        # fp32 accumulation over 256 and 128 terms against double: a few fp32 ulps of the sum's scale
        assert np.abs(y[t] - ref).max() <= 1e-5 * np.abs(ref).max() + 1e-7


def test_host_expert_ffn_zero_down_and_bad_shapes():
    H, I = 64, 32
    ent = mi.expert_entry(0, 0, 1, H, I).copy()
    ent[2 * I * H:] = 0  # W_down = 0 -> y = 0 exactly
    x = mi.activations(0, 1, 2, H)
    assert np.array_equal(moe.host_expert_ffn(ent, H, I, x), np.zeros((2, H), np.float32))
    with pytest.raises(moe.MoeError):
        moe.host_expert_ffn(ent, 60, I, x[:, :60])


def _brute_fills(bp, bh, m):
    """argmin over n in 0..m of max(n / bp, (m - n) / bh), ties to the larger n."""
    best, best_c = None, None
    for n in range(m + 1):
        c = max(n / bp, (m - n) / bh)
        if best_c is None or c <= best_c:
            best, best_c = n, c
    return best


def test_qstar_fills_is_the_minimiser_of_the_miss_time():
    rng = np.random.default_rng(3)
    for _ in range(400):
        bp, bh = rng.uniform(1, 200, 2)
        m = int(rng.integers(0, 40))
        assert moe.qstar_fills(bp, bh, m) == _brute_fills(bp, bh, m), (bp, bh, m)


def test_qstar_fills_closed_forms():
    assert moe.qstar_fills(50.0, 50.0, 6) == 3          # q* = 1/2
    assert moe.qstar_fills(50.0, 50.0, 5) == 3          # tie between 2 and 3 goes to the fill
    assert moe.qstar_fills(55.0, 110.0, 9) == 3         # q* = 1/3
    assert moe.qstar_fills(55.0, 0.0, 7) == 7           # no host path: every miss fills
    assert moe.qstar_fills(0.0, 30.0, 7) == 0           # no link: every miss runs on the host
    assert moe.qstar_fills(10.0, 10.0, 0) == 0
    with pytest.raises(moe.MoeError):
        moe.qstar_fills(0.0, 0.0, 3)
    with pytest.raises(moe.MoeError):
        moe.qstar_fills(1.0, 1.0, -1)


def _random_invocations(seed, n_inv, L, E, k_max):
    rng = np.random.default_rng(seed)
    invs = []
    for v in range(n_inv):
        l = v % L
        ex = np.sort(rng.choice(E, size=int(rng.integers(1, k_max + 1)), replace=False))
        invs.append([(l, int(e), int(rng.integers(1, 6))) for e in ex])
    return invs


def test_split_lru_is_classic_lru_on_the_kept_accesses():
    """Host-executed misses never enter the cache: the events of the accesses the split keeps are
    exactly the oracle's LRU events on that subsequence."""
    invs = _random_invocations(1, 300, 3, 24, 7)
    for q in (0.0, 0.3, 0.5, 1.0, -1.0):
        s, ev = moe.qstar_simulate(10, invs, q, 55.0, 80.0, 6500.0, 37748736.0, want_events=True)
        assert s["hits"] + s["fills"] + s["host_execs"] == s["expert_reads"] == sum(len(i) for i in invs)
        kept = ev[ev[:, 0] != moe.EV_HOST_EXEC]
        host = ev[ev[:, 0] == moe.EV_HOST_EXEC]
        assert len(host) == s["host_execs"] and np.all(host[:, 3] == -1)
        ref = oracle.lru_run(10, kept[:, 1], kept[:, 2])
        assert np.array_equal(kept, ref), q
        if q == 1.0:
            assert s["host_execs"] == 0
        if q == 0.0:
            assert s["fills"] == 0 and s["hits"] == 0  # nothing ever enters the cache


def test_split_takes_the_misses_with_most_tokens_and_counts_per_invocation():
    # one invocation, empty cache: 5 misses with tokens 1, 4, 2, 4, 3 (experts 0..4); the rule
    # fills 3 of them (q* = 1/2 of 5, tie up): the two with 4 tokens (ids 1, 3), then 3 tokens (id 4)
    inv = [[(0, 0, 1), (0, 1, 4), (0, 2, 2), (0, 3, 4), (0, 4, 3)]]
    s, ev = moe.qstar_simulate(8, inv, -1.0, 40.0, 40.0, 6500.0, 1e6, want_events=True)
    assert s["fills"] == 3 and s["host_execs"] == 2
    assert ev[:, 0].tolist() == [moe.EV_HOST_EXEC, moe.EV_FILL, moe.EV_HOST_EXEC, moe.EV_FILL, moe.EV_FILL]
    assert ev[:, 3].tolist() == [-1, 0, -1, 1, 2]  # fills take the lowest free slots in access order
    # modeled time: max(3 fills / 40 GB/s, 2 host / 40 GB/s) + 3 entries / 6500 GB/s, entry 1 MB
    assert s["modeled_ms"] == pytest.approx(1e3 * (3e6 / 40e9 + 3e6 / 6500e9), rel=1e-12)
    # a later invocation: the filled experts hit, the host-executed ones are misses again
    inv2 = inv + [[(0, 0, 1), (0, 1, 1)]]
    s2, ev2 = moe.qstar_simulate(8, inv2, -1.0, 40.0, 40.0, 6500.0, 1e6, want_events=True)
    assert ev2[5:, 0].tolist() == [moe.EV_FILL, moe.EV_HIT]  # one miss of one: ceil of 1/2 fills


def test_reuse_trace_simulation_orders_fill_fractions_sensibly():
    """On the 8-layer reuse trace (batch 8, p = 0.7 re-pick, 30 % cache) the modeled step time
    with the q* split is no worse than both extremes (all fills, all host) at these bandwidths."""
    W = mi.WORKLOADS["stream8"]
    steps, B = 24, 8
    bp = [mi.router_bias(W.seed, l, W.E, W.zipf_s) for l in range(W.L)]
    trace = mi.trace_reuse(W.seed, W.L, steps, B, W.E, W.k, W.zipf_s, 0.7, np.stack([p for _, p in bp]))
    invs = []
    for s in range(steps):
        for l in range(W.L):
            ex, cnt = np.unique(trace[s, l].ravel(), return_counts=True)
            invs.append([(l, int(e), int(c)) for e, c in zip(ex, cnt)])
    entry = 3 * W.H * W.I * 2
    res = {q: moe.qstar_simulate(W.C, invs, q, 55.0, 110.0, 6500.0, entry)[0] for q in (0.0, 1.0, -1.0)}
    assert res[-1.0]["modeled_ms"] <= min(res[0.0]["modeled_ms"], res[1.0]["modeled_ms"])
    assert res[1.0]["host_execs"] == 0 and res[0.0]["fills"] == 0
