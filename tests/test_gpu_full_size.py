"""GPU parity of the two multi-layer workloads at their full sizes, in the launch configuration
that `bench.py --workload stream8|stack48` times, on fewer steps:

* the 8-layer decode stream: hidden 4096, intermediate 1536, 256 experts top-6 per layer,
  batch 8, routing forced by the reuse trace (p = 0.7), one 614-entry LRU cache over the 2048
  (layer, expert) entries of a 77 GB pinned pool -- routing of every (step, layer) and the
  whole LRU trace bit-exact, outputs on sampled (step, layer) pairs;
* the 48-layer stack: hidden 2048, intermediate 768, 128 experts top-8 per layer, 1536-entry
  cache over a 58 GB pool; a 2048-token prefill with full-layer double buffering, then decode
  steps at batch 32 -- routing of every layer and step, the whole LRU trace with the prefetch
  events, outputs on sampled tokens of sampled layers.

The oracle computes every expected value from its own copy of the inputs."""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle
from tests import harness as hz

pytestmark = pytest.mark.gpu


def test_stream8_full_size():
    import torch
    W = mi.WORKLOADS["stream8"]
    B, steps = 8, 40
    ents = hz.OracleEntries(W)
    routers = [mi.router_weights(W.seed, l, W.E, W.H) for l in range(W.L)]
    biases, perms = zip(*[mi.router_bias(W.seed, l, W.E, W.zipf_s) for l in range(W.L)])
    trace = mi.trace_reuse(W.seed, W.L, steps, B, W.E, W.k, W.zipf_s, 0.7, np.stack(perms))
    sample = {(0, 0), (1, 0), (steps - 1, 0), (steps - 1, W.L - 1), (steps // 2, 3)}
    accesses = []
    with hz.make_cache(W, max_tokens=B) as cache:
        Wr_d = [hz.f32_dev(r) for r in routers]
        b_d = [hz.f32_dev(b) for b in biases]
        idx = torch.empty((B, W.k), dtype=torch.int32, device="cuda")
        w = torch.empty((B, W.k), dtype=torch.float32, device="cuda")
        out = torch.empty((B, W.H), dtype=torch.float32, device="cuda")
        for s in range(steps):
            for l in range(W.L):
                x = mi.activations(W.seed, 100000 + s * W.L + l, B, W.H)
                xd = hz.bf16_dev(x)
                sets = torch.from_numpy(np.ascontiguousarray(trace[s, l])).cuda()
                cache.route_forced(l, xd, Wr_d[l], b_d[l], sets, idx, w)
                resid = xd.float()
                cache.layer_forward(l, xd, resid, out, idx, w)
                cache.sync()
                z32, _ = oracle.router_logits(x, routers[l], biases[l], want_double=False)
                idx_o, w_o = oracle.forced_gates(z32, trace[s, l])
                assert np.array_equal(idx.cpu().numpy(), idx_o), (s, l)
                assert np.abs(w.cpu().numpy() - w_o).max() <= 1e-6
                if (s, l) in sample:
                    r = resid.cpu().numpy()
                    ref = oracle.moe_layer_rows(ents.layer(l), W.H, W.I, x, r, idx_o, w_o)
                    hz.assert_out_close(out.cpu().numpy(), ref, r)
                accesses += hz.routed_accesses(l, idx_o, W.E)
        st, tr = cache.stats(trace_cap=1 << 20)
    exp = hz.expected_trace(W.C, accesses)
    assert np.array_equal(tr, exp)
    assert st["expert_reads"] == len(accesses)
    assert st["evictions"] > 0  # the 614-entry cache filled up and the LRU chose victims


@pytest.mark.parametrize("fmt", ["bf16", "mxfp4"])
def test_stack48_full_size_prefill_then_decode(fmt):
    import torch
    W = mi.WORKLOADS["stack48"]
    T, B, steps = 2048, 32, 2
    ents = hz.OracleEntries(W, fp4=fmt == "mxfp4")
    fmt_flag = moe.MOE_MXFP4 if fmt == "mxfp4" else 0
    routers = [mi.router_weights(W.seed, l, W.E, W.H) for l in range(W.L)]
    biases = [mi.router_bias(W.seed, l, W.E, W.zipf_s)[0] for l in range(W.L)]
    check_layers = {0, 1, 24, W.L - 1}
    rows = np.arange(0, T, 97)  # sampled prefill tokens
    accesses = [(1, 0, e) for e in range(W.E)]
    with hz.make_cache(W, max_tokens=T, flags=moe.MOE_TRACE | moe.MOE_PREFILL_DB | fmt_flag) as cache:
        Wr_d = [hz.f32_dev(r) for r in routers]
        b_d = [hz.f32_dev(b) for b in biases]
        cache.cache_fill(0, None, moe.MOE_FILL_FULL_LAYER)
        keep, idxs, outs = [], [], []
        for l in range(W.L):
            x = mi.activations(W.seed, 200000 * W.L + l, T, W.H)
            xd = hz.bf16_dev(x)
            idx = torch.empty((T, W.k), dtype=torch.int32, device="cuda")
            w = torch.empty((T, W.k), dtype=torch.float32, device="cuda")
            o = torch.empty((T, W.H), dtype=torch.float32, device="cuda")
            resid = xd.float()
            cache.route(l, xd, Wr_d[l], b_d[l], idx, w)
            cache.layer_forward(l, xd, resid, o, idx, w)
            if l + 1 < W.L:
                cache.cache_fill(l + 1, None, moe.MOE_FILL_FULL_LAYER)
            keep.append((xd, resid, w))  # device inputs outlive the enqueued work (no sync between layers)
            idxs.append(idx)
            outs.append(o if l in check_layers else None)
        cache.sync()
        st = cache.stats()
        # every expert of every layer is prefetched before its layer computes, and no prefetch
        # finds its entry resident (a layer's entries are only ever brought in by its prefetch)
        assert st["misses"] == 0 and st["prefetch_fills"] == W.L * W.E and st["prefetch_hits"] == 0
        for l in range(W.L):
            x = mi.activations(W.seed, 200000 * W.L + l, T, W.H)
            idx_o, w_o, _, _ = oracle.route(x, routers[l], biases[l], W.k)
            assert np.array_equal(idxs[l].cpu().numpy(), idx_o), l
            accesses += hz.routed_accesses(l, idx_o, W.E)
            if l + 1 < W.L:
                accesses += [(1, l + 1, e) for e in range(W.E)]
            if l in check_layers:
                r = keep[l][1].cpu().numpy()
                ref = oracle.moe_layer_rows(ents.layer(l), W.H, W.I, x[rows], r[rows], idx_o[rows], w_o[rows])
                hz.assert_out_close(outs[l].cpu().numpy()[rows], ref, r[rows])
        del keep, outs
        idx = torch.empty((B, W.k), dtype=torch.int32, device="cuda")
        w = torch.empty((B, W.k), dtype=torch.float32, device="cuda")
        out = torch.empty((B, W.H), dtype=torch.float32, device="cuda")
        for s in range(steps):
            for l in range(W.L):
                x = mi.activations(W.seed, (300000 + s) * W.L + l, B, W.H)
                xd = hz.bf16_dev(x)
                cache.route(l, xd, Wr_d[l], b_d[l], idx, w)
                resid = xd.float()
                cache.layer_forward(l, xd, resid, out, idx, w)
                cache.sync()
                idx_o, w_o, _, _ = oracle.route(x, routers[l], biases[l], W.k)
                assert np.array_equal(idx.cpu().numpy(), idx_o), (s, l)
                if l in check_layers:
                    r = resid.cpu().numpy()
                    ref = oracle.moe_layer_rows(ents.layer(l), W.H, W.I, x, r, idx_o, w_o)
                    hz.assert_out_close(out.cpu().numpy(), ref, r)
                accesses += hz.routed_accesses(l, idx_o, W.E)
        st, tr = cache.stats(trace_cap=1 << 20)
    assert np.array_equal(tr, hz.expected_trace(W.C, accesses))
