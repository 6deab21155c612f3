"""GPU parity of multi-layer runs sharing one LRU cache of (layer, expert) entries.

* The 8-layer decode stream (256 experts top-6 per layer, batch 8, routing forced by a
  reuse trace: each token re-picks an expert of its previous step with p = 0.7, else Zipf;
  cache of 30% of the 2048 entries), at reduced hidden/intermediate sizes so the oracle runs
  every step: routing, outputs and the whole LRU trace.
* A 6-layer stack (128 experts top-8): a prefill with full-layer double buffering -- layer
  l+1's whole expert set is prefetched on the copy stream right after layer l's compute is
  enqueued -- then decode steps at batch 32. The trace includes the prefetch events. With bf16,
  MXFP4 and NVFP4 entries (the 4-bit prefill runs on the decode kernels, in token chunks).

Layer inputs are fresh seeded activations per (step, layer): the oracle never takes an
input from the GPU path.
"""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle
from tests import harness as hz

pytestmark = pytest.mark.gpu


def _bufs(T, W):
    import torch
    return (torch.empty((T, W.k), dtype=torch.int32, device="cuda"),
            torch.empty((T, W.k), dtype=torch.float32, device="cuda"),
            torch.empty((T, W.H), dtype=torch.float32, device="cuda"))


def test_decode_stream_8_layers():
    import torch
    base = mi.WORKLOADS["stream8"]
    W = mi.Workload("stream8-small", 256, 128, base.E, base.k, base.L, base.C, base.zipf_s)
    B, steps = 8, 24
    ents = hz.OracleEntries(W)
    routers = [mi.router_weights(W.seed, l, W.E, W.H) for l in range(W.L)]
    biases, perms = zip(*[mi.router_bias(W.seed, l, W.E, W.zipf_s) for l in range(W.L)])
    trace = mi.trace_reuse(W.seed, W.L, steps, B, W.E, W.k, W.zipf_s, 0.7, np.stack(perms))
    accesses = []
    with hz.make_cache(W, max_tokens=B) as cache:
        Wr_d = [hz.f32_dev(r) for r in routers]
        b_d = [hz.f32_dev(b) for b in biases]
        idx, w, out = _bufs(B, W)
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
                r = resid.cpu().numpy()
                if s % 4 == 0 or s == steps - 1:  # outputs on every 4th step (all layers)
                    ref = oracle.moe_layer_rows(ents.layer(l), W.H, W.I, x, r, idx_o, w_o)
                    hz.assert_out_close(out.cpu().numpy(), ref, r)
                accesses += hz.routed_accesses(l, idx_o, W.E)
        st, tr = cache.stats(trace_cap=1 << 20)
    exp = hz.expected_trace(W.C, accesses)
    assert np.array_equal(tr, exp)
    assert st["expert_reads"] == len(accesses)
    assert 0 < st["hits"] < st["expert_reads"]


FORMATS = {"bf16": 0, "mxfp4": moe.MOE_MXFP4, "nvfp4": moe.MOE_NVFP4}


def _layer_ref(fmt, ents, l, W, x, r, idx_o, w_o):
    """The oracle's layer on the format's own reading of the entries."""
    if fmt == "nvfp4":
        return oracle.moe_layer_rows_f64(ents.layer(l), W.H, W.I, x, r, idx_o, w_o)
    return oracle.moe_layer_rows(ents.layer(l), W.H, W.I, x, r, idx_o, w_o)


@pytest.mark.parametrize("fmt", list(FORMATS))
def test_stack_prefill_double_buffered_then_decode(fmt):
    import torch
    base = mi.WORKLOADS["stack48"]
    L = 6
    W = mi.Workload("stack-small", 256, 128, base.E, base.k, L, 2 * base.E, base.zipf_s)
    T_pre, B, steps = 256, 32, 3
    ents = hz.OracleEntries(W, fp4=fmt == "mxfp4", nvfp4=fmt == "nvfp4")
    routers = [mi.router_weights(W.seed, l, W.E, W.H) for l in range(L)]
    biases = [mi.router_bias(W.seed, l, W.E, W.zipf_s)[0] for l in range(L)]
    accesses = []
    with hz.make_cache(W, max_tokens=T_pre, flags=moe.MOE_TRACE | moe.MOE_PREFILL_DB | FORMATS[fmt]) as cache:
        Wr_d = [hz.f32_dev(r) for r in routers]
        b_d = [hz.f32_dev(b) for b in biases]
        # prefill: prefetch layer 0, then per layer: route, forward, prefetch the next layer
        cache.cache_fill(0, None, moe.MOE_FILL_FULL_LAYER)
        accesses += [(1, 0, e) for e in range(W.E)]
        idx, w, out = _bufs(T_pre, W)
        xs = [mi.activations(W.seed, 200000 + l, T_pre, W.H) for l in range(L)]
        outs, idxs, keep = [], [], []
        for l in range(L):
            xd = hz.bf16_dev(xs[l])
            keep.append(xd)  # device inputs must outlive the enqueued work (no sync between layers)
            cache.route(l, xd, Wr_d[l], b_d[l], idx, w)
            resid = xd.float()
            o = torch.empty_like(out)
            cache.layer_forward(l, xd, resid, o, idx, w)
            if l + 1 < L:
                cache.cache_fill(l + 1, None, moe.MOE_FILL_FULL_LAYER)
            outs.append((o, resid))
            idxs.append(idx.clone())
        cache.sync()
        st = cache.stats()
        assert st["misses"] == 0 and st["prefetch_fills"] == L * W.E
        for l in range(L):
            idx_o, w_o, _, _ = oracle.route(xs[l], routers[l], biases[l], W.k)
            assert np.array_equal(idxs[l].cpu().numpy(), idx_o), l
            accesses += hz.routed_accesses(l, idx_o, W.E)
            if l + 1 < L:
                accesses += [(1, l + 1, e) for e in range(W.E)]
            rows = np.arange(0, T_pre, 17)  # sampled tokens
            r = outs[l][1].cpu().numpy()
            ref = _layer_ref(fmt, ents, l, W, xs[l][rows], r[rows], idx_o[rows], w_o[rows])
            hz.assert_out_close(outs[l][0].cpu().numpy()[rows], ref, r[rows])
        # decode steps at batch 32 through every layer
        idx, w, out = _bufs(B, W)
        for s in range(steps):
            for l in range(L):
                x = mi.activations(W.seed, 300000 + s * L + l, B, W.H)
                xd = hz.bf16_dev(x)
                cache.route(l, xd, Wr_d[l], b_d[l], idx, w)
                resid = xd.float()
                cache.layer_forward(l, xd, resid, out, idx, w)
                cache.sync()
                idx_o, w_o, _, _ = oracle.route(x, routers[l], biases[l], W.k)
                assert np.array_equal(idx.cpu().numpy(), idx_o), (s, l)
                r = resid.cpu().numpy()
                ref = _layer_ref(fmt, ents, l, W, x, r, idx_o, w_o)
                hz.assert_out_close(out.cpu().numpy(), ref, r)
                accesses += hz.routed_accesses(l, idx_o, W.E)
        st, tr = cache.stats(trace_cap=1 << 20)
    assert np.array_equal(tr, hz.expected_trace(W.C, accesses))
