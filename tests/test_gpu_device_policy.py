"""GPU parity of the device-resident cache policy (MOE_DEVICE_POLICY): the LRU decisions, the
slot table, the counters, the trace and the fills all on the GPU, so a forward never waits on
the host and a decode step can be captured in a CUDA graph.

* the decode layer at full size (hidden 4096, intermediate 1536, 256 experts top-6, 64-entry
  cache), batches 1, 4, 16: routing, outputs against the oracle, and the whole LRU trace
  against the oracle's LRU;
* the same inputs through a host-policy context and a device-policy context give bitwise
  equal outputs and equal traces (same kernels, same K split rule);
* the 8-layer stream at reduced width, one whole decode step (8 layers of forced routing and
  forward) captured into a CUDA graph and replayed over many steps: outputs of every layer and
  the LRU trace against the oracle.
"""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle
from tests import harness as hz

pytestmark = pytest.mark.gpu


def _decode_batches(cache, W, steps_per_batch=3, check=True):
    import torch
    ents = hz.OracleEntries(W)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    Wrd, bd = hz.f32_dev(Wr), hz.f32_dev(b)
    outs, accesses = [], []
    for B in (1, 4, 16):
        for s in range(steps_per_batch):
            x = mi.activations(W.seed, 77000 + 1000 * B + s, B, W.H)
            xd = hz.bf16_dev(x)
            idx = torch.empty((B, W.k), dtype=torch.int32, device="cuda")
            w = torch.empty((B, W.k), dtype=torch.float32, device="cuda")
            resid = xd.float()
            out = torch.empty((B, W.H), dtype=torch.float32, device="cuda")
            cache.route(0, xd, Wrd, bd, idx, w)
            cache.layer_forward(0, xd, resid, out, idx, w)
            cache.sync()
            idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
            assert np.array_equal(idx.cpu().numpy(), idx_o)
            if check:
                r = resid.cpu().numpy()
                ref = oracle.moe_layer_rows(ents.layer(0), W.H, W.I, x, r, idx_o, w_o)
                hz.assert_out_close(out.cpu().numpy(), ref, r)
            outs.append(out.cpu().numpy())
            accesses += hz.routed_accesses(0, idx_o, W.E)
    return outs, accesses


def test_device_policy_decode_layer_matches_oracle_and_host_policy():
    W = mi.WORKLOADS["decode"]
    with hz.make_cache(W, max_tokens=16, flags=moe.MOE_TRACE | moe.MOE_DEVICE_POLICY) as cache:
        outs_d, accesses = _decode_batches(cache, W)
        st, tr = cache.stats(trace_cap=1 << 16)
    assert np.array_equal(tr, hz.expected_trace(W.C, accesses))
    assert st["expert_reads"] == len(accesses) and st["forwards"] == 9
    assert st["misses"] > 0 and st["hits"] > 0
    assert st["fill_bytes"] == st["misses"] * 3 * W.H * W.I * 2
    with hz.make_cache(W, max_tokens=16, flags=moe.MOE_TRACE) as cache:
        # the device policy runs gate/up and down as two launches with the host's two-launch
        # split rule, so its outputs equal the host policy's two-launch path bit for bit
        cache.set_path(moe.MOE_PATH_GEMV_UNFUSED)
        outs_h, _ = _decode_batches(cache, W, check=False)
        _, tr_h = cache.stats(trace_cap=1 << 16)
    assert np.array_equal(tr_h, tr)
    for a, b in zip(outs_d, outs_h):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_device_policy_decode_step_captured_in_a_cuda_graph():
    import torch
    base = mi.WORKLOADS["stream8"]
    W = mi.Workload("stream8-small", 256, 128, base.E, base.k, base.L, base.C, base.zipf_s)
    B, steps = 8, 12
    ents = hz.OracleEntries(W)
    routers = [mi.router_weights(W.seed, l, W.E, W.H) for l in range(W.L)]
    biases, perms = zip(*[mi.router_bias(W.seed, l, W.E, W.zipf_s) for l in range(W.L)])
    trace = mi.trace_reuse(W.seed, W.L, steps + 1, B, W.E, W.k, W.zipf_s, 0.7, np.stack(perms))
    accesses = []
    with hz.make_cache(W, max_tokens=B, flags=moe.MOE_TRACE | moe.MOE_DEVICE_POLICY) as cache:
        stream = cache.torch_stream
        Wr_d = [hz.f32_dev(r) for r in routers]
        b_d = [hz.f32_dev(b) for b in biases]
        # static buffers the graph reads and writes
        xs = [torch.empty((B, W.H), dtype=torch.bfloat16, device="cuda") for _ in range(W.L)]
        rs = [torch.empty((B, W.H), dtype=torch.float32, device="cuda") for _ in range(W.L)]
        sets = [torch.empty((B, W.k), dtype=torch.int32, device="cuda") for _ in range(W.L)]
        outs = [torch.empty((B, W.H), dtype=torch.float32, device="cuda") for _ in range(W.L)]
        idx = [torch.empty((B, W.k), dtype=torch.int32, device="cuda") for _ in range(W.L)]
        w = [torch.empty((B, W.k), dtype=torch.float32, device="cuda") for _ in range(W.L)]

        def load(s):
            xh = []
            for l in range(W.L):
                x = mi.activations(W.seed, 100000 + s * W.L + l, B, W.H)
                xh.append(x)
                xs[l].copy_(hz.bf16_dev(x))
                rs[l].copy_(xs[l].float())
                sets[l].copy_(torch.from_numpy(np.ascontiguousarray(trace[s, l])))
            return xh

        def step():
            for l in range(W.L):
                cache.route_forced(l, xs[l], Wr_d[l], b_d[l], sets[l], idx[l], w[l])
                cache.layer_forward(l, xs[l], rs[l], outs[l], idx[l], w[l])

        def check(s, xh):
            for l in range(W.L):
                z32, _ = oracle.router_logits(xh[l], routers[l], biases[l], want_double=False)
                idx_o, w_o = oracle.forced_gates(z32, trace[s, l])
                assert np.array_equal(idx[l].cpu().numpy(), idx_o), (s, l)
                r = rs[l].cpu().numpy()
                ref = oracle.moe_layer_rows(ents.layer(l), W.H, W.I, xh[l], r, idx_o, w_o)
                hz.assert_out_close(outs[l].cpu().numpy(), ref, r)
                accesses.extend(hz.routed_accesses(l, idx_o, W.E))

        xh = load(0)  # step 0 eagerly: first launches set kernel attributes outside the capture
        step()
        cache.sync()
        check(0, xh)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        # capturing enqueued nothing: the LRU has seen step 0 only
        assert cache.stats()["forwards"] == W.L
        for s in range(1, steps + 1):
            xh = load(s)
            g.replay()
            torch.cuda.synchronize()
            check(s, xh)
        cache.sync()
        st, tr = cache.stats(trace_cap=1 << 20)
    assert st["forwards"] == W.L * (steps + 1)
    assert np.array_equal(tr, hz.expected_trace(W.C, accesses))
