"""GPU parity on the decode layer at full size (hidden 4096, intermediate 1536, 256 experts,
top-6, Zipf(1.1) router bias, 64-entry cache): batches of 1, 4 and 16 tokens, the launch
configuration the benchmark times. Every output token is checked against the oracle;
logits bitwise, routing and the LRU trace bit-exact."""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle
from tests import harness as hz

pytestmark = pytest.mark.gpu
W = mi.WORKLOADS["decode"]


@pytest.fixture(scope="module")
def cache():
    c = hz.make_cache(W, max_tokens=16)
    yield c
    c.close()


def test_decode_batches(cache):
    import torch
    ents = hz.OracleEntries(W)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    Wrd, bd = hz.f32_dev(Wr), hz.f32_dev(b)
    cache.stats(reset=True)
    accesses = []
    for B, steps in [(1, 3), (4, 3), (16, 3)]:
        for s in range(steps):
            x = mi.activations(W.seed, 1000 * B + s, B, W.H)
            xd = hz.bf16_dev(x)
            idx = torch.empty((B, W.k), dtype=torch.int32, device="cuda")
            w = torch.empty((B, W.k), dtype=torch.float32, device="cuda")
            z = torch.empty((B, W.E), dtype=torch.float32, device="cuda")
            resid = xd.float()
            out = torch.empty((B, W.H), dtype=torch.float32, device="cuda")
            cache.route(0, xd, Wrd, bd, idx, w, z)
            cache.layer_forward(0, xd, resid, out, idx, w)
            cache.sync()
            z32, z64 = oracle.router_logits(x, Wr, b)
            assert np.array_equal(z.cpu().numpy().view(np.uint32), z32.view(np.uint32))
            idx_o, w_o = oracle.topk(z32, W.k)
            assert np.array_equal(idx.cpu().numpy(), idx_o)
            assert np.abs(w.cpu().numpy() - w_o).max() <= 1e-6
            r = resid.cpu().numpy()
            ref = oracle.moe_layer_rows(ents.layer(0), W.H, W.I, x, r, idx_o, w_o)
            hz.assert_out_close(out.cpu().numpy(), ref, r)
            accesses += hz.routed_accesses(0, idx_o, W.E)
    st, trace = cache.stats(trace_cap=1 << 16)
    assert np.array_equal(trace, hz.expected_trace(W.C, accesses))
    assert st["expert_reads"] == len(accesses)
