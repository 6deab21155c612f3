"""GPU parity of the MXFP4 expert path (MOE_MXFP4): 4-bit entries in the pinned pool and the
cache, expanded to bf16 on chip by the decode kernels.

* the tiny layer at batch sizes giving token chunks of every width and experts over several
  chunks, against the oracle's reading of the same MXFP4 entries;
* bitwise: a 4-bit context and a bf16 context whose pool holds the bf16 values the 4-bit
  entries encode give the same output bits (the on-chip expansion is exact and feeds the same
  tensor-core products);
* the decode layer at full size (hidden 4096, intermediate 1536, 256 experts top-6, 64-entry
  cache, 10 MB entries), batches 1, 4, 16: routing, outputs and the LRU trace, for the host
  and the device-resident policy.
"""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle
from tests import harness as hz

pytestmark = pytest.mark.gpu


def _forward(cache, W, x, Wr, b, T):
    import torch
    xd = hz.bf16_dev(x)
    idx = torch.empty((T, W.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, W.k), dtype=torch.float32, device="cuda")
    resid = xd.float()
    out = torch.empty((T, W.H), dtype=torch.float32, device="cuda")
    cache.route(0, xd, hz.f32_dev(Wr), hz.f32_dev(b), idx, w)
    cache.layer_forward(0, xd, resid, out, idx, w)
    cache.sync()
    return idx.cpu().numpy(), out.cpu().numpy(), resid.cpu().numpy()


@pytest.mark.parametrize("T", [1, 5, 17, 40, 100, 700])
def test_tiny_layer_fp4(T):
    W = mi.WORKLOADS["tiny"]
    ents = hz.OracleEntries(W, fp4=True)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    with hz.make_cache(W, max_tokens=T, capacity=16, flags=moe.MOE_TRACE | moe.MOE_MXFP4) as cache:
        assert cache.entry_bytes == mi.mxfp4_entry_bytes(W.H, W.I)
        x = mi.activations(W.seed, 850 + T, T, W.H)
        idx, out, resid = _forward(cache, W, x, Wr, b, T)
        idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
        assert np.array_equal(idx, idx_o)
        ref = oracle.moe_layer([ents(0, e) for e in range(W.E)], W.H, W.I, x, resid, idx_o, w_o)
        hz.assert_out_close(out, ref, resid)


def _dequantized_pool(cache, W, L):
    """bf16 pool holding exactly the values the MXFP4 entries encode."""
    for l in range(L):
        for e in range(W.E):
            vals = oracle.mxfp4_entry_as_bf16(mi.mxfp4_entry(W.seed, l, e, W.H, W.I), W.H, W.I)
            cache.host_entry_bytes(l, e)[:] = vals.view(np.uint8)


@pytest.mark.parametrize("name,T", [("tiny", 40), ("tiny", 300)])
def test_fp4_expansion_is_bitwise_the_bf16_path(name, T):
    W = mi.WORKLOADS[name]
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    x = mi.activations(W.seed, 990 + T, T, W.H)
    outs = []
    for flags, pool in [(moe.MOE_MXFP4, None), (0, _dequantized_pool)]:
        with hz.make_cache(W, max_tokens=T, capacity=16, flags=flags, pool=pool) as cache:
            cache.set_path(moe.MOE_PATH_GEMV_UNFUSED)  # the 4-bit kernels run gate/up and down as two launches
            outs.append(_forward(cache, W, x, Wr, b, T)[1])
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


@pytest.mark.parametrize("flags", [moe.MOE_TRACE | moe.MOE_MXFP4, moe.MOE_TRACE | moe.MOE_MXFP4 | moe.MOE_DEVICE_POLICY],
                         ids=["host", "device"])
def test_decode_layer_fp4_full_size(flags):
    W = mi.WORKLOADS["decode"]
    ents = hz.OracleEntries(W, fp4=True)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    accesses = []
    with hz.make_cache(W, max_tokens=16, flags=flags) as cache:
        for B, steps in [(1, 2), (4, 2), (16, 2)]:
            for s in range(steps):
                x = mi.activations(W.seed, 61000 + 100 * B + s, B, W.H)
                idx, out, resid = _forward(cache, W, x, Wr, b, B)
                idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
                assert np.array_equal(idx, idx_o)
                ref = oracle.moe_layer_rows(ents.layer(0), W.H, W.I, x, resid, idx_o, w_o)
                hz.assert_out_close(out, ref, resid)
                accesses += hz.routed_accesses(0, idx_o, W.E)
        st, tr = cache.stats(trace_cap=1 << 16)
    assert np.array_equal(tr, hz.expected_trace(W.C, accesses))
    assert st["fill_bytes"] == st["misses"] * mi.mxfp4_entry_bytes(W.H, W.I)
