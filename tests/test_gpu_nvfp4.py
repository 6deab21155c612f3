"""GPU parity of the NVFP4 expert path (MOE_NVFP4): 4-bit entries with E4M3 block scales (per 16
weights) and fp32 tensor scales (per matrix) in the pinned pool and the cache, expanded to bf16
on chip by the decode kernels, the tensor scales applied to the fp32 accumulators.

* the tiny layer at batch sizes giving token chunks of every width and experts over several
  chunks, against the oracle's float64 reading of the same NVFP4 entries;
* bitwise: with every tensor scale set to 1, a 4-bit context and a bf16 context whose pool holds
  the bf16 values the 4-bit entries encode give the same output bits (the expansion of code
  times block scale is exact and feeds the same tensor-core products);
* the decode layer at full size (hidden 4096, intermediate 1536, 256 experts top-6, 64-entry
  cache, 10.6 MB entries): routing, outputs and the LRU trace, for the host and the
  device-resident policy.
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
def test_tiny_layer_nvfp4(T):
    W = mi.WORKLOADS["tiny"]
    ents = hz.OracleEntries(W, nvfp4=True)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    with hz.make_cache(W, max_tokens=T, capacity=16, flags=moe.MOE_TRACE | moe.MOE_NVFP4) as cache:
        assert cache.entry_bytes == mi.nvfp4_entry_bytes(W.H, W.I)
        x = mi.activations(W.seed, 870 + T, T, W.H)
        idx, out, resid = _forward(cache, W, x, Wr, b, T)
        idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
        assert np.array_equal(idx, idx_o)
        ref = oracle.moe_layer_rows_f64(ents.layer(0), W.H, W.I, x, resid, idx_o, w_o)
        hz.assert_out_close(out, ref, resid)


def _unit_scale_entry(W, l, e):
    """The seeded NVFP4 entry with its three tensor scales replaced by 1.0."""
    ent = mi.nvfp4_entry(W.seed, l, e, W.H, W.I).copy()
    ent[-16:-4] = np.ones(3, np.float32).view(np.uint8)
    return ent


def _nv_unit_pool(cache, W, L):
    for l in range(L):
        for e in range(W.E):
            cache.host_entry_bytes(l, e)[:] = _unit_scale_entry(W, l, e)


def _bf16_of_unit_pool(cache, W, L):
    """bf16 pool holding exactly the values the unit-scale NVFP4 entries encode."""
    for l in range(L):
        for e in range(W.E):
            v = oracle.nvfp4_entry_as_f64(_unit_scale_entry(W, l, e), W.H, W.I)
            f = v.astype(np.float32)
            bits = f.view(np.uint32)
            assert np.array_equal(f.astype(np.float64), v) and not np.any(bits & 0xffff), "not exact in bf16"
            cache.host_entry_bytes(l, e)[:] = (bits >> 16).astype(np.uint16).view(np.uint8)


@pytest.mark.parametrize("T", [40, 300])
def test_nvfp4_expansion_is_bitwise_the_bf16_path(T):
    W = mi.WORKLOADS["tiny"]
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    x = mi.activations(W.seed, 995 + T, T, W.H)
    outs = []
    for flags, pool in [(moe.MOE_NVFP4, _nv_unit_pool), (0, _bf16_of_unit_pool)]:
        with hz.make_cache(W, max_tokens=T, capacity=16, flags=flags, pool=pool) as cache:
            cache.set_path(moe.MOE_PATH_GEMV_UNFUSED)  # the 4-bit kernels run gate/up and down as two launches
            outs.append(_forward(cache, W, x, Wr, b, T)[1])
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


@pytest.mark.parametrize("flags", [moe.MOE_TRACE | moe.MOE_NVFP4, moe.MOE_TRACE | moe.MOE_NVFP4 | moe.MOE_DEVICE_POLICY],
                         ids=["host", "device"])
def test_decode_layer_nvfp4_full_size(flags):
    W = mi.WORKLOADS["decode"]
    ents = hz.OracleEntries(W, nvfp4=True)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    accesses = []
    with hz.make_cache(W, max_tokens=16, flags=flags) as cache:
        for B, steps in [(1, 2), (4, 1), (16, 1)]:
            for s in range(steps):
                x = mi.activations(W.seed, 62000 + 100 * B + s, B, W.H)
                idx, out, resid = _forward(cache, W, x, Wr, b, B)
                idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
                assert np.array_equal(idx, idx_o)
                ref = oracle.moe_layer_rows_f64(ents.layer(0), W.H, W.I, x, resid, idx_o, w_o)
                hz.assert_out_close(out, ref, resid)
                accesses += hz.routed_accesses(0, idx_o, W.E)
        st, tr = cache.stats(trace_cap=1 << 16)
    assert np.array_equal(tr, hz.expected_trace(W.C, accesses))
    assert st["fill_bytes"] == st["misses"] * mi.nvfp4_entry_bytes(W.H, W.I)
