"""GPU parity of the elastic cache (moe_cache_resize) on the decode layer at full size
(hidden 4096, intermediate 1536, 256 experts top-6): decode steps at batches 1, 4 and 16 with
the capacity grown and shrunk between them, for the host policy and the device-resident policy,
with bf16 and with MXFP4 entries (a resize moves the surviving entries, whatever their size).
Outputs against the oracle, and the whole LRU trace -- including the entries a shrink evicts --
against the oracle's LRU run with the same capacity changes."""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle
from tests import harness as hz

pytestmark = pytest.mark.gpu

PLAN = [(16, 40), (4, None), (16, 96), (16, 24), (1, 8), (4, 8), (16, 64), (4, None)]  # (batch, resize after)


@pytest.mark.parametrize("fmt", ["bf16", "mxfp4"])
@pytest.mark.parametrize("flags", [moe.MOE_TRACE, moe.MOE_TRACE | moe.MOE_DEVICE_POLICY], ids=["host", "device"])
def test_resize_between_decode_steps(flags, fmt):
    import torch
    W = mi.WORKLOADS["decode"]
    fp4 = fmt == "mxfp4"
    if fp4:
        flags |= moe.MOE_MXFP4
    ents = hz.OracleEntries(W, fp4=fp4)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    Wrd, bd = hz.f32_dev(Wr), hz.f32_dev(b)
    ops = []  # (kind, layer, expert or capacity) for the oracle's LRU run
    with hz.make_cache(W, max_tokens=16, capacity=32, flags=flags) as cache:
        for i, (B, new_cap) in enumerate(PLAN):
            x = mi.activations(W.seed, 91000 + i, B, W.H)
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
            r = resid.cpu().numpy()
            ref = oracle.moe_layer_rows(ents.layer(0), W.H, W.I, x, r, idx_o, w_o)
            hz.assert_out_close(out.cpu().numpy(), ref, r)
            ops += [(0, 0, int(e)) for e in oracle.layer_accesses(idx_o, W.E)]
            if new_cap is not None:
                cache.resize(new_cap)
                ops.append((2, 0, new_cap))
        st, tr = cache.stats(trace_cap=1 << 16)
    a = np.array(ops, np.int32)
    exp = oracle.lru_run(32, a[:, 1], a[:, 2], a[:, 0])
    assert np.array_equal(tr, exp)
    assert st["resize_evictions"] == int((exp[:, 0] == moe.EV_RESIZE_EVICT).sum()) > 0
