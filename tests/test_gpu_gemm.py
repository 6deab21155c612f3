"""GPU parity of the prefill path: the tcgen05 grouped GEMM (gate/up with the SwiGLU epilogue,
down with the gate-weight epilogue). First on the tiny layer forced onto the GEMM path, then
on the full-size prefill layer (4096 tokens, 256 experts top-6, Zipf(1.1) router bias, every
routed expert resident) with routing and permutation bit-exact for all tokens and outputs
checked on sampled tokens."""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle
from tests import harness as hz

pytestmark = pytest.mark.gpu


def _run(cache, W, x, Wr, b, T, layer=0):
    import torch
    xd = hz.bf16_dev(x)
    idx = torch.empty((T, W.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, W.k), dtype=torch.float32, device="cuda")
    resid = xd.float()
    out = torch.empty((T, W.H), dtype=torch.float32, device="cuda")
    cache.route(layer, xd, hz.f32_dev(Wr), hz.f32_dev(b), idx, w)
    cache.layer_forward(layer, xd, resid, out, idx, w)
    cache.sync()
    return idx.cpu().numpy(), w.cpu().numpy(), out.cpu().numpy(), resid.cpu().numpy()


@pytest.mark.parametrize("T", [8, 64, 300])
def test_tiny_layer_on_gemm_path(T):
    W = mi.WORKLOADS["tiny"]
    ents = hz.OracleEntries(W)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b = np.zeros(W.E, np.float32)
    with hz.make_cache(W, max_tokens=T, capacity=16) as cache:
        cache.set_path(moe.MOE_PATH_GEMM)
        x = mi.activations(W.seed, 700 + T, T, W.H)
        idx, w, out, resid = _run(cache, W, x, Wr, b, T)
        idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
        assert np.array_equal(idx, idx_o)
        ref = oracle.moe_layer([ents(0, e) for e in range(W.E)], W.H, W.I, x, resid, idx_o, w_o)
        hz.assert_out_close(out, ref, resid)
        assert cache.kernel_stats is not None


def test_tiny_layer_auto_path_takes_the_gemm():
    """T = 450 on the tiny layer: 900 pairs, and one expert gets more than 64 tokens, so the AUTO
    path takes the grouped GEMM (reading the gathered rows)."""
    W = mi.WORKLOADS["tiny"]
    T = 450
    ents = hz.OracleEntries(W)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b = np.zeros(W.E, np.float32)
    x = mi.activations(W.seed, 700 + T, T, W.H)
    idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
    assert np.bincount(idx_o.ravel(), minlength=W.E).max() > 64
    with hz.make_cache(W, max_tokens=T, capacity=16, flags=moe.MOE_TRACE | moe.MOE_PROFILE) as cache:
        idx, w, out, resid = _run(cache, W, x, Wr, b, T)
        assert np.array_equal(idx, idx_o)
        ref = oracle.moe_layer([ents(0, e) for e in range(W.E)], W.H, W.I, x, resid, idx_o, w_o)
        hz.assert_out_close(out, ref, resid)
        ks = cache.kernel_stats()
        assert ks["gemm_gateup"]["launches"] == 1 and ks["decode_fused"]["launches"] == 0


def test_prefill_layer_full_size():
    W = mi.WORKLOADS["prefill"]
    T = 4096
    ents = hz.OracleEntries(W)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    x = mi.activations(W.seed, 9000, T, W.H)
    with hz.make_cache(W, max_tokens=T) as cache:
        idx, w, out, resid = _run(cache, W, x, Wr, b, T)
        z32, _ = oracle.router_logits(x, Wr, b, want_double=False)
        idx_o, w_o = oracle.topk(z32, W.k)
        assert np.array_equal(idx, idx_o)
        assert np.abs(w - w_o).max() <= 1e-6
        offs_o, perm_o = oracle.permute(idx_o, W.E)
        assert np.array_equal(cache.debug_read(moe.MOE_DBG_OFFSETS, W.E + 1), offs_o)
        assert np.array_equal(cache.debug_read(moe.MOE_DBG_PERM, T * W.k), perm_o)
        counts = np.diff(offs_o)
        assert counts.max() > 128  # several m-tiles for the most popular experts
        # sampled tokens: the first, the last, and tokens routed to the largest group
        rng = np.random.default_rng(0)
        big = int(np.argmax(counts))
        on_big = np.nonzero((idx_o == big).any(axis=1))[0]
        sample = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 40, replace=False),
                                           rng.choice(on_big, 20, replace=False)]))
        ref = oracle.moe_layer_rows(ents.layer(0), W.H, W.I, x[sample], resid[sample], idx_o[sample], w_o[sample])
        hz.assert_out_close(out[sample], ref, resid[sample])
        st = cache.stats()
        assert st["expert_reads"] == len(np.unique(idx_o))
