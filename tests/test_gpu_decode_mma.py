"""GPU parity of the tensor-core decode expert kernels (weights as the M = 128 side of
tcgen05.mma, tokens as N = 16..64), forced onto the decode path, both as one fused launch per
wave (gate/up units, then down units that wait for their h rows) and as two launches:

* the tiny layer at batch sizes that give experts of 1 to more than 64 tokens, so token
  chunks of every width (16, 32, 48, 64) and experts split over several chunks are covered;
* the decode-layer shape (hidden 4096, intermediate 1536, 256 experts top-6) at batch 1, whose
  down projection is split over K (too few tiles to fill the SMs), checked against the
  oracle and for bitwise repeatability (split partials are added in a fixed order);
* the smaller decode shape (hidden 2048, intermediate 768, 128 experts top-8) at batch 32.
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


@pytest.mark.parametrize("path", [moe.MOE_PATH_GEMV, moe.MOE_PATH_GEMV_UNFUSED], ids=["fused", "two-launch"])
@pytest.mark.parametrize("T", [1, 5, 17, 40, 100, 700])
def test_tiny_layer_decode_path_all_chunk_widths(T, path):
    W = mi.WORKLOADS["tiny"]
    ents = hz.OracleEntries(W)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    with hz.make_cache(W, max_tokens=T, capacity=16) as cache:
        cache.set_path(path)
        x = mi.activations(W.seed, 800 + T, T, W.H)
        idx, out, resid = _forward(cache, W, x, Wr, b, T)
        idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
        assert np.array_equal(idx, idx_o)
        ref = oracle.moe_layer([ents(0, e) for e in range(W.E)], W.H, W.I, x, resid, idx_o, w_o)
        hz.assert_out_close(out, ref, resid)
        if T == 700:
            assert np.bincount(idx_o.ravel()).max() > 64  # an expert spans several token chunks


def test_decode_layer_batch1_split_k_repeatable():
    W = mi.WORKLOADS["decode"]
    ents = hz.OracleEntries(W)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    with hz.make_cache(W, max_tokens=4, capacity=16) as cache:
        outs = []
        for rep in range(2):
            for s in range(3):
                x = mi.activations(W.seed, 4242 + s, 1, W.H)
                idx, out, resid = _forward(cache, W, x, Wr, b, 1)
                if rep == 0:
                    idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
                    assert np.array_equal(idx, idx_o)
                    ref = oracle.moe_layer_rows(ents.layer(0), W.H, W.I, x, resid, idx_o, w_o)
                    hz.assert_out_close(out, ref, resid)
                outs.append(out)
        for s in range(3):
            assert np.array_equal(outs[s].view(np.uint32), outs[3 + s].view(np.uint32))


@pytest.mark.parametrize("B", [1, 4, 16])
def test_decode_layer_fused_and_two_launch_agree(B):
    """The fused launch and the two-launch path on the same decode batches (every expert resident,
    then with fills in the wave): both within the oracle's tolerance and close to each other."""
    W = mi.WORKLOADS["decode"]
    ents = hz.OracleEntries(W)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    outs = {}
    for path in (moe.MOE_PATH_GEMV, moe.MOE_PATH_GEMV_UNFUSED):
        with hz.make_cache(W, max_tokens=16, capacity=64) as cache:
            cache.set_path(path)
            res = []
            for s in range(3):  # step 0 fills every routed expert; later steps mix hits and fills
                x = mi.activations(W.seed, 5150 + 10 * B + s, B, W.H)
                idx, out, resid = _forward(cache, W, x, Wr, b, B)
                idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
                assert np.array_equal(idx, idx_o)
                ref = oracle.moe_layer_rows(ents.layer(0), W.H, W.I, x, resid, idx_o, w_o)
                hz.assert_out_close(out, ref, resid)
                res.append(out)
            outs[path] = res
    for s in range(3):
        d = np.abs(outs[moe.MOE_PATH_GEMV][s] - outs[moe.MOE_PATH_GEMV_UNFUSED][s]).max()
        assert d <= 1e-3 * np.abs(outs[moe.MOE_PATH_GEMV_UNFUSED][s]).max()


def test_smaller_decode_shape_batch32():
    base = mi.WORKLOADS["stack48"]
    W = mi.Workload("stack-one-layer", base.H, base.I, base.E, base.k, 1, base.E, base.zipf_s)
    ents = hz.OracleEntries(W)
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b, _ = mi.router_bias(W.seed, 0, W.E, W.zipf_s)
    T = 32
    with hz.make_cache(W, max_tokens=T) as cache:
        x = mi.activations(W.seed, 31337, T, W.H)
        idx, out, resid = _forward(cache, W, x, Wr, b, T)
        idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
        assert np.array_equal(idx, idx_o)
        assert np.bincount(idx_o.ravel()).max() <= 64  # the AUTO path picks the decode kernels
        ref = oracle.moe_layer_rows(ents.layer(0), W.H, W.I, x, resid, idx_o, w_o)
        hz.assert_out_close(out, ref, resid)
