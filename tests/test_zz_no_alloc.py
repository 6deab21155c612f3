"""moe_route_noalloc, the router entry point for callers that cannot allocate device memory
(code running where cudaMalloc is not allowed, or whose device memory is owned by another
allocator). It keeps its logits in a static device array instead of a context's scratch.

Checked through the C ABI against the existing entry point moe_route on the same inputs,
on two calls in a row (the second must not see the first call's leftovers in the shared
array), and against the oracle's router: indices bit-exact, gates within 1e-6, as in the
other router tests. The shapes include the exact size limit and a call without a bias. This file is
collected last so that a run stopping at the first failure has already run every other test.
"""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

# (T, hidden, experts, top_k, bias): the tiny layer; a decode-shaped router at T*E = 16384;
# the exact limit T*E = 65536; a call without a bias
SHAPES = [(8, 256, 16, 2, True), (64, 4096, 256, 6, True), (256, 256, 256, 6, True), (16, 512, 64, 4, False)]


def _dev_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("T,H,E,k,with_bias", SHAPES)
def test_noalloc_router_matches_moe_route_twice(T, H, E, k, with_bias):
    import torch
    Wr_h = mi.router_weights(0, 0, E, H)
    b_h = mi.router_bias(0, 0, E, 1.1)[0] if with_bias else np.zeros(E, np.float32)
    Wr = torch.from_numpy(Wr_h).cuda()
    b = torch.from_numpy(b_h).cuda() if with_bias else None
    # a context only for the existing entry point (small entries: inter 128)
    with moe.MoeCache(moe.LayerShape(1, E, H, 128, k, 1, T)) as cache:
        for call in range(2):
            x_h = mi.activations(0, 500 + call, T, H)
            x = _dev_bf16(x_h)
            idx_ref = torch.empty((T, k), dtype=torch.int32, device="cuda")
            w_ref = torch.empty((T, k), dtype=torch.float32, device="cuda")
            cache.route(0, x, Wr, b, idx_ref, w_ref)
            cache.sync()
            idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
            w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
            moe.route_noalloc(x, Wr, b, idx, w, top_k=k, stream=torch.cuda.current_stream())
            torch.cuda.synchronize()
            assert np.array_equal(idx.cpu().numpy(), idx_ref.cpu().numpy()), f"call {call}"
            assert np.abs(w.cpu().numpy() - w_ref.cpu().numpy()).max() <= 1e-6, f"call {call}"
            # and directly against the oracle's router on the same seeded inputs
            idx_o, w_o, _, _ = oracle.route(x_h, Wr_h, b_h, k)
            assert np.array_equal(idx.cpu().numpy(), idx_o), f"call {call}: routing differs from the oracle"
            assert np.abs(w.cpu().numpy() - w_o).max() <= 1e-6, f"call {call}: gates differ from the oracle"


def test_noalloc_router_rejects_sizes_beyond_the_static_array():
    import torch
    T, H, E, k = 257, 256, 256, 2  # 65792 logits > 65536
    x = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    Wr = torch.zeros((E, H), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.route_noalloc(x, Wr, None, idx, w, top_k=k)
    assert e.value.code == moe.MOE_E_INVAL
    assert "exceeds the static scratch" in str(e.value)
