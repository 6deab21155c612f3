"""GPU parity of the router on its own: fp32 logits bitwise equal to the oracle's fixed
evaluation order, and top-k indices bit-exact, for every router kernel variant -- the
shared-memory kernels of small batches (T <= 32) and the register-tiled kernel of large
batches (32-token x 32-expert tiles, the lanes of the order split over warps) -- including
ragged tiles (T and E not multiples of the tile) and several chunks of 256 hidden columns."""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # (T, E, H, k)
    (1, 256, 4096, 6), (2, 256, 4096, 6), (3, 16, 256, 2), (8, 256, 4096, 6), (13, 100, 512, 4),
    (16, 256, 4096, 6), (32, 128, 2048, 8), (33, 256, 4096, 6), (77, 100, 768, 5), (300, 16, 256, 2),
    (1000, 256, 4096, 6), (4096, 256, 4096, 6), (65, 70, 256, 3), (130, 200, 1024, 8),
]


@pytest.mark.parametrize("T,E,H,k", CASES)
def test_router_logits_bitwise(T, E, H, k):
    import torch
    seed = 11
    x = mi.activations(seed, 40 + T, T, H)
    Wr = mi.router_weights(seed, 0, E, H)
    b, _ = mi.router_bias(seed, 0, E, 1.1)
    with moe.MoeCache(moe.LayerShape(1, E, H, 128, k, 1, T)) as cache:
        xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        z = torch.empty((T, E), dtype=torch.float32, device="cuda")
        cache.route(0, xd, torch.from_numpy(Wr).cuda(), torch.from_numpy(b).cuda(), idx, w, z)
        cache.sync()
        z32, _ = oracle.router_logits(x, Wr, b, want_double=False)
        zg = z.cpu().numpy()
        bad = np.nonzero(zg.view(np.uint32) != z32.view(np.uint32))
        assert bad[0].size == 0, f"{bad[0].size} logits differ, first at {bad[0][0]},{bad[1][0]}"
        idx_o, w_o = oracle.topk(z32, k)
        assert np.array_equal(idx.cpu().numpy(), idx_o)
        assert np.abs(w.cpu().numpy() - w_o).max() <= 1e-6
