"""GPU parity of the permutation on its own: offsets, perm, inv_perm, the active list and its
length bit-exact with the oracle's stable counting sort, and the permuted gates and token rows
bit-exact with the pairs they come from, for the one-launch kernel (up to 1024 pairs: ranks
counted per pair, rows gathered in the same launch) and the many-CTA kernels (more pairs:
per-CTA counts, a scan by the last CTA to finish, placement, then a row gather), at the
boundary between them, with ragged last CTAs, a single pair, a single expert, 1024 experts,
expert counts that are not powers of two, and heavy collisions (few experts, many pairs)."""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import oracle

pytestmark = pytest.mark.gpu

CASES = [
    # (T, E, k)
    (1, 1, 1), (170, 16, 6), (171, 16, 6), (1024, 1, 1), (1025, 1, 1), (500, 1000, 8), (3000, 7, 3),
    (4096, 256, 6), (2731, 1024, 3), (1, 1024, 8), (16, 256, 6), (128, 64, 8), (7, 3, 2),
]


def _forced_sets(rng, T, E, k, zipf):
    """k distinct experts per token; with zipf, popular experts dominate (many equal ids per warp)."""
    if not zipf:
        return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    p = 1.0 / np.arange(1, E + 1) ** 1.1
    p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k", CASES)
@pytest.mark.parametrize("zipf", [False, True])
def test_permutation_bit_exact(T, E, k, zipf):
    import torch
    H, I = 256, 128
    rng = np.random.default_rng(T * 7919 + E * 31 + k + (1 if zipf else 0))
    sets = _forced_sets(rng, T, E, k, zipf)
    with moe.MoeCache(moe.LayerShape(1, E, H, I, k, E, T)) as cache:
        x = torch.randn(T, H, device="cuda").to(torch.bfloat16)
        Wr = torch.randn(E, H, device="cuda") * 0.02
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        out = torch.empty((T, H), dtype=torch.float32, device="cuda")
        cache.route_forced(0, x, Wr, None, torch.from_numpy(sets).cuda(), idx, w)
        cache.layer_forward(0, x, x.float(), out, idx, w)
        cache.sync()
        idx_h = idx.cpu().numpy()
        assert np.array_equal(np.sort(idx_h, axis=1), np.sort(sets, axis=1))
        offs_o, perm_o = oracle.permute(idx_h, E)
        P = T * k
        assert np.array_equal(cache.debug_read(moe.MOE_DBG_OFFSETS, E + 1), offs_o)
        perm = cache.debug_read(moe.MOE_DBG_PERM, P)
        assert np.array_equal(perm, perm_o)
        inv = cache.debug_read(moe.MOE_DBG_INV_PERM, P)
        assert np.array_equal(inv[perm_o], np.arange(P))
        active_o = np.nonzero(np.diff(offs_o))[0]
        n_act = int(cache.debug_read(moe.MOE_DBG_N_ACTIVE, 1)[0])
        assert n_act == active_o.size
        assert np.array_equal(cache.debug_read(moe.MOE_DBG_ACTIVE, E)[:n_act], active_o)
        # gates and token rows follow their pairs, bit for bit
        w_perm = cache.debug_read(moe.MOE_DBG_W_PERM, P, "float32")
        assert np.array_equal(w_perm.view(np.uint32), w.cpu().numpy().ravel()[perm_o].view(np.uint32))
        x_perm = cache.debug_read(moe.MOE_DBG_X_PERM, P * H, "uint16").reshape(P, H)
        x_h = x.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(x_perm, x_h[perm_o // k])
