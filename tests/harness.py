"""Test harness shared by the GPU tests and the smoke check: builds a library context whose
pinned pool holds the seeded entries, moves seeded inputs to the device, and compares
library results with the oracle (which regenerates its own copy of every input)."""
from __future__ import annotations

import numpy as np

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle


def bf16_dev(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def f32_dev(a: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def make_cache(W: mi.Workload, max_tokens: int, L: int | None = None, capacity: int | None = None,
               flags: int = moe.MOE_TRACE, pool=None) -> moe.MoeCache:
    import torch
    L = W.L if L is None else L
    # one stream for torch's work (inputs, resid = x.float(), ...) and the library's compute,
    # so everything the tests enqueue is ordered
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    cache = moe.MoeCache(moe.LayerShape(L, W.E, W.H, W.I, W.k, W.C if capacity is None else capacity, max_tokens),
                         flags=flags, stream_compute=stream)
    cache.torch_stream = stream
    if pool is None:
        fill_pool(cache, W, L)
    else:
        pool(cache, W, L)
    return cache


def fill_pool(cache: moe.MoeCache, W: mi.Workload, L: int):
    """Write every seeded entry into the context's pinned pool, with the GPU build of the input
    generator (the same bits as the CPU build, which the oracle uses for its own copy): bf16, or
    MXFP4 for a context created with MOE_MXFP4."""
    keys = [(l, e) for l in range(L) for e in range(W.E)]
    ptrs = [cache.host_entry(l, e) for l, e in keys]
    if cache.shape_flags & moe.MOE_MXFP4:
        mi.gpu_fill_mxfp4_entries(W.seed, keys, W.H, W.I, ptrs)
    elif cache.shape_flags & moe.MOE_NVFP4:
        mi.gpu_fill_nvfp4_entries(W.seed, keys, W.H, W.I, ptrs)
    else:
        mi.gpu_fill_entries(W.seed, keys, W.H, W.I, ptrs)


class OracleEntries:
    """The oracle's own copy of the expert entries, regenerated from the seed (bf16; or the
    MXFP4 entries read back by the oracle as the bf16 values they encode, when fp4; or the
    NVFP4 entries read back as float64 weights, when nvfp4 -- use oracle.moe_layer_rows_f64)."""

    def __init__(self, W: mi.Workload, fp4: bool = False, nvfp4: bool = False):
        self.W = W
        self.fp4 = fp4
        self.nvfp4 = nvfp4
        self.cache = {}

    def __call__(self, layer: int, expert: int) -> np.ndarray:
        key = (layer, expert)
        if key not in self.cache:
            W = self.W
            if self.fp4:
                self.cache[key] = oracle.mxfp4_entry_as_bf16(mi.mxfp4_entry(W.seed, layer, expert, W.H, W.I), W.H, W.I)
            elif self.nvfp4:
                self.cache[key] = oracle.nvfp4_entry_as_f64(mi.nvfp4_entry(W.seed, layer, expert, W.H, W.I), W.H, W.I)
            else:
                self.cache[key] = mi.expert_entry(W.seed, layer, expert, W.H, W.I)
        return self.cache[key]

    def layer(self, layer: int):
        return lambda e: self(layer, e)


def out_tolerance(ref: np.ndarray) -> float:
    """max|gpu - oracle| <= 1e-2 * max|oracle| + 1e-3 (bf16 weights, fp32 accumulation)."""
    return 1e-2 * float(np.abs(ref).max()) + 1e-3


def assert_out_close(gpu: np.ndarray, ref: np.ndarray, resid: np.ndarray):
    err = float(np.abs(gpu - ref).max())
    tol = out_tolerance(ref)
    assert err <= tol, f"max|gpu-oracle| = {err:.3e} > {tol:.3e}"
    # stricter check on the MoE contribution alone (out - resid): bf16 rounding of the SwiGLU
    # activations bounds its relative error near 2^-9, far inside 5e-3
    dg, dr = gpu - resid, ref - resid
    err_d = float(np.abs(dg - dr).max())
    tol_d = 5e-3 * float(np.abs(dr).max()) + 1e-4
    assert err_d <= tol_d, f"MoE delta error {err_d:.3e} > {tol_d:.3e}"
    return err, tol


def expected_trace(capacity: int, accesses) -> np.ndarray:
    """accesses: list of (kind 0/1, layer, expert) in the order the library makes them."""
    if not accesses:
        return np.zeros((0, 6), np.int32)
    a = np.array(accesses, np.int32)
    return oracle.lru_run(capacity, a[:, 1], a[:, 2], a[:, 0])


def routed_accesses(layer: int, idx: np.ndarray, E: int):
    return [(0, layer, int(e)) for e in oracle.layer_accesses(idx, E)]
