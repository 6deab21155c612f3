"""The GPU build of the seeded input generator writes exactly the bits of the CPU build, so a
pool filled on the GPU and the oracle's own CPU copy of the same entries are identical."""
import numpy as np
import pytest

import moe_inputs as mi

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("H,I", [(256, 128), (4096, 1536), (2048, 768)])
def test_gpu_generator_is_bitwise_the_cpu_generator(H, I):
    keys = [(0, 0), (0, 5), (3, 255), (47, 127)]
    bufs = [np.empty(3 * H * I, np.uint16) for _ in keys]
    mi.gpu_fill_entries(0, keys, H, I, [b.ctypes.data for b in bufs])
    for (l, e), b in zip(keys, bufs):
        ref = mi.expert_entry(0, l, e, H, I)
        diff = np.nonzero(b != ref)[0]
        assert diff.size == 0, f"entry {(l, e)}: {diff.size} elements differ, first at {diff[0]}"


@pytest.mark.parametrize("H,I", [(256, 128), (4096, 1536)])
def test_gpu_mxfp4_entries_are_bitwise_the_cpu_ones(H, I):
    keys = [(0, 1), (2, 200)]
    bufs = [np.empty(mi.mxfp4_entry_bytes(H, I), np.uint8) for _ in keys]
    mi.gpu_fill_mxfp4_entries(0, keys, H, I, [b.ctypes.data for b in bufs])
    for (l, e), b in zip(keys, bufs):
        ref = mi.mxfp4_entry(0, l, e, H, I)
        diff = np.nonzero(b != ref)[0]
        assert diff.size == 0, f"entry {(l, e)}: {diff.size} bytes differ, first at {diff[0]}"


@pytest.mark.parametrize("H,I", [(256, 128), (4096, 1536)])
def test_gpu_nvfp4_entries_are_bitwise_the_cpu_ones(H, I):
    keys = [(0, 3), (1, 77)]
    bufs = [np.empty(mi.nvfp4_entry_bytes(H, I), np.uint8) for _ in keys]
    mi.gpu_fill_nvfp4_entries(0, keys, H, I, [b.ctypes.data for b in bufs])
    for (l, e), b in zip(keys, bufs):
        ref = mi.nvfp4_entry(0, l, e, H, I)
        diff = np.nonzero(b != ref)[0]
        assert diff.size == 0, f"entry {(l, e)}: {diff.size} bytes differ, first at {diff[0]}"
