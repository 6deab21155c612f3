"""The q-star split's measurements on the GPU machine: pinned host-to-device copies of whole entries
and the host expert FFN on the same entry (moe_measure_bandwidth), then the split rule and the
simulation fed with them. Nothing here runs an expert on the host inside a forward."""
import os

import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle
from tests import harness as hz

pytestmark = pytest.mark.gpu


def test_measured_bandwidths_drive_the_split():
    base = mi.WORKLOADS["decode"]
    W = mi.Workload("one-expert", base.H, base.I, 1, 1, 1, 1, None)  # one 36 MiB entry
    with hz.make_cache(W, max_tokens=1, capacity=1, L=1) as cache:
        bw = cache.measure_bandwidth(len(os.sched_getaffinity(0)), reps=3)
        # the host FFN read entry (0, 0) from the pinned pool: check it against the oracle there
        ent = cache.host_entry_array(0, 0).copy()
    assert bw["entry_bytes"] == 3 * W.H * W.I * 2
    assert 1.0 < bw["pcie_h2d_gbps"] < 1000.0
    assert 0.01 < bw["host_expert_gbps"] < 10000.0
    x = mi.activations(0, 77, 2, W.H)
    y = moe.host_expert_ffn(ent, W.H, W.I, x, threads=len(os.sched_getaffinity(0)))
    for t in range(2):
        ref = oracle.expert_ffn(ent, W.H, W.I, x[t])
        assert np.abs(y[t] - ref).max() <= 1e-4 * np.abs(ref).max()
    n = moe.qstar_fills(bw["pcie_h2d_gbps"], bw["host_expert_gbps"], 10)
    q = bw["pcie_h2d_gbps"] / (bw["pcie_h2d_gbps"] + bw["host_expert_gbps"])
    assert abs(n - 10 * q) <= 1.0
