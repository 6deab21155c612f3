"""GPU edge cases on the tiny layer: empty calls, size limits, forced-routing validation,
host-side fault injection (a fill that fails, a host wait that times out), explicit fills,
capacity errors and run-to-run determinism. Nothing here faults the GPU: failures are
injected on the host or reported by kernels through the device status word."""
import numpy as np
import pytest

import moe_expert_layer_10_b300 as moe
import moe_inputs as mi
import oracle
from tests import harness as hz

pytestmark = pytest.mark.gpu
W = mi.WORKLOADS["tiny"]


def _bufs(T):
    import torch
    idx = torch.empty((max(T, 1), W.k), dtype=torch.int32, device="cuda")
    w = torch.empty((max(T, 1), W.k), dtype=torch.float32, device="cuda")
    out = torch.empty((max(T, 1), W.H), dtype=torch.float32, device="cuda")
    return idx, w, out


def _layer(cache, x, T):
    Wr = mi.router_weights(W.seed, 0, W.E, W.H)
    b = np.zeros(W.E, np.float32)
    xd = hz.bf16_dev(x)
    idx, w, out = _bufs(T)
    cache.route(0, xd, hz.f32_dev(Wr), hz.f32_dev(b), idx, w)
    resid = xd.float()
    cache.layer_forward(0, xd, resid, out, idx, w)
    cache.sync()
    return idx.cpu().numpy(), w.cpu().numpy(), out.cpu().numpy(), resid.cpu().numpy(), Wr, b


def test_empty_and_oversized_calls():
    with hz.make_cache(W, max_tokens=8) as c:
        x = hz.bf16_dev(mi.activations(0, 0, 1, W.H))
        idx, w, out = _bufs(0)
        Wr = hz.f32_dev(mi.router_weights(0, 0, W.E, W.H))
        c.route(0, x, Wr, None, idx, w, T=0)
        c.layer_forward(0, x, out, out, idx, w, T=0)
        c.sync()
        assert c.stats()["forwards"] == 0
        with pytest.raises(moe.MoeError) as e:
            c.route(0, x, Wr, None, idx, w, T=9)
        assert e.value.code == moe.MOE_E_INVAL
        with pytest.raises(moe.MoeError):
            c.route(1, x, Wr, None, idx, w, T=1)  # layer out of range


def test_forced_set_with_repeat_raises_device_status():
    import torch
    with hz.make_cache(W, max_tokens=8) as c:
        x = hz.bf16_dev(mi.activations(0, 1, 2, W.H))
        Wr = hz.f32_dev(mi.router_weights(0, 0, W.E, W.H))
        idx, w, _ = _bufs(2)
        bad = torch.tensor([[3, 3], [1, 2]], dtype=torch.int32, device="cuda")
        c.route_forced(0, x, Wr, None, bad, idx, w)
        with pytest.raises(moe.MoeError) as e:
            c.sync()
        assert e.value.code == moe.MOE_E_DEVICE
        c.sync()  # the status was consumed; the context stays usable
        good = torch.tensor([[5, 1], [0, 15]], dtype=torch.int32, device="cuda")
        c.route_forced(0, x, Wr, None, good, idx, w)
        c.sync()
        assert sorted(idx.cpu().numpy()[0].tolist()) == [1, 5]


def test_injected_fill_failure_keeps_lru_consistent():
    ents = hz.OracleEntries(W)
    with hz.make_cache(W, max_tokens=8) as c:
        x = mi.activations(0, 2, 8, W.H)
        c.debug_inject(1, 1)
        with pytest.raises(moe.MoeError) as e:
            _layer(c, x, 8)
        assert e.value.code == moe.MOE_E_CUDA
        st = c.stats()
        assert st["misses"] == 0 and st["fill_bytes"] == 0
        for e_ in range(W.E):
            assert c.resident_slot(0, e_) == -1
        idx, w, out, resid, Wr, b = _layer(c, x, 8)  # the injection was one-shot
        idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
        assert np.array_equal(idx, idx_o)
        ref = oracle.moe_layer([ents(0, e) for e in range(W.E)], W.H, W.I, x, resid, idx_o, w_o)
        hz.assert_out_close(out, ref, resid)


def test_injected_host_timeout():
    with hz.make_cache(W, max_tokens=8) as c:
        x = mi.activations(0, 3, 4, W.H)
        c.debug_inject(2, 1)
        with pytest.raises(moe.MoeError) as e:
            _layer(c, x, 4)
        assert e.value.code == moe.MOE_E_TIMEOUT
        c.sync()
        _layer(c, x, 4)


def test_explicit_fills_and_capacity_errors():
    with hz.make_cache(W, max_tokens=8, capacity=4) as c:
        with pytest.raises(moe.MoeError) as e:
            c.cache_fill(0, None, moe.MOE_FILL_FULL_LAYER)  # 16 experts > 4 slots
        assert e.value.code == moe.MOE_E_CAPACITY
        with pytest.raises(moe.MoeError) as e:
            c.cache_fill(0, np.arange(5), moe.MOE_FILL_DEMAND)
        assert e.value.code == moe.MOE_E_CAPACITY
        c.cache_fill(0, np.array([7, 3, 7, 9]), moe.MOE_FILL_DEMAND)
        c.sync()
        _, tr = c.stats(trace_cap=64)
        assert np.array_equal(tr, hz.expected_trace(4, [(0, 0, 3), (0, 0, 7), (0, 0, 9)]))
        assert [c.resident_slot(0, e) for e in (3, 7, 9)] == [0, 1, 2]
    with hz.make_cache(W, max_tokens=8, capacity=32) as c:
        c.cache_fill(0, None, moe.MOE_FILL_FULL_LAYER)
        c.sync()
        st, tr = c.stats(trace_cap=64)
        assert st["prefetch_fills"] == W.E and st["expert_reads"] == 0
        assert np.array_equal(tr, hz.expected_trace(32, [(1, 0, e) for e in range(W.E)]))
        table = c.debug_read(moe.MOE_DBG_SLOT_TABLE, W.E)
        assert table.tolist() == list(range(W.E))  # uploaded before the next compute; read after sync


def test_prefill_db_needs_two_layers_of_capacity():
    with pytest.raises(moe.MoeError) as e:
        moe.MoeCache(moe.LayerShape(2, 16, 256, 128, 2, 31, 8), flags=moe.MOE_PREFILL_DB)
    assert e.value.code == moe.MOE_E_CAPACITY


def test_deterministic_outputs():
    x = mi.activations(0, 4, 8, W.H)
    with hz.make_cache(W, max_tokens=8) as c:
        o1 = _layer(c, x, 8)[2]
        o2 = _layer(c, x, 8)[2]
    assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32))


def test_device_fill_wait_deadline_reports_and_recovers():
    """A decode wave whose kernels wait for a fill generation that is never written (injected
    on the host) gives up after its device-side deadline, raises the device status, and
    leaves the context usable: the next forward matches the oracle."""
    ents = hz.OracleEntries(W)
    with hz.make_cache(W, max_tokens=8) as c:
        x = mi.activations(0, 5, 8, W.H)
        c.debug_inject(3, 1)
        with pytest.raises(moe.MoeError) as e:
            _layer(c, x, 8)  # 8 tokens top-2 over 16 experts with 4 empty slots: fills happen
        assert e.value.code == moe.MOE_E_DEVICE
        assert "5" in str(e.value)
        x2 = mi.activations(0, 6, 8, W.H)
        idx, w, out, resid, Wr, b = _layer(c, x2, 8)
        idx_o, w_o, _, _ = oracle.route(x2, Wr, b, W.k)
        assert np.array_equal(idx, idx_o)
        ref = oracle.moe_layer([ents(0, e_) for e_ in range(W.E)], W.H, W.I, x2, resid, idx_o, w_o)
        hz.assert_out_close(out, ref, resid)


def test_fill_failing_after_its_copy_evicts_the_overwritten_entry():
    """A fill whose copy was already enqueued when it failed (an injected fill-flag write error)
    leaves neither the old nor the new entry resident in that slot: the old entry's bytes are
    being overwritten, so a later hit on it must not read the slot. The next forward refills
    what it needs and matches the oracle."""
    ents = hz.OracleEntries(W)
    with hz.make_cache(W, max_tokens=8, capacity=4) as c:
        c.cache_fill(0, np.array([1, 2, 3, 4]), moe.MOE_FILL_DEMAND)
        c.sync()
        assert [c.resident_slot(0, e) for e in (1, 2, 3, 4)] == [0, 1, 2, 3]
        c.debug_inject(4, 1)
        with pytest.raises(moe.MoeError) as e:
            c.cache_fill(0, np.array([9]), moe.MOE_FILL_DEMAND)  # evicts expert 1 from slot 0
        assert e.value.code == moe.MOE_E_CUDA
        c.sync()
        assert c.resident_slot(0, 1) == -1 and c.resident_slot(0, 9) == -1
        assert [c.resident_slot(0, e) for e in (2, 3, 4)] == [1, 2, 3]
        c.cache_fill(0, np.array([1]), moe.MOE_FILL_DEMAND)  # the freed slot is taken first
        c.sync()
        assert c.resident_slot(0, 1) == 0
        x = mi.activations(0, 7, 8, W.H)
        idx, w, out, resid, Wr, b = _layer(c, x, 8)
        idx_o, w_o, _, _ = oracle.route(x, Wr, b, W.k)
        assert np.array_equal(idx, idx_o)
        ref = oracle.moe_layer([ents(0, e_) for e_ in range(W.E)], W.H, W.I, x, resid, idx_o, w_o)
        hz.assert_out_close(out, ref, resid)
