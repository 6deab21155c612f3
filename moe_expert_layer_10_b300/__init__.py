"""Python binding of libmoe_b300.so: the routed-MoE layer with a shared VRAM LRU cache of
whole (layer, expert) entries and the complete expert pool in pinned host memory.

Argument marshalling only: every step of the hot path runs in the library's CUDA kernels.
The names mirror include/moe.h (moe_cache_init -> MoeCache, moe_route -> MoeCache.route, ...).
Device buffers are torch CUDA tensors, passed as raw pointers; torch provides memory and
streams, nothing else. There is no CPU fallback: if the library is missing this module
raises at import of the library handle.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_b300.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "moe.h")

MOE_OK, MOE_E_INVAL, MOE_E_NOMEM, MOE_E_CUDA, MOE_E_TIMEOUT, MOE_E_CAPACITY, MOE_E_DEVICE = 0, -1, -2, -3, -4, -5, -6
MOE_TRACE, MOE_PROFILE, MOE_PREFILL_DB, MOE_DEVICE_POLICY, MOE_MXFP4, MOE_NVFP4 = 1, 2, 4, 8, 16, 32
MOE_FILL_DEMAND, MOE_FILL_FULL_LAYER = 0, 1
MOE_PATH_AUTO, MOE_PATH_GEMV, MOE_PATH_GEMM, MOE_PATH_GEMV_UNFUSED = 0, 1, 2, 3
EV_HIT, EV_FILL, EV_PREFETCH_FILL, EV_PREFETCH_HIT, EV_RESIZE_EVICT, EV_HOST_EXEC = 0, 1, 2, 3, 4, 5

# every symbol include/moe.h declares
EXPORTS = ["moe_cache_init", "moe_cache_destroy", "moe_host_entry", "moe_entry_bytes", "moe_route",
           "moe_route_forced", "moe_cache_fill", "moe_layer_forward", "moe_stats", "moe_last_error",
           "moe_set_path", "moe_set_profile", "moe_sync", "moe_resident_slot", "moe_kernel_stats", "moe_lru_simulate",
           "moe_debug_inject", "moe_debug_read", "moe_route_noalloc", "moe_cache_resize", "moe_measure_bandwidth",
           "moe_host_expert_ffn", "moe_qstar_fills", "moe_qstar_simulate", "moe_fused_schedule"]
MOE_NOALLOC_MAX_LOGITS = 65536
MOE_DBG_OFFSETS, MOE_DBG_PERM, MOE_DBG_INV_PERM, MOE_DBG_ACTIVE, MOE_DBG_N_ACTIVE, MOE_DBG_SLOT_TABLE, \
    MOE_DBG_H_PERM, MOE_DBG_X_PERM, MOE_DBG_W_PERM = range(9)


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where} failed ({code}): {msg}")
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_experts", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("top_k", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("flags", ctypes.c_uint32), ("trace_capacity", ctypes.c_uint64)]


class Stats(ctypes.Structure):
    _fields_ = [("expert_reads", ctypes.c_uint64), ("hits", ctypes.c_uint64), ("misses", ctypes.c_uint64),
                ("prefetch_fills", ctypes.c_uint64), ("prefetch_hits", ctypes.c_uint64),
                ("evictions", ctypes.c_uint64), ("fill_bytes", ctypes.c_uint64), ("fill_ms", ctypes.c_double),
                ("trace_len", ctypes.c_uint64), ("forwards", ctypes.c_uint64), ("waves", ctypes.c_uint64),
                ("resize_evictions", ctypes.c_uint64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class Event(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("layer", ctypes.c_int32), ("expert", ctypes.c_int32),
                ("slot", ctypes.c_int32), ("ev_layer", ctypes.c_int32), ("ev_expert", ctypes.c_int32)]


class Bandwidth(ctypes.Structure):
    _fields_ = [("pcie_h2d_gbps", ctypes.c_double), ("host_expert_gbps", ctypes.c_double),
                ("host_threads", ctypes.c_int32), ("pad", ctypes.c_int32), ("entry_bytes", ctypes.c_double)]


class QstarSim(ctypes.Structure):
    _fields_ = [("expert_reads", ctypes.c_uint64), ("hits", ctypes.c_uint64), ("fills", ctypes.c_uint64),
                ("host_execs", ctypes.c_uint64), ("evictions", ctypes.c_uint64), ("events", ctypes.c_uint64),
                ("modeled_ms", ctypes.c_double), ("link_ms", ctypes.c_double), ("host_ms", ctypes.c_double)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class KernelStat(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_uint64), ("total_ms", ctypes.c_double),
                ("bytes", ctypes.c_double), ("flops", ctypes.c_double)]


_lib = None


def lib():
    """Load libmoe_b300.so (raises if it was not built: there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing; build it with `python -m moe_expert_layer_10_b300.build`")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
    L.moe_cache_init.argtypes = [ctypes.POINTER(Config), vp, vp, ctypes.POINTER(vp)]
    L.moe_cache_destroy.argtypes = [vp]
    L.moe_cache_destroy.restype = None
    L.moe_host_entry.argtypes = [vp, i32, i32]
    L.moe_host_entry.restype = vp
    L.moe_entry_bytes.argtypes = [vp]
    L.moe_entry_bytes.restype = u64
    L.moe_route.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, vp]
    L.moe_route_forced.argtypes = [vp, i32, vp, i32, vp, vp, vp, vp, vp, vp]
    L.moe_cache_fill.argtypes = [vp, i32, vp, i32, i32]
    L.moe_layer_forward.argtypes = [vp, i32, vp, vp, vp, i32, vp, vp]
    L.moe_stats.argtypes = [vp, ctypes.POINTER(Stats), vp, u64, i32]
    L.moe_last_error.restype = ctypes.c_char_p
    L.moe_set_path.argtypes = [vp, i32]
    L.moe_set_profile.argtypes = [vp, i32]
    L.moe_sync.argtypes = [vp]
    L.moe_resident_slot.argtypes = [vp, i32, i32]
    L.moe_kernel_stats.argtypes = [vp, vp, i32, i32]
    L.moe_lru_simulate.argtypes = [i32, i32, vp, vp, vp, vp, u64]
    L.moe_cache_resize.argtypes = [vp, i32]
    L.moe_debug_inject.argtypes = [vp, i32, i32]
    L.moe_debug_read.argtypes = [vp, i32, vp, u64]
    L.moe_route_noalloc.argtypes = [vp, i32, i32, i32, i32, vp, vp, vp, vp, vp]
    dbl = ctypes.c_double
    L.moe_measure_bandwidth.argtypes = [vp, i32, i32, ctypes.POINTER(Bandwidth)]
    L.moe_host_expert_ffn.argtypes = [vp, i32, i32, vp, i32, vp, i32]
    L.moe_qstar_fills.argtypes = [dbl, dbl, i32]
    L.moe_fused_schedule.argtypes = [i32, i32, i32, i32, i32, vp, i32]
    L.moe_qstar_simulate.argtypes = [i32, i32, vp, vp, vp, vp, dbl, dbl, dbl, dbl, dbl, ctypes.POINTER(QstarSim),
                                     vp, u64]
    _lib = L
    return L


def last_error() -> str:
    return lib().moe_last_error().decode(errors="replace")


def _check(rc: int, where: str) -> int:
    if rc < 0:
        raise MoeError(rc, where, last_error())
    return rc


def _ptr(t) -> int:
    """Raw data pointer of a torch tensor (or an int / None)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_handle(stream) -> int:
    if stream is None:
        return 0
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def lru_simulate(capacity: int, layers, experts, kinds=None):
    """Run the library's host LRU policy on an operation sequence (no GPU): kind 0 routed
    access, 1 prefetch, 2 capacity change to experts[i] slots. Returns rows (kind, layer,
    expert, slot, evicted_layer, evicted_expert), one per access and one per entry evicted by
    a capacity change (kind 4)."""
    import numpy as np
    l = np.ascontiguousarray(layers, dtype=np.int32)
    e = np.ascontiguousarray(experts, dtype=np.int32)
    n = len(l)
    k = np.ascontiguousarray(np.zeros(n) if kinds is None else kinds, dtype=np.int32)
    cap_max = int(max([capacity] + [int(x) for x, kk in zip(e, k) if kk == 2]))
    m = n + cap_max * int(np.sum(k == 2)) + 1
    ev = (Event * m)()
    got = _check(lib().moe_lru_simulate(capacity, n, l.ctypes.data, e.ctypes.data, k.ctypes.data,
                                        ctypes.addressof(ev), m), "moe_lru_simulate")
    return np.array([[ev[i].kind, ev[i].layer, ev[i].expert, ev[i].slot, ev[i].ev_layer, ev[i].ev_expert]
                     for i in range(got)], dtype=np.int32).reshape(got, 6)


def route_noalloc(x, router_w, router_b, topk_idx, topk_w, top_k: int, stream=None, T: Optional[int] = None):
    """moe_route_noalloc: the router without a context or any allocation (see include/moe.h)."""
    T = x.shape[0] if T is None else T
    _check(lib().moe_route_noalloc(_ptr(x), T, x.shape[1], router_w.shape[0], top_k, _ptr(router_w), _ptr(router_b),
                                   _ptr(topk_idx), _ptr(topk_w), _stream_handle(stream)), "moe_route_noalloc")


def host_expert_ffn(entry_bf16, hidden: int, inter: int, x_bf16, threads: int = 1):
    """moe_host_expert_ffn: the expert FFN on the host cores (numpy uint16 entry and tokens [n x hidden]);
    returns fp32 [n x hidden]."""
    import numpy as np
    e = np.ascontiguousarray(entry_bf16, dtype=np.uint16)
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16).reshape(-1, hidden)
    y = np.empty((x.shape[0], hidden), dtype=np.float32)
    _check(lib().moe_host_expert_ffn(e.ctypes.data, hidden, inter, x.ctypes.data, x.shape[0], y.ctypes.data, threads),
           "moe_host_expert_ffn")
    return y


def fused_schedule(units_gu: int, units_d: int, kb_gu: int, kb_d: int, grid: int, cap: int = 1024):
    """moe_fused_schedule: (keep, pool_off, pool) of the fused decode launch's unit schedule, or
    None when the plain round robin is as level."""
    import numpy as np
    buf = np.zeros(max(cap, 1), np.int32)
    n = _check(lib().moe_fused_schedule(int(units_gu), int(units_d), int(kb_gu), int(kb_d), int(grid),
                                        buf.ctypes.data, int(cap)), "moe_fused_schedule")
    if n == 0:
        return None
    keep, off = buf[:grid].copy(), buf[grid:2 * grid + 1].copy()
    return keep, off, buf[2 * grid + 1:2 * grid + 1 + off[grid]].copy()


def qstar_fills(pcie_gbps: float, host_gbps: float, n_miss: int) -> int:
    """moe_qstar_fills: how many of n_miss misses fill under the q-star split."""
    return _check(lib().moe_qstar_fills(float(pcie_gbps), float(host_gbps), int(n_miss)), "moe_qstar_fills")


def qstar_simulate(capacity: int, invocations, q: float, pcie_gbps: float, host_gbps: float, hbm_gbps: float,
                   entry_bytes: float, want_events: bool = False):
    """moe_qstar_simulate on a list of invocations, each a list of (layer, expert, n_tok) in
    ascending expert id. q < 0 uses the bandwidth rule. Returns (summary dict, events or None)."""
    import numpy as np
    offs = np.zeros(len(invocations) + 1, np.int32)
    rows = []
    for v, inv in enumerate(invocations):
        rows += list(inv)
        offs[v + 1] = len(rows)
    a = np.array(rows, np.int32).reshape(-1, 3) if rows else np.zeros((0, 3), np.int32)
    lay, exp_, ntk = (np.ascontiguousarray(a[:, i]) for i in range(3))
    s = QstarSim()
    cap = len(rows) + 1 if want_events else 0
    ev = (Event * cap)() if want_events else None
    got = _check(lib().moe_qstar_simulate(capacity, len(invocations), offs.ctypes.data, lay.ctypes.data,
                                          exp_.ctypes.data, ntk.ctypes.data, float(q), float(pcie_gbps),
                                          float(host_gbps), float(hbm_gbps), float(entry_bytes), ctypes.byref(s),
                                          ctypes.addressof(ev) if want_events else None, cap), "moe_qstar_simulate")
    events = None
    if want_events:
        events = np.array([[ev[i].kind, ev[i].layer, ev[i].expert, ev[i].slot, ev[i].ev_layer, ev[i].ev_expert]
                           for i in range(got)], dtype=np.int32).reshape(got, 6)
    return s.as_dict(), events


@dataclass
class LayerShape:
    num_layers: int
    num_experts: int
    hidden: int
    inter: int
    top_k: int
    capacity: int
    max_tokens: int


class MoeCache:
    """One moe_ctx: pinned host pool, VRAM slot arena, LRU, streams and scratch."""

    def __init__(self, shape: LayerShape, flags: int = 0, trace_capacity: int = 0, stream_compute=None,
                 stream_copy=None):
        self.shape = shape
        self.shape_flags = flags
        cfg = Config(shape.num_layers, shape.num_experts, shape.hidden, shape.inter, shape.top_k, shape.capacity,
                     shape.max_tokens, flags, trace_capacity)
        h = ctypes.c_void_p()
        _check(lib().moe_cache_init(ctypes.byref(cfg), _stream_handle(stream_compute), _stream_handle(stream_copy),
                                    ctypes.byref(h)), "moe_cache_init")
        self._h = h
        self.entry_bytes = int(lib().moe_entry_bytes(h))

    # -- lifetime
    def close(self):
        if self._h:
            lib().moe_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # -- pool
    def host_entry(self, layer: int, expert: int) -> int:
        p = lib().moe_host_entry(self._h, layer, expert)
        if not p:
            raise MoeError(MOE_E_INVAL, "moe_host_entry", f"({layer}, {expert}) out of range")
        return p

    def host_entry_bytes(self, layer: int, expert: int):
        """The pinned pool's entry (layer, expert) as a writable uint8 numpy view."""
        import numpy as np
        return np.ctypeslib.as_array((ctypes.c_uint8 * self.entry_bytes).from_address(self.host_entry(layer, expert)))

    def host_entry_array(self, layer: int, expert: int):
        """numpy uint16 view of entry (layer, expert) in the pinned pool (writable in place)."""
        import numpy as np
        n = self.entry_bytes // 2
        buf = (ctypes.c_uint16 * n).from_address(self.host_entry(layer, expert))
        return np.ctypeslib.as_array(buf)

    # -- hot path
    def route(self, layer, x, router_w, router_b, topk_idx, topk_w, logits=None, T: Optional[int] = None):
        T = x.shape[0] if T is None else T
        _check(lib().moe_route(self._h, layer, _ptr(x), T, _ptr(router_w), _ptr(router_b), _ptr(topk_idx),
                               _ptr(topk_w), _ptr(logits)), "moe_route")

    def route_forced(self, layer, x, router_w, router_b, forced_sets, topk_idx, topk_w, logits=None,
                     T: Optional[int] = None):
        T = x.shape[0] if T is None else T
        _check(lib().moe_route_forced(self._h, layer, _ptr(x), T, _ptr(router_w), _ptr(router_b),
                                      _ptr(forced_sets), _ptr(topk_idx), _ptr(topk_w), _ptr(logits)),
               "moe_route_forced")

    def cache_fill(self, layer: int, topk_idx_host=None, mode: int = MOE_FILL_DEMAND):
        import numpy as np
        if topk_idx_host is None:
            return _check(lib().moe_cache_fill(self._h, layer, None, 0, mode), "moe_cache_fill")
        a = np.ascontiguousarray(topk_idx_host, dtype=np.int32).ravel()
        return _check(lib().moe_cache_fill(self._h, layer, a.ctypes.data, a.size, mode), "moe_cache_fill")

    def layer_forward(self, layer, x, resid, out, topk_idx, topk_w, T: Optional[int] = None):
        T = x.shape[0] if T is None else T
        _check(lib().moe_layer_forward(self._h, layer, _ptr(x), _ptr(resid), _ptr(out), T, _ptr(topk_idx),
                                       _ptr(topk_w)), "moe_layer_forward")

    def resize(self, capacity: int):
        """Elastic cache: change the capacity at a safe point (waits for enqueued work)."""
        _check(lib().moe_cache_resize(self._h, capacity), "moe_cache_resize")

    def set_path(self, path: int):
        _check(lib().moe_set_path(self._h, path), "moe_set_path")

    def set_profile(self, on: bool):
        _check(lib().moe_set_profile(self._h, 1 if on else 0), "moe_set_profile")

    def sync(self):
        _check(lib().moe_sync(self._h), "moe_sync")

    def resident_slot(self, layer: int, expert: int) -> int:
        return int(lib().moe_resident_slot(self._h, layer, expert))

    def debug_inject(self, kind: int, count: int):
        _check(lib().moe_debug_inject(self._h, kind, count), "moe_debug_inject")

    def debug_read(self, what: int, count: int, dtype="int32"):
        import numpy as np
        out = np.empty(count, dtype=dtype)
        _check(lib().moe_debug_read(self._h, what, out.ctypes.data, out.nbytes), "moe_debug_read")
        return out

    # -- introspection
    def stats(self, reset: bool = False, trace_cap: int = 0):
        import numpy as np
        s = Stats()
        if trace_cap:
            ev = (Event * trace_cap)()
            n = _check(lib().moe_stats(self._h, ctypes.byref(s), ctypes.addressof(ev), trace_cap, int(reset)),
                       "moe_stats")
            tr = np.array([[ev[i].kind, ev[i].layer, ev[i].expert, ev[i].slot, ev[i].ev_layer, ev[i].ev_expert]
                           for i in range(n)], dtype=np.int32).reshape(n, 6)
            return s.as_dict(), tr
        _check(lib().moe_stats(self._h, ctypes.byref(s), None, 0, int(reset)), "moe_stats")
        return s.as_dict()

    def measure_bandwidth(self, host_threads: int, reps: int = 5):
        """moe_measure_bandwidth: pinned H2D and host expert-FFN bandwidth (GB/s) on entry (0, 0)."""
        b = Bandwidth()
        _check(lib().moe_measure_bandwidth(self._h, host_threads, reps, ctypes.byref(b)), "moe_measure_bandwidth")
        return {"pcie_h2d_gbps": b.pcie_h2d_gbps, "host_expert_gbps": b.host_expert_gbps,
                "host_threads": b.host_threads, "entry_bytes": b.entry_bytes}

    def kernel_stats(self, reset: bool = False):
        arr = (KernelStat * 16)()
        n = _check(lib().moe_kernel_stats(self._h, ctypes.addressof(arr), 16, int(reset)), "moe_kernel_stats")
        return {arr[i].name.decode(): {"launches": arr[i].launches, "total_ms": arr[i].total_ms,
                                       "bytes": arr[i].bytes, "flops": arr[i].flops} for i in range(n)}
