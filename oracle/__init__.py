"""CPU oracle for the routed-MoE layer with a shared LRU cache of (layer, expert) entries.

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()`` and by the
CPU-baseline leg of ``bench.py``; never by the library.  Thin ctypes wrapper over
oracle.cpp (plain C++, double accumulation), which shares no code with the CUDA path.
See oracle.cpp for the definitions, the page sections they follow and the readings taken
where the pages are silent.  Every function here is pinned by tests/test_oracle_*.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_SO = os.path.join(_HERE, "liboracle.so")

EV_HIT, EV_FILL, EV_PREFETCH_FILL, EV_PREFETCH_HIT = 0, 1, 2, 3
ACCESS_ROUTED, ACCESS_PREFETCH = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.cpp (g++ -O2, OpenMP, no FP contraction, no fast-math)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", _SRC, "-o", tmp])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        i32, dbl, vp = ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.orc_num_threads.restype = i32
        L.orc_set_num_threads.restype = i32
        L.orc_set_num_threads.argtypes = [i32]
        L.orc_router_logits.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp]
        L.orc_topk.argtypes = [vp, i32, i32, i32, vp, vp]
        L.orc_forced_gates.argtypes = [vp, vp, i32, i32, i32, vp, vp]
        L.orc_forced_gates.restype = i32
        L.orc_near_ties.argtypes = [vp, i32, i32, i32, dbl, vp]
        L.orc_near_ties.restype = i32
        L.orc_permute.argtypes = [vp, i32, i32, i32, vp, vp]
        L.orc_permute.restype = i32
        L.orc_expert_ffn.argtypes = [vp, i32, i32, vp, vp]
        L.orc_moe_layer.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, vp, vp]
        L.orc_moe_dense.argtypes = [vp, i32, i32, i32, vp, vp, i32, i32, vp, vp, vp]
        L.orc_mxfp4_dequant.argtypes = [vp, vp, ctypes.c_int64, vp]
        L.orc_mxfp4_dequant.restype = ctypes.c_int64
        L.orc_nvfp4_dequant.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_float, vp]
        L.orc_nvfp4_dequant.restype = ctypes.c_int64
        L.orc_expert_ffn_f64.argtypes = [vp, i32, i32, vp, vp]
        L.orc_moe_layer_f64.argtypes = [vp, i32, i32, vp, vp, i32, i32, vp, vp, vp]
        L.orc_layer_accesses.argtypes = [vp, i32, i32, i32, vp]
        L.orc_layer_accesses.restype = i32
        L.orc_lru_run.argtypes = [i32, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]
        L.orc_lru_run.restype = i32
        _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a) -> int:
    return a.ctypes.data if a is not None else 0


def num_threads() -> int:
    return int(lib().orc_num_threads())


def set_num_threads(n: int) -> int:
    """Threads of the oracle's later parallel regions; returns the previous count."""
    return int(lib().orc_set_num_threads(int(n)))


def router_logits(x_bf16: np.ndarray, Wr: np.ndarray, b: np.ndarray, want_double: bool = True):
    """Router logits (T, E): fp32 in the fixed order, and the same sum in double."""
    x = _c(x_bf16, np.uint16)
    T, H = x.shape
    Wr = _c(Wr, np.float32)
    E = Wr.shape[0]
    if H % 256:
        raise ValueError("hidden size must be a multiple of 256")
    z32 = np.empty((T, E), dtype=np.float32)
    z64 = np.empty((T, E), dtype=np.float64) if want_double else None
    lib().orc_router_logits(_p(x), _p(Wr), _p(_c(b, np.float32)), T, H, E, _p(z32), _p(z64))
    return z32, z64


def topk(z32: np.ndarray, k: int):
    z = _c(z32, np.float32)
    T, E = z.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    lib().orc_topk(_p(z), T, E, k, _p(idx), _p(w))
    return idx, w


def forced_gates(z32: np.ndarray, sets: np.ndarray):
    z = _c(z32, np.float32)
    s = _c(sets, np.int32)
    T, E = z.shape
    k = s.shape[1]
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    if lib().orc_forced_gates(_p(z), _p(s), T, E, k, _p(idx), _p(w)) != 0:
        raise ValueError("forced sets must hold k distinct experts in [0, E)")
    return idx, w


def near_ties(z64: np.ndarray, k: int, eps: float = 1e-5) -> np.ndarray:
    z = _c(z64, np.float64)
    T, E = z.shape
    flag = np.empty(T, dtype=np.int32)
    lib().orc_near_ties(_p(z), T, E, k, eps, _p(flag))
    return flag.astype(bool)


def permute(idx: np.ndarray, E: int):
    i = _c(idx, np.int32)
    T, k = i.shape
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(T * k, dtype=np.int32)
    if lib().orc_permute(_p(i), T, k, E, _p(offsets), _p(perm)) != 0:
        raise ValueError("expert index out of range")
    return offsets, perm


def expert_ffn(entry: np.ndarray, H: int, I: int, x_row: np.ndarray) -> np.ndarray:
    e = _c(entry, np.uint16)
    x = _c(x_row, np.uint16)
    y = np.empty(H, dtype=np.float64)
    lib().orc_expert_ffn(_p(e), H, I, _p(x), _p(y))
    return y


def _entry_table(entries):
    arrs = [_c(e, np.uint16) for e in entries]
    table = (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])
    return table, arrs


def moe_layer(entries, H: int, I: int, x_bf16, resid, idx, w) -> np.ndarray:
    """Sparse routed layer. entries: per-expert bf16 entries of this layer (sequence or dict-like
    indexable by expert id)."""
    x = _c(x_bf16, np.uint16)
    T = x.shape[0]
    idx = _c(idx, np.int32)
    k = idx.shape[1]
    E = int(idx.max()) + 1 if not hasattr(entries, "__len__") else len(entries)
    table, keep = _entry_table([entries[e] for e in range(E)])
    out = np.empty((T, H), dtype=np.float64)
    lib().orc_moe_layer(ctypes.addressof(table), H, I, _p(x), _p(_c(resid, np.float32)), T, k, _p(idx),
                        _p(_c(w, np.float64)), _p(out))
    del keep
    return out


def moe_layer_rows(entry_of, H: int, I: int, x_bf16, resid, idx, w) -> np.ndarray:
    """Sparse routed layer where entry_of(e) returns expert e's entry (only routed experts are fetched)."""
    x = _c(x_bf16, np.uint16)
    T = x.shape[0]
    idx = _c(idx, np.int32)
    k = idx.shape[1]
    used = sorted(set(int(e) for e in idx.ravel()))
    E = max(used) + 1
    cache = {e: _c(entry_of(e), np.uint16) for e in used}
    dummy = np.zeros(1, dtype=np.uint16)
    table = (ctypes.c_void_p * E)(*[(cache[e].ctypes.data if e in cache else dummy.ctypes.data) for e in range(E)])
    out = np.empty((T, H), dtype=np.float64)
    lib().orc_moe_layer(ctypes.addressof(table), H, I, _p(x), _p(_c(resid, np.float32)), T, k, _p(idx),
                        _p(_c(w, np.float64)), _p(out))
    del cache
    return out


def moe_dense(entries, H: int, I: int, x_bf16, resid, idx, w) -> np.ndarray:
    x = _c(x_bf16, np.uint16)
    T = x.shape[0]
    idx = _c(idx, np.int32)
    k = idx.shape[1]
    E = len(entries)
    table, keep = _entry_table(list(entries))
    out = np.empty((T, H), dtype=np.float64)
    lib().orc_moe_dense(ctypes.addressof(table), H, I, E, _p(x), _p(_c(resid, np.float32)), T, k, _p(idx),
                        _p(_c(w, np.float64)), _p(out))
    del keep
    return out


def mxfp4_dequant(q: np.ndarray, s: np.ndarray, n: int) -> np.ndarray:
    """MXFP4 elements (E2M1 bytes q, E8M0 scales s per 32) -> exact bf16 bit patterns."""
    qq, ss = _c(q, np.uint8), _c(s, np.uint8)
    out = np.empty(n, np.uint16)
    bad = lib().orc_mxfp4_dequant(_p(qq), _p(ss), n, _p(out))
    if bad:
        raise ValueError(f"{bad} MXFP4 values are not exact in bf16")
    return out


def mxfp4_entry_as_bf16(entry: np.ndarray, H: int, I: int) -> np.ndarray:
    """An MXFP4 expert entry as the bf16 entry (W_gate | W_up | W_down, row-major) of the same
    values, for the bf16 expert FFN. Entry layout, in stages of 4096 code bytes + 256 scale
    bytes: for W_gate/W_up, per 64-row tile and 64-column slab: gate rows (64 x 32 bytes), up
    rows (64 x 32), gate scales (64 x 2), up scales (64 x 2); then for W_down, per 128-row tile
    and slab: rows (128 x 32), scales (128 x 2). A row's 32 bytes hold its two 32-blocks of the
    slab, with the scale bytes in the same order."""
    st = 4352
    gu = (I // 64) * (H // 64) * st
    a = entry[:gu].reshape(I // 64, H // 64, st)
    gate_q = a[:, :, :2048].reshape(I // 64, H // 64, 64, 32).transpose(0, 2, 1, 3).reshape(I, H // 2)
    up_q = a[:, :, 2048:4096].reshape(I // 64, H // 64, 64, 32).transpose(0, 2, 1, 3).reshape(I, H // 2)
    gate_s = a[:, :, 4096:4224].reshape(I // 64, H // 64, 64, 2).transpose(0, 2, 1, 3).reshape(I, H // 32)
    up_s = a[:, :, 4224:4352].reshape(I // 64, H // 64, 64, 2).transpose(0, 2, 1, 3).reshape(I, H // 32)
    d = entry[gu:].reshape(H // 128, I // 64, st)
    down_q = d[:, :, :4096].reshape(H // 128, I // 64, 128, 32).transpose(0, 2, 1, 3).reshape(H, I // 2)
    down_s = d[:, :, 4096:].reshape(H // 128, I // 64, 128, 2).transpose(0, 2, 1, 3).reshape(H, I // 32)
    q = np.concatenate([gate_q.ravel(), up_q.ravel(), down_q.ravel()])
    s = np.concatenate([gate_s.ravel(), up_s.ravel(), down_s.ravel()])
    return mxfp4_dequant(q, s, 3 * H * I)


def nvfp4_dequant(q: np.ndarray, s: np.ndarray, n: int, tensor_scale: float) -> np.ndarray:
    """NVFP4 elements of one matrix (E2M1 bytes q, E4M3 scales s per 16, fp32 tensor scale)
    -> their exact values in float64."""
    qq, ss = _c(q, np.uint8), _c(s, np.uint8)
    out = np.empty(n, np.float64)
    bad = lib().orc_nvfp4_dequant(_p(qq), _p(ss), n, float(tensor_scale), _p(out))
    if bad:
        raise ValueError(f"{bad} NVFP4 block scales are not valid E4M3 scales")
    return out


def nvfp4_entry_as_f64(entry: np.ndarray, H: int, I: int) -> np.ndarray:
    """An NVFP4 expert entry as the float64 weights W_gate | W_up | W_down (row-major). Entry
    layout, in stages of 4096 code bytes + 512 scale bytes: for W_gate/W_up, per 64-row tile
    and 64-column slab: gate rows (64 x 32 bytes), up rows (64 x 32), gate scales (64 x 4), up
    scales (64 x 4); then for W_down, per 128-row tile and slab: rows (128 x 32), scales
    (128 x 4); then the fp32 tensor scales of W_gate, W_up, W_down and 4 zero bytes."""
    st = 4608
    gu = (I // 64) * (H // 64) * st
    a = entry[:gu].reshape(I // 64, H // 64, st)
    gate_q = a[:, :, :2048].reshape(I // 64, H // 64, 64, 32).transpose(0, 2, 1, 3).reshape(I, H // 2)
    up_q = a[:, :, 2048:4096].reshape(I // 64, H // 64, 64, 32).transpose(0, 2, 1, 3).reshape(I, H // 2)
    gate_s = a[:, :, 4096:4352].reshape(I // 64, H // 64, 64, 4).transpose(0, 2, 1, 3).reshape(I, H // 16)
    up_s = a[:, :, 4352:4608].reshape(I // 64, H // 64, 64, 4).transpose(0, 2, 1, 3).reshape(I, H // 16)
    dn = (H // 128) * (I // 64) * st
    d = entry[gu:gu + dn].reshape(H // 128, I // 64, st)
    down_q = d[:, :, :4096].reshape(H // 128, I // 64, 128, 32).transpose(0, 2, 1, 3).reshape(H, I // 2)
    down_s = d[:, :, 4096:].reshape(H // 128, I // 64, 128, 4).transpose(0, 2, 1, 3).reshape(H, I // 16)
    t = np.frombuffer(entry[gu + dn:gu + dn + 12].tobytes(), dtype=np.float32)
    return np.concatenate([nvfp4_dequant(gate_q, gate_s, I * H, t[0]), nvfp4_dequant(up_q, up_s, I * H, t[1]),
                           nvfp4_dequant(down_q, down_s, H * I, t[2])])


def expert_ffn_f64(W: np.ndarray, H: int, I: int, x_row: np.ndarray) -> np.ndarray:
    """orc_expert_ffn with float64 weights W_gate | W_up | W_down (row-major)."""
    w = _c(W, np.float64)
    x = _c(x_row, np.uint16)
    y = np.empty(H, dtype=np.float64)
    lib().orc_expert_ffn_f64(_p(w), H, I, _p(x), _p(y))
    return y


def moe_layer_rows_f64(entry_of, H: int, I: int, x_bf16, resid, idx, w) -> np.ndarray:
    """moe_layer_rows for experts given as float64 weights: entry_of(e) returns expert e's
    W_gate | W_up | W_down as float64 (e.g. nvfp4_entry_as_f64); only routed experts are fetched."""
    x = _c(x_bf16, np.uint16)
    T = x.shape[0]
    idx = _c(idx, np.int32)
    k = idx.shape[1]
    used = sorted(set(int(e) for e in idx.ravel()))
    E = max(used) + 1
    cache = {e: _c(entry_of(e), np.float64) for e in used}
    dummy = np.zeros(1, dtype=np.float64)
    table = (ctypes.c_void_p * E)(*[(cache[e].ctypes.data if e in cache else dummy.ctypes.data) for e in range(E)])
    out = np.empty((T, H), dtype=np.float64)
    lib().orc_moe_layer_f64(ctypes.addressof(table), H, I, _p(x), _p(_c(resid, np.float32)), T, k, _p(idx),
                            _p(_c(w, np.float64)), _p(out))
    del cache
    return out


def layer_accesses(idx: np.ndarray, E: int) -> np.ndarray:
    i = _c(idx, np.int32)
    T, k = i.shape
    out = np.empty(E, dtype=np.int32)
    n = lib().orc_layer_accesses(_p(i), T, k, E, _p(out))
    return out[:n].copy()


def lru_run(capacity: int, layers, experts, kinds=None) -> np.ndarray:
    """Run the LRU over an operation sequence (kind 0 routed access, 1 prefetch, 2 capacity
    change to `experts[i]` slots). Returns events as an int32 array (n_events, 6):
    (kind, layer, expert, slot, evicted_layer, evicted_expert); kind 4 = evicted by a
    capacity change."""
    l = _c(layers, np.int32)
    e = _c(experts, np.int32)
    n = len(l)
    kd = _c(np.zeros(n) if kinds is None else kinds, np.int32)
    cap_max = int(max([capacity] + [int(x) for x, k in zip(e, kd) if k == 2]))
    m = n + cap_max * int(np.sum(kd == 2)) + 1
    outs = [np.empty(m, np.int32) for _ in range(6)]
    got = lib().orc_lru_run(capacity, n, _p(l), _p(e), _p(kd), m, *[_p(o) for o in outs])
    if got < 0:
        raise ValueError("capacity must be >= 1")
    return np.stack([o[:got] for o in outs], axis=1)


def route(x_bf16, Wr, b, k):
    """Router + top-k + gates for one layer: (idx, w, z32, z64)."""
    z32, z64 = router_logits(x_bf16, Wr, b)
    idx, w = topk(z32, k)
    return idx, w, z32, z64
