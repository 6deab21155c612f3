"""Seeded synthetic inputs shared by the CUDA library's tests/bench and the CPU oracle.

Holds no arithmetic of the MoE method: it only draws random numbers (Philox-4x32-10,
Salmon et al., SC'11) and lays them out.  Both sides of every parity check consume
the identical bytes produced here.

Tensor streams (one Philox stream per tensor):
  expert entry (l, e)   -> N(0, 0.02) bf16, 3*H*I elements laid out [W_gate I*H | W_up I*H | W_down H*I]
  router weights (l)    -> N(0, 0.02) fp32 [E*H]
  activations (step)    -> N(0, 1) bf16 [T*H]
  router bias (l)       -> ln of Zipf(s) rank probabilities under a seeded permutation, fp32 [E]
  reuse trace           -> forced top-k sets for the multi-layer decode stream
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libmoe_inputs.so")
_SRC = os.path.join(_HERE, "gen.c")

KIND_EXPERT, KIND_ROUTER, KIND_X, KIND_PERM, KIND_TRACE = 1, 2, 3, 4, 5


def build(force: bool = False) -> str:
    """Compile gen.c into libmoe_inputs.so next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        u64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        L.mi_philox4x32_10.argtypes = [vp, vp, vp]
        L.mi_normal_bf16.argtypes = [u64, u64, u64, u64, dbl, vp]
        L.mi_normal_f32.argtypes = [u64, u64, u64, u64, dbl, vp]
        L.mi_uniform_u32.argtypes = [u64, u64, u64, u64, vp]
        L.mi_zipf_bias.argtypes = [u64, u64, i32, dbl, vp, vp]
        L.mi_trace_reuse.argtypes = [u64, u64, i32, i32, i32, i32, i32, dbl, dbl, vp, vp]
        L.mi_trace_reuse.restype = i32
        L.mi_f32_to_bf16.argtypes = [ctypes.c_float]
        L.mi_f32_to_bf16.restype = ctypes.c_uint16
        _lib = L
    return _lib


def stream_id(kind: int, a: int = 0, b: int = 0) -> int:
    assert 0 <= a < (1 << 28) and 0 <= b < (1 << 28)
    return (kind << 56) | (a << 28) | b


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().mi_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def normal_bf16(seed: int, stream: int, n: int, std: float, first: int = 0, out: Optional[np.ndarray] = None) -> np.ndarray:
    if out is None:
        out = np.empty(n, dtype=np.uint16)
    lib().mi_normal_bf16(seed, stream, first, n, std, _ptr(out))
    return out


def normal_f32(seed: int, stream: int, n: int, std: float, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    lib().mi_normal_f32(seed, stream, first, n, std, _ptr(out))
    return out


def uniform_u32(seed: int, stream: int, n: int, first: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    lib().mi_uniform_u32(seed, stream, first, n, _ptr(out))
    return out


def f32_to_bf16_bits(x: float) -> int:
    return int(lib().mi_f32_to_bf16(float(x)))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------- tensors
def expert_entry(seed: int, layer: int, expert: int, H: int, I: int) -> np.ndarray:
    """Entry (layer, expert): bf16 bits [W_gate (I,H) | W_up (I,H) | W_down (H,I)], N(0, 0.02)."""
    return normal_bf16(seed, stream_id(KIND_EXPERT, layer, expert), 3 * H * I, 0.02)


def fill_entry_at(ptr: int, seed: int, layer: int, expert: int, H: int, I: int) -> None:
    """Write entry (layer, expert) straight into host memory at `ptr` (3*H*I bf16)."""
    lib().mi_normal_bf16(seed, stream_id(KIND_EXPERT, layer, expert), 0, 3 * H * I, 0.02, ptr)


def router_weights(seed: int, layer: int, E: int, H: int) -> np.ndarray:
    """Router matrix W_r (E, H) fp32, N(0, 0.02)."""
    return normal_f32(seed, stream_id(KIND_ROUTER, layer), E * H, 0.02).reshape(E, H)


def router_bias(seed: int, layer: int, E: int, zipf_s: Optional[float]):
    """(bias fp32 [E], perm int32 [E] rank->expert).  zipf_s None -> zero bias, identity perm."""
    if zipf_s is None:
        return np.zeros(E, dtype=np.float32), np.arange(E, dtype=np.int32)
    perm = np.empty(E, dtype=np.int32)
    bias = np.empty(E, dtype=np.float32)
    lib().mi_zipf_bias(seed, stream_id(KIND_PERM, layer), E, float(zipf_s), _ptr(perm), _ptr(bias))
    return bias, perm


def activations(seed: int, step: int, T: int, H: int) -> np.ndarray:
    """Activations x (T, H) as bf16 bits, N(0, 1); a fresh stream per step."""
    return normal_bf16(seed, stream_id(KIND_X, step), T * H, 1.0).reshape(T, H)


def trace_reuse(seed: int, L: int, steps: int, B: int, E: int, k: int, zipf_s: float, p_reuse: float,
                perms: np.ndarray) -> np.ndarray:
    """Forced top-k sets [steps, L, B, k] with step-to-step reuse (see gen.c)."""
    perms = np.ascontiguousarray(perms, dtype=np.int32).reshape(L, E)
    out = np.empty((steps, L, B, k), dtype=np.int32)
    rc = lib().mi_trace_reuse(seed, stream_id(KIND_TRACE), L, steps, B, E, k, float(zipf_s), float(p_reuse),
                              _ptr(perms), _ptr(out))
    if rc != 0:
        raise ValueError("trace_reuse: k must be in [1, E]")
    return out


# ----------------------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Workload:
    """One synthetic workload, named by what it is."""
    name: str
    H: int          # hidden size
    I: int          # expert SwiGLU intermediate size
    E: int          # routed experts per layer
    k: int          # experts per token
    L: int          # layers sharing the cache
    C: int          # cache capacity in whole (layer, expert) entries
    zipf_s: Optional[float]   # router-bias Zipf exponent (None: zero bias)
    seed: int = 0

    @property
    def entry_elems(self) -> int:
        return 3 * self.H * self.I

    @property
    def entry_bytes(self) -> int:
        return 2 * self.entry_elems


WORKLOADS = {
    # single layer, hidden 256, intermediate 128, 16 experts, top-2, 8 tokens, 4 cache slots
    "tiny": Workload("tiny", 256, 128, 16, 2, 1, 4, None),
    # decode layer, hidden 4096, intermediate 1536, 256 experts top-6, 64-entry cache, batch 1/4/16
    "decode": Workload("decode", 4096, 1536, 256, 6, 1, 64, 1.1),
    # prefill layer of the same shape, 4096 tokens, every expert resident
    "prefill": Workload("prefill", 4096, 1536, 256, 6, 1, 256, 1.1),
    # 8-layer decode stream, batch 8, 512 steps, cache of 30% of 2048 entries
    "stream8": Workload("stream8", 4096, 1536, 256, 6, 8, int(0.3 * 2048), 1.1),
    # 48-layer stack, 128 experts top-8, hidden 2048, intermediate 768, cache of 25% of entries
    "stack48": Workload("stack48", 2048, 768, 128, 8, 48, int(0.25 * 48 * 128), 1.1),
}
