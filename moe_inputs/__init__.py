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


_CORE = os.path.join(_HERE, "normal_core.h")
_CORE_FP4 = os.path.join(_HERE, "mxfp4_core.h")
_CORE_NVFP4 = os.path.join(_HERE, "nvfp4_core.h")
_SO_FMA = os.path.join(_HERE, "libmoe_inputs_fma.so")


def _cpu_has_fma() -> bool:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("flags"):
                    return " fma " in line + " "
    except OSError:
        pass
    return False
_GPU_SRC = os.path.join(_HERE, "gen_gpu.cu")
_GPU_SO = os.path.join(_HERE, "libmoe_inputs_gpu.so")
_NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _stale(out: str, *srcs: str) -> bool:
    return not os.path.exists(out) or os.path.getmtime(out) < max(os.path.getmtime(s) for s in srcs)


def build(force: bool = False) -> str:
    """Compile gen.c into libmoe_inputs.so (gcc, OpenMP) and gen_gpu.cu into
    libmoe_inputs_gpu.so (nvcc, sm_103a) next to them. Neither build contracts a*b+c."""
    # two CPU builds: one that calls fma() from libm, and one that uses the FMA instruction
    # (loaded only on CPUs that have it); fused multiply-add rounds once either way, so the
    # bits are the same
    for so, extra in ((_SO, []), (_SO_FMA, ["-mfma"])):
        if force or _stale(so, _SRC, _CORE, _CORE_FP4, _CORE_NVFP4):
            tmp = so + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC", "-std=c11"] +
                                  extra + [_SRC, "-o", tmp, "-lm"])
            os.replace(tmp, so)
    if os.path.exists(_NVCC) and (force or _stale(_GPU_SO, _GPU_SRC, _CORE, _CORE_FP4, _CORE_NVFP4)):
        tmp = _GPU_SO + f".tmp{os.getpid()}"
        subprocess.check_call([_NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false",
                               "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
                               "-cudart", "shared", _GPU_SRC, "-o", tmp])
        os.replace(tmp, _GPU_SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO_FMA if _cpu_has_fma() else _SO)
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
        L.mi_mxfp4_entry.argtypes = [u64, u64, i32, i32, vp]
        L.mi_mxfp4_block32.argtypes = [vp, vp, vp]
        L.mi_nvfp4_entry.argtypes = [u64, u64, i32, i32, vp]
        L.mi_nvfp4_block16.argtypes = [vp, ctypes.c_float, vp, vp]
        L.mi_e4m3_encode.argtypes = [ctypes.c_float]
        L.mi_e4m3_encode.restype = ctypes.c_uint8
        L.mi_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.mi_e4m3_decode.restype = ctypes.c_float
        L.mi_nvfp4_tscale.argtypes = [ctypes.c_float]
        L.mi_nvfp4_tscale.restype = ctypes.c_float
        L.mi_nvfp4_bytes.argtypes = [i32, i32]
        L.mi_nvfp4_bytes.restype = u64
        L.mi_log_unit.argtypes = [dbl]
        L.mi_log_unit.restype = dbl
        L.mi_sincos_2pi.argtypes = [dbl, vp, vp]
        _lib = L
    return _lib


_gpu_lib = None


def gpu_lib():
    """The GPU build of the generator (needs a CUDA device at call time)."""
    global _gpu_lib
    if _gpu_lib is None:
        build()
        L = ctypes.CDLL(_GPU_SO)
        L.mi_gpu_normal_bf16_to_host.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64,
                                                 ctypes.c_double, ctypes.c_void_p, ctypes.c_char_p, ctypes.c_int]
        L.mi_gpu_mxfp4_entries_to_host.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_char_p,
                                                   ctypes.c_int]
        L.mi_gpu_nvfp4_entries_to_host.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
                                                   ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_char_p,
                                                   ctypes.c_int]
        _gpu_lib = L
    return _gpu_lib


def log_unit(x: float) -> float:
    """The generator's own series logarithm (the one its normal transform uses)."""
    return float(lib().mi_log_unit(float(x)))


def sincos_turn(u: float):
    """(sin, cos) of 2*pi*u by the generator's own series (u in [0, 1))."""
    s, c = ctypes.c_double(), ctypes.c_double()
    lib().mi_sincos_2pi(float(u), ctypes.byref(s), ctypes.byref(c))
    return s.value, c.value


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


def mxfp4_entry_bytes(H: int, I: int) -> int:
    """Bytes of one MXFP4 entry: E2M1 pairs (3*H*I/2) then E8M0 scales (3*H*I/32)."""
    return 3 * H * I // 2 + 3 * H * I // 32


def mxfp4_entry(seed: int, layer: int, expert: int, H: int, I: int) -> np.ndarray:
    """Entry (layer, expert) quantized to MXFP4 (uint8 bytes; layout in gen.c)."""
    out = np.empty(mxfp4_entry_bytes(H, I), np.uint8)
    lib().mi_mxfp4_entry(seed, stream_id(KIND_EXPERT, layer, expert), H, I, _ptr(out))
    return out


def mxfp4_block(x_bf16_bits: np.ndarray):
    """Quantize one block of 32 bf16 values: (16 bytes of E2M1 pairs, E8M0 scale byte)."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    assert x.size == 32
    q = np.empty(16, np.uint8)
    s = np.empty(1, np.uint8)
    lib().mi_mxfp4_block32(_ptr(x), _ptr(q), _ptr(s))
    return q, int(s[0])


def nvfp4_entry_bytes(H: int, I: int) -> int:
    """Bytes of one NVFP4 entry: E2M1 pairs (3*H*I/2), E4M3 scales (3*H*I/16), 16-byte trailer."""
    return int(lib().mi_nvfp4_bytes(H, I))


def nvfp4_entry(seed: int, layer: int, expert: int, H: int, I: int) -> np.ndarray:
    """Entry (layer, expert) quantized to NVFP4 (uint8 bytes; layout in nvfp4_core.h)."""
    out = np.empty(nvfp4_entry_bytes(H, I), np.uint8)
    lib().mi_nvfp4_entry(seed, stream_id(KIND_EXPERT, layer, expert), H, I, _ptr(out))
    return out


def nvfp4_block(x_bf16_bits: np.ndarray, tensor_scale: float):
    """Quantize one block of 16 bf16 values: (8 bytes of E2M1 pairs, E4M3 scale byte)."""
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    assert x.size == 16
    q = np.empty(8, np.uint8)
    s = np.empty(1, np.uint8)
    lib().mi_nvfp4_block16(_ptr(x), float(tensor_scale), _ptr(q), _ptr(s))
    return q, int(s[0])


def e4m3_encode(v: float) -> int:
    """The quantizer's E4M3 code of v >= 0 (round to nearest even, saturating at 448)."""
    return int(lib().mi_e4m3_encode(float(v)))


def e4m3_decode(c: int) -> float:
    """The quantizer's value of an E4M3 code (used when it divides by the stored scale)."""
    return float(lib().mi_e4m3_decode(int(c)))


def nvfp4_tensor_scale(amax: float) -> float:
    """The quantizer's tensor scale for a matrix whose largest magnitude is amax."""
    return float(lib().mi_nvfp4_tscale(float(amax)))


def fill_mxfp4_entry_at(ptr: int, seed: int, layer: int, expert: int, H: int, I: int) -> None:
    """Write the MXFP4 entry (layer, expert) straight into host memory at `ptr`."""
    lib().mi_mxfp4_entry(seed, stream_id(KIND_EXPERT, layer, expert), H, I, ptr)


def fill_entry_at(ptr: int, seed: int, layer: int, expert: int, H: int, I: int) -> None:
    """Write entry (layer, expert) straight into host memory at `ptr` (3*H*I bf16)."""
    lib().mi_normal_bf16(seed, stream_id(KIND_EXPERT, layer, expert), 0, 3 * H * I, 0.02, ptr)


def gpu_fill_entries(seed: int, keys, H: int, I: int, ptrs) -> None:
    """Write entries keys[i] = (layer, expert) into host memory at ptrs[i] using the GPU build
    of this generator (same bits as fill_entry_at; the current CUDA device does the work)."""
    keys = list(keys)
    if not keys:
        return
    streams = (ctypes.c_uint64 * len(keys))(*[stream_id(KIND_EXPERT, l, e) for l, e in keys])
    dsts = (ctypes.c_void_p * len(keys))(*[int(p) for p in ptrs])
    err = ctypes.create_string_buffer(256)
    rc = gpu_lib().mi_gpu_normal_bf16_to_host(seed, len(keys), streams, 3 * H * I, 0.02, dsts, err, 256)
    if rc != 0:
        raise RuntimeError("GPU input generator: " + err.value.decode(errors="replace"))


def gpu_fill_mxfp4_entries(seed: int, keys, H: int, I: int, ptrs) -> None:
    """Write MXFP4 entries keys[i] = (layer, expert) into host memory at ptrs[i] with the GPU
    build of this generator (the same bytes as fill_mxfp4_entry_at)."""
    keys = list(keys)
    if not keys:
        return
    streams = (ctypes.c_uint64 * len(keys))(*[stream_id(KIND_EXPERT, l, e) for l, e in keys])
    dsts = (ctypes.c_void_p * len(keys))(*[int(p) for p in ptrs])
    err = ctypes.create_string_buffer(256)
    rc = gpu_lib().mi_gpu_mxfp4_entries_to_host(seed, len(keys), streams, H, I, 0.02, dsts, err, 256)
    if rc != 0:
        raise RuntimeError("GPU input generator: " + err.value.decode(errors="replace"))


def gpu_fill_nvfp4_entries(seed: int, keys, H: int, I: int, ptrs) -> None:
    """Write NVFP4 entries keys[i] = (layer, expert) into host memory at ptrs[i] with the GPU
    build of this generator (the same bytes as nvfp4_entry)."""
    keys = list(keys)
    if not keys:
        return
    streams = (ctypes.c_uint64 * len(keys))(*[stream_id(KIND_EXPERT, l, e) for l, e in keys])
    dsts = (ctypes.c_void_p * len(keys))(*[int(p) for p in ptrs])
    err = ctypes.create_string_buffer(256)
    rc = gpu_lib().mi_gpu_nvfp4_entries_to_host(seed, len(keys), streams, H, I, 0.02, dsts, err, 256)
    if rc != 0:
        raise RuntimeError("GPU input generator: " + err.value.decode(errors="replace"))


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
