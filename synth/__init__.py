"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

The one source of input tensors for tests and the benchmark. It holds none of
the method's arithmetic: counter-based splitmix64 streams, Box-Muller normals
and fp32->bf16 rounding (see gen.c). The workload shapes follow the PulseInfer
pages (PulseInfer Guide, "The Long-Context Decoding Memory Wall" and "SoloHead
Sparse Selection"): Llama-3-shaped attention, K/V ~ N(0,1), a fraction of
heavy-hitter blocks with shifted keys, and AR(1) decode-step queries.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "libsynth.so")

KIND_K, KIND_V, KIND_Q, KIND_HEAVY, KIND_DIR = 1, 2, 3, 4, 5
KIND_RESIDENT, KIND_BUDGET, KIND_FRAC, KIND_MISC = 6, 7, 8, 9


def build(force: bool = False) -> str:
    """Compile gen.c into libsynth.so next to it (gcc, OpenMP)."""
    src = os.path.join(_HERE, "gen.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        u64, i32, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        L.sy_tid.restype = u64
        L.sy_tid.argtypes = [i32, i32, i32]
        L.sy_u64.restype = u64
        L.sy_u64.argtypes = [u64, u64, u64]
        L.sy_normal.restype = dbl
        L.sy_normal.argtypes = [u64, u64, u64]
        L.sy_normal_bf16.restype = None
        L.sy_normal_bf16.argtypes = [u64, u64, u64, i64, vp]
        L.sy_heavy_mask.restype = i32
        L.sy_heavy_mask.argtypes = [u64, i32, i32, i32, dbl, vp]
        L.sy_direction.restype = None
        L.sy_direction.argtypes = [u64, i32, i32, i32, i32, vp]
        L.sy_fill_kv.restype = i32
        L.sy_fill_kv.argtypes = [u64, i32, i32, i32, i32, i32, i32, i32, dbl, dbl, vp]
        L.sy_token_kv.restype = None
        L.sy_token_kv.argtypes = [u64, i32, i32, i32, i32, i32, vp, vp]
        L.sy_q_ar1.restype = None
        L.sy_q_ar1.argtypes = [u64, i32, i32, i32, i32, i32, dbl, vp, i64]
        L.sy_uniform_int.restype = i64
        L.sy_uniform_int.argtypes = [u64, i32, i32, i32, u64, i64, i64]
        L.sy_uniform_real.restype = dbl
        L.sy_uniform_real.argtypes = [u64, i32, i32, i32, u64, dbl, dbl]
        L.sy_sample_sorted.restype = i32
        L.sy_sample_sorted.argtypes = [u64, i32, i32, i32, i32, i32, vp, vp]
        L.sy_bf16_of_double.restype = ctypes.c_uint16
        L.sy_bf16_of_double.argtypes = [dbl]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- bf16 helpers
def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact widening)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest even (finite values)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    return ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)


# ---------------------------------------------------------------- streams
def normal_bf16(seed: int, kind: int, a: int, b: int, n: int, start: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    L = lib()
    L.sy_normal_bf16(seed, L.sy_tid(kind, a, b), start, n, _ptr(out))
    return out


def normal_f64(seed: int, kind: int, a: int, b: int, idx: int) -> float:
    L = lib()
    return L.sy_normal(seed, L.sy_tid(kind, a, b), idx)


def uniform_int(seed: int, kind: int, a: int, b: int, idx: int, lo: int, hi: int) -> int:
    return int(lib().sy_uniform_int(seed, kind, a, b, idx, lo, hi))


def uniform_real(seed: int, kind: int, a: int, b: int, idx: int, lo: float, hi: float) -> float:
    return float(lib().sy_uniform_real(seed, kind, a, b, idx, lo, hi))


def heavy_mask(seed: int, hl: int, r: int, nb: int, frac: float) -> np.ndarray:
    m = np.zeros(max(nb, 1), dtype=np.uint8)
    rc = lib().sy_heavy_mask(seed, hl, r, nb, frac, _ptr(m))
    if rc < 0:
        raise MemoryError("heavy mask")
    return m[:nb].astype(bool)


def direction(seed: int, hl: int, r: int, g: int, D: int) -> np.ndarray:
    u = np.empty(D, dtype=np.float64)
    lib().sy_direction(seed, hl, r, g, D, _ptr(u))
    return u


def sample_sorted(seed: int, kind: int, a: int, b: int, nb: int, n: int) -> np.ndarray:
    """n distinct block ids of 0..nb-1, ascending (seeded partial Fisher-Yates)."""
    out = np.empty(max(nb, 1), dtype=np.int32)
    scratch = np.empty(max(nb, 1), dtype=np.int32)
    m = lib().sy_sample_sorted(seed, kind, a, b, nb, n, _ptr(out), _ptr(scratch))
    return out[:m].copy()


# ---------------------------------------------------------------- tensors
def fill_kv(ptr: int, seed: int, hl: int, r: int, ntok: int, max_blocks: int, hkv: int, B: int, D: int,
            heavy_frac: float = 0.0, heavy_shift: float = 0.0) -> None:
    """Fill one (host layer, request) region [max_blocks][hkv][2][B][D] bf16 at a raw pointer."""
    rc = lib().sy_fill_kv(seed, hl, r, ntok, max_blocks, hkv, B, D, heavy_frac, heavy_shift, ptr)
    if rc != 0:
        raise ValueError(f"sy_fill_kv failed ({rc})")


def kv_region(seed: int, hl: int, r: int, ntok: int, max_blocks: int, hkv: int, B: int, D: int,
              heavy_frac: float = 0.0, heavy_shift: float = 0.0) -> np.ndarray:
    out = np.empty((max_blocks, hkv, 2, B, D), dtype=np.uint16)
    fill_kv(_ptr(out), seed, hl, r, ntok, max_blocks, hkv, B, D, heavy_frac, heavy_shift)
    return out


def token_kv(seed: int, hl: int, r: int, tt: int, hkv: int, D: int):
    """(k[hkv][D], v[hkv][D]) bf16 bits of token position tt (no heavy shift)."""
    k = np.empty((hkv, D), dtype=np.uint16)
    v = np.empty((hkv, D), dtype=np.uint16)
    lib().sy_token_kv(seed, hl, r, tt, hkv, D, _ptr(k), _ptr(v))
    return k, v


def q_ar1(seed: int, layers: int, R: int, hq: int, D: int, steps: int, rho: float) -> np.ndarray:
    """Queries [steps][layers][R][hq][D] bf16 bits; AR(1) per element across steps."""
    out = np.empty((steps, layers, R, hq, D), dtype=np.uint16)
    L = lib()
    stride = layers * R * hq * D
    for l in range(layers):
        for r in range(R):
            view = out[0, l, r]
            L.sy_q_ar1(seed, l, r, hq, D, steps, rho, view.ctypes.data, stride)
    return out
