"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no arithmetic of the reshard method: it only produces
buffer contents, request lengths and page free lists.  Buffer contents are a
counter-based function of the 16-bit element index, so any element can be
recomputed on the host without materialising the buffer:

    u64(seed, i) = splitmix64_mix(seed + (i + 1) * 0x9E3779B97F4A7C15)

(the SplitMix64 generator of Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014, in its counter form).  Mode RAW
keeps the low 16 bits (arbitrary bf16 bit patterns, NaN and Inf included);
mode NORMAL maps the top 16 bits through a 65,536-entry table of bf16 values
of sigma * Phi^-1((k + 0.5) / 65536), i.e. bf16 samples of N(0, sigma^2).

The device twin of ``fill_host`` is the CUDA kernel in ``synth_fill.cu``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from statistics import NormalDist

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
M1 = np.uint64(0xBF58476D1CE4E5B9)
M2 = np.uint64(0x94D049BB133111EB)

RAW = 0
NORMAL = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_CU = os.path.join(_HERE, "synth_fill.cu")
_SO = os.path.join(_HERE, "libsynth.so")


def splitmix64(seed: int, idx: np.ndarray) -> np.ndarray:
    """Counter-form SplitMix64 over an array of indices (uint64, wrapping)."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (idx + np.uint64(1)) * GAMMA
        z = (z ^ (z >> np.uint64(30))) * M1
        z = (z ^ (z >> np.uint64(27))) * M2
        z = z ^ (z >> np.uint64(31))
    return z


def _f32_to_bf16_rne(x: np.ndarray) -> np.ndarray:
    b = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (b >> np.uint64(16)) & np.uint64(1)
    b = (b + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return b.astype(np.uint16)


_tables: dict[float, np.ndarray] = {}


def normal_table(sigma: float) -> np.ndarray:
    """bf16 bit patterns of sigma * Phi^-1((k + 0.5) / 65536), k = 0..65535
    (quantiles in double, then rounded to f32 and to bf16, both to nearest-even)."""
    if sigma not in _tables:
        nd = NormalDist()
        q = np.array([nd.inv_cdf((k + 0.5) / 65536.0) for k in range(65536)], dtype=np.float64)
        _tables[sigma] = _f32_to_bf16_rne((q * sigma).astype(np.float32))
    return _tables[sigma]


def values_at(seed: int, idx: np.ndarray, mode: int = RAW, sigma: float = 1.0) -> np.ndarray:
    """uint16 contents of element indices ``idx`` of a buffer filled by ``fill``."""
    z = splitmix64(seed, idx)
    if mode == RAW:
        return (z & np.uint64(0xFFFF)).astype(np.uint16)
    return normal_table(sigma)[(z >> np.uint64(48)).astype(np.int64)]


def fill_host(n: int, seed: int, mode: int = RAW, sigma: float = 1.0, base: int = 0) -> np.ndarray:
    """Host buffer of n uint16 elements with indices base..base+n-1."""
    out = np.empty(n, dtype=np.uint16)
    step = 1 << 24
    for s in range(0, n, step):
        e = min(n, s + step)
        out[s:e] = values_at(seed, np.arange(base + s, base + e, dtype=np.uint64), mode, sigma)
    return out


# ---------------------------------------------------------------- device twin

def build(force: bool = False) -> str:
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_CU):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["nvcc", "-O3", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-shared", "-Xcompiler", "-fPIC", "-o", tmp, _CU])
        os.replace(tmp, _SO)
    return _SO


_dev = None


def _devlib():
    global _dev
    if _dev is None:
        build()
        L = ctypes.CDLL(_SO)
        L.synth_fill_u16.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                     ctypes.c_uint64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        L.synth_fill_u16.restype = ctypes.c_int
        _dev = L
    return _dev


def fill_device(ptr: int, n: int, seed: int, mode: int = RAW, table_ptr: int = 0,
                base: int = 0, stream: int = 0) -> None:
    """Fill n uint16 elements at device address ``ptr`` with indices base.. .
    NORMAL mode needs ``table_ptr``: the device copy of ``normal_table``."""
    rc = _devlib().synth_fill_u16(ptr, n, base, seed & 0xFFFFFFFFFFFFFFFF, mode,
                                  table_ptr or None, stream or None)
    if rc != 0:
        raise RuntimeError(f"synth_fill_u16 failed with CUDA error {rc}")


# ---------------------------------------------------------------- request mixes

def rng(seed: int, purpose: int) -> np.random.Generator:
    """Independent stream per purpose (1 lengths, 2 source pages, 3 dest pages,
    4 later dest pages, 5 queries, ...)."""
    return np.random.default_rng([seed, purpose])


def lengths_uniform(seed: int, R: int, lo: int, hi: int) -> np.ndarray:
    return rng(seed, 1).integers(lo, hi + 1, R).astype(np.int32)


def lengths_lognormal(seed: int, R: int, median: float, sigma: float, cap: int) -> np.ndarray:
    x = np.exp(rng(seed, 1).normal(math.log(median), sigma, R))
    return np.clip(np.round(x), 1, cap).astype(np.int32)


def npages(lens: np.ndarray, ps: int) -> np.ndarray:
    return (np.asarray(lens, dtype=np.int64) + ps - 1) // ps


def permutation(seed: int, purpose: int, n: int, rows: int = 1) -> np.ndarray:
    """rows independent random permutations of 0..n-1 (page free lists)."""
    g = rng(seed, purpose)
    return np.stack([g.permutation(n) for _ in range(rows)]).astype(np.int32)
