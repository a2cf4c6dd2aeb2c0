"""Seeded synthetic inputs (Philox4x32-10 + Box-Muller), shared by tests and bench.

Holds no arithmetic of the draft-tree method: it only maps (seed, stream,
counter) to numbers. Both the oracle side and the CUDA side of a test consume
the same arrays produced here. bf16 arrays are returned as numpy uint16 bit
patterns. The C source is compiled in place on first use (gcc, -O2, OpenMP
when available).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_synth.so")
_lib = None

F32, BF16 = 0, 1
STREAM_DRAFT, STREAM_TARGET, STREAM_Q, STREAM_K, STREAM_V, STREAM_SEQ, STREAM_VERIFY = 1, 2, 3, 4, 5, 6, 7
STREAM_HIDDEN, STREAM_LMHEAD = 8, 9  # frontier hidden states, LM-head weights
STREAM_GUMBEL = 10  # uniform words of sampled drafting


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so next to it (idempotent)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        p, i64, u64, u32, i32, f64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                      ctypes.c_int, ctypes.c_double)
        lib.synth_philox4x32_10.argtypes = [p, p, p]
        lib.synth_normal4.argtypes = [p, i32, i64, i64, i64, i64, p, i32, u64, u32]
        lib.synth_plant.argtypes = [p, i32, i64, i64, i64, i64, f64, f64, u64, u32]
        lib.synth_kv_region.argtypes = [p, i32, i64, i32, i32, i32, i32, u32, u32, f64, u64, u32]
        lib.synth_words.argtypes = [p, i64, i64, u32, u64, u32]
        lib.synth_seq_params.argtypes = [i32, i32, i32, f64, f64, u64, p, p]
        lib.synth_threads.restype = i32
        lib.synth_gumbel_words.argtypes = [p, i32, i32, i32, u32, u32, u64]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def philox(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    _load().synth_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def normal4(shape, dtype: int, scale, seed: int, stream: int, scale_axis: int = -1, out=None) -> np.ndarray:
    """Array of shape (n3, n2, n1, n0) (leading dims may be dropped) of scale*N(0,1).

    The element at index [i3, i2, i1, i0] is drawn at Philox counter (i0, i1, i2, i3).
    ``scale_axis`` 2 or 3 takes a per-i2 / per-i3 scale vector (per-sequence sharpness).
    """
    shape = tuple(int(s) for s in shape)
    full = (1,) * (4 - len(shape)) + shape
    n3, n2, n1, n0 = full
    sc = np.ascontiguousarray(np.atleast_1d(np.asarray(scale, dtype=np.float32)))
    if out is None:
        out = np.empty(shape, dtype=np.float32 if dtype == F32 else np.uint16)
    _load().synth_normal4(_ptr(out), dtype, n0, n1, n2, n3, _ptr(sc), scale_axis, seed, stream)
    return out


def plant(arr: np.ndarray, dtype: int, value: float, seed: int, stream: int, frac: float = 1.0) -> np.ndarray:
    """In place: one token per row (Philox-chosen) gets logit ``value`` (rows kept with prob ``frac``)."""
    full = (1,) * (4 - arr.ndim) + arr.shape
    n3, n2, n1, n0 = full
    _load().synth_plant(_ptr(arr), dtype, n0, n1, n2, n3, float(value), float(frac), seed, stream)
    return arr


def kv_region(base: np.ndarray, dtype: int, offset: int, pos_stride: int, hkv: int, d: int, pos0: int, pos1: int,
              layer: int, b: int, seed: int, stream: int, scale: float = 1.0) -> None:
    """Fill positions [pos0, pos1) of one (sequence, layer, K|V) region starting at element ``offset``."""
    esz = 4 if dtype == F32 else 2
    assert base.flags["C_CONTIGUOUS"]
    addr = base.ctypes.data + offset * esz
    _load().synth_kv_region(ctypes.c_void_p(addr), dtype, pos_stride, hkv, d, pos0, pos1, layer, b, scale, seed,
                            stream)


def words(n1: int, n0: int, c2: int, seed: int, stream: int = STREAM_VERIFY) -> np.ndarray:
    out = np.empty((n1, n0), dtype=np.uint32)
    _load().synth_words(_ptr(out), n0, n1, c2, seed, stream)
    return out


def gumbel_words(B: int, k: int, V: int, step: int, cycle: int, seed: int) -> np.ndarray:
    """[B, k, V] uniform words of sampled drafting for one draft step: element
    (b, f, x) is word x & 3 of Philox4x32-10 at counter (x >> 2, b * k + f,
    step, cycle), key (seed_lo ^ 10, seed_hi)."""
    out = np.empty((B, k, V), dtype=np.uint32)
    _load().synth_gumbel_words(_ptr(out), B, k, V, step, cycle, seed)
    return out


def seq_params(batch: int, lmin: int, lspan: int, smin: float, sspan: float, seed: int):
    L = np.empty(batch, dtype=np.int32)
    s = np.empty(batch, dtype=np.float32)
    _load().synth_seq_params(batch, lmin, lspan, smin, sspan, seed, _ptr(L), _ptr(s))
    return L, s


def threads() -> int:
    return int(_load().synth_threads())


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (a.astype(np.uint32) << 16).view(np.float32)
