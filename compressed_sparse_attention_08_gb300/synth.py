"""Seeded synthetic input generator shared by the CUDA path's tests/bench and the oracle.

This module makes inputs only. It holds none of the attention method's arithmetic:
no softmax, no norm, no RoPE, no scoring, no selection. Both sides of every parity
check receive the exact same bytes from here.

Definition (counter-based, so any element can be produced independently and the
stream is identical on every machine):

* stream key      ``k = mix64(seed * G ^ mix64(tensor_id + 1))``
* element ``i``   pair ``j = i // 2``;
  ``h1 = mix64(k + (2j + 1) * G)``, ``h2 = mix64(k + (2j + 2) * G)``
* uniforms        ``u1 = ((h1 >> 11) + 0.5) * 2**-53``  (open interval, never 0),
  ``u2 = (h2 >> 11) * 2**-53``
* Box-Muller      ``r = sqrt(-2 ln u1)``, ``phi = 2 pi u2``;
  even ``i`` takes ``r cos phi``, odd ``i`` takes ``r sin phi``
* value           ``mean + std * z`` in float64, rounded to float32 (round to
  nearest even), then to bfloat16 (round to nearest even) where bf16 is asked for.

``mix64`` is the SplitMix64 output function (Steele, Lea, Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014) and ``G = 0x9E3779B97F4A7C15`` its
increment. Box and Muller, "A note on the generation of random normal deviates",
Ann. Math. Statist. 1958.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # elements per vectorised chunk (bounds host memory)


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _stream_key(seed: int, tensor_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        a = _mix64(np.array([tensor_id + 1], dtype=np.uint64))[0]
        s = np.uint64(seed) * _G
        return np.uint64(_mix64(np.array([s ^ a], dtype=np.uint64))[0])


def _normals_f64(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Standard normals for element indices [start, start + count) of a stream."""
    i0 = start - (start & 1)
    i1 = start + count + ((start + count) & 1)
    pairs = np.arange(i0 // 2, i1 // 2, dtype=np.uint64)
    with np.errstate(over="ignore"):
        c1 = key + (pairs * np.uint64(2) + np.uint64(1)) * _G
        c2 = key + (pairs * np.uint64(2) + np.uint64(2)) * _G
        h1 = _mix64(c1)
        h2 = _mix64(c2)
    u1 = ((h1 >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    u2 = (h2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    r = np.sqrt(-2.0 * np.log(u1))
    phi = (2.0 * np.pi) * u2
    out = np.empty(2 * len(pairs), dtype=np.float64)
    out[0::2] = r * np.cos(phi)
    out[1::2] = r * np.sin(phi)
    off = start - i0
    return out[off:off + count]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        r = ((u + rounding) >> np.uint32(16)).astype(np.uint16)
    r[nan] = np.uint16(0x7FC0)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


_HERE = os.path.dirname(os.path.abspath(__file__))
_FILL_SRC = os.path.join(_HERE, "synth_fill.c")
_FILL_LIB = os.path.join(_HERE, "_synth_fill.so")
_fill = None


def _fill_lib():
    """The multithreaded C fill (same stream, same bits); None if it cannot be built."""
    global _fill
    if _fill is None:
        try:
            if not os.path.exists(_FILL_LIB) or os.path.getmtime(_FILL_LIB) < os.path.getmtime(_FILL_SRC):
                tmp = _FILL_LIB + f".tmp{os.getpid()}"
                subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                                       "-pthread", _FILL_SRC, "-o", tmp, "-lm"])
                os.replace(tmp, _FILL_LIB)
            lib = ctypes.CDLL(_FILL_LIB)
            for f in (lib.synth_normal_bf16, lib.synth_normal_f32):
                f.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                              ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
                f.restype = None
            _fill = lib
        except (OSError, subprocess.CalledProcessError):
            _fill = False
    return _fill or None


def _threads():
    return max(1, min(32, os.cpu_count() or 1))


def normal_f32_numpy(seed: int, tensor_id: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """float32 array of N(mean, std) draws for stream (seed, tensor_id) (numpy implementation)."""
    n = int(np.prod(shape)) if len(shape) else 1
    key = _stream_key(seed, tensor_id)
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = (mean + std * _normals_f64(key, s, c)).astype(np.float32)
    return out.reshape(shape)


def normal_bf16_numpy(seed: int, tensor_id: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """bfloat16 bit patterns of N(mean, std) draws for stream (seed, tensor_id) (numpy)."""
    n = int(np.prod(shape)) if len(shape) else 1
    key = _stream_key(seed, tensor_id)
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = f32_to_bf16_bits((mean + std * _normals_f64(key, s, c)).astype(np.float32))
    return out.reshape(shape)


def normal_f32(seed: int, tensor_id: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """float32 array of N(mean, std) draws for stream (seed, tensor_id)."""
    lib = _fill_lib()
    if lib is None:
        return normal_f32_numpy(seed, tensor_id, shape, mean, std)
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float32)
    lib.synth_normal_f32(int(_stream_key(seed, tensor_id)), 0, n, float(mean), float(std),
                         out.ctypes.data, _threads())
    return out.reshape(shape)


def normal_bf16(seed: int, tensor_id: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """bfloat16 bit patterns (uint16 array) of N(mean, std) draws for stream (seed, tensor_id)."""
    lib = _fill_lib()
    if lib is None:
        return normal_bf16_numpy(seed, tensor_id, shape, mean, std)
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.uint16)
    lib.synth_normal_bf16(int(_stream_key(seed, tensor_id)), 0, n, float(mean), float(std),
                          out.ctypes.data, _threads())
    return out.reshape(shape)


def uniform_index_sets(seed: int, tensor_id: int, rows: int, n_valid, k: int) -> np.ndarray:
    """Per row r, ``min(k, n_valid[r])`` distinct indices in [0, n_valid[r]) in ascending
    order, padded with -1 to length ``k`` (int32 [rows, k]).  A seeded permutation stands in
    for an index list produced upstream; it is input data, not a selection rule."""
    rng = np.random.Generator(np.random.PCG64([seed, tensor_id]))
    out = np.full((rows, k), -1, dtype=np.int32)
    for r in range(rows):
        n = int(n_valid[r])
        t = min(k, n)
        if t > 0:
            out[r, :t] = np.sort(rng.choice(n, size=t, replace=False)).astype(np.int32)
    return out
