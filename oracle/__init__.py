"""Oracle for the CSA decode step: ctypes wrapper around ``csa_oracle.cpp``.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package. The CUDA
library never loads it and there is no CPU fallback built on it.

Arrays in and out are numpy; bf16 tensors travel as uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "csa_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle_csa.so")
_lib = None


def compile_oracle(src: str, out: str) -> str:
    """Compile an oracle source with g++ (-O2, no fast-math, no FMA contraction)."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC",
                           "-shared", src, "-o", tmp])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build the oracle library next to its source (if missing or stale)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_oracle(SOURCE, _LIB)
    return _LIB


def use_library(path: str | None) -> None:
    """Point this module at another build of the oracle (tests plant mistakes in copies
    of the source to prove that the pins catch them); None restores the default."""
    global _lib
    _lib = None if path is None else _bind(ctypes.CDLL(path))


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_compress.argtypes = [P, P, P, P, P, I, I, I, I, I, D, D, P, P]
    lib.oracle_compress_overlap.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, D, D, P, P]
    lib.oracle_index_scores.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P]
    lib.oracle_topk.argtypes = [P, P, I, I, I, P]
    lib.oracle_topk_f32.argtypes = [P, P, I, I, I, P]
    lib.oracle_sparse_attn.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I,
                                       I, D, P, P, P]
    lib.oracle_quantize_rows_e4m3.argtypes = [P, I, I, P, P]
    lib.oracle_quantize_rows_e4m3.restype = ctypes.c_int
    lib.oracle_quantize_kv_mixed.argtypes = [P, I, I, I, P, P, P]
    lib.oracle_quantize_kv_mixed.restype = ctypes.c_int
    lib.oracle_dequant_kv_mixed.argtypes = [P, P, P, I, I, I, P]
    lib.oracle_dequant_kv_mixed.restype = ctypes.c_int
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = D
    lib.oracle_e4m3_from_double.argtypes = [D]
    lib.oracle_e4m3_from_double.restype = ctypes.c_uint8
    lib.oracle_index_scores_fp8.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, P, P]
    lib.oracle_index_scores_fp8.restype = ctypes.c_int
    lib.oracle_inverse_rope.argtypes = [P, P, I, I, I, I, D, P, P]
    lib.oracle_inverse_rope.restype = ctypes.c_int
    lib.oracle_max_comp.argtypes = [ctypes.c_int64, I]
    lib.oracle_max_comp.restype = ctypes.c_int64
    lib.oracle_visible_entries.argtypes = [ctypes.c_int64, ctypes.c_int64, I]
    lib.oracle_visible_entries.restype = ctypes.c_int64
    lib.oracle_double_to_bf16.argtypes = [D]
    lib.oracle_double_to_bf16.restype = ctypes.c_uint16
    for f in (lib.oracle_compress, lib.oracle_compress_overlap, lib.oracle_index_scores, lib.oracle_topk,
              lib.oracle_topk_f32, lib.oracle_sparse_attn):
        f.restype = ctypes.c_int
    return lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def compress(C, Z, bias, gamma, pos0, ratio, rope_dim=64, theta=10000.0, eps=1e-6):
    """Block compressor + RMSNorm + RoPE.  C, Z: uint16 [B, T, d]; bias fp32 [ratio, d];
    gamma fp32 [d]; pos0 int64 [B].  Returns (bf16 bits [B, T/ratio, d], float64 same)."""
    lib = _load()
    C = _c(C, np.uint16); Z = _c(Z, np.uint16)
    bias = _c(bias, np.float32); gamma = _c(gamma, np.float32); pos0 = _c(pos0, np.int64)
    B, T, d = C.shape
    out = np.zeros((B, T // ratio, d), np.uint16)
    out64 = np.zeros((B, T // ratio, d), np.float64)
    rc = lib.oracle_compress(_p(C), _p(Z), _p(bias), _p(gamma), _p(pos0), B, T, d, ratio,
                             rope_dim, float(theta), float(eps), _p(out), _p(out64))
    if rc != 0:
        raise ValueError(f"oracle_compress: bad arguments (rc={rc})")
    return out, out64


def compress_overlap(C, Z, bias, gamma, pos0, ratio, prev_C=None, prev_Z=None, rope_dim=64,
                     theta=10000.0, eps=1e-6):
    """Overlapped two-stream (CSA) compressor + RMSNorm + RoPE.  C, Z: uint16 [B, T, 2d]
    (stream a = channels [0, d), stream b = [d, 2d)); bias fp32 [ratio, 2d]; gamma fp32 [d];
    pos0 int64 [B]; prev_C, prev_Z uint16 [B, ratio, 2d] or None (the block before C's first
    block).  Returns (bf16 bits [B, T/ratio, d], float64 same)."""
    lib = _load()
    C = _c(C, np.uint16); Z = _c(Z, np.uint16)
    prev_C = _c(prev_C, np.uint16); prev_Z = _c(prev_Z, np.uint16)
    bias = _c(bias, np.float32); gamma = _c(gamma, np.float32); pos0 = _c(pos0, np.int64)
    B, T, w = C.shape
    d = w // 2
    out = np.zeros((B, T // ratio, d), np.uint16)
    out64 = np.zeros((B, T // ratio, d), np.float64)
    rc = lib.oracle_compress_overlap(_p(C), _p(Z), _p(prev_C), _p(prev_Z), _p(bias), _p(gamma),
                                     _p(pos0), B, T, d, ratio, rope_dim, float(theta), float(eps),
                                     _p(out), _p(out64))
    if rc != 0:
        raise ValueError(f"oracle_compress_overlap: bad arguments (rc={rc})")
    return out, out64


def index_scores(q, w, keys, n_comp, ratio=4, q_pos=None):
    """Indexer scores.  q uint16 [B, n_q, H, Di]; w fp32 [B, n_q, H]; keys uint16
    [B, max_comp, Di]; n_comp int32 [B]; q_pos int64 [B, n_q] or None.
    Returns (float64 [B, n_q, max_comp] with -inf past the visible count, int32 n_vis [B, n_q])."""
    lib = _load()
    q = _c(q, np.uint16); w = _c(w, np.float32); keys = _c(keys, np.uint16)
    n_comp = _c(n_comp, np.int32); q_pos = _c(q_pos, np.int64)
    B, n_q, H, Di = q.shape
    max_comp = keys.shape[1]
    scores = np.empty((B, n_q, max_comp), np.float64)
    n_vis = np.empty((B, n_q), np.int32)
    rc = lib.oracle_index_scores(_p(q), _p(w), _p(keys), _p(n_comp), _p(q_pos), B, n_q, H, Di,
                                 max_comp, ratio, _p(scores), _p(n_vis))
    if rc != 0:
        raise ValueError(f"oracle_index_scores: bad arguments (rc={rc})")
    return scores, n_vis


def topk(scores, n_vis, top_k):
    """Top-k over the last axis (ties -> lower index), ascending, -1 padded.
    scores float64 or float32 [..., max_comp]; n_vis int32 [...]."""
    lib = _load()
    lead = scores.shape[:-1]
    max_comp = scores.shape[-1]
    rows = int(np.prod(lead)) if lead else 1
    n_vis = _c(np.broadcast_to(n_vis, lead), np.int32)
    idx = np.empty(lead + (top_k,), np.int32)
    if scores.dtype == np.float32:
        s = _c(scores, np.float32)
        rc = lib.oracle_topk_f32(_p(s), _p(n_vis), rows, max_comp, top_k, _p(idx))
    else:
        s = _c(scores, np.float64)
        rc = lib.oracle_topk(_p(s), _p(n_vis), rows, max_comp, top_k, _p(idx))
    if rc != 0:
        raise ValueError(f"oracle_topk: bad arguments (rc={rc})")
    return idx


def sparse_attn(q, sink, comp_kv, n_comp, idx, win, win_len, top_k, window=128, ratio=4,
                scale=None, q_pos=None, q_abs=None, n_q_total=None, want_gather=False):
    """Gather + sink attention.  q uint16 [B, n_q, H, D]; sink fp32 [H]; comp_kv uint16
    [B, max_comp, D]; n_comp int32 [B]; idx int32 [B, n_q, top_k] or None (dense; top_k must
    be max_comp); win uint16 [B, win_rows, D]; win_len int32 [B].
    Returns (bf16 bits [B, n_q, H, D], float64 same, gather bits or None)."""
    lib = _load()
    q = _c(q, np.uint16); sink = _c(sink, np.float32); comp_kv = _c(comp_kv, np.uint16)
    n_comp = _c(n_comp, np.int32); idx = _c(idx, np.int32); win = _c(win, np.uint16)
    win_len = _c(win_len, np.int32); q_pos = _c(q_pos, np.int64); q_abs = _c(q_abs, np.int32)
    B, n_q, H, D = q.shape
    max_comp = comp_kv.shape[1]
    win_rows = win.shape[1]
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    if n_q_total is None:
        n_q_total = n_q
    out = np.zeros((B, n_q, H, D), np.uint16)
    out64 = np.zeros((B, n_q, H, D), np.float64)
    gather = np.zeros((B, n_q, top_k + window, D), np.uint16) if want_gather else None
    rc = lib.oracle_sparse_attn(_p(q), _p(sink), _p(comp_kv), _p(n_comp), _p(idx), _p(q_pos),
                                _p(win), _p(win_len), _p(q_abs), B, n_q, n_q_total, H, D,
                                max_comp, top_k, window, win_rows, ratio, float(scale),
                                _p(out), _p(out64), _p(gather))
    if rc != 0:
        raise ValueError(f"oracle_sparse_attn: bad arguments (rc={rc})")
    return out, out64, gather


def e4m3_encode(x):
    """FP8 E4M3 codes (round to nearest even, saturating) of float64 values, elementwise."""
    lib = _load()
    x = np.asarray(x, np.float64)
    return np.array([lib.oracle_e4m3_from_double(float(v)) for v in x.ravel()], np.uint8).reshape(x.shape)


def e4m3_decode(c):
    lib = _load()
    c = np.asarray(c, np.uint8)
    return np.array([lib.oracle_e4m3_to_double(int(v)) for v in c.ravel()], np.float64).reshape(c.shape)


def quantize_kv_mixed(x, rope_dim=64):
    """Mixed compressed-KV storage of fp32 rows x [..., dim]: (nope codes uint8 [..., dim -
    rope_dim], scale fp32 [...], rope bf16 bits uint16 [..., rope_dim])."""
    lib = _load()
    x = np.ascontiguousarray(x, np.float32)
    shape = x.shape
    rows = int(np.prod(shape[:-1]))
    dim = shape[-1]
    nope = np.zeros(shape[:-1] + (dim - rope_dim,), np.uint8)
    sc = np.zeros(shape[:-1], np.float32)
    rope = np.zeros(shape[:-1] + (rope_dim,), np.uint16)
    rc = lib.oracle_quantize_kv_mixed(_p(x), rows, dim, rope_dim, _p(nope), _p(sc), _p(rope))
    if rc != 0:
        raise ValueError("oracle_quantize_kv_mixed: bad arguments")
    return nope, sc, rope


def dequant_kv_mixed(nope, scale, rope):
    """bf16 bits [..., dim] of the rows the attention multiplies (see quantize_kv_mixed)."""
    lib = _load()
    nope = np.ascontiguousarray(nope, np.uint8)
    scale = np.ascontiguousarray(scale, np.float32)
    rope = np.ascontiguousarray(rope, np.uint16)
    rope_dim = rope.shape[-1]
    dim = nope.shape[-1] + rope_dim
    rows = int(np.prod(nope.shape[:-1]))
    out = np.zeros(nope.shape[:-1] + (dim,), np.uint16)
    rc = lib.oracle_dequant_kv_mixed(_p(nope), _p(scale), _p(rope), rows, dim, rope_dim, _p(out))
    if rc != 0:
        raise ValueError("oracle_dequant_kv_mixed: bad arguments")
    return out


def quantize_rows_e4m3(x):
    """Per-row FP8 E4M3 quantization of fp32 rows x [..., dim]: (codes uint8, scale fp32 [...])."""
    lib = _load()
    x = np.ascontiguousarray(x, np.float32)
    shape = x.shape
    rows = int(np.prod(shape[:-1]))
    q = np.zeros(shape, np.uint8)
    sc = np.zeros(shape[:-1], np.float32)
    rc = lib.oracle_quantize_rows_e4m3(_p(x), rows, shape[-1], _p(q), _p(sc))
    if rc != 0:
        raise ValueError(f"oracle_quantize_rows_e4m3: bad arguments (rc={rc})")
    return q, sc


def index_scores_fp8(q, q_scale, w, keys, k_scale, n_comp, ratio=4, q_pos=None):
    """Indexer scores of FP8 rows.  q uint8 [B, n_q, H, Di], q_scale fp32 [B, n_q, H], w fp32
    [B, n_q, H], keys uint8 [B, max_comp, Di], k_scale fp32 [B, max_comp]; as index_scores."""
    lib = _load()
    q = _c(q, np.uint8); q_scale = _c(q_scale, np.float32); w = _c(w, np.float32)
    keys = _c(keys, np.uint8); k_scale = _c(k_scale, np.float32)
    n_comp = _c(n_comp, np.int32); q_pos = _c(q_pos, np.int64)
    B, n_q, H, Di = q.shape
    max_comp = keys.shape[1]
    scores = np.empty((B, n_q, max_comp), np.float64)
    n_vis = np.empty((B, n_q), np.int32)
    rc = lib.oracle_index_scores_fp8(_p(q), _p(q_scale), _p(w), _p(keys), _p(k_scale), _p(n_comp),
                                     _p(q_pos), B, n_q, H, Di, max_comp, ratio, _p(scores), _p(n_vis))
    if rc != 0:
        raise ValueError(f"oracle_index_scores_fp8: bad arguments (rc={rc})")
    return scores, n_vis


def inverse_rope(x, pos, rope_dim=64, theta=10000.0):
    """Inverse RoPE of attention outputs.  x float64 [rows, heads, D] (any leading shape that
    flattens to rows x heads); pos int64 [rows].  Returns (bf16 bits, float64) of x's shape."""
    lib = _load()
    x = np.asarray(x, np.float64)
    shape = x.shape
    D, H = shape[-1], shape[-2]
    rows = int(np.prod(shape[:-2])) if len(shape) > 2 else 1
    xf = np.ascontiguousarray(x.reshape(rows, H, D))
    pos = _c(np.asarray(pos).reshape(rows), np.int64)
    out = np.zeros((rows, H, D), np.uint16)
    out64 = np.zeros((rows, H, D), np.float64)
    rc = lib.oracle_inverse_rope(_p(xf), _p(pos), rows, H, D, rope_dim, float(theta), _p(out), _p(out64))
    if rc != 0:
        raise ValueError(f"oracle_inverse_rope: bad arguments (rc={rc})")
    return out.reshape(shape), out64.reshape(shape)


def max_comp(max_context, ratio):
    return int(_load().oracle_max_comp(int(max_context), int(ratio)))


def visible_entries(n_comp, p, ratio):
    return int(_load().oracle_visible_entries(int(n_comp), int(p), int(ratio)))


def double_to_bf16(x):
    return int(_load().oracle_double_to_bf16(float(x)))
