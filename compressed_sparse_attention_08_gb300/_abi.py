"""ctypes mirror of include/dsv4.h and tensor-to-argument marshalling.

Each ``dsv4_*`` function takes torch tensors, checks dtype/device/contiguity/shape, fills
the C argument struct with their data pointers, and calls the library on the current (or
given) CUDA stream. A non-zero status raises :class:`Dsv4Error`.
"""
from __future__ import annotations

import ctypes
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))

DSV4_OK = 0
DSV4_ERR_INVALID_ARG = 1
DSV4_ERR_LAUNCH = 2
DSV4_ERR_BAD_INDEX = 3
DSV4_ERR_TIMEOUT = 4
DSV4_ERR_UNSUPPORTED = 5
DSV4_EWORD_BAD_INDEX = 0x1
DSV4_EWORD_TIMEOUT = 0x2
DSV4_WAIT_FAULT_NONE = 0
DSV4_WAIT_FAULT_SCORER_STAGE = 1
DSV4_WAIT_FAULT_ATTN_QUERY = 2

EXPORTED_SYMBOLS = (
    "dsv4_compress", "dsv4_compress_step", "dsv4_quantize_rows_fp8", "dsv4_indexer_topk_workspace_size",
    "dsv4_indexer_topk",
    "dsv4_index_score_workspace_size", "dsv4_index_score",
    "dsv4_topk_workspace_size", "dsv4_topk", "dsv4_topk_noalloc", "dsv4_sparse_attn_workspace_size",
    "dsv4_sparse_attn_decode", "dsv4_csa_decode_workspace_size", "dsv4_csa_decode",
    "dsv4_status_string", "dsv4_read_error_word", "dsv4_last_launch_count", "dsv4_max_comp",
    "dsv4_test_wait_fault", "dsv4_copy_async",
)

P = ctypes.c_void_p
I = ctypes.c_int


class CompressArgs(ctypes.Structure):
    _fields_ = [("C", P), ("Z", P), ("bias", P), ("gamma", P), ("pos0", P), ("out", P),
                ("out_row0", P), ("batch", I), ("tokens", I), ("dim", I), ("ratio", I),
                ("rope_dim", I), ("out_rows", I), ("eps", ctypes.c_float),
                ("rope_theta", ctypes.c_double), ("overlap", I), ("prev_C", P), ("prev_Z", P),
                ("out_fp8", I), ("out_scale", P), ("out_rope", P)]


class StepArgs(ctypes.Structure):
    _fields_ = [("C", P), ("Z", P), ("bias", P), ("gamma", P), ("pos", P), ("stage", P),
                ("fill", P), ("n_comp", P), ("out", P), ("batch", I), ("dim", I), ("ratio", I),
                ("rope_dim", I), ("out_rows", I), ("overlap", I), ("eps", ctypes.c_float),
                ("rope_theta", ctypes.c_double), ("out_fp8", I), ("out_scale", P), ("out_rope", P)]


class IndexArgs(ctypes.Structure):
    _fields_ = [("q", P), ("w", P), ("keys", P), ("n_comp", P), ("q_pos", P), ("idx_out", P),
                ("scores_out", P), ("batch", I), ("n_q", I), ("heads", I), ("dim", I),
                ("max_comp", I), ("top_k", I), ("ratio", I), ("key_fp8", I), ("q_scale", P),
                ("key_scale", P)]


class TopkArgs(ctypes.Structure):
    _fields_ = [("scores", P), ("n_vis", P), ("idx_out", P), ("rows", I), ("max_comp", I),
                ("top_k", I)]


class AttnArgs(ctypes.Structure):
    _fields_ = [("q", P), ("sink", P), ("comp_kv", P), ("n_comp", P), ("idx", P), ("q_pos", P),
                ("win", P), ("win_len", P), ("gather", P), ("out", P), ("batch", I), ("n_q", I),
                ("heads", I), ("dim", I), ("max_comp", I), ("top_k", I), ("window", I),
                ("win_rows", I), ("ratio", I), ("scale", ctypes.c_float), ("out_rope_pos", P),
                ("out_rope_dim", I), ("out_rope_theta", ctypes.c_double), ("kv_fp8", I),
                ("kv_nope", P), ("kv_scale", P), ("kv_rope", P), ("kv_rope_dim", I)]


class CsaArgs(ctypes.Structure):
    _fields_ = [("compress_kv", ctypes.POINTER(CompressArgs)),
                ("compress_keys", ctypes.POINTER(CompressArgs)),
                ("index", ctypes.POINTER(IndexArgs)), ("attn", ctypes.POINTER(AttnArgs))]


class Dsv4Error(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {dsv4_status_string(status)} (status {status})")


_lib = None


def library_path() -> str:
    return os.path.join(HERE, "libdsv4.so")


def library():
    """The loaded CUDA library. Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"CSA CUDA library not built ({path}); run "
                               "`python -m compressed_sparse_attention_08_gb300._build`")
        lib = ctypes.CDLL(path)
        lib.dsv4_compress.argtypes = [ctypes.POINTER(CompressArgs), P]
        lib.dsv4_compress_step.argtypes = [ctypes.POINTER(StepArgs), P]
        lib.dsv4_quantize_rows_fp8.argtypes = [P, I, I, P, P, P]
        lib.dsv4_indexer_topk_workspace_size.argtypes = [ctypes.POINTER(IndexArgs)]
        lib.dsv4_indexer_topk_workspace_size.restype = ctypes.c_size_t
        lib.dsv4_indexer_topk.argtypes = [ctypes.POINTER(IndexArgs), P, ctypes.c_size_t, P]
        lib.dsv4_index_score_workspace_size.argtypes = [ctypes.POINTER(IndexArgs)]
        lib.dsv4_index_score_workspace_size.restype = ctypes.c_size_t
        lib.dsv4_index_score.argtypes = [ctypes.POINTER(IndexArgs), P, ctypes.c_size_t, P]
        lib.dsv4_topk_workspace_size.argtypes = [ctypes.POINTER(TopkArgs)]
        lib.dsv4_topk_workspace_size.restype = ctypes.c_size_t
        lib.dsv4_topk.argtypes = [ctypes.POINTER(TopkArgs), P, ctypes.c_size_t, P]
        lib.dsv4_topk_noalloc.argtypes = [ctypes.POINTER(TopkArgs), P]
        lib.dsv4_topk_noalloc.restype = I
        lib.dsv4_sparse_attn_workspace_size.argtypes = [ctypes.POINTER(AttnArgs)]
        lib.dsv4_sparse_attn_workspace_size.restype = ctypes.c_size_t
        lib.dsv4_sparse_attn_decode.argtypes = [ctypes.POINTER(AttnArgs), P, ctypes.c_size_t, P]
        lib.dsv4_csa_decode_workspace_size.argtypes = [ctypes.POINTER(CsaArgs)]
        lib.dsv4_csa_decode_workspace_size.restype = ctypes.c_size_t
        lib.dsv4_csa_decode.argtypes = [ctypes.POINTER(CsaArgs), P, ctypes.c_size_t, P]
        lib.dsv4_status_string.argtypes = [I]
        lib.dsv4_status_string.restype = ctypes.c_char_p
        lib.dsv4_read_error_word.argtypes = [P, P, ctypes.POINTER(ctypes.c_uint32)]
        lib.dsv4_last_launch_count.restype = I
        lib.dsv4_max_comp.argtypes = [ctypes.c_int64, I]
        lib.dsv4_max_comp.restype = ctypes.c_int64
        lib.dsv4_test_wait_fault.argtypes = [I, ctypes.c_uint32]
        lib.dsv4_test_wait_fault.restype = I
        lib.dsv4_copy_async.argtypes = [P, P, ctypes.c_size_t, P]
        lib.dsv4_copy_async.restype = I
        for f in ("dsv4_compress", "dsv4_indexer_topk", "dsv4_index_score", "dsv4_topk", "dsv4_sparse_attn_decode",
                  "dsv4_csa_decode", "dsv4_read_error_word"):
            getattr(lib, f).restype = I
        _lib = lib
    return _lib


# ------------------------------------------------------------------ marshalling helpers
def _ptr(t, dtype=None, name="tensor", optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status, what):
    if status != DSV4_OK:
        raise Dsv4Error(status, what)


def _dt():
    import torch
    return torch.bfloat16, torch.float32, torch.int32, torch.int64


# ------------------------------------------------------------------ argument builders
def compress_args(C, Z, bias, gamma, pos0, out, *, ratio, rope_dim=64, eps=1e-6,
                  rope_theta=10000.0, out_row0=None, overlap=False, prev_C=None, prev_Z=None,
                  out_scale=None, out_rope=None):
    """overlap=True: the two-stream (CSA) form, C and Z [B, T, 2*dim], bias [ratio, 2*dim],
    optional prev_C / prev_Z [B, ratio, 2*dim] (the block before C's first block).
    out_scale given: FP8 entries, out uint8 [B, rows, dim] and out_scale fp32 [B, rows].
    out_scale and out_rope given: the mixed KV storage, out uint8 [B, rows, dim - rope_dim]
    codes, out_scale fp32 [B, rows], out_rope bf16 [B, rows, rope_dim]."""
    import torch
    bf16, f32, i32, i64 = _dt()
    B, T, w = C.shape
    d = w // 2 if overlap else w
    fp8 = out_scale is not None
    mode = 2 if (fp8 and out_rope is not None) else (1 if fp8 else 0)
    return CompressArgs(_ptr(C, bf16, "C"), _ptr(Z, bf16, "Z"), _ptr(bias, f32, "bias"),
                        _ptr(gamma, f32, "gamma"), _ptr(pos0, i64, "pos0"),
                        _ptr(out, torch.uint8 if fp8 else bf16, "out"),
                        _ptr(out_row0, i32, "out_row0", True), B, T, d, ratio, rope_dim,
                        out.shape[1], eps, rope_theta, 1 if overlap else 0,
                        _ptr(prev_C, bf16, "prev_C", True), _ptr(prev_Z, bf16, "prev_Z", True),
                        mode, _ptr(out_scale, f32, "out_scale", True),
                        _ptr(out_rope, bf16, "out_rope", True))


def index_args(q, w, keys, n_comp, idx_out, *, ratio, q_pos=None, scores_out=None, q_scale=None,
               key_scale=None):
    """q_scale / key_scale given: q and keys are FP8 E4M3 codes (uint8), as
    dsv4_quantize_rows_fp8 writes them."""
    bf16, f32, i32, i64 = _dt()
    import torch
    fp8 = q_scale is not None
    kt = torch.uint8 if fp8 else bf16
    B, n_q, H, Di = q.shape
    return IndexArgs(_ptr(q, kt, "q"), _ptr(w, f32, "w"), _ptr(keys, kt, "keys"),
                     _ptr(n_comp, i32, "n_comp"), _ptr(q_pos, i64, "q_pos", True),
                     _ptr(idx_out, i32, "idx_out"), _ptr(scores_out, f32, "scores_out", True),
                     B, n_q, H, Di, keys.shape[1], idx_out.shape[-1], ratio, 1 if fp8 else 0,
                     _ptr(q_scale, f32, "q_scale", True), _ptr(key_scale, f32, "key_scale", True))


def topk_args(scores, n_vis, idx_out):
    bf16, f32, i32, i64 = _dt()
    rows = n_vis.numel()
    return TopkArgs(_ptr(scores, f32, "scores"), _ptr(n_vis, i32, "n_vis"),
                    _ptr(idx_out, i32, "idx_out"), rows, scores.shape[-1], idx_out.shape[-1])


def attn_args(q, sink, comp_kv, n_comp, win, win_len, out, *, idx=None, top_k=None, window=128,
              ratio=4, q_pos=None, gather=None, scale=None, out_rope_pos=None, out_rope_dim=64,
              out_rope_theta=10000.0, kv_nope=None, kv_scale=None, kv_rope=None):
    """out_rope_pos (int64 [B, n_q]): rotate the output's last out_rope_dim channels back at
    these positions (inverse RoPE). comp_kv None and kv_nope / kv_scale / kv_rope given: the
    mixed FP8 / bf16 compressed KV (codes uint8 [B, max_comp, D - rd], scales fp32
    [B, max_comp], RoPE part bf16 [B, max_comp, rd])."""
    import torch
    bf16, f32, i32, i64 = _dt()
    B, n_q, H, D = q.shape
    kv_fp8 = comp_kv is None
    max_comp = kv_nope.shape[1] if kv_fp8 else comp_kv.shape[1]
    if top_k is None:
        top_k = idx.shape[-1] if idx is not None else max_comp
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return AttnArgs(_ptr(q, bf16, "q"), _ptr(sink, f32, "sink"), _ptr(comp_kv, bf16, "comp_kv", kv_fp8),
                    _ptr(n_comp, i32, "n_comp"), _ptr(idx, i32, "idx", True),
                    _ptr(q_pos, i64, "q_pos", True), _ptr(win, bf16, "win"),
                    _ptr(win_len, i32, "win_len"), _ptr(gather, bf16, "gather", True),
                    _ptr(out, bf16, "out"), B, n_q, H, D, max_comp, top_k, window, win.shape[1],
                    ratio, scale, _ptr(out_rope_pos, i64, "out_rope_pos", True),
                    out_rope_dim if out_rope_pos is not None else 0, out_rope_theta,
                    1 if kv_fp8 else 0, _ptr(kv_nope, torch.uint8, "kv_nope", True),
                    _ptr(kv_scale, f32, "kv_scale", True), _ptr(kv_rope, bf16, "kv_rope", True),
                    kv_rope.shape[-1] if kv_fp8 else 0)


# ------------------------------------------------------------------ entry points
def dsv4_compress(C, Z, bias, gamma, pos0, out, *, ratio, rope_dim=64, eps=1e-6,
                  rope_theta=10000.0, out_row0=None, overlap=False, prev_C=None, prev_Z=None,
                  out_scale=None, out_rope=None, stream=None):
    a = compress_args(C, Z, bias, gamma, pos0, out, ratio=ratio, rope_dim=rope_dim, eps=eps,
                      rope_theta=rope_theta, out_row0=out_row0, overlap=overlap, prev_C=prev_C,
                      prev_Z=prev_Z, out_scale=out_scale, out_rope=out_rope)
    _check(library().dsv4_compress(ctypes.byref(a), _stream(stream)), "dsv4_compress")


def dsv4_quantize_rows_fp8(x, q, scale, *, stream=None):
    """FP8 E4M3 rows: x bf16 [..., dim] -> q uint8 [..., dim], scale fp32 [...]."""
    import torch
    bf16, f32, i32, i64 = _dt()
    dim = x.shape[-1]
    rows = x.numel() // dim
    _check(library().dsv4_quantize_rows_fp8(_ptr(x, bf16, "x"), rows, dim, _ptr(q, torch.uint8, "q"),
                                            _ptr(scale, f32, "scale"), _stream(stream)),
           "dsv4_quantize_rows_fp8")


def compress_step_state(batch, dim, ratio, *, overlap=False, device="cuda"):
    """Zeroed state for dsv4_compress_step: (stage, fill, n_comp)."""
    import torch
    w = 2 * dim if overlap else dim
    return (torch.zeros(batch, 2, 2, ratio, w, dtype=torch.bfloat16, device=device),
            torch.zeros(batch, dtype=torch.int32, device=device),
            torch.zeros(batch, dtype=torch.int32, device=device))


def dsv4_compress_step(C, Z, bias, gamma, pos, stage, fill, n_comp, out, *, ratio, rope_dim=64,
                       eps=1e-6, rope_theta=10000.0, overlap=False, out_scale=None, out_rope=None,
                       stream=None):
    """One decode token per sequence: C, Z [B, w] (w = dim, or 2*dim two-stream); pos int64 [B];
    state stage / fill / n_comp (see compress_step_state) updated on the device; a completed
    block goes to out[s, n_comp[s]]. out_scale (and out_rope): the FP8 (mixed) cache formats,
    as compress_args."""
    import torch
    bf16, f32, i32, i64 = _dt()
    B, w = C.shape
    fp8 = out_scale is not None
    mode = 2 if (fp8 and out_rope is not None) else (1 if fp8 else 0)
    d = out.shape[2] + (out_rope.shape[2] if mode == 2 else 0)
    a = StepArgs(_ptr(C, bf16, "C"), _ptr(Z, bf16, "Z"), _ptr(bias, f32, "bias"), _ptr(gamma, f32, "gamma"),
                 _ptr(pos, i64, "pos"), _ptr(stage, bf16, "stage"), _ptr(fill, i32, "fill"),
                 _ptr(n_comp, i32, "n_comp"), _ptr(out, torch.uint8 if fp8 else bf16, "out"), B, d, ratio,
                 rope_dim, out.shape[1], 1 if overlap else 0, eps, rope_theta, mode,
                 _ptr(out_scale, f32, "out_scale", True), _ptr(out_rope, bf16, "out_rope", True))
    _check(library().dsv4_compress_step(ctypes.byref(a), _stream(stream)), "dsv4_compress_step")


def dsv4_indexer_topk_workspace_size(q, w, keys, n_comp, idx_out, *, ratio, q_pos=None,
                                     scores_out=None, q_scale=None, key_scale=None):
    a = index_args(q, w, keys, n_comp, idx_out, ratio=ratio, q_pos=q_pos, scores_out=scores_out,
                   q_scale=q_scale, key_scale=key_scale)
    return int(library().dsv4_indexer_topk_workspace_size(ctypes.byref(a)))


def dsv4_indexer_topk(q, w, keys, n_comp, idx_out, ws, *, ratio, q_pos=None, scores_out=None,
                      q_scale=None, key_scale=None, stream=None):
    """q_scale / key_scale given: FP8 E4M3 queries and keys (see index_args)."""
    a = index_args(q, w, keys, n_comp, idx_out, ratio=ratio, q_pos=q_pos, scores_out=scores_out,
                   q_scale=q_scale, key_scale=key_scale)
    _check(library().dsv4_indexer_topk(ctypes.byref(a), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                       _stream(stream)), "dsv4_indexer_topk")


def dsv4_index_score_workspace_size(q, w, keys, n_comp, scores_out, *, ratio, q_pos=None,
                                    q_scale=None, key_scale=None):
    import torch
    idx = torch.empty(1, dtype=torch.int32, device=q.device)
    a = index_args(q, w, keys, n_comp, idx, ratio=ratio, q_pos=q_pos, scores_out=scores_out,
                   q_scale=q_scale, key_scale=key_scale)
    a.top_k = 1
    return int(library().dsv4_index_score_workspace_size(ctypes.byref(a)))


def dsv4_index_score(q, w, keys, n_comp, scores_out, ws, *, ratio, q_pos=None, q_scale=None,
                     key_scale=None, stream=None):
    """Scores only (no top-k): scores_out [B, n_q, max_comp] fp32 gets the visible scores."""
    import torch
    idx = torch.empty(1, dtype=torch.int32, device=q.device)
    a = index_args(q, w, keys, n_comp, idx, ratio=ratio, q_pos=q_pos, scores_out=scores_out,
                   q_scale=q_scale, key_scale=key_scale)
    a.top_k = 1
    _check(library().dsv4_index_score(ctypes.byref(a), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                      _stream(stream)), "dsv4_index_score")


def dsv4_topk_workspace_size(scores, n_vis, idx_out):
    a = topk_args(scores, n_vis, idx_out)
    return int(library().dsv4_topk_workspace_size(ctypes.byref(a)))


def dsv4_topk(scores, n_vis, idx_out, ws, *, stream=None):
    a = topk_args(scores, n_vis, idx_out)
    _check(library().dsv4_topk(ctypes.byref(a), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                               _stream(stream)), "dsv4_topk")


def dsv4_topk_noalloc(scores, n_vis, idx_out, *, stream=None):
    """dsv4_topk without a workspace, for callers that cannot allocate device memory: the
    library's fixed 16 MiB per-GPU scratch array is used instead. Calls must not overlap on
    the GPU; sizes needing more scratch than the array holds raise Dsv4Error
    (DSV4_ERR_INVALID_ARG)."""
    a = topk_args(scores, n_vis, idx_out)
    _check(library().dsv4_topk_noalloc(ctypes.byref(a), _stream(stream)), "dsv4_topk_noalloc")


def dsv4_sparse_attn_workspace_size(q, sink, comp_kv, n_comp, win, win_len, out, **kw):
    a = attn_args(q, sink, comp_kv, n_comp, win, win_len, out, **kw)
    return int(library().dsv4_sparse_attn_workspace_size(ctypes.byref(a)))


def dsv4_sparse_attn_decode(q, sink, comp_kv, n_comp, win, win_len, out, ws, *, stream=None, **kw):
    a = attn_args(q, sink, comp_kv, n_comp, win, win_len, out, **kw)
    _check(library().dsv4_sparse_attn_decode(ctypes.byref(a), _ptr(ws, None, "ws"),
                                             ws.numel() * ws.element_size(), _stream(stream)),
           "dsv4_sparse_attn_decode")


def _csa(compress_kv, compress_keys, index, attn):
    keep = (compress_kv, compress_keys, index, attn)
    c = CsaArgs(ctypes.pointer(compress_kv) if compress_kv is not None else None,
                ctypes.pointer(compress_keys) if compress_keys is not None else None,
                ctypes.pointer(index) if index is not None else None, ctypes.pointer(attn))
    return c, keep


def dsv4_csa_decode_workspace_size(*, attn, index=None, compress_kv=None, compress_keys=None):
    c, _keep = _csa(compress_kv, compress_keys, index, attn)
    return int(library().dsv4_csa_decode_workspace_size(ctypes.byref(c)))


def dsv4_csa_decode(ws, *, attn, index=None, compress_kv=None, compress_keys=None, stream=None):
    """One decode step from prepared argument structs (see compress_args / index_args /
    attn_args); the structs keep raw pointers, so the tensors must outlive the call."""
    c, _keep = _csa(compress_kv, compress_keys, index, attn)
    _check(library().dsv4_csa_decode(ctypes.byref(c), _ptr(ws, None, "ws"),
                                     ws.numel() * ws.element_size(), _stream(stream)),
           "dsv4_csa_decode")


def dsv4_read_error_word(ws, stream=None):
    v = ctypes.c_uint32(0)
    st = library().dsv4_read_error_word(_ptr(ws, None, "ws"), _stream(stream), ctypes.byref(v))
    return st, int(v.value)


def dsv4_status_string(status):
    try:
        return library().dsv4_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def dsv4_last_launch_count():
    return int(library().dsv4_last_launch_count())


def dsv4_max_comp(max_context, ratio):
    return int(library().dsv4_max_comp(int(max_context), int(ratio)))


def dsv4_copy_async(dst, src, stream=None):
    """Copies tensor src into dst (same byte size, contiguous; each on the GPU or in pinned host
    memory) with the library's copy kernel, after the kernel before it on the stream."""
    import torch
    for t, name in ((dst, "dst"), (src, "src")):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device.type != "cuda" and not t.is_pinned():
            raise ValueError(f"{name} must be on the GPU or in pinned host memory")
    nbytes = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != nbytes:
        raise ValueError("dst and src differ in size")
    _check(library().dsv4_copy_async(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), nbytes,
                                     _stream(stream)), "dsv4_copy_async")


def dsv4_test_wait_fault(which, wait_limit_us=0):
    """Test support: from now on every launch of kernel `which` (DSV4_WAIT_FAULT_*) leaves one
    copy unissued so its bounded wait runs out after wait_limit_us microseconds (0: the
    default 2 s); DSV4_WAIT_FAULT_NONE restores normal launches."""
    _check(library().dsv4_test_wait_fault(int(which), int(wait_limit_us)), "dsv4_test_wait_fault")
