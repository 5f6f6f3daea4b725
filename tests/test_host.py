"""CPU-only checks of the C ABI library: it builds for sm_103a, loads without a GPU, exports
every function that include/dsv4.h declares, rejects bad arguments on the host before any
CUDA call, and sizes workspaces sensibly. No compute calls are made here."""
from __future__ import annotations

import ctypes
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from compressed_sparse_attention_08_gb300 import _build, _abi
    _build.build()
    return _abi.library()


def header_functions():
    with open(os.path.join(ROOT, "include", "dsv4.h")) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsv4_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_function(lib):
    names = header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/dsv4.h but not exported"
    from compressed_sparse_attention_08_gb300 import EXPORTED_SYMBOLS
    assert sorted(EXPORTED_SYMBOLS) == names


def test_status_strings_and_sizing(lib):
    from compressed_sparse_attention_08_gb300 import _abi
    for s in range(6):
        assert _abi.dsv4_status_string(s)
    with open(os.path.join(ROOT, "tests", "golden", "page_sizes.json")) as fh:
        g = json.load(fh)
    for case in g["max_comp"]:
        assert _abi.dsv4_max_comp(case["context"], case["ratio"]) == case["entries"]
    assert _abi.dsv4_max_comp(10, 4) == 3 and _abi.dsv4_max_comp(8, 0) == -1


FAKE = 0x7F0000000000   # aligned fake device addresses: never dereferenced on the host path


def _p(i):
    return ctypes.c_void_p(FAKE + 4096 * i)


def _index_args(**over):
    from compressed_sparse_attention_08_gb300._abi import IndexArgs
    a = dict(q=_p(1), w=_p(2), keys=_p(3), n_comp=_p(4), q_pos=None, idx_out=_p(5), scores_out=None,
             batch=4, n_q=1, heads=64, dim=128, max_comp=262144, top_k=2048, ratio=4)
    a.update(over)
    return IndexArgs(**a)


def _attn_args(**over):
    from compressed_sparse_attention_08_gb300._abi import AttnArgs
    a = dict(q=_p(1), sink=_p(2), comp_kv=_p(3), n_comp=_p(4), idx=_p(5), q_pos=None, win=_p(6),
             win_len=_p(7), gather=None, out=_p(8), batch=4, n_q=1, heads=64, dim=512,
             max_comp=262144, top_k=2048, window=128, win_rows=128, ratio=4, scale=0.0442)
    a.update(over)
    return AttnArgs(**a)


@pytest.mark.parametrize("bad", [
    dict(top_k=300000), dict(top_k=0), dict(dim=64), dict(heads=12), dict(heads=72),
    dict(q=None), dict(q=ctypes.c_void_p(FAKE + 8)), dict(n_q=0), dict(ratio=0), dict(max_comp=0),
])
def test_indexer_rejects_on_host(lib, bad):
    a = _index_args(**bad)
    ws_bytes = lib.dsv4_indexer_topk_workspace_size(ctypes.byref(a))
    rc = lib.dsv4_indexer_topk(ctypes.byref(a), _p(9), ws_bytes, None)
    assert rc == 1


def test_indexer_rejects_small_workspace(lib):
    a = _index_args()
    need = lib.dsv4_indexer_topk_workspace_size(ctypes.byref(a))
    # scores (4 MiB) + the top-k's per-row histograms (4096 + 4096 + 256 bins)
    assert need >= 4 * 262144 * 4 + 4 * 8448 * 4
    assert lib.dsv4_indexer_topk(ctypes.byref(a), _p(9), need - 1, None) == 1


def _align256(n):
    return (n + 255) // 256 * 256


def _split_ws(rows, chunks, heads, dim):
    """The split form's partials: (m, l) and the fp32 O per (row, chunk, head)."""
    hs = (heads + 31) // 32 * 32 if heads % 32 == 0 else (heads + 15) // 16 * 16
    return _align256(rows * chunks * hs * 2 * 4) + _align256(rows * chunks * hs * dim * 4)


def test_attention_workspace_split_and_walk(lib):
    """Decode (few query rows) splits each row into 128-slot chunks and needs partials; from
    304 (query row, head group) pairs on, one CTA walks each row and needs the header only."""
    header = lib.dsv4_sparse_attn_workspace_size(ctypes.byref(_attn_args(batch=1, n_q=2048, top_k=1024,
                                                                         max_comp=16896, q_pos=_p(10))))
    assert header == 256
    # the bench decode: 4 rows x 17 chunks x 64 heads x 512 dims
    need = lib.dsv4_sparse_attn_workspace_size(ctypes.byref(_attn_args()))
    assert need == header + _split_ws(4, 17, 64, 512)
    # the threshold: 64 heads = 2 groups of 32, 16 heads = 1 group
    for heads, rows_split in ((64, 151), (16, 303)):
        a = _attn_args(batch=1, n_q=rows_split, heads=heads, q_pos=_p(10))
        assert lib.dsv4_sparse_attn_workspace_size(ctypes.byref(a)) == header + _split_ws(rows_split, 17, heads, 512)
        a = _attn_args(batch=1, n_q=rows_split + 1, heads=heads, q_pos=_p(10))
        assert lib.dsv4_sparse_attn_workspace_size(ctypes.byref(a)) == header
    # 48 heads: three groups of 16
    a = _attn_args(batch=3, n_q=1, heads=48, dim=256, top_k=48, window=64, max_comp=200)
    assert lib.dsv4_sparse_attn_workspace_size(ctypes.byref(a)) == header + _split_ws(3, 1, 48, 256)


@pytest.mark.parametrize("bad", [
    dict(dim=100), dict(heads=0), dict(heads=65), dict(idx=None),   # dense needs top_k == max_comp
    dict(top_k=262145), dict(win_rows=0), dict(scale=float("inf")), dict(out=None),
    dict(gather=ctypes.c_void_p(FAKE + 4)),
    dict(out_rope_pos=_p(11), out_rope_dim=0), dict(out_rope_pos=_p(11), out_rope_dim=63),
    dict(out_rope_pos=_p(11), out_rope_dim=256), dict(out_rope_pos=_p(11), out_rope_dim=64, out_rope_theta=0.0),
    dict(out_rope_pos=ctypes.c_void_p(FAKE + 4096 * 11 + 4), out_rope_dim=64, out_rope_theta=1e4),
    # mixed FP8 / bf16 KV: comp_kv must be NULL, the three parts given, the RoPE part 8..dim-8
    dict(kv_fp8=1, kv_nope=_p(12), kv_scale=_p(13), kv_rope=_p(14), kv_rope_dim=64),
    dict(comp_kv=None, kv_fp8=1, kv_nope=_p(12), kv_scale=_p(13), kv_rope=None, kv_rope_dim=64),
    dict(comp_kv=None, kv_fp8=1, kv_nope=_p(12), kv_scale=_p(13), kv_rope=_p(14), kv_rope_dim=60),
    dict(comp_kv=None, kv_fp8=1, kv_nope=_p(12), kv_scale=_p(13), kv_rope=_p(14), kv_rope_dim=512),
    dict(comp_kv=None, kv_fp8=2, kv_nope=_p(12), kv_scale=_p(13), kv_rope=_p(14), kv_rope_dim=64),
    dict(kv_nope=_p(12)),
])
def test_attention_rejects_on_host(lib, bad):
    a = _attn_args(**bad)
    rc = lib.dsv4_sparse_attn_decode(ctypes.byref(a), _p(9), 1 << 40, None)
    assert rc == 1


def test_compress_rejects_on_host(lib):
    from compressed_sparse_attention_08_gb300._abi import CompressArgs
    base = dict(C=_p(1), Z=_p(2), bias=_p(3), gamma=_p(4), pos0=_p(5), out=_p(6), out_row0=None,
                batch=4, tokens=16, dim=512, ratio=4, rope_dim=64, out_rows=4, eps=1e-6,
                rope_theta=10000.0)
    for bad in (dict(tokens=15), dict(rope_dim=63), dict(rope_dim=1024), dict(dim=2048),
                dict(out_rows=3), dict(eps=-1.0), dict(C=None), dict(ratio=0), dict(overlap=2),
                dict(overlap=1, prev_C=_p(7)), dict(overlap=0, prev_C=_p(7), prev_Z=_p(8)),
                dict(overlap=1, prev_C=_p(7), prev_Z=ctypes.c_void_p(FAKE + 4096 * 9 + 8)),
                dict(out_fp8=3, out_scale=_p(7)), dict(out_fp8=1), dict(out_scale=_p(7)),
                dict(out_fp8=1, out_scale=ctypes.c_void_p(FAKE + 4096 * 7 + 4)),
                dict(out_fp8=2, out_scale=_p(7)), dict(out_fp8=1, out_scale=_p(7), out_rope=_p(8)),
                dict(out_rope=_p(8)), dict(out_fp8=2, out_scale=_p(7), out_rope=_p(8), rope_dim=512)):
        a = CompressArgs(**{**base, **bad})
        assert lib.dsv4_compress(ctypes.byref(a), None) == 1, bad


def test_compress_step_rejects_on_host(lib):
    from compressed_sparse_attention_08_gb300._abi import StepArgs
    base = dict(C=_p(1), Z=_p(2), bias=_p(3), gamma=_p(4), pos=_p(5), stage=_p(6), fill=_p(7),
                n_comp=_p(8), out=_p(9), batch=4, dim=512, ratio=4, rope_dim=64, out_rows=10,
                overlap=0, eps=1e-6, rope_theta=10000.0)
    for bad in (dict(stage=None), dict(fill=None), dict(n_comp=None), dict(ratio=0),
                dict(dim=2048), dict(rope_dim=65), dict(out_rows=0), dict(overlap=3),
                dict(rope_theta=-1.0), dict(pos=ctypes.c_void_p(FAKE + 4)),
                dict(out_fp8=3, out_scale=_p(10)), dict(out_fp8=1), dict(out_scale=_p(10)),
                dict(out_fp8=2, out_scale=_p(10)), dict(out_rope=_p(11)),
                dict(out_fp8=2, out_scale=_p(10), out_rope=_p(11), rope_dim=512)):
        a = StepArgs(**{**base, **bad})
        assert lib.dsv4_compress_step(ctypes.byref(a), None) == 1, bad


def test_fused_requires_consistent_stages(lib):
    from compressed_sparse_attention_08_gb300._abi import CsaArgs, IndexArgs, AttnArgs
    ia = _index_args()
    aa = _attn_args(idx=ia.idx_out)
    c = CsaArgs(None, None, ctypes.pointer(ia), ctypes.pointer(aa))
    need = lib.dsv4_csa_decode_workspace_size(ctypes.byref(c))
    assert need >= lib.dsv4_indexer_topk_workspace_size(ctypes.byref(ia))
    aa2 = _attn_args(idx=_p(42))          # attention must read the indexer's output
    c2 = CsaArgs(None, None, ctypes.pointer(ia), ctypes.pointer(aa2))
    assert lib.dsv4_csa_decode(ctypes.byref(c2), _p(9), need, None) == 1


def test_fused_key_cache_format_must_match(lib):
    """A key cache written in the step is scored in the format it was written in."""
    from compressed_sparse_attention_08_gb300._abi import CsaArgs, CompressArgs
    ia = _index_args(key_fp8=1, q_scale=_p(20), key_scale=_p(21))
    aa = _attn_args(idx=ia.idx_out)
    base = dict(C=_p(1), Z=_p(2), bias=_p(3), gamma=_p(4), pos0=_p(5), out=ia.keys, out_row0=None,
                batch=4, tokens=16, dim=128, ratio=4, rope_dim=64, out_rows=262144, eps=1e-6,
                rope_theta=10000.0)
    for bad in (dict(), dict(out_fp8=1, out_scale=_p(22))):   # bf16 entries; another scale array
        cq = CompressArgs(**{**base, **bad})
        c = CsaArgs(None, ctypes.pointer(cq), ctypes.pointer(ia), ctypes.pointer(aa))
        need = lib.dsv4_csa_decode_workspace_size(ctypes.byref(c))
        assert lib.dsv4_csa_decode(ctypes.byref(c), _p(9), need, None) == 1, bad


def test_binding_refuses_without_library(tmp_path, monkeypatch):
    from compressed_sparse_attention_08_gb300 import _abi
    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi, "library_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _abi.library()


@pytest.mark.parametrize("dst, src, nbytes", [
    (None, _p(1), 16),                              # null
    (_p(0), ctypes.c_void_p(FAKE + 4096 + 8), 16),  # unaligned source
    (_p(0), _p(1), 24),                             # not a multiple of 16
    (_p(0), ctypes.c_void_p(FAKE + 64), 128),       # overlapping ranges
])
def test_copy_rejects_on_host(lib, dst, src, nbytes):
    """dsv4_copy_async refuses bad arguments before touching the device."""
    assert lib.dsv4_copy_async(dst, src, nbytes, None) == 1


def test_copy_of_nothing_is_a_no_op(lib):
    assert lib.dsv4_copy_async(_p(0), _p(1), 0, None) == 0
