"""GPU parity: every stage of the CSA step against the fp64 oracle on seeded inputs.

Runs through the C ABI (ctypes binding) on cuda:0. Sizes: the five workloads at full size
(the oracle checks sampled sequences/queries where a full check would take minutes), plus
small ragged and degenerate cases.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from compressed_sparse_attention_08_gb300 import synth
from compressed_sparse_attention_08_gb300.workloads import WORKLOADS, make_inputs
from helpers import (assert_bf16_close, check_topk_row, dev, dev_bf16, host_bf16,
                     topk_valid_for_scores, bf16_to_f64)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_sparse_attention_08_gb300 import _build
    _build.build()


def csa():
    import compressed_sparse_attention_08_gb300 as m
    return m


def ws_tensor(nbytes):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


_INPUTS = {}


def inputs(cfg):
    if cfg not in _INPUTS:
        _INPUTS[cfg] = make_inputs(WORKLOADS[cfg])
    return _INPUTS[cfg]


def _oracle_keys(x, wl):
    """Compressed indexer keys for workloads that compress the whole context (oracle)."""
    bits, _ = oracle.compress(x["C_I"], x["Z_I"], x["bias_I"], x["gamma_I"], x["pos0"], wl.ratio,
                              wl.rope_dim)
    return bits


def _oracle_kv(x, wl, seqs=None):
    C, Z, pos0 = x["C"], x["Z"], x["pos0"]
    if seqs is not None:
        C, Z, pos0 = C[seqs], Z[seqs], pos0[seqs]
    return oracle.compress(C, Z, x["bias"], x["gamma"], pos0, wl.ratio, wl.rope_dim)


def _gpu_compress(C, Z, bias, gamma, pos0, ratio, out_rows=None, out_row0=None, out=None, rope_dim=64):
    m = csa()
    B, T, d = C.shape
    if out is None:
        out = torch.zeros(B, out_rows or T // ratio, d, dtype=torch.bfloat16, device="cuda")
    m.dsv4_compress(dev_bf16(C), dev_bf16(Z), dev(bias), dev(gamma), dev(pos0), out, ratio=ratio,
                    rope_dim=rope_dim, out_row0=None if out_row0 is None else dev(out_row0))
    torch.cuda.synchronize()
    return out


# ------------------------------------------------------------------ stage 1: compressor
@pytest.mark.parametrize("cfg", [0, 1])
def test_compress_full_context(cfg):
    wl = WORKLOADS[cfg]
    x = inputs(cfg)
    got = host_bf16(_gpu_compress(x["C"], x["Z"], x["bias"], x["gamma"], x["pos0"], wl.ratio))
    seqs = None if cfg == 0 else [0, 7, 15]
    _, ref = _oracle_kv(x, wl, seqs)
    assert_bf16_close(got if seqs is None else got[seqs], ref, f"cfg{cfg} main KV")
    gk = host_bf16(_gpu_compress(x["C_I"], x["Z_I"], x["bias_I"], x["gamma_I"], x["pos0"], wl.ratio))
    _, rk = oracle.compress(x["C_I"], x["Z_I"], x["bias_I"], x["gamma_I"], x["pos0"], wl.ratio, wl.rope_dim)
    assert_bf16_close(gk, rk, f"cfg{cfg} indexer keys")


def test_compress_hca_ratio128():
    wl = WORKLOADS[2]
    x = inputs(2)
    got = host_bf16(_gpu_compress(x["C"], x["Z"], x["bias"], x["gamma"], x["pos0"], wl.ratio))
    seqs = [0, 31, 63]
    _, ref = _oracle_kv(x, wl, seqs)
    assert got.shape == (64, 64, 512)
    assert_bf16_close(got[seqs], ref, "HCA ratio 128")


def test_compress_newest_block_into_cache():
    """1M context: the newest block of each sequence lands in row n_comp - 1 of the cache."""
    wl = WORKLOADS[3]
    x = inputs(3)
    cache = torch.zeros(4, wl.max_comp, 512, dtype=torch.bfloat16, device="cuda")
    _gpu_compress(x["C"], x["Z"], x["bias"], x["gamma"], x["pos0"], wl.ratio, out=cache,
                  out_row0=x["append_row"])
    _, ref = _oracle_kv(x, wl)
    rows = host_bf16(cache[:, wl.max_comp - 1:wl.max_comp]).reshape(4, 1, 512)
    assert_bf16_close(rows, ref, "newest block")
    assert int(torch.count_nonzero(cache[:, :wl.max_comp - 1].view(torch.int16))) == 0


def test_compress_prefill_chunk():
    wl = WORKLOADS[4]
    x = inputs(4)
    cache = torch.zeros(1, wl.max_comp, 512, dtype=torch.bfloat16, device="cuda")
    _gpu_compress(x["C"], x["Z"], x["bias"], x["gamma"], x["pos0"], wl.ratio, out=cache,
                  out_row0=x["append_row"])
    _, ref = _oracle_kv(x, wl)
    got = host_bf16(cache[:, 16384:])
    assert_bf16_close(got, ref, "prefill chunk entries")


# ------------------------------------------------------------------ stage 1, two-stream (CSA) form
def _overlap_inputs(seed, B, T, d, ratio, prev=False):
    C = synth.normal_bf16(seed, 101, (B, T, 2 * d))
    Z = synth.normal_bf16(seed, 102, (B, T, 2 * d))
    bias = synth.bf16_bits_to_f32(synth.normal_bf16(seed, 103, (ratio, 2 * d), 0.0, 0.5))
    gamma = synth.bf16_bits_to_f32(synth.normal_bf16(seed, 104, (d,), 1.0, 0.1))
    pC = synth.normal_bf16(seed, 105, (B, ratio, 2 * d)) if prev else None
    pZ = synth.normal_bf16(seed, 106, (B, ratio, 2 * d)) if prev else None
    return C, Z, bias, gamma, pC, pZ


def _gpu_compress_overlap(C, Z, bias, gamma, pos0, ratio, prev_C=None, prev_Z=None, out=None,
                          out_row0=None, rope_dim=64):
    m = csa()
    B, T, w = C.shape
    if out is None:
        out = torch.zeros(B, T // ratio, w // 2, dtype=torch.bfloat16, device="cuda")
    m.dsv4_compress(dev_bf16(C), dev_bf16(Z), dev(bias), dev(gamma), dev(pos0), out, ratio=ratio,
                    rope_dim=rope_dim, out_row0=None if out_row0 is None else dev(out_row0),
                    overlap=True, prev_C=None if prev_C is None else dev_bf16(prev_C),
                    prev_Z=None if prev_Z is None else dev_bf16(prev_Z))
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("d", [512, 128])
def test_compress_overlap_full_context(d):
    """8192 tokens -> 2048 entries per sequence, the sequence's first block without stream a."""
    B, T, r = 2, 8192, 4
    C, Z, bias, gamma, _, _ = _overlap_inputs(1, B, T, d, r)
    pos0 = np.zeros(B, np.int64)
    got = host_bf16(_gpu_compress_overlap(C, Z, bias, gamma, pos0, r))
    _, ref = oracle.compress_overlap(C, Z, bias, gamma, pos0, r)
    assert_bf16_close(got, ref, f"two-stream compressor d={d}")


def test_compress_overlap_newest_block_with_previous_block():
    """Decode: the newest block (stream b) plus the block before it (stream a, from the
    previous-block buffer) into row n_comp - 1 of a cache."""
    B, r, d, n_rows = 4, 4, 512, 1000
    C, Z, bias, gamma, pC, pZ = _overlap_inputs(3, B, r, d, r, prev=True)
    pos0 = np.array([3996, 396, 1200, 8], np.int64)
    row0 = (pos0 // r).astype(np.int32)
    cache = torch.zeros(B, n_rows, d, dtype=torch.bfloat16, device="cuda")
    _gpu_compress_overlap(C, Z, bias, gamma, pos0, r, pC, pZ, out=cache, out_row0=row0)
    _, ref = oracle.compress_overlap(C, Z, bias, gamma, pos0, r, pC, pZ)
    got = host_bf16(cache)
    for b in range(B):
        assert_bf16_close(got[b, row0[b]:row0[b] + 1], ref[b], f"seq {b}")
        others = np.delete(got[b], row0[b], axis=0)
        assert not np.any(others), f"seq {b}: rows other than the newest were written"


def test_compress_overlap_long_blocks():
    """ratio 16 and 40 (not multiples of the 8-token load chunk), previous block given."""
    for r in (16, 40):
        B, T, d = 2, 4 * r, 256
        C, Z, bias, gamma, pC, pZ = _overlap_inputs(4 + r, B, T, d, r, prev=True)
        pos0 = np.array([r * 9, r * 100], np.int64)
        got = host_bf16(_gpu_compress_overlap(C, Z, bias, gamma, pos0, r, pC, pZ))
        _, ref = oracle.compress_overlap(C, Z, bias, gamma, pos0, r, pC, pZ)
        assert_bf16_close(got, ref, f"ratio {r}")


# ------------------------------------------------------------------ stage 1 at decode time: one token per call
@pytest.mark.parametrize("overlap", [False, True])
def test_compress_step_matches_block_compressor(overlap):
    """Token by token through the device-side step (state on the device, one launch per token)
    for 3 sequences over 30 tokens with ratio 4: the cache rows and counts equal the oracle's
    compression of the whole token history."""
    m = csa()
    B, d, r, T = 3, 512, 4, 30
    w = 2 * d if overlap else d
    C = synth.normal_bf16(7, 111, (B, T, w))
    Z = synth.normal_bf16(7, 112, (B, T, w))
    bias = synth.bf16_bits_to_f32(synth.normal_bf16(7, 113, (r, w), 0.0, 0.5))
    gamma = synth.bf16_bits_to_f32(synth.normal_bf16(7, 114, (d,), 1.0, 0.1))
    pos0 = np.array([0, 4096, 1048000], np.int64)                 # block-aligned starts
    stage, fill, n_comp = m.compress_step_state(B, d, r, overlap=overlap)
    cache = torch.zeros(B, 16, d, dtype=torch.bfloat16, device="cuda")
    Cd, Zd, bd, gd = dev_bf16(C), dev_bf16(Z), dev(bias), dev(gamma)
    for t in range(T):
        pos = dev(pos0 + t)
        m.dsv4_compress_step(Cd[:, t].contiguous(), Zd[:, t].contiguous(), bd, gd, pos, stage, fill,
                             n_comp, cache, ratio=r, overlap=overlap)
    torch.cuda.synchronize()
    nb = T // r
    assert n_comp.cpu().tolist() == [nb] * B and fill.cpu().tolist() == [T % r] * B
    Tb = nb * r
    if overlap:
        _, ref = oracle.compress_overlap(C[:, :Tb], Z[:, :Tb], bias, gamma, pos0, r)
    else:
        _, ref = oracle.compress(C[:, :Tb], Z[:, :Tb], bias, gamma, pos0, r, 64)
    got = host_bf16(cache)
    assert_bf16_close(got[:, :nb], ref, "step compressor")
    assert not np.any(got[:, nb:]), "rows past n_comp were written"


@pytest.mark.parametrize("mode", ["fp8", "mixed"])
def test_compress_step_fp8_outputs(mode):
    """The device-side decode compressor writing an FP8 key cache (128-wide entries) or the
    mixed KV storage (512-wide entries), token by token, against the oracle's compression of
    the whole token history quantized by the oracle."""
    m = csa()
    B, r, T = 3, 4, 24
    d = 128 if mode == "fp8" else 512
    rd = 64
    C = synth.normal_bf16(9, 131, (B, T, d))
    Z = synth.normal_bf16(9, 132, (B, T, d))
    bias = synth.bf16_bits_to_f32(synth.normal_bf16(9, 133, (r, d), 0.0, 0.5))
    gamma = synth.bf16_bits_to_f32(synth.normal_bf16(9, 134, (d,), 1.0, 0.1))
    pos0 = np.array([0, 8192, 1048000], np.int64)
    stage, fill, n_comp = m.compress_step_state(B, d, r)
    rows = 8
    qd = d if mode == "fp8" else d - rd
    out = torch.zeros(B, rows, qd, dtype=torch.uint8, device="cuda")
    sc = torch.full((B, rows), float("nan"), dtype=torch.float32, device="cuda")
    rope = torch.zeros(B, rows, rd, dtype=torch.bfloat16, device="cuda") if mode == "mixed" else None
    Cd, Zd, bd, gd = dev_bf16(C), dev_bf16(Z), dev(bias), dev(gamma)
    for t in range(T):
        m.dsv4_compress_step(Cd[:, t].contiguous(), Zd[:, t].contiguous(), bd, gd, dev(pos0 + t), stage, fill,
                             n_comp, out, ratio=r, rope_dim=rd, out_scale=sc, out_rope=rope)
    torch.cuda.synchronize()
    nb = T // r
    assert n_comp.cpu().tolist() == [nb] * B
    _, ref = oracle.compress(C, Z, bias, gamma, pos0, r, rd)
    _check_fp8_cache(out.cpu().numpy()[:, :nb], sc.cpu().numpy()[:, :nb], ref[..., :qd], f"step {mode}")
    if mode == "mixed":
        assert_bf16_close(host_bf16(rope)[:, :nb], ref[..., qd:], "step mixed: RoPE part")
    assert not np.any(out.cpu().numpy()[:, nb:]), "rows past n_comp were written"


def test_compress_step_graph_replay_and_full_cache():
    """One captured graph replayed for every token (inputs copied into fixed buffers); a cache
    that is full keeps its rows and its count."""
    m = csa()
    B, d, r, T, rows = 2, 128, 4, 24, 5
    C = synth.normal_bf16(8, 121, (B, T, d))
    Z = synth.normal_bf16(8, 122, (B, T, d))
    bias = synth.bf16_bits_to_f32(synth.normal_bf16(8, 123, (r, d), 0.0, 0.5))
    gamma = synth.bf16_bits_to_f32(synth.normal_bf16(8, 124, (d,), 1.0, 0.1))
    pos0 = np.array([8, 800], np.int64)
    stage, fill, n_comp = m.compress_step_state(B, d, r)
    cache = torch.zeros(B, rows, d, dtype=torch.bfloat16, device="cuda")
    Cd, Zd = dev_bf16(C), dev_bf16(Z)
    tok_c = torch.empty(B, d, dtype=torch.bfloat16, device="cuda")
    tok_z = torch.empty_like(tok_c)
    pos = torch.empty(B, dtype=torch.int64, device="cuda")
    posd = dev(pos0)
    bd, gd = dev(bias), dev(gamma)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            m.dsv4_compress_step(tok_c, tok_z, bd, gd, pos, stage, fill, n_comp, cache, ratio=r, stream=s)
        for t in range(T):
            tok_c.copy_(Cd[:, t])
            tok_z.copy_(Zd[:, t])
            pos.copy_(posd + t)
            g.replay()
    torch.cuda.synchronize()
    assert n_comp.cpu().tolist() == [rows] * B                   # 6 blocks completed, 5 rows kept
    _, ref = oracle.compress(C[:, :rows * r], Z[:, :rows * r], bias, gamma, pos0, r, 64)
    assert_bf16_close(host_bf16(cache), ref, "graph-replayed step compressor")


# ------------------------------------------------------------------ stage 2: indexer + top-k
def _run_indexer(q, w, keys, n_comp, top_k, ratio=4, q_pos=None, want_scores=True):
    m = csa()
    B, n_q = q.shape[:2]
    max_comp = keys.shape[1]
    qd, wd, kd, nd = dev_bf16(q), dev(w), dev_bf16(keys), dev(n_comp)
    pd = None if q_pos is None else dev(q_pos)
    idx = torch.empty(B, n_q, top_k, dtype=torch.int32, device="cuda")
    sc = torch.full((B, n_q, max_comp), float("nan"), dtype=torch.float32, device="cuda") if want_scores else None
    nbytes = m.dsv4_indexer_topk_workspace_size(qd, wd, kd, nd, idx, ratio=ratio, q_pos=pd, scores_out=sc)
    ws = ws_tensor(nbytes)
    m.dsv4_indexer_topk(qd, wd, kd, nd, idx, ws, ratio=ratio, q_pos=pd, scores_out=sc)
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    assert ew == 0, f"device error word {ew:#x}"
    return idx.cpu().numpy(), (sc.cpu().numpy() if sc is not None else None)


def _check_scores(got, ref, n_vis):
    g = got[:n_vis].astype(np.float64)
    r = ref[:n_vis]
    scale = np.mean(np.abs(r)) + 1e-30
    err = np.abs(g - r)
    assert np.all(err <= 2e-5 * scale + 2e-5 * np.abs(r)), f"scores: max err {err.max():.3e} (scale {scale:.3e})"


@pytest.mark.parametrize("cfg", [0, 1])
def test_indexer_topk_decode(cfg):
    wl = WORKLOADS[cfg]
    x = inputs(cfg)
    keys = _oracle_keys(x, wl)
    idx, sc = _run_indexer(x["q_I"], x["w"], keys, x["n_comp"], wl.top_k)
    ref_s, nv = oracle.index_scores(x["q_I"], x["w"], keys, x["n_comp"], wl.ratio)
    ref_i = oracle.topk(ref_s, nv, wl.top_k)
    swaps = 0
    for b in range(wl.batch):
        _check_scores(sc[b, 0], ref_s[b, 0], nv[b, 0])
        swaps += check_topk_row(idx[b, 0], ref_i[b, 0], ref_s[b, 0], nv[b, 0], wl.top_k, f"b{b}")
        topk_valid_for_scores(idx[b, 0], sc[b, 0], nv[b, 0], wl.top_k, f"b{b}")
    assert swaps <= wl.batch


def test_indexer_topk_1m_context():
    """262,144 keys per sequence, top-2048: the long-row selection path."""
    wl = WORKLOADS[3]
    x = inputs(3)
    idx, sc = _run_indexer(x["q_I"], x["w"], x["keys"], x["n_comp"], wl.top_k)
    for b in range(4):
        topk_valid_for_scores(idx[b, 0], sc[b, 0], wl.n_comp, wl.top_k, f"b{b}")
    for b in (0, 3):
        ref_s, nv = oracle.index_scores(x["q_I"][b:b + 1], x["w"][b:b + 1], x["keys"][b:b + 1],
                                        x["n_comp"][b:b + 1], wl.ratio)
        ref_i = oracle.topk(ref_s, nv, wl.top_k)
        _check_scores(sc[b, 0], ref_s[0, 0], nv[0, 0])
        check_topk_row(idx[b, 0], ref_i[0, 0], ref_s[0, 0], nv[0, 0], wl.top_k, f"b{b}")


def test_indexer_topk_prefill_causal():
    """2048 queries over 16,896 keys with the causal block rule; sampled queries vs oracle."""
    wl = WORKLOADS[4]
    x = inputs(4)
    idx, sc = _run_indexer(x["q_I"], x["w"], x["keys"], x["n_comp"], wl.top_k, q_pos=x["q_pos"])
    sample = np.array([0, 1, 2, 3, 4, 777, 1024, 2045, 2046, 2047])
    ref_s, nv = oracle.index_scores(x["q_I"][:, sample], x["w"][:, sample], x["keys"], x["n_comp"],
                                    wl.ratio, q_pos=x["q_pos"][:, sample])
    ref_i = oracle.topk(ref_s, nv, wl.top_k)
    for j, t in enumerate(sample):
        assert nv[0, j] == 16384 + (t + 1) // 4
        _check_scores(sc[0, t], ref_s[0, j], nv[0, j])
        check_topk_row(idx[0, t], ref_i[0, j], ref_s[0, j], nv[0, j], wl.top_k, f"q{t}")
    for t in range(0, 2048, 97):
        n = 16384 + (t + 1) // 4
        topk_valid_for_scores(idx[0, t], sc[0, t], n, wl.top_k, f"q{t}")


def test_indexer_small_heads_ragged():
    """8 heads (N = 16 UMMA with zero-padded queries), ragged n_comp, fewer keys than top_k."""
    rng = np.random.default_rng(5)
    B, H, N, k = 4, 8, 700, 96
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, 1, H, 128)).astype(np.float32))
    keys = synth.f32_to_bf16_bits(rng.standard_normal((B, N, 128)).astype(np.float32))
    w = rng.standard_normal((B, 1, H)).astype(np.float32)
    n_comp = np.array([700, 0, 50, 129], np.int32)
    idx, sc = _run_indexer(q, w, keys, n_comp, k)
    ref_s, nv = oracle.index_scores(q, w, keys, n_comp, 4)
    ref_i = oracle.topk(ref_s, nv, k)
    for b in range(B):
        if nv[b, 0]:
            _check_scores(sc[b, 0], ref_s[b, 0], nv[b, 0])
        check_topk_row(idx[b, 0], ref_i[b, 0], ref_s[b, 0], nv[b, 0], k, f"b{b}")


def test_indexer_cache_shorter_than_one_tile():
    """A 100-row key cache: every key tile reaches past the cache's end."""
    rng = np.random.default_rng(6)
    B, H, N, k = 2, 16, 100, 32
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, 1, H, 128)).astype(np.float32))
    keys = synth.f32_to_bf16_bits(rng.standard_normal((B, N, 128)).astype(np.float32))
    w = rng.standard_normal((B, 1, H)).astype(np.float32)
    n_comp = np.array([100, 37], np.int32)
    idx, sc = _run_indexer(q, w, keys, n_comp, k)
    ref_s, nv = oracle.index_scores(q, w, keys, n_comp, 4)
    ref_i = oracle.topk(ref_s, nv, k)
    for b in range(B):
        _check_scores(sc[b, 0], ref_s[b, 0], nv[b, 0])
        check_topk_row(idx[b, 0], ref_i[b, 0], ref_s[b, 0], nv[b, 0], k, f"b{b}")


@pytest.mark.parametrize("n_q,H,N", [(2, 64, 700), (3, 40, 700), (4, 64, 700), (5, 64, 700), (6, 32, 700),
                                     (7, 40, 700), (12, 16, 700), (5, 64, 100)])
def test_indexer_several_queries_per_mma(n_q, H, N):
    """More query rows than SMs and no histogram: two (n_q 2, 3) or four queries share each
    key tile's MMA, the last unit of a sequence ragged (n_q 5, 7); causal positions give every
    query its own visible count, some inside a tile, some past the cache's ragged end (a cache
    of 100 rows: the only tile reaches past it)."""
    rng = np.random.default_rng(70 + n_q + N)
    B, k = 152 // n_q + 1, 64
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, n_q, H, 128)).astype(np.float32))
    keys = synth.f32_to_bf16_bits(rng.standard_normal((B, N, 128)).astype(np.float32))
    w = rng.standard_normal((B, n_q, H)).astype(np.float32)
    n_comp = rng.integers(0, N + 1, B).astype(np.int32)
    n_comp[0], n_comp[-1] = N, 0
    q_pos = rng.integers(0, 4 * N, B).astype(np.int64)[:, None] + np.arange(n_q, dtype=np.int64)[None, :]
    idx, sc = _run_indexer(q, w, keys, n_comp, k, q_pos=q_pos)
    ref_s, nv = oracle.index_scores(q, w, keys, n_comp, 4, q_pos=q_pos)
    ref_i = oracle.topk(ref_s, nv, k)
    for b in range(B):
        for t in range(n_q):
            if nv[b, t]:
                _check_scores(sc[b, t], ref_s[b, t], nv[b, t])
            check_topk_row(idx[b, t], ref_i[b, t], ref_s[b, t], nv[b, t], k, f"b{b} q{t}")


# ------------------------------------------------------------------ FP8 index keys
def test_quantize_rows_fp8_matches_oracle():
    """The GPU quantizer's codes and scales equal the oracle's bit for bit (rows of 32..1024)."""
    m = csa()
    rng = np.random.default_rng(21)
    for rows, dim in ((1000, 128), (64, 512), (3, 32), (5, 1024)):
        x = synth.f32_to_bf16_bits((rng.standard_normal((rows, dim)) * rng.uniform(0.01, 100, (rows, 1))).astype(np.float32))
        x[0] = 0                                     # an all-zero row: scale 1
        xd = dev_bf16(x)
        q = torch.empty(rows, dim, dtype=torch.uint8, device="cuda")
        sc = torch.empty(rows, dtype=torch.float32, device="cuda")
        m.dsv4_quantize_rows_fp8(xd, q, sc)
        torch.cuda.synchronize()
        want_q, want_s = oracle.quantize_rows_e4m3(synth.bf16_bits_to_f32(x))
        assert np.array_equal(q.cpu().numpy(), want_q), f"codes differ ({rows}x{dim})"
        assert np.array_equal(sc.cpu().numpy(), want_s), f"scales differ ({rows}x{dim})"


def _fp8_rows(x_bits):
    """Oracle quantization of bf16 rows (the inputs of the FP8 scorer come from the oracle)."""
    return oracle.quantize_rows_e4m3(synth.bf16_bits_to_f32(x_bits))


def _run_indexer_fp8(q8, qs, w, k8, ks, n_comp, top_k, ratio=4):
    m = csa()
    B, n_q = q8.shape[:2]
    max_comp = k8.shape[1]
    qd, kd = dev(q8), dev(k8)
    qsd, ksd, wd, nd = dev(qs), dev(ks), dev(w), dev(n_comp)
    idx = torch.empty(B, n_q, top_k, dtype=torch.int32, device="cuda")
    sc = torch.full((B, n_q, max_comp), float("nan"), dtype=torch.float32, device="cuda")
    kw = dict(ratio=ratio, scores_out=sc, q_scale=qsd, key_scale=ksd)
    ws = ws_tensor(m.dsv4_indexer_topk_workspace_size(qd, wd, kd, nd, idx, **kw))
    m.dsv4_indexer_topk(qd, wd, kd, nd, idx, ws, **kw)
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    assert ew == 0, f"device error word {ew:#x}"
    return idx.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("cfg", [1, 3])
def test_indexer_fp8_keys(cfg):
    """FP8 E4M3 queries and keys (oracle-quantized): scores against the oracle's FP8 scores,
    top-k exact up to near ties; at 1M context the selection is also checked against its own
    scores on every sequence."""
    wl = WORKLOADS[cfg]
    x = inputs(cfg)
    keys = _oracle_keys(x, wl) if cfg == 1 else x["keys"]
    q8, qs = _fp8_rows(x["q_I"])
    k8, ks = _fp8_rows(keys)
    idx, sc = _run_indexer_fp8(q8, qs, x["w"], k8, ks, x["n_comp"], wl.top_k)
    seqs = [0, 9, 15] if cfg == 1 else [0, 3]
    for b in seqs:
        ref_s, nv = oracle.index_scores_fp8(q8[b:b + 1], qs[b:b + 1], x["w"][b:b + 1], k8[b:b + 1],
                                            ks[b:b + 1], x["n_comp"][b:b + 1], wl.ratio)
        ref_i = oracle.topk(ref_s, nv, wl.top_k)
        _check_scores(sc[b, 0], ref_s[0, 0], nv[0, 0])
        check_topk_row(idx[b, 0], ref_i[0, 0], ref_s[0, 0], nv[0, 0], wl.top_k, f"b{b}")
    for b in range(wl.batch):
        topk_valid_for_scores(idx[b, 0], sc[b, 0], x["n_comp"][b], wl.top_k, f"b{b}")


def test_indexer_fp8_ragged_and_short():
    """FP8 keys: 8 heads, ragged n_comp (0 included), a cache that ends inside a 512-key stage."""
    rng = np.random.default_rng(22)
    B, H, N, k = 4, 8, 700, 96
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, 1, H, 128)).astype(np.float32))
    keys = synth.f32_to_bf16_bits(rng.standard_normal((B, N, 128)).astype(np.float32))
    w = rng.standard_normal((B, 1, H)).astype(np.float32)
    n_comp = np.array([700, 0, 50, 513], np.int32)
    q8, qs = _fp8_rows(q)
    k8, ks = _fp8_rows(keys)
    idx, sc = _run_indexer_fp8(q8, qs, w, k8, ks, n_comp, k)
    ref_s, nv = oracle.index_scores_fp8(q8, qs, w, k8, ks, n_comp, 4)
    ref_i = oracle.topk(ref_s, nv, k)
    for b in range(B):
        if nv[b, 0]:
            _check_scores(sc[b, 0], ref_s[b, 0], nv[b, 0])
        check_topk_row(idx[b, 0], ref_i[b, 0], ref_s[b, 0], nv[b, 0], k, f"b{b}")


def test_indexer_fp8_many_rows_causal():
    """FP8 keys with more query rows than SMs (4 per sequence, causal positions): the CTAs'
    contiguous shares of (row, stage) pairs cross row boundaries, so the head weights and the
    key-scale row change inside a CTA; every row against the oracle's FP8 scores."""
    rng = np.random.default_rng(23)
    B, n_q, H, N, k = 40, 4, 64, 700, 64
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, n_q, H, 128)).astype(np.float32))
    keys = synth.f32_to_bf16_bits(rng.standard_normal((B, N, 128)).astype(np.float32))
    w = rng.standard_normal((B, n_q, H)).astype(np.float32)
    n_comp = rng.integers(0, N + 1, B).astype(np.int32)
    n_comp[0], n_comp[1] = N, 0
    q_pos = rng.integers(0, 4 * N, B).astype(np.int64)[:, None] + np.arange(n_q, dtype=np.int64)[None, :]
    q8, qs = _fp8_rows(q)
    k8, ks = _fp8_rows(keys)
    m = csa()
    qd, kd, qsd, ksd, wd, nd, pd = dev(q8), dev(k8), dev(qs), dev(ks), dev(w), dev(n_comp), dev(q_pos)
    idx = torch.empty(B, n_q, k, dtype=torch.int32, device="cuda")
    sc = torch.full((B, n_q, N), float("nan"), dtype=torch.float32, device="cuda")
    kw = dict(ratio=4, q_pos=pd, scores_out=sc, q_scale=qsd, key_scale=ksd)
    ws = ws_tensor(m.dsv4_indexer_topk_workspace_size(qd, wd, kd, nd, idx, **kw))
    m.dsv4_indexer_topk(qd, wd, kd, nd, idx, ws, **kw)
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    assert ew == 0, f"device error word {ew:#x}"
    got_i, got_s = idx.cpu().numpy(), sc.cpu().numpy()
    ref_s, nv = oracle.index_scores_fp8(q8, qs, w, k8, ks, n_comp, 4, q_pos=q_pos)
    ref_i = oracle.topk(ref_s, nv, k)
    for b in range(B):
        for t in range(n_q):
            if nv[b, t]:
                _check_scores(got_s[b, t], ref_s[b, t], nv[b, t])
            check_topk_row(got_i[b, t], ref_i[b, t], ref_s[b, t], nv[b, t], k, f"b{b} q{t}")


def _e4m3_ord(codes):
    """E4M3 codes as signed ordinals (sign-magnitude -> integer line; +0 and -0 both 0)."""
    c = np.asarray(codes, np.int32)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def _e4m3_step(codes):
    """Spacing of the E4M3 grid at each code's magnitude: 2^(max(e, 1) - 10)."""
    e = (np.asarray(codes, np.int32) & 0x7F) >> 3
    return np.ldexp(1.0, np.maximum(e, 1) - 10)


def _check_fp8_cache(got8, got_s, ref_f64, what):
    """An FP8 cache written from entries computed in fp32 against the oracle's fp64 entries
    quantized the same way: scales within 1e-5 relative, codes within one E4M3 step, and
    almost all codes equal (a code can move only where fp32 and fp64 round across a grid
    midpoint). Returns the keys whose row differs from the oracle's."""
    d = ref_f64.shape[-1]
    want8, want_s = oracle.quantize_rows_e4m3(ref_f64.astype(np.float32).reshape(-1, d))
    want8 = want8.reshape(got8.shape)
    want_s = want_s.reshape(got_s.shape)
    rel = np.abs(got_s.astype(np.float64) - want_s) / want_s
    assert np.all(rel <= 1e-5), f"{what}: scale rel err {rel.max():.2e}"
    dist = np.abs(_e4m3_ord(got8) - _e4m3_ord(want8))
    assert dist.max() <= 1, f"{what}: a code moved {dist.max()} steps"
    frac = np.count_nonzero(dist) / dist.size
    assert frac <= 1e-3, f"{what}: {frac:.2e} of the codes differ"
    return want8, want_s, np.any(dist, axis=-1)


def _gpu_compress_fp8(C, Z, bias, gamma, pos0, ratio, overlap=False, prev_C=None, prev_Z=None):
    m = csa()
    B, T, w = C.shape
    d = w // 2 if overlap else w
    out = torch.zeros(B, T // ratio, d, dtype=torch.uint8, device="cuda")
    sc = torch.full((B, T // ratio), float("nan"), dtype=torch.float32, device="cuda")
    m.dsv4_compress(dev_bf16(C), dev_bf16(Z), dev(bias), dev(gamma), dev(pos0), out, ratio=ratio,
                    overlap=overlap, out_scale=sc,
                    prev_C=None if prev_C is None else dev_bf16(prev_C),
                    prev_Z=None if prev_Z is None else dev_bf16(prev_Z))
    torch.cuda.synchronize()
    return out.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("cfg", [0, 1])
def test_compress_fp8_key_cache(cfg):
    """The compressor writing the indexer's key cache in FP8 (codes + per-entry scale) against
    the oracle's entries quantized by the oracle."""
    wl = WORKLOADS[cfg]
    x = inputs(cfg)
    got8, got_s = _gpu_compress_fp8(x["C_I"], x["Z_I"], x["bias_I"], x["gamma_I"], x["pos0"], wl.ratio)
    _, ref = oracle.compress(x["C_I"], x["Z_I"], x["bias_I"], x["gamma_I"], x["pos0"], wl.ratio,
                             wl.rope_dim)
    _check_fp8_cache(got8, got_s, ref, f"fp8 keys cfg{cfg}")


def test_compress_overlap_fp8_key_cache():
    """Two-stream compressor, 128-dim keys, previous block given, FP8 output."""
    B, r, d = 3, 4, 128
    C, Z, bias, gamma, pC, pZ = _overlap_inputs(31, B, 64 * r, d, r, prev=True)
    pos0 = np.array([4 * r, 1000 * r, 0], np.int64)
    got8, got_s = _gpu_compress_fp8(C, Z, bias, gamma, pos0, r, overlap=True, prev_C=pC, prev_Z=pZ)
    _, ref = oracle.compress_overlap(C, Z, bias, gamma, pos0, r, pC, pZ)
    _check_fp8_cache(got8, got_s, ref, "fp8 two-stream keys")


def test_indexer_fp8_one_bin_long_rows():
    """FP8 keys, 153 rows (more rows than SMs: each CTA scores a contiguous run of stages of
    one row, up to 257 stages of 512 keys) with every score equal: every key of a row lands in
    one histogram bin, more than a 16-bit count holds between flushes unless the scorer
    flushes often enough. The selection must be the first top_k keys (ties: lower index)."""
    m = csa()
    B, H, N, k = 153, 8, 131072, 64
    one = 0x38                                          # E4M3 code of 1.0
    q8 = torch.full((B, 1, H, 128), one, dtype=torch.uint8, device="cuda")
    qs = torch.ones(B, 1, H, dtype=torch.float32, device="cuda")
    k8 = torch.full((B, N, 128), one, dtype=torch.uint8, device="cuda")
    ks = torch.ones(B, N, dtype=torch.float32, device="cuda")
    w = torch.full((B, 1, H), 1.0 / H, dtype=torch.float32, device="cuda")
    n_comp = torch.full((B,), N, dtype=torch.int32, device="cuda")
    idx = torch.empty(B, 1, k, dtype=torch.int32, device="cuda")
    kw = dict(ratio=4, q_scale=qs, key_scale=ks)
    ws = ws_tensor(m.dsv4_indexer_topk_workspace_size(q8, w, k8, n_comp, idx, **kw))
    m.dsv4_indexer_topk(q8, w, k8, n_comp, idx, ws, **kw)
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    assert ew == 0, f"device error word {ew:#x}"
    want = np.broadcast_to(np.arange(k, dtype=np.int32), (B, k))
    assert np.array_equal(idx[:, 0].cpu().numpy(), want)
    del k8


# ------------------------------------------------------------------ stage 3 alone: exact top-k
def _run_topk(scores, n_vis, k):
    m = csa()
    sd, nd = dev(scores.astype(np.float32)), dev(n_vis.astype(np.int32))
    idx = torch.empty(scores.shape[0], k, dtype=torch.int32, device="cuda")
    ws = ws_tensor(m.dsv4_topk_workspace_size(sd, nd, idx))
    m.dsv4_topk(sd, nd, idx, ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy()


@pytest.mark.parametrize("max_comp,k", [(33, 8), (700, 96), (2048, 512), (2048, 2047), (3000, 64), (40000, 2048),
                                         (262144, 2048)])
def test_topk_exact_with_planted_ties(max_comp, k):
    rows = 6
    s = synth.normal_f32(11, 18, (rows, max_comp), 0.0, 8.0)
    s[0] = np.round(s[0] * 4) / 4                    # heavy ties everywhere
    s[1, ::3] = 0.0
    s[1, 1::3] = -0.0                                 # +0 and -0 must tie
    s[2] = 1.5                                        # every score equal
    s[3, : max_comp // 2] = s[3, max_comp // 2:][: max_comp // 2]   # duplicated halves
    n_vis = np.array([max_comp, max_comp - 1, max_comp, max_comp // 3 + 1, k, 5], np.int32)
    got = _run_topk(s, n_vis, k)
    want = oracle.topk(s, n_vis, k)
    for r in range(rows):
        assert np.array_equal(got[r], want[r]), f"row {r}: first diff at {np.argmax(got[r] != want[r])}"


# ------------------------------------------------------------------ stage 4: gather + attention
def _run_attn(x, wl, idx, want_gather=True, top_k=None, out_rope_pos=None):
    m = csa()
    q, sink = dev_bf16(x["q"]), dev(x["sink"])
    kv = dev_bf16(x["comp_kv_dev"])
    n_comp, win, win_len = dev(x["n_comp"]), dev_bf16(x["win"]), dev(x["win_len"])
    B, n_q, H, D = x["q"].shape
    top_k = top_k or (idx.shape[-1] if idx is not None else kv.shape[1])
    out = torch.empty(B, n_q, H, D, dtype=torch.bfloat16, device="cuda")
    gather = torch.full((B, n_q, top_k + wl.window, D), 7.0, dtype=torch.bfloat16, device="cuda") if want_gather else None
    kw = dict(idx=None if idx is None else dev(idx), top_k=top_k, window=wl.window, ratio=wl.ratio,
              q_pos=None if x.get("q_pos") is None else dev(x["q_pos"]), gather=gather)
    if out_rope_pos is not None:
        kw["out_rope_pos"] = dev(np.ascontiguousarray(out_rope_pos, np.int64))
    ws = ws_tensor(m.dsv4_sparse_attn_workspace_size(q, sink, kv, n_comp, win, win_len, out, **kw))
    m.dsv4_sparse_attn_decode(q, sink, kv, n_comp, win, win_len, out, ws, **kw)
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    return host_bf16(out), (host_bf16(gather) if gather is not None else None), ew


def _attn_case(cfg):
    wl = WORKLOADS[cfg]
    x = dict(inputs(cfg))
    if wl.pregen_cache:
        x["comp_kv_dev"] = x["comp_kv"]
    else:
        x["comp_kv_dev"] = _oracle_kv(x, wl)[0]
    return wl, x


@pytest.mark.parametrize("cfg", [0, 1, 3])
def test_sparse_attention_decode(cfg):
    wl, x = _attn_case(cfg)
    B = wl.batch
    idx = synth.uniform_index_sets(wl.seed, 17, B, x["n_comp"], wl.top_k).reshape(B, 1, wl.top_k)
    got, gat, ew = _run_attn(x, wl, idx)
    assert ew == 0
    seqs = list(range(B)) if B <= 4 else [0, 5, 15]
    ref_bits, ref, ref_g = oracle.sparse_attn(x["q"][seqs], x["sink"], x["comp_kv_dev"][seqs],
                                              x["n_comp"][seqs], idx[seqs], x["win"][seqs],
                                              x["win_len"][seqs], wl.top_k, wl.window, wl.ratio,
                                              want_gather=True)
    assert_bf16_close(got[seqs], ref, f"cfg{cfg} attention")
    assert np.array_equal(gat[seqs], ref_g), "gather buffer differs"


def _mixed_kv(comp_bits, rope_dim=64):
    """The mixed FP8 / bf16 storage of bf16 cache rows (the oracle's quantization), and the
    bf16 rows the attention then multiplies (the oracle's dequantization)."""
    nope, sc, rope = oracle.quantize_kv_mixed(synth.bf16_bits_to_f32(comp_bits), rope_dim)
    return (nope, sc, rope), oracle.dequant_kv_mixed(nope, sc, rope)


def _run_attn_mixed(x, wl, idx, mixed, top_k=None, q_pos=None):
    m = csa()
    nope, sc, rope = mixed
    q, sink = dev_bf16(x["q"]), dev(x["sink"])
    n_comp, win, win_len = dev(x["n_comp"]), dev_bf16(x["win"]), dev(x["win_len"])
    B, n_q, H, D = x["q"].shape
    top_k = top_k or (idx.shape[-1] if idx is not None else nope.shape[1])
    out = torch.empty(B, n_q, H, D, dtype=torch.bfloat16, device="cuda")
    gather = torch.full((B, n_q, top_k + wl.window, D), 7.0, dtype=torch.bfloat16, device="cuda")
    kw = dict(idx=None if idx is None else dev(idx), top_k=top_k, window=wl.window, ratio=wl.ratio,
              gather=gather, kv_nope=dev(nope), kv_scale=dev(sc), kv_rope=dev_bf16(rope),
              q_pos=None if q_pos is None else dev(q_pos))
    ws = ws_tensor(m.dsv4_sparse_attn_workspace_size(q, sink, None, n_comp, win, win_len, out, **kw))
    m.dsv4_sparse_attn_decode(q, sink, None, n_comp, win, win_len, out, ws, **kw)
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    return host_bf16(out), host_bf16(gather), ew


@pytest.mark.parametrize("cfg", [1, 3])
def test_sparse_attention_decode_mixed_kv(cfg):
    """Compressed rows in the mixed FP8 / bf16 storage: the gather buffer holds exactly the
    oracle's dequantized rows (and the window rows), the output matches the oracle's attention
    over them."""
    wl, x = _attn_case(cfg)
    B = wl.batch
    seqs = [0, 3] if cfg == 3 else [0, 5, 15]
    comp = x["comp_kv_dev"]
    if cfg == 3:
        mixed, deq = _mixed_kv(comp[:, : 40000])              # the first 40,000 rows suffice
        n_comp = np.minimum(x["n_comp"], 40000).astype(np.int32)
        x = dict(x, n_comp=n_comp)
    else:
        mixed, deq = _mixed_kv(comp)
    idx = synth.uniform_index_sets(wl.seed, 19, B, x["n_comp"], wl.top_k).reshape(B, 1, wl.top_k)
    got, gat, ew = _run_attn_mixed(x, wl, idx, mixed)
    assert ew == 0
    _, ref, ref_g = oracle.sparse_attn(x["q"][seqs], x["sink"], deq[seqs], x["n_comp"][seqs], idx[seqs],
                                       x["win"][seqs], x["win_len"][seqs], wl.top_k, wl.window, wl.ratio,
                                       want_gather=True)
    assert np.array_equal(gat[seqs], ref_g), "gather buffer differs from the dequantized rows"
    assert_bf16_close(got[seqs], ref, f"cfg{cfg} attention over mixed KV")


def test_hca_dense_attention_mixed_kv():
    """The dense (HCA) form over the mixed storage, every compressed row and the window."""
    wl, x = _attn_case(2)
    mixed, deq = _mixed_kv(x["comp_kv_dev"])
    got, gat, ew = _run_attn_mixed(x, wl, None, mixed)
    assert ew == 0
    seqs = [0, 17, 63]
    _, ref, ref_g = oracle.sparse_attn(x["q"][seqs], x["sink"], deq[seqs], x["n_comp"][seqs], None,
                                       x["win"][seqs], x["win_len"][seqs], wl.max_comp, wl.window,
                                       wl.ratio, want_gather=True)
    assert np.array_equal(gat[seqs], ref_g)
    assert_bf16_close(got[seqs], ref, "HCA attention over mixed KV")


def test_compress_mixed_kv_cache():
    """The compressor writing the mixed storage (codes and scale of the 448 channels without
    RoPE, bf16 RoPE part) against the oracle's entries quantized by the oracle."""
    wl = WORKLOADS[1]
    x = inputs(1)
    m = csa()
    B, T, D = x["C"].shape
    rows, rd = T // wl.ratio, wl.rope_dim
    nope = torch.zeros(B, rows, D - rd, dtype=torch.uint8, device="cuda")
    sc = torch.full((B, rows), float("nan"), dtype=torch.float32, device="cuda")
    rope = torch.zeros(B, rows, rd, dtype=torch.bfloat16, device="cuda")
    m.dsv4_compress(dev_bf16(x["C"]), dev_bf16(x["Z"]), dev(x["bias"]), dev(x["gamma"]), dev(x["pos0"]),
                    nope, ratio=wl.ratio, rope_dim=rd, out_scale=sc, out_rope=rope)
    torch.cuda.synchronize()
    _, ref = oracle.compress(x["C"], x["Z"], x["bias"], x["gamma"], x["pos0"], wl.ratio, rd)
    got8, got_s = nope.cpu().numpy(), sc.cpu().numpy()
    _check_fp8_cache(got8, got_s, ref[..., : D - rd], "mixed KV: part without RoPE")
    assert_bf16_close(host_bf16(rope), ref[..., D - rd:], "mixed KV: RoPE part")


def _plain_inputs(seed, B, T, d, r):
    C = synth.normal_bf16(seed, 201, (B, T, d))
    Z = synth.normal_bf16(seed, 202, (B, T, d))
    bias = synth.bf16_bits_to_f32(synth.normal_bf16(seed, 203, (r, d), 0.0, 0.5))
    gamma = synth.bf16_bits_to_f32(synth.normal_bf16(seed, 204, (d,), 1.0, 0.1))
    return C, Z, bias, gamma


@pytest.mark.parametrize("mode", ["fp8", "mixed"])
def test_compress_long_blocks_fp8_outputs(mode):
    """Ratio 128 with few entries (two per sequence) and FP8 or mixed outputs: the one-CTA wide
    pooling (few bf16 entries take the 2-CTA channel split instead, which writes bf16 only)."""
    B, r, d, rd = 8, 128, 512, 64
    C, Z, bias, gamma = _plain_inputs(41, B, 2 * r, d, r)
    pos0 = (np.arange(B, dtype=np.int64) * 37 + 3) * r
    _, ref = oracle.compress(C, Z, bias, gamma, pos0, r, rd)
    if mode == "fp8":
        got8, got_s = _gpu_compress_fp8(C, Z, bias, gamma, pos0, r)
        _check_fp8_cache(got8, got_s, ref, "ratio 128, FP8 output")
        return
    m = csa()
    nope = torch.zeros(B, 2, d - rd, dtype=torch.uint8, device="cuda")
    sc = torch.full((B, 2), float("nan"), dtype=torch.float32, device="cuda")
    rope = torch.zeros(B, 2, rd, dtype=torch.bfloat16, device="cuda")
    m.dsv4_compress(dev_bf16(C), dev_bf16(Z), dev(bias), dev(gamma), dev(pos0), nope, ratio=r, rope_dim=rd,
                    out_scale=sc, out_rope=rope)
    torch.cuda.synchronize()
    _check_fp8_cache(nope.cpu().numpy(), sc.cpu().numpy(), ref[..., : d - rd], "ratio 128, mixed: part without RoPE")
    assert_bf16_close(host_bf16(rope), ref[..., d - rd:], "ratio 128, mixed: RoPE part")


@pytest.mark.parametrize("d, split", [(100, False), (512, True)])
def test_compress_long_blocks_pooling_forms(d, split):
    """Ratio 16 in bf16: 100 channels (not a multiple of 8) take the per-channel pooling; 512
    channels with few entries take the 2-CTA channel split, the newest block written into a
    cache row at a device offset (the HCA decode step's form)."""
    B, r = 3, 16
    T = r if split else 4 * r
    C, Z, bias, gamma = _plain_inputs(43 + d, B, T, d, r)
    pos0 = np.array([5 * r, 700 * r, 0], np.int64)
    _, ref = oracle.compress(C, Z, bias, gamma, pos0, r, 64)
    if not split:
        got = host_bf16(_gpu_compress(C, Z, bias, gamma, pos0, r))
        assert_bf16_close(got, ref, f"ratio {r}, {d} channels")
        return
    row0 = np.array([5, 700, 0], np.int32)
    cache = torch.zeros(B, 1000, d, dtype=torch.bfloat16, device="cuda")
    _gpu_compress(C, Z, bias, gamma, pos0, r, out=cache, out_row0=row0)
    got = host_bf16(cache)
    for b in range(B):
        assert_bf16_close(got[b, row0[b]:row0[b] + 1], ref[b], f"seq {b}")
        assert not np.any(np.delete(got[b], row0[b], axis=0)), f"seq {b}: other rows were written"


def test_hca_dense_attention():
    wl, x = _attn_case(2)
    got, gat, ew = _run_attn(x, wl, None)
    assert ew == 0
    seqs = [0, 17, 63]
    _, ref, ref_g = oracle.sparse_attn(x["q"][seqs], x["sink"], x["comp_kv_dev"][seqs],
                                       x["n_comp"][seqs], None, x["win"][seqs], x["win_len"][seqs],
                                       wl.max_comp, wl.window, wl.ratio, want_gather=True)
    assert_bf16_close(got[seqs], ref, "HCA attention")
    assert np.array_equal(gat[seqs], ref_g)


def test_dense_attention_many_chunks():
    """The dense form over 39,999 compressed rows and a full window: 314 chunks of 128 slots,
    more than the combine holds in registers (it loops over the rest)."""
    from types import SimpleNamespace
    rng = np.random.default_rng(31)
    H, D, N = 8, 128, 40000
    wl = SimpleNamespace(window=128, ratio=4)
    x = {"q": synth.f32_to_bf16_bits(rng.standard_normal((1, 1, H, D)).astype(np.float32)),
         "sink": rng.standard_normal(H).astype(np.float32),
         "comp_kv_dev": synth.f32_to_bf16_bits(rng.standard_normal((1, N, D)).astype(np.float32)),
         "n_comp": np.array([N - 1], np.int32),
         "win": synth.f32_to_bf16_bits(rng.standard_normal((1, 128, D)).astype(np.float32)),
         "win_len": np.array([128], np.int32), "q_pos": None}
    got, gat, ew = _run_attn(x, wl, None)
    assert ew == 0
    _, ref, ref_g = oracle.sparse_attn(x["q"], x["sink"], x["comp_kv_dev"], x["n_comp"], None, x["win"],
                                       x["win_len"], N, 128, 4, want_gather=True)
    assert np.array_equal(gat, ref_g)
    assert_bf16_close(got, ref, "dense attention over 314 chunks")


def test_prefill_attention_sampled_queries():
    wl, x = _attn_case(4)
    nvis = np.array([16384 + (t + 1) // 4 for t in range(2048)], np.int32)
    idx = synth.uniform_index_sets(4, 17, 2048, nvis, wl.top_k).reshape(1, 2048, wl.top_k)
    got, gat, ew = _run_attn(x, wl, idx, want_gather=False)
    assert ew == 0
    sample = np.array([0, 1, 126, 127, 128, 1000, 2047], np.int32)
    _, ref, _ = oracle.sparse_attn(x["q"][:, sample], x["sink"], x["comp_kv_dev"], x["n_comp"],
                                   idx[:, sample], x["win"], x["win_len"], wl.top_k, wl.window,
                                   wl.ratio, q_pos=x["q_pos"][:, sample], q_abs=sample,
                                   n_q_total=2048)
    assert_bf16_close(got[:, sample], ref, "prefill attention")


@pytest.mark.parametrize("cfg", [0, 1])
def test_attention_output_inverse_rope(cfg):
    """The output rotated back at the query positions (64 rope dims): decode with D = 128
    (pairs split across neighbouring threads) and D = 512; positions up to 2^20."""
    wl, x = _attn_case(cfg)
    B = wl.batch
    idx = synth.uniform_index_sets(wl.seed, 17, B, x["n_comp"], wl.top_k).reshape(B, 1, wl.top_k)
    pos = (np.array([1048575, 8192, 123457, 3, 0, 65536, 777, 4095, 1, 2, 9, 99, 999, 9999, 99999, 524288],
                    np.int64)[:B]).reshape(B, 1)
    got, _, ew = _run_attn(x, wl, idx, want_gather=False, out_rope_pos=pos)
    assert ew == 0
    seqs = list(range(B)) if B <= 4 else [0, 5, 15]
    _, ref, _ = oracle.sparse_attn(x["q"][seqs], x["sink"], x["comp_kv_dev"][seqs], x["n_comp"][seqs],
                                   idx[seqs], x["win"][seqs], x["win_len"][seqs], wl.top_k, wl.window,
                                   wl.ratio)
    _, ref_rot = oracle.inverse_rope(ref, pos[seqs].reshape(-1), 64)
    assert_bf16_close(got[seqs], ref_rot, f"cfg{cfg} attention + inverse RoPE")


def test_prefill_attention_inverse_rope_sampled_queries():
    wl, x = _attn_case(4)
    nvis = np.array([16384 + (t + 1) // 4 for t in range(2048)], np.int32)
    idx = synth.uniform_index_sets(4, 17, 2048, nvis, wl.top_k).reshape(1, 2048, wl.top_k)
    got, _, ew = _run_attn(x, wl, idx, want_gather=False, out_rope_pos=x["q_pos"])
    assert ew == 0
    sample = np.array([0, 127, 1000, 2047], np.int32)
    _, ref, _ = oracle.sparse_attn(x["q"][:, sample], x["sink"], x["comp_kv_dev"], x["n_comp"],
                                   idx[:, sample], x["win"], x["win_len"], wl.top_k, wl.window,
                                   wl.ratio, q_pos=x["q_pos"][:, sample], q_abs=sample,
                                   n_q_total=2048)
    _, ref_rot = oracle.inverse_rope(ref, x["q_pos"][0, sample], 64)
    assert_bf16_close(got[:, sample], ref_rot, "prefill attention + inverse RoPE")


def test_attention_edge_cases_and_bad_index():
    """Ragged n_comp (including 0), short and empty windows, -1 padding, and an index past the
    visible range (masked, reported as DSV4_EWORD_BAD_INDEX)."""
    rng = np.random.default_rng(8)
    B, H, D, N, k, W = 4, 64, 512, 300, 64, 128
    x = {"q": synth.f32_to_bf16_bits(rng.standard_normal((B, 1, H, D)).astype(np.float32)),
         "sink": rng.standard_normal(H).astype(np.float32),
         "comp_kv_dev": synth.f32_to_bf16_bits(rng.standard_normal((B, N, D)).astype(np.float32)),
         "n_comp": np.array([300, 0, 37, 129], np.int32),
         "win": synth.f32_to_bf16_bits(rng.standard_normal((B, W, D)).astype(np.float32)),
         "win_len": np.array([128, 0, 5, 128], np.int32)}

    class WL:
        window, ratio = W, 4

    idx = synth.uniform_index_sets(3, 17, B, x["n_comp"], k).reshape(B, 1, k)
    got, gat, ew = _run_attn(x, WL, idx)
    assert ew == 0
    _, ref, ref_g = oracle.sparse_attn(x["q"], x["sink"], x["comp_kv_dev"], x["n_comp"], idx,
                                       x["win"], x["win_len"], k, W, 4, want_gather=True)
    assert_bf16_close(got, ref, "edge cases")
    assert np.array_equal(gat, ref_g)
    bad = idx.copy()
    bad[2, 0, 3] = 200                      # sequence 2 has only 37 visible entries
    got2, _, ew2 = _run_attn(x, WL, bad)
    assert ew2 & csa().DSV4_EWORD_BAD_INDEX
    masked = bad.copy()
    masked[2, 0, 3] = -1
    _, ref2, _ = oracle.sparse_attn(x["q"], x["sink"], x["comp_kv_dev"], x["n_comp"], masked,
                                    x["win"], x["win_len"], k, W, 4)
    assert_bf16_close(got2, ref2, "masked bad index")


def _walk_case(seed=41):
    """Many query rows per sequence (4 x 40 rows x 2 head groups: one CTA walks each row's
    chunks): ragged causal visibility (n_comp 300, 0, 37, 129 capped by the query positions),
    windows of 168, 0, 45 and 100 rows, 64 selected slots and 128 window slots per row."""
    rng = np.random.default_rng(seed)
    B, n_q, H, D, N, k, W = 4, 40, 64, 512, 300, 64, 128
    q_pos = (np.array([1160, 0, 100, 400], np.int64)[:, None] + np.arange(n_q, dtype=np.int64)[None, :])
    x = {"q": synth.f32_to_bf16_bits(rng.standard_normal((B, n_q, H, D)).astype(np.float32)),
         "sink": rng.standard_normal(H).astype(np.float32),
         "comp_kv_dev": synth.f32_to_bf16_bits(rng.standard_normal((B, N, D)).astype(np.float32)),
         "n_comp": np.array([300, 0, 37, 129], np.int32),
         "win": synth.f32_to_bf16_bits(rng.standard_normal((B, W + n_q, D)).astype(np.float32)),
         "win_len": np.array([W + n_q, 0, 45, 100], np.int32),
         "q_pos": q_pos}
    nvis = np.minimum(x["n_comp"][:, None], (q_pos + 1) // 4).reshape(-1).astype(np.int32)
    idx = synth.uniform_index_sets(seed, 17, B * n_q, nvis, k).reshape(B, n_q, k)

    class WL:
        window, ratio = W, 4

    return WL, x, idx, nvis


def test_attention_row_walk_edge_cases():
    """The row-walking kernel: outputs and the gather buffer of every row against the oracle,
    then an index past a row's visible range (masked, reported as DSV4_EWORD_BAD_INDEX)."""
    wl, x, idx, nvis = _walk_case()
    got, gat, ew = _run_attn(x, wl, idx)
    assert ew == 0
    _, ref, ref_g = oracle.sparse_attn(x["q"], x["sink"], x["comp_kv_dev"], x["n_comp"], idx, x["win"],
                                       x["win_len"], 64, wl.window, 4, q_pos=x["q_pos"], want_gather=True)
    assert np.array_equal(gat, ref_g), "gather buffer differs"
    assert_bf16_close(got, ref, "row-walk attention")
    bad = idx.copy()
    bad[2, 5, 3] = int(nvis[2 * 40 + 5]) + 2             # past that row's visible entries
    got2, _, ew2 = _run_attn(x, wl, bad, want_gather=False)
    assert ew2 & csa().DSV4_EWORD_BAD_INDEX
    masked = bad.copy()
    masked[2, 5, 3] = -1
    _, ref2, _ = oracle.sparse_attn(x["q"], x["sink"], x["comp_kv_dev"], x["n_comp"], masked, x["win"],
                                    x["win_len"], 64, wl.window, 4, q_pos=x["q_pos"])
    assert_bf16_close(got2, ref2, "row-walk attention, masked bad index")


def test_attention_row_walk_mixed_kv():
    """The row-walking kernel over the mixed FP8 / bf16 storage: the gather buffer holds the
    oracle's dequantized rows, the output matches the oracle's attention over them."""
    wl, x, idx, _ = _walk_case(43)
    mixed, deq = _mixed_kv(x["comp_kv_dev"])
    got, gat, ew = _run_attn_mixed(x, wl, idx, mixed, q_pos=x["q_pos"])
    assert ew == 0
    _, ref, ref_g = oracle.sparse_attn(x["q"], x["sink"], deq, x["n_comp"], idx, x["win"], x["win_len"],
                                       64, wl.window, 4, q_pos=x["q_pos"], want_gather=True)
    assert np.array_equal(gat, ref_g), "gather buffer differs"
    assert_bf16_close(got, ref, "row-walk attention over mixed KV")


def test_attention_row_walk_small_heads_inverse_rope():
    """The row-walking kernel with D = 128 and 8 heads (one group of 16, half empty), 320 query
    rows, a ragged last chunk (40 + 128 slots), and the output rotated back (each RoPE pair
    split across neighbouring lanes)."""
    rng = np.random.default_rng(45)
    n_q, H, D, N, k, W = 320, 8, 128, 256, 40, 128
    q_pos = 704 + np.arange(n_q, dtype=np.int64)[None, :]
    x = {"q": synth.f32_to_bf16_bits(rng.standard_normal((1, n_q, H, D)).astype(np.float32)),
         "sink": rng.standard_normal(H).astype(np.float32),
         "comp_kv_dev": synth.f32_to_bf16_bits(rng.standard_normal((1, N, D)).astype(np.float32)),
         "n_comp": np.array([256], np.int32),
         "win": synth.f32_to_bf16_bits(rng.standard_normal((1, W + n_q, D)).astype(np.float32)),
         "win_len": np.array([W + n_q], np.int32), "q_pos": q_pos}
    nvis = np.minimum(256, (q_pos[0] + 1) // 4).astype(np.int32)
    idx = synth.uniform_index_sets(45, 17, n_q, nvis, k).reshape(1, n_q, k)

    class WL:
        window, ratio = W, 4

    got, gat, ew = _run_attn(x, WL, idx, out_rope_pos=q_pos)
    assert ew == 0
    _, ref, ref_g = oracle.sparse_attn(x["q"], x["sink"], x["comp_kv_dev"], x["n_comp"], idx, x["win"],
                                       x["win_len"], k, W, 4, q_pos=q_pos, want_gather=True)
    assert np.array_equal(gat, ref_g), "gather buffer differs"
    _, ref_rot = oracle.inverse_rope(ref.reshape(n_q, H, D), q_pos[0], 64)
    assert_bf16_close(got.reshape(n_q, H, D), ref_rot, "row-walk attention + inverse RoPE, D = 128")


@pytest.mark.parametrize("late", ["scaled", "aligned", "aligned3"])
def test_attention_row_walk_64_heads_late_maximum(late):
    """The 64-head walking kernel (160 rows x 64 heads, 512 dims: one CTA per row), whose
    running O^T stays in TMEM and whose per-head reference maximum moves only when some score
    of a chunk exceeds its head's by more than 64 in base-2 units (then every head whose chunk
    maximum exceeds its reference by more than 8 in natural units takes it), with the largest
    scores in the last of three chunks (the window): "scaled" multiplies the window rows by 3
    (scores up to ~6 above the earlier chunks': P up to ~e^6 in bf16); "aligned" makes query t's
    own window row a copy of its query for head t mod 64 (that head's score ~22, ~33 in base-2
    units, above ~3 before: P up to ~2^33, no new reference); "aligned3" makes it three times
    the query (~68, ~98 in base-2 units: that head's maximum moves and its O^T columns and sum
    are rescaled, the other heads' stay)."""
    rng = np.random.default_rng({"scaled": 61, "aligned": 62, "aligned3": 64}[late])
    n_q, H, D, N, k, W = 160, 64, 512, 300, 256, 128
    q_pos = 4000 + np.arange(n_q, dtype=np.int64)[None, :]
    q = synth.f32_to_bf16_bits(rng.standard_normal((1, n_q, H, D)).astype(np.float32))
    win = synth.f32_to_bf16_bits(rng.standard_normal((1, W + n_q, D)).astype(np.float32) *
                                 np.float32(3.0 if late == "scaled" else 1.0))
    if late != "scaled":
        qf = (q.astype(np.uint32) << 16).view(np.float32)
        mult = np.float32(1.0 if late == "aligned" else 3.0)
        for t in range(n_q):
            win[0, t + W] = synth.f32_to_bf16_bits(mult * qf[0, t, t % H])   # query t's newest window row
    x = {"q": q, "sink": rng.standard_normal(H).astype(np.float32),
         "comp_kv_dev": synth.f32_to_bf16_bits(rng.standard_normal((1, N, D)).astype(np.float32)),
         "n_comp": np.array([N], np.int32), "win": win,
         "win_len": np.array([W + n_q], np.int32), "q_pos": q_pos}
    nvis = np.full(n_q, N, np.int32)
    idx = synth.uniform_index_sets(63, 17, n_q, nvis, k).reshape(1, n_q, k)

    class WL:
        window, ratio = W, 4

    got, gat, ew = _run_attn(x, WL, idx)
    assert ew == 0
    _, ref, ref_g = oracle.sparse_attn(x["q"], x["sink"], x["comp_kv_dev"], x["n_comp"], idx, x["win"],
                                       x["win_len"], k, W, 4, q_pos=q_pos, want_gather=True)
    assert np.array_equal(gat, ref_g), "gather buffer differs"
    assert_bf16_close(got, ref, f"64-head row walk, late maximum ({late})")


@pytest.mark.parametrize("form", ["split", "walk", "walk_mixed"])
def test_attention_d256_three_head_groups(form):
    """D = 256 and 48 heads (three groups of 16), a 64-row window, ragged visibility: decode
    (one CTA per chunk, partials and combine; 3 query rows) and many query rows (one CTA walks
    each row; 2 x 60 rows), the latter also over the mixed FP8 / bf16 storage."""
    rng = np.random.default_rng({"split": 51, "walk": 52, "walk_mixed": 53}[form])
    H, D, N, k, W = 48, 256, 200, 48, 64
    B, n_q = (3, 1) if form == "split" else (2, 60)
    x = {"q": synth.f32_to_bf16_bits(rng.standard_normal((B, n_q, H, D)).astype(np.float32)),
         "sink": rng.standard_normal(H).astype(np.float32),
         "comp_kv_dev": synth.f32_to_bf16_bits(rng.standard_normal((B, N, D)).astype(np.float32)),
         "n_comp": np.array([200, 31, 120][:B], np.int32),
         "win": synth.f32_to_bf16_bits(rng.standard_normal((B, W + n_q, D)).astype(np.float32)),
         "win_len": np.array([W + n_q, 20, 50][:B], np.int32)}
    if n_q > 1:
        x["q_pos"] = np.array([700, 90], np.int64)[:, None] + np.arange(n_q, dtype=np.int64)[None, :]
        nvis = np.minimum(x["n_comp"][:, None], (x["q_pos"] + 1) // 4).reshape(-1).astype(np.int32)
    else:
        nvis = x["n_comp"]
    idx = synth.uniform_index_sets(54, 17, B * n_q, nvis, k).reshape(B, n_q, k)

    class WL:
        window, ratio = W, 4

    kv = x["comp_kv_dev"]
    if form == "walk_mixed":
        mixed, kv = _mixed_kv(x["comp_kv_dev"])
        got, gat, ew = _run_attn_mixed(x, WL, idx, mixed, q_pos=x["q_pos"])
    else:
        got, gat, ew = _run_attn(x, WL, idx)
    assert ew == 0
    _, ref, ref_g = oracle.sparse_attn(x["q"], x["sink"], kv, x["n_comp"], idx, x["win"], x["win_len"], k, W, 4,
                                       q_pos=x.get("q_pos"), want_gather=True)
    assert np.array_equal(gat, ref_g), "gather buffer differs"
    assert_bf16_close(got, ref, f"D = 256, 48 heads ({form})")


# ------------------------------------------------------------------ the fused decode step
def _fused_step(x, wl, graph=False, fp8=False, mixed=False):
    """Compress (whole context) + indexer top-k + gather/attention in one dsv4_csa_decode.
    fp8: the key cache is written and scored in FP8 E4M3 (queries quantized by the oracle),
    and the step also returns its scores."""
    m = csa()
    from compressed_sparse_attention_08_gb300 import _abi
    B, T, D = x["C"].shape
    Di = x["C_I"].shape[2]
    t = {}
    fkw, ikw = {}, {}
    if fp8:
        q8, qs = _fp8_rows(x["q_I"])
        t["q8"], t["qs"] = dev(q8), dev(qs)
        t["key_scale"] = torch.full((B, wl.max_comp), float("nan"), dtype=torch.float32, device="cuda")
        t["scores"] = torch.full((B, 1, wl.max_comp), float("nan"), dtype=torch.float32, device="cuda")
        fkw = dict(out_scale=t["key_scale"])
        ikw = dict(q_scale=t["qs"], key_scale=t["key_scale"], scores_out=t["scores"])
    t["C"], t["Z"] = dev_bf16(x["C"]), dev_bf16(x["Z"])
    t["CI"], t["ZI"] = dev_bf16(x["C_I"]), dev_bf16(x["Z_I"])
    t["bias"], t["gamma"] = dev(x["bias"]), dev(x["gamma"])
    t["biasI"], t["gammaI"] = dev(x["bias_I"]), dev(x["gamma_I"])
    t["pos0"] = dev(x["pos0"])
    rd = wl.rope_dim
    if mixed:
        # the KV cache in the mixed FP8 / bf16 storage, written by the step's compressor
        t["kv"] = torch.zeros(B, wl.max_comp, D - rd, dtype=torch.uint8, device="cuda")
        t["kv_scale"] = torch.full((B, wl.max_comp), float("nan"), dtype=torch.float32, device="cuda")
        t["kv_rope"] = torch.zeros(B, wl.max_comp, rd, dtype=torch.bfloat16, device="cuda")
    else:
        t["kv"] = torch.zeros(B, wl.max_comp, D, dtype=torch.bfloat16, device="cuda")
    t["keys"] = torch.zeros(B, wl.max_comp, Di, dtype=torch.uint8 if fp8 else torch.bfloat16, device="cuda")
    t["q_I"], t["w"] = dev_bf16(x["q_I"]), dev(x["w"])
    t["n_comp"] = dev(x["n_comp"])
    t["idx"] = torch.empty(B, 1, wl.top_k, dtype=torch.int32, device="cuda")
    t["q"], t["sink"] = dev_bf16(x["q"]), dev(x["sink"])
    t["win"], t["win_len"] = dev_bf16(x["win"]), dev(x["win_len"])
    t["out"] = torch.empty(B, 1, wl.heads, D, dtype=torch.bfloat16, device="cuda")
    t["gather"] = torch.empty(B, 1, wl.top_k + wl.window, D, dtype=torch.bfloat16, device="cuda")
    mkw = dict(out_scale=t["kv_scale"], out_rope=t["kv_rope"]) if mixed else {}
    ck = _abi.compress_args(t["C"], t["Z"], t["bias"], t["gamma"], t["pos0"], t["kv"], ratio=wl.ratio, **mkw)
    cq = _abi.compress_args(t["CI"], t["ZI"], t["biasI"], t["gammaI"], t["pos0"], t["keys"], ratio=wl.ratio,
                            **fkw)
    ia = _abi.index_args(t["q8"] if fp8 else t["q_I"], t["w"], t["keys"], t["n_comp"], t["idx"],
                         ratio=wl.ratio, **ikw)
    akw = dict(kv_nope=t["kv"], kv_scale=t["kv_scale"], kv_rope=t["kv_rope"]) if mixed else {}
    aa = _abi.attn_args(t["q"], t["sink"], None if mixed else t["kv"], t["n_comp"], t["win"], t["win_len"],
                        t["out"], idx=t["idx"], window=wl.window, ratio=wl.ratio, gather=t["gather"], **akw)
    ws = ws_tensor(m.dsv4_csa_decode_workspace_size(attn=aa, index=ia, compress_kv=ck, compress_keys=cq))
    m.dsv4_csa_decode(ws, attn=aa, index=ia, compress_kv=ck, compress_keys=cq)
    torch.cuda.synchronize()
    launches = m.dsv4_last_launch_count()
    return t, (ck, cq, ia, aa, ws), launches


def _gather_copy(kv_bits, idx, win, win_len, top_k, window, n_comp=None):
    """The gather buffer a decode step (one query per sequence) must hold, as a plain copy of
    the step's own rows: slot j < top_k the cache row idx[b, 0, j] (zeros for -1; with idx
    None, the dense form, row j for j < n_comp[b]), slot top_k + i the i-th of the window rows
    the query sees (the last `window` of its win_len rows, in order; zeros past them). Data
    movement only: none of the method's arithmetic."""
    B, _, D = kv_bits.shape
    g = np.zeros((B, 1, top_k + window, D), np.uint16)
    for b in range(B):
        if idx is None:
            n = int(n_comp[b])
            g[b, 0, :n] = kv_bits[b, :n]
        else:
            sel = idx[b, 0]
            ok = sel >= 0
            g[b, 0, :top_k][ok] = kv_bits[b, sel[ok]]
        wl_b = min(int(win_len[b]), win.shape[1])
        lo = max(wl_b - window, 0)
        g[b, 0, top_k:top_k + wl_b - lo] = win[b, lo:wl_b]
    return g


def _score_band(keys_bits, q_I, w):
    """Per key, a bound on how far its score moves when each element of the key moves by one
    bf16 step: sum_h |w_h| sum_d |q_hd| ulp(k_d). [B, n_keys]."""
    ulp = np.abs(bf16_to_f64(keys_bits)) * 2.0 ** -7 + 1e-38
    qa = np.abs(bf16_to_f64(q_I))                       # [B,1,H,Di]
    wa = np.abs(w.astype(np.float64))                   # [B,1,H]
    return np.einsum("bd,bsd->bs", np.einsum("bh,bhd->bd", wa[:, 0], qa[:, 0]), ulp)


def _check_selection(idx, ref_s, ref_i, nv, band, top_k, what, extra_ok=None):
    """A decode step's selection against the oracle's: ascending valid indices then -1
    padding, and equal to the oracle's top-k except for keys whose oracle score lies within
    the band of the k-th score (the step scores its own bf16 keys, whose elements may differ
    from the oracle's by one rounding step) or that extra_ok(b, diff) allows."""
    for b in range(idx.shape[0]):
        n = int(nv[b, 0])
        t = min(top_k, n)
        sel = idx[b, 0]
        assert np.all(sel[t:] == -1), f"{what} b{b}: padding"
        assert np.all(sel[:t] >= 0) and np.all(sel[:t] < n), f"{what} b{b}: range"
        assert np.all(np.diff(sel[:t]) > 0), f"{what} b{b}: not ascending"
        if np.array_equal(sel, ref_i[b, 0]):
            continue
        s = ref_s[b, 0, :n]
        kth = np.sort(s)[::-1][t - 1]
        diff = np.setxor1d(sel[:t], ref_i[b, 0][:t])
        ok = np.abs(s[diff] - kth) <= 2 * band[b, diff].max() + 1e-5 * abs(kth)
        if extra_ok is not None:
            ok |= extra_ok(b, diff)
        assert np.all(ok), f"{what} b{b}: selection differs beyond near ties at {diff[~ok][:8]}"


def _check_fused_attention(t, x, wl, kv_ref_bits, idx, kv_step_bits, what, seqs=None):
    """Attention output and gather buffer of a fused decode step, every sequence in `seqs`
    (all by default), never skipped: the oracle's attention over the oracle's cache rows with
    the step's own selection (already checked against the oracle's top-k: where several
    selections are valid, the attention of the one made is compared), within the bf16
    tolerance; the gather buffer within the same tolerance against the oracle's gather, and
    bit for bit against a plain copy of the step's own cache rows."""
    seqs = list(range(wl.batch)) if seqs is None else list(seqs)
    dense = idx is None
    k = wl.max_comp if dense else wl.top_k
    _, ref_o, ref_g = oracle.sparse_attn(x["q"][seqs], x["sink"], kv_ref_bits, x["n_comp"][seqs],
                                         None if dense else idx[seqs], x["win"][seqs], x["win_len"][seqs],
                                         k, wl.window, wl.ratio, want_gather=True)
    assert_bf16_close(host_bf16(t["out"])[seqs], ref_o, f"{what}: attention output")
    gat = host_bf16(t["gather"])[seqs]
    assert_bf16_close(gat, bf16_to_f64(ref_g), f"{what}: gather buffer against the oracle's")
    want = _gather_copy(kv_step_bits, None if dense else idx[seqs], x["win"][seqs], x["win_len"][seqs], k,
                        wl.window, x["n_comp"][seqs])
    assert np.array_equal(gat, want), f"{what}: gather buffer is not a copy of the step's rows"


@pytest.mark.parametrize("cfg", [0, 1])
def test_fused_decode_step(cfg):
    """The fused step (compress the whole context into both caches, indexer top-k, gather +
    attention) against the oracle: the caches, the selection (exact up to near ties), and for
    every sequence the attention output and the gather buffer."""
    wl = WORKLOADS[cfg]
    x = inputs(cfg)
    t, (ck, cq, ia, aa, ws), launches = _fused_step(x, wl)
    assert launches >= 5
    st, ew = csa().dsv4_read_error_word(ws)
    assert ew == 0, f"device error word {ew:#x}"
    kv_bits = host_bf16(t["kv"])
    keys_bits = host_bf16(t["keys"])
    ref_kv_bits, ref_kv = _oracle_kv(x, wl)
    ref_keys_bits, ref_keys = oracle.compress(x["C_I"], x["Z_I"], x["bias_I"], x["gamma_I"],
                                              x["pos0"], wl.ratio, wl.rope_dim)
    assert_bf16_close(kv_bits, ref_kv, "fused: compressed KV")
    assert_bf16_close(keys_bits, ref_keys, "fused: indexer keys")
    ref_s, nv = oracle.index_scores(x["q_I"], x["w"], ref_keys_bits, x["n_comp"], wl.ratio)
    ref_i = oracle.topk(ref_s, nv, wl.top_k)
    idx = t["idx"].cpu().numpy()
    _check_selection(idx, ref_s, ref_i, nv, _score_band(ref_keys_bits, x["q_I"], x["w"]), wl.top_k, "fused")
    _check_fused_attention(t, x, wl, ref_kv_bits, idx, kv_bits, "fused")


def test_fused_decode_step_hca():
    """The dense (HCA) form of the fused step as the benchmark runs it: ratio 128, 64 entries
    per sequence, no indexer (index = NULL). The caches hold the first 63 blocks (compressed by
    dsv4_compress beforehand); the step compresses the newest 128-token block into row 63 and
    attends over every compressed row plus the 128-row window. Every sequence runs on the GPU;
    the oracle checks three: the whole cache (new row included), the gather buffer of all
    64 + 128 rows and the attention output."""
    m = csa()
    from compressed_sparse_attention_08_gb300 import _abi
    wl = WORKLOADS[2]
    x = inputs(2)
    B, T, D = x["C"].shape
    r = wl.ratio
    kv = torch.zeros(B, wl.max_comp, D, dtype=torch.bfloat16, device="cuda")
    bias, gamma = dev(x["bias"]), dev(x["gamma"])
    m.dsv4_compress(dev_bf16(x["C"][:, :T - r]), dev_bf16(x["Z"][:, :T - r]), bias, gamma, dev(x["pos0"]), kv,
                    ratio=r)
    Cn, Zn = dev_bf16(x["C"][:, T - r:]), dev_bf16(x["Z"][:, T - r:])
    pos_n = torch.full((B,), T - r, dtype=torch.int64, device="cuda")
    row_n = torch.full((B,), wl.n_comp - 1, dtype=torch.int32, device="cuda")
    q, sink, n_comp = dev_bf16(x["q"]), dev(x["sink"]), dev(x["n_comp"])
    win, win_len = dev_bf16(x["win"]), dev(x["win_len"])
    out = torch.empty(B, 1, wl.heads, D, dtype=torch.bfloat16, device="cuda")
    gather = torch.full((B, 1, wl.max_comp + wl.window, D), 7.0, dtype=torch.bfloat16, device="cuda")
    ck = _abi.compress_args(Cn, Zn, bias, gamma, pos_n, kv, ratio=r, out_row0=row_n)
    aa = _abi.attn_args(q, sink, kv, n_comp, win, win_len, out, idx=None, top_k=wl.max_comp,
                        window=wl.window, ratio=r, gather=gather)
    ws = ws_tensor(m.dsv4_csa_decode_workspace_size(attn=aa, compress_kv=ck))
    m.dsv4_csa_decode(ws, attn=aa, compress_kv=ck)
    torch.cuda.synchronize()
    assert m.dsv4_last_launch_count() >= 2
    st, ew = m.dsv4_read_error_word(ws)
    assert ew == 0, f"device error word {ew:#x}"
    seqs = [0, 31, 63]
    ref_kv_bits, ref_kv = _oracle_kv(x, wl, seqs)
    kv_bits = host_bf16(kv)
    assert_bf16_close(kv_bits[seqs], ref_kv, "fused HCA: compressed KV (63 earlier rows and the new one)")
    t = {"out": out, "gather": gather}
    _check_fused_attention(t, x, wl, ref_kv_bits, None, kv_bits[seqs], "fused HCA", seqs=seqs)


@pytest.mark.parametrize("cfg", [0, 1])
def test_fused_decode_step_fp8_keys(cfg):
    """The fused step with the index-key cache in FP8: the compressor writes codes + scales, the
    scorer reads them. Cache against the oracle's quantized entries; scores against the
    oracle's FP8 scores (exactly where the cache row equals the oracle's, else within the
    shift one E4M3 step per element can cause); the selection is the exact top-k of the
    step's own scores and equals the oracle's up to near ties and moved keys; attention
    output against the oracle on the step's selection."""
    wl = WORKLOADS[cfg]
    x = inputs(cfg)
    t, (ck, cq, ia, aa, ws), _ = _fused_step(x, wl, fp8=True)
    st, ew = csa().dsv4_read_error_word(ws)
    assert ew == 0, f"device error word {ew:#x}"
    ref_kv_bits, ref_kv = _oracle_kv(x, wl)
    assert_bf16_close(host_bf16(t["kv"]), ref_kv, "fused fp8: compressed KV")
    _, ref_keys = oracle.compress(x["C_I"], x["Z_I"], x["bias_I"], x["gamma_I"], x["pos0"], wl.ratio,
                                  wl.rope_dim)
    nc = ref_keys.shape[1]
    got8 = t["keys"].cpu().numpy()
    got_s = t["key_scale"].cpu().numpy()
    k8, ks, moved = _check_fp8_cache(got8[:, :nc], got_s[:, :nc], ref_keys, "fused fp8: key cache")
    q8, qs = _fp8_rows(x["q_I"])
    ref_s, nv = oracle.index_scores_fp8(q8, qs, x["w"], k8, ks, x["n_comp"], wl.ratio)
    ref_i = oracle.topk(ref_s, nv, wl.top_k)
    # bound on the score shift of a key whose codes moved by one step: every element moving
    coef = np.einsum("bh,bhd->bd", np.abs(x["w"][:, 0].astype(np.float64) * qs[:, 0]),
                     np.abs(oracle.e4m3_decode(q8[:, 0])))
    band = np.einsum("bd,bsd->bs", coef, _e4m3_step(k8)) * ks
    sc = t["scores"].cpu().numpy()
    idx = t["idx"].cpu().numpy()
    for b in range(wl.batch):
        n = nv[b, 0]
        g, r = sc[b, 0, :n].astype(np.float64), ref_s[b, 0, :n]
        tol = 2e-5 * (np.mean(np.abs(r)) + 1e-30) + 2e-5 * np.abs(r)
        tol = np.where(moved[b, :n], tol + band[b, :n], tol)
        assert np.all(np.abs(g - r) <= tol), f"b{b}: scores"
        topk_valid_for_scores(idx[b, 0], sc[b, 0], n, wl.top_k, f"b{b}")
        if np.array_equal(idx[b, 0], ref_i[b, 0]):
            continue
        kth = np.sort(r)[::-1][min(wl.top_k, n) - 1]
        diff = np.setxor1d(idx[b, 0][idx[b, 0] >= 0], ref_i[b, 0][ref_i[b, 0] >= 0])
        slack = 1e-5 * abs(kth) + np.where(moved[b, diff], band[b, diff], 0.0) + band[b, moved[b, :n]].max(initial=0.0)
        assert np.all(np.abs(r[diff] - kth) <= slack), f"b{b}: selection"
    # the attention output and gather buffer of every sequence, on the step's (checked) selection
    _check_fused_attention(t, x, wl, ref_kv_bits, idx, host_bf16(t["kv"]), "fused fp8")


@pytest.mark.parametrize("cfg", [0, 1])
def test_fused_decode_step_mixed_kv(cfg):
    """The fused step with the KV cache in the mixed FP8 / bf16 storage: the compressor writes
    it, the attention reads it. Cache against the oracle's quantized entries; the selection
    against the oracle's top-k (exact up to near ties); for every sequence the output against
    the oracle's attention over the oracle's dequantized rows with the step's selection, and
    the gather buffer against those rows."""
    wl = WORKLOADS[cfg]
    x = inputs(cfg)
    t, (ck, cq, ia, aa, ws), _ = _fused_step(x, wl, mixed=True)
    st, ew = csa().dsv4_read_error_word(ws)
    assert ew == 0, f"device error word {ew:#x}"
    D, rd = x["C"].shape[2], wl.rope_dim
    _, ref_kv = _oracle_kv(x, wl)
    nc = ref_kv.shape[1]
    _check_fp8_cache(t["kv"].cpu().numpy()[:, :nc], t["kv_scale"].cpu().numpy()[:, :nc],
                     ref_kv[..., : D - rd], "fused mixed KV")
    assert_bf16_close(host_bf16(t["kv_rope"])[:, :nc], ref_kv[..., D - rd:], "fused mixed KV: RoPE part")
    # the oracle's storage of its own entries (the fp32 value of each, as the compressor's)
    deq = oracle.dequant_kv_mixed(*oracle.quantize_kv_mixed(ref_kv.astype(np.float32), rd))
    ref_keys_bits, ref_keys = oracle.compress(x["C_I"], x["Z_I"], x["bias_I"], x["gamma_I"], x["pos0"],
                                              wl.ratio, wl.rope_dim)
    assert_bf16_close(host_bf16(t["keys"]), ref_keys, "fused mixed KV: indexer keys")
    ref_s, nv = oracle.index_scores(x["q_I"], x["w"], ref_keys_bits, x["n_comp"], wl.ratio)
    ref_i = oracle.topk(ref_s, nv, wl.top_k)
    idx = t["idx"].cpu().numpy()
    _check_selection(idx, ref_s, ref_i, nv, _score_band(ref_keys_bits, x["q_I"], x["w"]), wl.top_k,
                     "fused mixed KV")
    # every sequence: the oracle's attention over its dequantized rows with the step's selection
    _, ref_o, ref_g = oracle.sparse_attn(x["q"], x["sink"], deq, x["n_comp"], idx, x["win"], x["win_len"],
                                         wl.top_k, wl.window, wl.ratio, want_gather=True)
    assert_bf16_close(host_bf16(t["out"]), ref_o, "fused mixed KV: attention output")
    # the gather buffer holds the dequantized rows: against the oracle's wherever the entry's
    # codes equal the oracle's (a code one E4M3 step away moves its channel by up to 1/8)
    _, _, moved = _check_fp8_cache(t["kv"].cpu().numpy()[:, :nc], t["kv_scale"].cpu().numpy()[:, :nc],
                                   ref_kv[..., : D - rd], "fused mixed KV")
    gat = host_bf16(t["gather"])
    keep = np.ones(gat.shape[:3], bool)
    for b in range(wl.batch):
        sel = idx[b, 0]
        keep[b, 0, :wl.top_k] = (sel < 0) | ~moved[b, np.maximum(sel, 0)]
    assert keep.mean() > 0.9
    assert_bf16_close(gat[keep], bf16_to_f64(ref_g)[keep], "fused mixed KV: gather buffer")


def test_fused_decode_step_1m_context_as_benchmarked():
    """The fused step exactly as the benchmark runs it (1M-token context, batch 4, the caches
    pre-filled, the newest block compressed into the last row of both caches in the step,
    stage claims, one CUDA graph), checked on sequences 0 and 3: the new cache rows against
    the oracle's compression of the newest block; the selection against the oracle's top-k
    over the input keys with the oracle's newest key (exact up to near ties and the bf16
    rounding of that one key); the attention output and the gather buffer against the oracle
    on the step's selection, for both sequences."""
    m = csa()
    from compressed_sparse_attention_08_gb300 import _abi
    wl = WORKLOADS[3]
    x = inputs(3)
    B, D, Di = wl.batch, wl.head_dim, wl.idx_dim
    t = {k: dev_bf16(x[k]) for k in ("C", "Z", "C_I", "Z_I", "q_I", "q", "win")}
    t.update({k: dev(x[k]) for k in ("bias", "gamma", "bias_I", "gamma_I", "pos0", "append_row", "w",
                                     "n_comp", "sink", "win_len")})
    t["kv"], t["keys"] = dev_bf16(x["comp_kv"]), dev_bf16(x["keys"])
    t["idx"] = torch.empty(B, 1, wl.top_k, dtype=torch.int32, device="cuda")
    t["out"] = torch.empty(B, 1, wl.heads, D, dtype=torch.bfloat16, device="cuda")
    t["gather"] = torch.empty(B, 1, wl.top_k + wl.window, D, dtype=torch.bfloat16, device="cuda")
    ck = _abi.compress_args(t["C"], t["Z"], t["bias"], t["gamma"], t["pos0"], t["kv"], ratio=wl.ratio,
                            out_row0=t["append_row"])
    cq = _abi.compress_args(t["C_I"], t["Z_I"], t["bias_I"], t["gamma_I"], t["pos0"], t["keys"],
                            ratio=wl.ratio, out_row0=t["append_row"])
    ia = _abi.index_args(t["q_I"], t["w"], t["keys"], t["n_comp"], t["idx"], ratio=wl.ratio)
    aa = _abi.attn_args(t["q"], t["sink"], t["kv"], t["n_comp"], t["win"], t["win_len"], t["out"],
                        idx=t["idx"], window=wl.window, ratio=wl.ratio, gather=t["gather"])
    ws = ws_tensor(m.dsv4_csa_decode_workspace_size(attn=aa, index=ia, compress_kv=ck, compress_keys=cq))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        m.dsv4_csa_decode(ws, attn=aa, index=ia, compress_kv=ck, compress_keys=cq, stream=s)
    s.synchronize()
    row = int(x["append_row"][0])
    eager = {k: t[k].clone() for k in ("out", "idx", "gather")}
    eager["kv"], eager["keys"] = t["kv"][:, row].clone(), t["keys"][:, row].clone()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            m.dsv4_csa_decode(ws, attn=aa, index=ia, compress_kv=ck, compress_keys=cq, stream=s)
        g.replay()
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    assert ew == 0, f"device error word {ew:#x}"
    # deterministic: the replay (stages claimed by other CTAs, counts summed by atomics in
    # another order) gives the eager step's bytes
    for k, v in eager.items():
        now = t[k][:, row] if k in ("kv", "keys") else t[k]
        assert torch.equal(now.view(torch.int16) if now.dtype == torch.bfloat16 else now,
                           v.view(torch.int16) if v.dtype == torch.bfloat16 else v), f"1M step not deterministic: {k}"
    seqs = [0, 3]
    new_kv_bits, new_kv = oracle.compress(x["C"][seqs], x["Z"][seqs], x["bias"], x["gamma"], x["pos0"][seqs],
                                          wl.ratio, wl.rope_dim)
    new_key_bits, new_key = oracle.compress(x["C_I"][seqs], x["Z_I"][seqs], x["bias_I"], x["gamma_I"],
                                            x["pos0"][seqs], wl.ratio, wl.rope_dim)
    kv_rows = t["kv"][seqs, row].cpu().view(torch.int16).numpy().view(np.uint16)
    key_rows = t["keys"][seqs, row].cpu().view(torch.int16).numpy().view(np.uint16)
    assert_bf16_close(kv_rows[:, None], new_kv, "newest KV row")
    assert_bf16_close(key_rows[:, None], new_key, "newest key row")
    idx = t["idx"].cpu().numpy()
    for j, b in enumerate(seqs):
        keys_b = x["keys"][b:b + 1].copy()
        keys_b[0, row] = new_key_bits[j, 0]
        ref_s, nv = oracle.index_scores(x["q_I"][b:b + 1], x["w"][b:b + 1], keys_b, x["n_comp"][b:b + 1], wl.ratio)
        ref_i = oracle.topk(ref_s, nv, wl.top_k)
        # exact up to near ties, or the newest key (its bf16 entry may differ by one rounding step)
        band = np.zeros((1, wl.n_comp))
        _check_selection(idx[b:b + 1], ref_s, ref_i, nv, band, wl.top_k, f"1M b{b}",
                         extra_ok=lambda _b, diff: diff == row)
        # the attention output and gather buffer, on the step's (checked) selection: the
        # oracle's cache is the input cache with its own newest row; the step's is the input
        # cache with the step's newest row
        kv_b = x["comp_kv"][b:b + 1].copy()
        kv_b[0, row] = new_kv_bits[j, 0]
        kv_step = x["comp_kv"][b:b + 1].copy()
        kv_step[0, row] = kv_rows[j]
        sub = {"out": t["out"][b:b + 1], "gather": t["gather"][b:b + 1]}
        xb = {k: (x[k][b:b + 1] if k != "sink" else x[k]) for k in ("q", "sink", "n_comp", "win", "win_len")}
        wl1 = type("W", (), dict(batch=1, top_k=wl.top_k, window=wl.window, ratio=wl.ratio, max_comp=wl.max_comp))
        _check_fused_attention(sub, xb, wl1, kv_b, idx[b:b + 1], kv_step, f"1M b{b}")


@pytest.mark.parametrize("cfg", [0, 1])
def test_fused_decode_graph_replay_matches_eager(cfg):
    """The whole step captured in a CUDA graph replays to the eager result, bit for bit,
    after the inputs are changed in place (at the 8K-context batch-16 size as well: several
    scoring CTAs per row, the combine of five chunk partials, 64-head attention tiles on a
    152-SM device): every stage is deterministic."""
    wl = WORKLOADS[cfg]
    x = inputs(cfg)
    m = csa()
    t, (ck, cq, ia, aa, ws), _ = _fused_step(x, wl)
    eager = {k: t[k].clone() for k in ("out", "idx", "gather", "kv", "keys")}
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            m.dsv4_csa_decode(ws, attn=aa, index=ia, compress_kv=ck, compress_keys=cq, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for k in ("out", "idx", "gather"):
        t[k].zero_()
    g.replay()
    torch.cuda.synchronize()
    for k, v in eager.items():
        assert torch.equal(t[k].view(torch.int16) if t[k].dtype == torch.bfloat16 else t[k],
                           v.view(torch.int16) if v.dtype == torch.bfloat16 else v), k
    # new query, same graph
    q2 = synth.normal_bf16(99, 12, x["q"].shape)
    t["q"].copy_(dev_bf16(q2))
    g.replay()
    torch.cuda.synchronize()
    out_graph = t["out"].clone()
    m.dsv4_csa_decode(ws, attn=aa, index=ia, compress_kv=ck, compress_keys=cq)
    torch.cuda.synchronize()
    assert torch.equal(out_graph.view(torch.int16), t["out"].view(torch.int16))


def test_invalid_arguments_rejected_before_launch():
    m = csa()
    q = torch.zeros(1, 1, 64, 128, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(1, 1, 64, dtype=torch.float32, device="cuda")
    keys = torch.zeros(1, 100, 128, dtype=torch.bfloat16, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx = torch.empty(1, 1, 200, dtype=torch.int32, device="cuda")   # top_k > max_comp
    ws = ws_tensor(1 << 20)
    with pytest.raises(m.Dsv4Error) as e:
        m.dsv4_indexer_topk(q, w, keys, n, idx, ws, ratio=4)
    assert e.value.status == m.DSV4_ERR_INVALID_ARG
