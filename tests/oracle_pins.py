"""Pins for the oracle: facts fixed by the pages and by mathematics, not by the oracle.

Each ``pin_*`` function raises AssertionError when the oracle currently loaded in the
``oracle`` module disagrees with the fact it checks. The pins are also run against
copies of the oracle with planted mistakes (test_oracle_mutants.py) to show that they
bite. Sources, by page title and section:

  [A] "nvfp4-megamoe-kernel: compare v0.1-e2e-working...v-c1-c2-c3-20260602"
  [B] "nvfp4-megamoe-kernel: compare master..pure-nvfp4"
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
from scipy.special import expit, softmax

import oracle
from compressed_sparse_attention_08_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf(x):
    return synth.f32_to_bf16_bits(np.asarray(x, np.float32))


def _f(b):
    return synth.bf16_bits_to_f32(np.asarray(b, np.uint16)).astype(np.float64)


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol=1e-12, atol=1e-12, msg=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, (a.shape, b.shape, msg)
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    assert np.all(err <= lim), f"{msg}: max err {err.max():.3e} (worst at {np.unravel_index(np.argmax(err - lim), err.shape)})"


# ------------------------------------------------------------------ bf16 rounding
def pin_bf16_rounding():
    """Round-to-nearest-even to 8 significant bits: exact ties and known patterns, plus
    agreement with an integer-bit implementation on random float32 values."""
    cases = {1.0: 0x3F80, -2.0: 0xC000, 1.0 + 2.0 ** -8: 0x3F80, 1.0 + 3 * 2.0 ** -8: 0x3F82,
             1.0 + 2.0 ** -8 + 2.0 ** -30: 0x3F81, 0.0: 0x0000, 3.0e38: 0x7F62,
             3.4e38: 0x7F80, 2.0 ** -133: 0x0001}
    for x, bits in cases.items():
        assert oracle.double_to_bf16(x) == bits, (x, hex(oracle.double_to_bf16(x)), hex(bits))
    xs = _rng(1).standard_normal(4000).astype(np.float32) * np.float32(37.0)
    ref = synth.f32_to_bf16_bits(xs)
    got = np.array([oracle.double_to_bf16(float(v)) for v in xs], np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ compressor
def _compress(C, Z, bias, gamma=None, pos0=None, ratio=4, rope_dim=0, theta=10000.0, eps=1e-6):
    B, T, d = C.shape
    gamma = np.ones(d, np.float32) if gamma is None else gamma
    pos0 = np.zeros(B, np.int64) if pos0 is None else pos0
    return oracle.compress(C, Z, bias, gamma, pos0, ratio, rope_dim, theta, eps)


def _int_block_mean_tokens(rng, B, nb, ratio, d):
    """bf16-exact tokens whose per-block, per-channel mean is an exact integer m:
    tokens m+a, m-a, m+b, m-b (ratio 4)."""
    assert ratio == 4
    m = rng.integers(-40, 41, size=(B, nb, 1, d))
    a = rng.integers(-20, 21, size=(B, nb, 1, d))
    b = rng.integers(-20, 21, size=(B, nb, 1, d))
    tok = np.concatenate([m + a, m - a, m + b, m - b], axis=2).astype(np.float32)
    C = _bf(tok.reshape(B, nb * ratio, d))
    Cmean = _bf(np.repeat(m, ratio, axis=2).astype(np.float32).reshape(B, nb * ratio, d))
    return C, Cmean


def pin_compress_equal_logits_block_mean():
    """Equal logits along the block => the compressed entry is the block mean of C
    (softmax of a constant is uniform). Compared with a block whose tokens are all the mean,
    where any logits give the same result."""
    rng = _rng(2)
    B, nb, r, d = 2, 5, 4, 16
    C, Cmean = _int_block_mean_tokens(rng, B, nb, r, d)
    zrow = rng.standard_normal((B, nb, 1, d)).astype(np.float32)
    Zeq = _bf(np.repeat(zrow, r, axis=2).reshape(B, nb * r, d))
    bias0 = np.zeros((r, d), np.float32)
    _, got = _compress(C, Zeq, bias0)
    Zrand = _bf(rng.standard_normal((B, nb * r, d)) * 3)
    _, ref = _compress(Cmean, Zrand, bias0)
    _close(got, ref, msg="equal logits -> block mean")


def pin_compress_bias_not_on_C():
    """C = 0 => output 0 for any logits and any bias ([B] commit "Fix two correctness bugs",
    item 1: the positional bias enters the logits Z+B only, never the content C)."""
    rng = _rng(3)
    B, T, d, r = 2, 16, 32, 4
    C = np.zeros((B, T, d), np.uint16)
    Z = _bf(rng.standard_normal((B, T, d)))
    bias = _f(_bf(rng.standard_normal((r, d)) * 0.5)).astype(np.float32)
    bits, out = _compress(C, Z, bias, rope_dim=16, pos0=np.array([5, 77], np.int64))
    assert np.all(out == 0.0), "bias leaked into the content"


def pin_compress_bias_shift_invariance():
    """A bias constant along the block's tokens changes nothing (softmax shift invariance)."""
    rng = _rng(4)
    B, T, d, r = 1, 32, 24, 4
    C = _bf(rng.standard_normal((B, T, d)))
    Z = _bf(rng.standard_normal((B, T, d)))
    beta = _f(_bf(rng.standard_normal((1, d)) * 2)).astype(np.float32)
    _, a = _compress(C, Z, np.repeat(beta, r, axis=0))
    _, b = _compress(C, Z, np.zeros((r, d), np.float32))
    _close(a, b, rtol=1e-12, atol=1e-13, msg="constant bias")


def pin_compress_bias_row_selects_token():
    """A large bias on row t* makes the softmax one-hot on token t* of every block: the
    entry equals the entry of a block made of copies of token t* (bias row t pairs with the
    block's t-th token)."""
    rng = _rng(5)
    B, nb, r, d = 1, 6, 4, 8
    T = nb * r
    C = _bf(rng.standard_normal((B, T, d)))
    Z = _bf(rng.standard_normal((B, T, d)))
    for t_star in range(r):
        bias = np.zeros((r, d), np.float32)
        bias[t_star, :] = 200.0
        _, got = _compress(C, Z, bias)
        Ct = C.reshape(B, nb, r, d)[:, :, t_star:t_star + 1, :]
        Crep = np.repeat(Ct, r, axis=2).reshape(B, T, d)
        _, ref = _compress(Crep, Z, np.zeros((r, d), np.float32))
        _close(got, ref, rtol=1e-12, atol=1e-12, msg=f"bias row {t_star}")


def pin_compress_ratio_one_is_identity_reduce():
    """ratio 1: the softmax runs over a single token, so the logits do not matter."""
    rng = _rng(6)
    C = _bf(rng.standard_normal((1, 9, 16)))
    _, a = _compress(C, _bf(rng.standard_normal((1, 9, 16)) * 5), np.zeros((1, 16), np.float32), ratio=1)
    _, b = _compress(C, _bf(rng.standard_normal((1, 9, 16)) * 5), np.zeros((1, 16), np.float32), ratio=1)
    _close(a, b, msg="ratio 1")


def pin_rmsnorm():
    """[A] compressor_reduce.cu apply_kv_norm_kernel: y = x * rsqrt(mean(x^2) + 1e-6) * g.
    With every token of a block equal to m, x = m; then y is parallel to m with
    mean(y^2) = ms / (ms + eps), ms = mean(m^2); gamma multiplies channelwise afterwards."""
    rng = _rng(7)
    B, nb, r, d = 1, 4, 4, 32
    for scale in (1.0, 1e-3, 30.0):
        m = _f(_bf(rng.standard_normal((B, nb, 1, d)) * scale))
        C = _bf(np.repeat(m, r, axis=2).reshape(B, nb * r, d))
        Z = _bf(rng.standard_normal((B, nb * r, d)))
        _, y = _compress(C, Z, np.zeros((r, d), np.float32))
        m2 = m.reshape(nb, d)
        y2 = y.reshape(nb, d)
        ms = np.mean(m2 ** 2, axis=1)
        _close(np.mean(y2 ** 2, axis=1), ms / (ms + 1e-6), rtol=1e-12, msg="mean(y^2)")
        k = y2 / m2
        _close(k, np.repeat(k[:, :1], d, axis=1), rtol=1e-12, msg="y parallel to x")
        assert np.all(k > 0)
        g = _f(_bf(1.0 + 0.1 * rng.standard_normal(d))).astype(np.float32)
        _, yg = _compress(C, Z, np.zeros((r, d), np.float32), gamma=g)
        _close(yg.reshape(nb, d), y2 * g[None, :].astype(np.float64), rtol=1e-12, msg="gamma")


def _pair_angle(v, d0):
    return np.arctan2(v[..., d0 + 1], v[..., d0])


def pin_rope_identity_and_norms():
    """RoPE leaves the first d - rope_dim channels alone, is the identity at position 0 and
    preserves the length of every (2j, 2j+1) pair ([A] PERFORMANCE_AUDIT.md "P5")."""
    rng = _rng(8)
    B, T, d, r, rd = 2, 12, 96, 4, 64
    C = _bf(rng.standard_normal((B, T, d)))
    Z = _bf(rng.standard_normal((B, T, d)))
    bias = np.zeros((r, d), np.float32)
    pos0 = np.array([0, 1000003], np.int64)
    _, plain = _compress(C, Z, bias, pos0=pos0, rope_dim=0)
    _, rot = _compress(C, Z, bias, pos0=pos0, rope_dim=rd)
    _close(rot[..., :d - rd], plain[..., :d - rd], rtol=0, atol=0, msg="nope dims untouched")
    _close(rot[0, 0], plain[0, 0], rtol=0, atol=1e-15, msg="position 0 is the identity")
    pr = rot[..., d - rd:].reshape(B, T // r, rd // 2, 2)
    pp = plain[..., d - rd:].reshape(B, T // r, rd // 2, 2)
    _close(np.hypot(pr[..., 0], pr[..., 1]), np.hypot(pp[..., 0], pp[..., 1]), rtol=1e-12,
           msg="pair norms")


def pin_rope_direction_and_frequencies():
    """Forward rotation angle of pair j at position p is +p * theta^(-2j/rope_dim).
    The page prints the inverse (e' = e c + o s, o' = -e s + o c), so the forward turns the
    pair (e, o) counter-clockwise. With theta = 2^32 and rope_dim 64, theta^(-2j/64) = 2^-j:
    pair j at position P*2^j turns exactly as far as pair 0 at position P, and pair 0 at
    position 1 turns by exactly 1 radian. Pairs are adjacent channels (2j, 2j+1) of the
    last 64."""
    rng = _rng(9)
    d, rd, r = 64, 64, 1
    C = _bf(rng.standard_normal((1, 1, d)))
    C = np.repeat(C, 3, axis=0)
    Z = np.zeros_like(C)
    bias = np.zeros((r, d), np.float32)
    P = 3
    for j in (1, 5, 17, 31):
        pos0 = np.array([1, P, P * 2 ** j], np.int64)
        _, plain = _compress(C, Z, bias, pos0=pos0, ratio=r, rope_dim=0, theta=2.0 ** 32)
        _, rot = _compress(C, Z, bias, pos0=pos0, ratio=r, rope_dim=rd, theta=2.0 ** 32)
        turn = lambda s, pair: (_pair_angle(rot[s, 0], 2 * pair) - _pair_angle(plain[s, 0], 2 * pair)) % (2 * np.pi)
        assert abs(turn(0, 0) - 1.0) < 1e-12, turn(0, 0)
        assert abs(turn(1, 0) - turn(2, j)) < 1e-9, (j, turn(1, 0), turn(2, j))
        assert abs(turn(1, 0) - P % (2 * np.pi)) < 1e-12


def pin_rope_relative_position():
    """<rope(x, p), rope(y, p')> over the rope channels depends only on p - p'."""
    rng = _rng(10)
    d, rd, r = 64, 64, 1
    C = _bf(rng.standard_normal((4, 1, d)))
    C[2:] = C[:2]
    Z = np.zeros_like(C)
    bias = np.zeros((r, d), np.float32)
    pos0 = np.array([10, 3, 10 + 9999, 3 + 9999], np.int64)
    _, rot = _compress(C, Z, bias, pos0=pos0, ratio=r, rope_dim=rd)
    a = float(np.dot(rot[0, 0], rot[1, 0]))
    b = float(np.dot(rot[2, 0], rot[3, 0]))
    assert abs(a - b) < 1e-9 * max(1.0, abs(a)), (a, b)
    pos0b = np.array([10, 3, 10, 5], np.int64)
    _, rot2 = _compress(C, Z, bias, pos0=pos0b, ratio=r, rope_dim=rd)
    c = float(np.dot(rot2[2, 0], rot2[3, 0]))
    assert abs(a - c) > 1e-6, "the score must depend on the relative position"


def pin_compress_block_positions():
    """Entry b of a sequence sits at position pos0 + b*ratio (its first token): entry b of a
    sequence starting at 0 rotates exactly like entry 0 of a sequence starting at b*ratio."""
    rng = _rng(11)
    d, rd, r, nb = 64, 64, 4, 5
    blk = _bf(rng.standard_normal((1, r, d)))
    C = np.concatenate([np.tile(blk, (1, nb, 1)), np.tile(blk, (1, nb, 1))], axis=0)
    Zb = _bf(rng.standard_normal((1, r, d)))
    Z = np.concatenate([np.tile(Zb, (1, nb, 1))] * 2, axis=0)
    bias = np.zeros((r, d), np.float32)
    _, a = _compress(C, Z, bias, pos0=np.array([0, 3 * r], np.int64), rope_dim=rd)
    _close(a[0, 3], a[1, 0], rtol=1e-12, atol=1e-14, msg="entry position")


# ------------------------------------------------------------------ indexer scores
def pin_scores_one_hot_weight():
    """w = e_h => I[s] = ReLU(q_h . K[s]) ([A] ARCHITECTURE_AND_MEMORY_AUDIT.md "F3")."""
    rng = _rng(12)
    H, Di, N = 6, 32, 40
    q = _bf(rng.standard_normal((1, 1, H, Di)))
    keys = _bf(rng.standard_normal((1, N, Di)))
    for h in (0, 3, 5):
        w = np.zeros((1, 1, H), np.float32)
        w[0, 0, h] = 1.0
        s, nv = oracle.index_scores(q, w, keys, np.array([N], np.int32))
        ref = np.maximum(0.0, _f(keys[0]) @ _f(q[0, 0, h]))
        _close(s[0, 0], ref, rtol=1e-13, atol=1e-12, msg=f"one-hot head {h}")
        assert nv[0, 0] == N


def pin_scores_linear_when_positive():
    """Non-negative w, q and keys make every dot product non-negative, so ReLU is the
    identity and I = (w^T Q) . K: one shared key per block for every head (MQA), no scale."""
    rng = _rng(13)
    H, Di, N = 8, 16, 50
    q = _bf(np.abs(rng.standard_normal((1, 1, H, Di))))
    keys = _bf(np.abs(rng.standard_normal((1, N, Di))))
    w = np.abs(rng.standard_normal((1, 1, H))).astype(np.float32)
    s, _ = oracle.index_scores(q, w, keys, np.array([N], np.int32))
    ref = _f(keys[0]) @ (w[0, 0].astype(np.float64) @ _f(q[0, 0]))
    _close(s[0, 0], ref, rtol=1e-12, msg="linear regime")


def pin_scores_relu_kills_negative():
    """Keys anti-aligned with every head give no score; orthogonal keys give zero."""
    H, Di = 4, 8
    qv = np.zeros((1, 1, H, Di), np.float32)
    qv[0, 0, :, 0] = [1, 2, 3, 4]
    q = _bf(qv)
    kv = np.zeros((1, 3, Di), np.float32)
    kv[0, 0, 0] = -2.0        # anti-aligned
    kv[0, 1, 1] = 5.0         # orthogonal
    kv[0, 2, 0] = 0.5         # aligned
    w = np.array([[[1.0, -1.0, 0.5, 2.0]]], np.float32)
    s, _ = oracle.index_scores(q, w, _bf(kv), np.array([3], np.int32))
    assert s[0, 0, 0] == 0.0 and s[0, 0, 1] == 0.0
    assert s[0, 0, 2] == 0.5 * (1 * 1.0 - 2 * 1.0 + 3 * 0.5 + 4 * 2.0)


def pin_visibility_rule():
    """Block j covers tokens [j*r, (j+1)*r - 1] and is visible to a query at position p iff
    it ends at or before p ([A] archived_plans/NEXT_STEPS.md "Issue 2"). Counted by
    enumerating the blocks one by one."""
    for r in (1, 4, 128):
        for n_comp in (0, 3, 17):
            for p in range(-2, 20 * r):
                brute = sum(1 for j in range(n_comp) if (j + 1) * r - 1 <= p)
                assert oracle.visible_entries(n_comp, p, r) == brute, (r, n_comp, p)
    rng = _rng(14)
    H, Di, N, r = 2, 8, 12, 4
    q = _bf(rng.standard_normal((1, 3, H, Di)))
    keys = _bf(rng.standard_normal((1, N, Di)))
    w = np.ones((1, 3, H), np.float32)
    q_pos = np.array([[6, 7, 100]], np.int64)
    s, nv = oracle.index_scores(q, w, keys, np.array([10], np.int32), ratio=r, q_pos=q_pos)
    assert list(nv[0]) == [1, 2, 10]
    assert np.all(np.isneginf(s[0, 0, 1:])) and np.all(np.isneginf(s[0, 2, 10:]))


# ------------------------------------------------------------------ top-k
def _topk_valid(scores, n, k, idx):
    """The selected set S is valid iff |S| = min(k, n), S within [0, n), ascending, -1 padded,
    and every member outranks every non-member under (score desc, index asc)."""
    t = min(k, n)
    sel = list(idx[:t])
    assert all(i == -1 for i in idx[t:]), "padding"
    assert sel == sorted(sel) and len(set(sel)) == t, "ascending, distinct"
    assert all(0 <= i < n for i in sel), "range"
    inside = set(sel)
    worst_in = min(((scores[i], -i) for i in sel), default=None)
    best_out = max(((scores[j], -j) for j in range(n) if j not in inside), default=None)
    if worst_in is not None and best_out is not None:
        assert worst_in > best_out, (worst_in, best_out)


def pin_topk_brute_force_and_ties():
    """Top-k with planted ties: equal scores rank by lower index; +0.0 and -0.0 are equal;
    top_k >= n gives every index; n = 0 gives only padding."""
    rng = _rng(15)
    for trial in range(60):
        n = int(rng.integers(0, 40))
        k = int(rng.integers(1, 12))
        vals = rng.integers(-3, 4, size=n).astype(np.float64)   # many exact ties
        if n and trial % 3 == 0:
            vals[vals == 0] = -0.0
        scores = np.full((1, 48), -np.inf)
        scores[0, :n] = vals
        idx = oracle.topk(scores, np.array([n], np.int32), k)[0]
        _topk_valid(scores[0], n, k, idx)
        brute = sorted(range(n), key=lambda i: (-vals[i], i))[:min(k, n)]
        assert list(idx[:min(k, n)]) == sorted(brute)
        idx32 = oracle.topk(scores.astype(np.float32), np.array([n], np.int32), k)[0]
        assert np.array_equal(idx32, idx)
    scores = np.zeros((1, 5))
    scores[0] = [0.0, -0.0, 0.0, -0.0, 0.0]
    assert list(oracle.topk(scores, np.array([5], np.int32), 2)[0]) == [0, 1]
    assert list(oracle.topk(scores, np.array([3], np.int32), 8)[0]) == [0, 1, 2, -1, -1, -1, -1, -1]
    assert list(oracle.topk(scores, np.array([0], np.int32), 3)[0]) == [-1, -1, -1]


# ------------------------------------------------------------------ attention
def _attn_case(rng, B=1, n_q=1, H=4, D=32, max_comp=20, n_comp=20, k=6, W=8, win_len=8):
    q = _bf(rng.standard_normal((B, n_q, H, D)))
    kv = _bf(rng.standard_normal((B, max_comp, D)))
    win = _bf(rng.standard_normal((B, W, D)))
    sink = rng.standard_normal(H).astype(np.float32)
    idx = synth.uniform_index_sets(99, 1, B * n_q, [n_comp] * (B * n_q), k).reshape(B, n_q, k)
    return q, kv, win, sink, idx


def pin_attention_zero_query():
    """q = 0 makes every logit 0: o = (sum of the rows) / (n_rows + e^sink) — the sink adds
    to the denominator only ([A] fmha_6warp_tma_multirow_multitile.cuh "Sink bias
    correction"), and V is the gathered K row itself ([A] PERFORMANCE_AUDIT.md "P4")."""
    rng = _rng(16)
    q, kv, win, sink, idx = _attn_case(rng)
    q = np.zeros_like(q)
    for wl in (8, 3, 0):
        _, o, _ = oracle.sparse_attn(q, sink, kv, np.array([20], np.int32), idx, win,
                                     np.array([wl], np.int32), top_k=6, window=8)
        rows = np.concatenate([_f(kv[0, idx[0, 0]]), _f(win[0, :wl])], axis=0)
        ref = rows.sum(0)[None, :] / (len(rows) + np.exp(sink.astype(np.float64)))[:, None]
        _close(o[0, 0], ref, rtol=1e-12, atol=1e-14, msg=f"zero query, window {wl}")


def pin_attention_no_sink_is_softmax():
    """A sink of -1e30 contributes nothing: plain softmax attention with scale 1/sqrt(D)
    ([B] single_shot_inference.py eager_attention), computed with a library softmax."""
    rng = _rng(17)
    q, kv, win, sink, idx = _attn_case(rng, H=3, D=16)
    sink = np.full(3, -1e30, np.float32)
    _, o, _ = oracle.sparse_attn(q, sink, kv, np.array([20], np.int32), idx, win,
                                 np.array([8], np.int32), top_k=6, window=8)
    rows = np.concatenate([_f(kv[0, idx[0, 0]]), _f(win[0])], axis=0)
    for h in range(3):
        p = softmax(rows @ _f(q[0, 0, h]) / math.sqrt(16))
        _close(o[0, 0, h], p @ rows, rtol=1e-11, atol=1e-13, msg=f"softmax head {h}")


def pin_attention_single_row():
    """One row v: o = v * sigmoid(s - sink), s = q.v / sqrt(D)."""
    rng = _rng(18)
    H, D = 5, 64
    q = _bf(rng.standard_normal((1, 1, H, D)) * 0.3)
    kv = _bf(rng.standard_normal((1, 4, D)))
    win = np.zeros((1, 2, D), np.uint16)
    sink = rng.standard_normal(H).astype(np.float32)
    idx = np.array([[[2, -1, -1]]], np.int32)
    _, o, _ = oracle.sparse_attn(q, sink, kv, np.array([4], np.int32), idx, win,
                                 np.array([0], np.int32), top_k=3, window=2)
    v = _f(kv[0, 2])
    for h in range(H):
        s = float(v @ _f(q[0, 0, h])) / math.sqrt(D)
        _close(o[0, 0, h], v * expit(s - float(sink[h])), rtol=1e-12, atol=1e-15, msg=f"head {h}")


def pin_attention_permutation_and_gather():
    """The output does not depend on the order of the index list or of the window rows;
    the gather buffer holds comp_kv[idx] (zeros for -1) then the window rows."""
    rng = _rng(19)
    q, kv, win, sink, idx = _attn_case(rng, k=7, n_comp=15)
    idx[0, 0, 5:] = -1
    perm = idx.copy()
    perm[0, 0, :5] = perm[0, 0, :5][::-1]
    perm[0, 0] = np.roll(perm[0, 0], 2)
    n_comp = np.array([15], np.int32)
    win_len = np.array([8], np.int32)
    _, a, g = oracle.sparse_attn(q, sink, kv, n_comp, idx, win, win_len, top_k=7, window=8,
                                 want_gather=True)
    _, b, _ = oracle.sparse_attn(q, sink, kv, n_comp, perm, win[:, ::-1], win_len, top_k=7,
                                 window=8)
    _close(a, b, rtol=1e-12, atol=1e-14, msg="permutation")
    for j in range(7):
        e = idx[0, 0, j]
        want = kv[0, e] if e >= 0 else np.zeros(kv.shape[-1], np.uint16)
        assert np.array_equal(g[0, 0, j], want)
    assert np.array_equal(g[0, 0, 7:], win[0])


def pin_attention_prefill_window_rows():
    """Chunked prefill: query t of n_q sees the `window` rows ending at its own row, the
    query tokens being the last n_q rows of the window buffer. With q = 0 the output is the
    sum of exactly those rows over (n + e^sink)."""
    rng = _rng(20)
    B, n_q, H, D, W = 1, 5, 2, 16, 3
    rows = W + n_q
    q = np.zeros((B, n_q, H, D), np.uint16)
    kv = _bf(rng.standard_normal((B, 8, D)))
    win = _bf(rng.standard_normal((B, rows, D)))
    sink = np.array([0.3, -1.2], np.float32)
    idx = np.full((B, n_q, 2), -1, np.int32)
    _, o, g = oracle.sparse_attn(q, sink, kv, np.array([8], np.int32), idx, win,
                                 np.array([rows], np.int32), top_k=2, window=W, want_gather=True)
    for t in range(n_q):
        lo, hi = t + 1, t + W            # own row is t + rows - n_q = t + W
        sel = _f(win[0, lo:hi + 1])
        ref = sel.sum(0)[None, :] / (len(sel) + np.exp(sink.astype(np.float64)))[:, None]
        _close(o[0, t], ref, rtol=1e-12, atol=1e-14, msg=f"query {t}")
        assert np.array_equal(g[0, t, 2:], win[0, lo:hi + 1])


def pin_dense_equals_full_topk():
    """top_k >= n_comp selects every entry, so CSA attention equals the HCA form (dense over
    every compressed entry plus the window), and the indexer+top-k then gives 0..n-1."""
    rng = _rng(21)
    B, H, D, N = 2, 4, 32, 10
    q = _bf(rng.standard_normal((B, 1, H, D)))
    kv = _bf(rng.standard_normal((B, N, D)))
    win = _bf(rng.standard_normal((B, 6, D)))
    sink = rng.standard_normal(H).astype(np.float32)
    n_comp = np.array([N, 7], np.int32)
    qi = _bf(rng.standard_normal((B, 1, 3, 16)))
    keys = _bf(rng.standard_normal((B, N, 16)))
    wts = rng.standard_normal((B, 1, 3)).astype(np.float32)
    s, nv = oracle.index_scores(qi, wts, keys, n_comp)
    idx = oracle.topk(s, nv, N)
    assert list(idx[0, 0]) == list(range(N)) and list(idx[1, 0]) == list(range(7)) + [-1] * 3
    win_len = np.array([6, 4], np.int32)
    _, a, _ = oracle.sparse_attn(q, sink, kv, n_comp, idx, win, win_len, top_k=N, window=6)
    _, b, _ = oracle.sparse_attn(q, sink, kv, n_comp, None, win, win_len, top_k=N, window=6)
    _close(a, b, rtol=0, atol=0, msg="dense == full top-k")


# ------------------------------------------------------------------ page-printed sizes
def pin_page_sizes():
    """Numbers the pages print for the cache sizes (tests/golden/page_sizes.json)."""
    with open(os.path.join(GOLDEN, "page_sizes.json")) as fh:
        g = json.load(fh)
    for case in g["max_comp"]:
        assert oracle.max_comp(case["context"], case["ratio"]) == case["entries"], case
    for case in g["bytes_per_layer"]:
        n = oracle.max_comp(case["context"], case["ratio"])
        assert n * case["row_bytes"] == case["bytes"], case
    # a partial last block still needs a row: the smallest n with n * ratio >= context
    for r in (1, 4, 128):
        for ctx in range(0, 3 * r + 2):
            assert oracle.max_comp(ctx, r) == next(n for n in range(ctx + 1) if n * r >= ctx)


# ------------------------------------------------------------------ a1, CSA form: overlapped
# [A] compressor_reduce.cu "CSA compressor reduce kernel": entry i pools block i-1 from stream a
# (channels [0, d)) and block i from stream b (channels [d, 2d)); entry 0 has only stream b.
def _overlap(C, Z, bias, prev_C=None, prev_Z=None, pos0=None, ratio=4, rope_dim=0, gamma=None):
    B, T, w = C.shape
    d = w // 2
    gamma = np.ones(d, np.float32) if gamma is None else gamma
    pos0 = np.zeros(B, np.int64) if pos0 is None else pos0
    return oracle.compress_overlap(C, Z, bias, gamma, pos0, ratio, prev_C, prev_Z, rope_dim)


def _unit_rms(v, eps=1e-6):
    v = np.asarray(v, np.float64)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps)


def pin_overlap_first_entry_is_plain_stream_b():
    """With no block before it, entry 0 of the two-stream form is the plain compressor applied
    to stream b alone (C, Z and bias columns [d, 2d)), RMSNorm and RoPE included."""
    rng = _rng(41)
    B, r, d = 2, 4, 64
    C = _bf(rng.standard_normal((B, 3 * r, 2 * d)))
    Z = _bf(rng.standard_normal((B, 3 * r, 2 * d)))
    bias = _f(_bf(rng.standard_normal((r, 2 * d)) * 0.5)).astype(np.float32)
    gamma = _f(_bf(1 + 0.1 * rng.standard_normal(d))).astype(np.float32)
    pos0 = np.array([0, 640], np.int64)
    _, got = _overlap(C, Z, bias, pos0=pos0, rope_dim=16, gamma=gamma)
    _, want = oracle.compress(C[:, :r, d:], Z[:, :r, d:], bias[:, d:], gamma, pos0, r, 16)
    _close(got[:, 0], want[:, 0], rtol=1e-14, atol=1e-14, msg="entry 0 vs plain on stream b")


def pin_overlap_equal_logits_pool_both_blocks():
    """Equal logits (Z = 0, bias = 0): entry i >= 1 is the mean of block i-1's stream-a values
    and block i's stream-b values (2 x ratio tokens), then unit RMS."""
    rng = _rng(42)
    B, r, d, nb = 2, 4, 32, 5
    C = _bf(rng.integers(-64, 65, size=(B, nb * r, 2 * d)).astype(np.float32))
    Z = np.zeros_like(C)
    bias = np.zeros((r, 2 * d), np.float32)
    _, got = _overlap(C, Z, bias)
    c = _f(C)
    for i in range(1, nb):
        pooled = np.concatenate([c[:, (i - 1) * r:i * r, :d], c[:, i * r:(i + 1) * r, d:]], axis=1)
        _close(got[:, i], _unit_rms(pooled.mean(axis=1)), rtol=1e-12, atol=1e-12, msg=f"entry {i}")


def pin_overlap_bias_not_on_C():
    """C = 0 => every entry is 0, for any logits and any bias in either stream ([B] commit
    "Fix two correctness bugs", item 1)."""
    rng = _rng(43)
    B, r, d = 2, 4, 32
    C = np.zeros((B, 4 * r, 2 * d), np.uint16)
    Z = _bf(rng.standard_normal((B, 4 * r, 2 * d)))
    bias = _f(_bf(rng.standard_normal((r, 2 * d)))).astype(np.float32)
    prev = _bf(rng.standard_normal((B, r, 2 * d)))
    _, got = _overlap(C, Z, bias, prev_C=np.zeros_like(prev), prev_Z=prev, rope_dim=8)
    assert np.all(got == 0.0), "bias leaked into the content"


def pin_overlap_streams_come_from_the_right_blocks():
    """A dominant bias on row t0 of one stream's half selects that single token: stream a
    yields C[block i-1, token t0, channels < d], stream b yields C[block i, token t0,
    channels >= d]; for entry 0 with a previous block, stream a reads that block."""
    rng = _rng(44)
    B, r, d, nb = 2, 4, 32, 3
    C = _bf(rng.standard_normal((B, nb * r, 2 * d)))
    Z = _bf(0.1 * rng.standard_normal((B, nb * r, 2 * d)))
    prev_C = _bf(rng.standard_normal((B, r, 2 * d)))
    prev_Z = _bf(0.1 * rng.standard_normal((B, r, 2 * d)))
    c, pc = _f(C), _f(prev_C)
    for t0 in (0, 3):
        bias = np.zeros((r, 2 * d), np.float32)
        bias[t0, :d] = 80.0                                       # stream a, row t0
        _, got = _overlap(C, Z, bias, prev_C=prev_C, prev_Z=prev_Z)
        _close(got[:, 0], _unit_rms(pc[:, t0, :d]), rtol=1e-9, atol=1e-9, msg=f"a, entry 0, t0={t0}")
        for i in range(1, nb):
            _close(got[:, i], _unit_rms(c[:, (i - 1) * r + t0, :d]), rtol=1e-9, atol=1e-9,
                   msg=f"a, entry {i}, t0={t0}")
        bias = np.zeros((r, 2 * d), np.float32)
        bias[t0, d:] = 80.0                                       # stream b, row t0
        _, got = _overlap(C, Z, bias, prev_C=prev_C, prev_Z=prev_Z)
        for i in range(nb):
            _close(got[:, i], _unit_rms(c[:, i * r + t0, d:]), rtol=1e-9, atol=1e-9,
                   msg=f"b, entry {i}, t0={t0}")


def pin_overlap_previous_block_pointer_matches_longer_buffer():
    """Passing block 0 as the previous block and the rest as the buffer gives the entries of
    the longer buffer from entry 1 on, positions shifted by one block (RoPE included)."""
    rng = _rng(45)
    B, r, d, nb = 2, 4, 64, 4
    C = _bf(rng.standard_normal((B, nb * r, 2 * d)))
    Z = _bf(rng.standard_normal((B, nb * r, 2 * d)))
    bias = _f(_bf(0.5 * rng.standard_normal((r, 2 * d)))).astype(np.float32)
    pos0 = np.array([0, 4096], np.int64)
    _, full = _overlap(C, Z, bias, pos0=pos0, rope_dim=64)
    _, tail = _overlap(C[:, r:], Z[:, r:], bias, prev_C=C[:, :r], prev_Z=Z[:, :r], pos0=pos0 + r,
                       rope_dim=64)
    _close(tail, full[:, 1:], rtol=1e-14, atol=1e-14, msg="previous-block pointer")


# ------------------------------------------------------------------ inverse RoPE on the output
def pin_inverse_rope_closed_form():
    """Unit pairs rotate backwards: (1, 0) -> (cos a, -sin a) and (0, 1) -> (sin a, cos a) with
    a = pos * theta^(-2j/rope_dim); position 0 and channels before the rope part are untouched."""
    D, rd, H = 96, 64, 2
    pos = np.array([0, 1, 777, 1048576], np.int64)
    for e_first in (True, False):
        x = np.zeros((len(pos), H, D))
        for j in range(rd // 2):
            x[:, :, D - rd + 2 * j + (0 if e_first else 1)] = 1.0
        x[:, :, : D - rd] = 0.25
        _, got = oracle.inverse_rope(x, pos, rd)
        for r, p in enumerate(pos):
            a = p * 10000.0 ** (-2.0 * np.arange(rd // 2) / rd)
            want_e, want_o = (np.cos(a), -np.sin(a)) if e_first else (np.sin(a), np.cos(a))
            # angles reach 1e6 rad: one ulp of the angle is ~1e-10 there
            _close(got[r, :, D - rd::2], np.broadcast_to(want_e, (H, rd // 2)), 1e-9, 1e-9, "even")
            _close(got[r, :, D - rd + 1::2], np.broadcast_to(want_o, (H, rd // 2)), 1e-9, 1e-9, "odd")
            assert np.all(got[r, :, : D - rd] == 0.25)


def pin_inverse_rope_undoes_the_compressor_rotation():
    """The inverse rotation at the entry's position recovers the compressor's output before
    RoPE (the forward rotation is pinned above)."""
    rng = _rng(51)
    B, r, d = 2, 4, 128
    C = _bf(rng.standard_normal((B, 3 * r, d)))
    Z = _bf(rng.standard_normal((B, 3 * r, d)))
    bias = _f(_bf(0.5 * rng.standard_normal((r, d)))).astype(np.float32)
    pos0 = np.array([12, 90000], np.int64)
    _, rot = _compress(C, Z, bias, pos0=pos0, rope_dim=64)
    _, plain = _compress(C, Z, bias, pos0=pos0, rope_dim=0)
    pos = pos0[:, None] + r * np.arange(3)[None, :]
    _, back = oracle.inverse_rope(rot.reshape(B * 3, 1, d), pos.reshape(-1), 64)
    _close(back.reshape(B, 3, d), plain, 1e-11, 1e-11, "inverse after forward")


# ------------------------------------------------------------------ FP8 E4M3 index keys
def pin_e4m3_codes_from_the_format():
    """Codes worked out by hand from the E4M3 format (bias 7, 3 mantissa bits, subnormals
    m * 2^-9, largest finite 448 = 0x7E, round to nearest even, saturating)."""
    table = [(0.0, 0x00), (-0.0, 0x80), (1.0, 0x38), (1.125, 0x39), (1.0625, 0x38),
             (1.1875, 0x3A), (-2.0, 0xC0), (240.0, 0x77), (448.0, 0x7E), (464.0, 0x7E),
             (1e6, 0x7E), (-1e6, 0xFE), (2.0 ** -6, 0x08), (2.0 ** -9, 0x01), (2.0 ** -10, 0x00),
             (3 * 2.0 ** -10, 0x02), (0.1, 0x1D), (7 * 2.0 ** -9, 0x07), (15 * 2.0 ** -10, 0x08)]
    got = oracle.e4m3_encode([v for v, _ in table])
    for (v, want), g in zip(table, got):
        assert int(g) == want, f"{v}: got {int(g):#04x}, want {want:#04x}"
    dec = oracle.e4m3_decode(np.array([0x38, 0x7E, 0x01, 0x08, 0xC0, 0x1D], np.uint8))
    _close(dec, [1.0, 448.0, 2.0 ** -9, 2.0 ** -6, -2.0, 0.1015625], 0, 0, "decode")


def pin_e4m3_round_trip_and_order():
    """Every finite code decodes and re-encodes to itself; encoding is monotonic; the relative
    error of a normal value is at most 2^-4."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.e4m3_decode(codes)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)
    rng = _rng(61)
    x = np.sort(rng.uniform(-500, 500, 4000))
    dq = oracle.e4m3_decode(oracle.e4m3_encode(x))
    assert np.all(np.diff(dq) >= 0), "not monotonic"
    normal = (np.abs(x) >= 2.0 ** -6) & (np.abs(x) <= 448)
    assert np.all(np.abs(dq[normal] - x[normal]) <= 2.0 ** -4 * np.abs(x[normal]))


def pin_quantize_rows_scale():
    """Each row's largest magnitude maps to +-448 (code 0x7E / 0xFE); an all-zero row has scale
    1 and zero codes."""
    rng = _rng(62)
    x = rng.standard_normal((5, 128)).astype(np.float32)
    x[3] = 0.0
    q, sc = oracle.quantize_rows_e4m3(x)
    for r in (0, 1, 2, 4):
        i = int(np.argmax(np.abs(x[r])))
        assert q[r, i] == (0x7E if x[r, i] > 0 else 0xFE)
        assert sc[r] == np.float32(np.float32(np.abs(x[r, i])) / np.float32(448.0))
    assert sc[3] == 1.0 and not np.any(q[3])


def pin_fp8_scores_equal_plain_scores_on_exact_rows():
    """Rows whose values are E4M3 values with largest magnitude 448 quantize exactly (scale 1),
    so the FP8 scores equal the plain scores of the same values."""
    rng = _rng(63)
    B, H, Di, N = 2, 8, 128, 40
    codes = rng.integers(0, 0x7E, size=(B, 1, H, Di)).astype(np.uint8) | (rng.integers(0, 2, size=(B, 1, H, Di)) << 7).astype(np.uint8)
    kcodes = rng.integers(0, 0x7E, size=(B, N, Di)).astype(np.uint8) | (rng.integers(0, 2, size=(B, N, Di)) << 7).astype(np.uint8)
    codes[..., 0] = 0x7E
    kcodes[..., 0] = 0x7E
    qv = oracle.e4m3_decode(codes).astype(np.float32)
    kv = oracle.e4m3_decode(kcodes).astype(np.float32)
    q8, qs = oracle.quantize_rows_e4m3(qv)
    k8, ks = oracle.quantize_rows_e4m3(kv)
    assert np.array_equal(q8, codes) and np.array_equal(k8, kcodes) and np.all(qs == 1) and np.all(ks == 1)
    w = rng.standard_normal((B, 1, H)).astype(np.float32)
    n_comp = np.array([N, 17], np.int32)
    got, nv8 = oracle.index_scores_fp8(q8, qs, w, k8, ks, n_comp)
    # the plain scorer takes bf16 inputs: scale both sides by 1/64 so every E4M3 value is bf16-exact
    want, nv = oracle.index_scores(_bf(qv / 64), w, _bf(kv / 64), n_comp)
    assert np.array_equal(nv8, nv)
    _close(got[np.isfinite(got)], 4096.0 * want[np.isfinite(want)], 1e-12, 1e-12, "fp8 vs plain")


def pin_fp8_scores_scale_with_the_rows():
    """Scaling a key row by 4 or a query head by 8 (powers of two: exact in fp32) leaves the
    codes unchanged and multiplies the scale; the key's scores then grow 4 times, and head h's
    share of every score 8 times (ReLU is positively homogeneous)."""
    rng = _rng(64)
    B, H, Di, N = 1, 4, 128, 30
    qv = rng.standard_normal((B, 1, H, Di)).astype(np.float32)
    kv = rng.standard_normal((B, N, Di)).astype(np.float32)
    w = np.abs(rng.standard_normal((B, 1, H))).astype(np.float32)
    n_comp = np.array([N], np.int32)
    q8, qs = oracle.quantize_rows_e4m3(qv)
    k8, ks = oracle.quantize_rows_e4m3(kv)
    base, _ = oracle.index_scores_fp8(q8, qs, w, k8, ks, n_comp)
    kv2 = kv.copy()
    kv2[0, 5] *= 4
    k82, ks2 = oracle.quantize_rows_e4m3(kv2)
    assert np.array_equal(k82, k8) and ks2[0, 5] == 4 * ks[0, 5]
    got, _ = oracle.index_scores_fp8(q8, qs, w, k82, ks2, n_comp)
    _close(got[0, 0, 5], 4 * base[0, 0, 5], 1e-12, 1e-12, "key scale")
    _close(np.delete(got[0, 0], 5), np.delete(base[0, 0], 5), 0, 0, "other keys")
    # head 2 alone, then head 2 scaled by 8
    w1 = np.zeros_like(w)
    w1[..., 2] = 1.0
    one, _ = oracle.index_scores_fp8(q8, qs, w1, k8, ks, n_comp)
    qv2 = qv.copy()
    qv2[0, 0, 2] *= 8
    q82, qs2 = oracle.quantize_rows_e4m3(qv2)
    assert np.array_equal(q82, q8) and qs2[0, 0, 2] == 8 * qs[0, 0, 2]
    got2, _ = oracle.index_scores_fp8(q82, qs2, w, k8, ks, n_comp)
    _close(got2, base + 7.0 * float(w[0, 0, 2]) * one, 1e-11, 1e-11, "query scale")


# ------------------------------------------------------------------ mixed FP8 / bf16 KV cache
def pin_kv_mixed_exact_rows_round_trip():
    """An entry whose part without RoPE holds E4M3 values with largest magnitude 448 (scale 1)
    and whose RoPE part holds bf16 values comes back bit for bit; the RoPE part is not folded
    into the scale even when it is the larger part."""
    rng = _rng(71)
    rows, dim, rd = 6, 512, 64
    codes = rng.integers(0, 0x7E, size=(rows, dim - rd)).astype(np.uint8) | \
        (rng.integers(0, 2, size=(rows, dim - rd)) << 7).astype(np.uint8)
    codes[:, 3] = 0x7E
    nope_v = oracle.e4m3_decode(codes).astype(np.float32)
    rope_bits = _bf(rng.standard_normal((rows, rd)) * 1000.0)      # larger than 448
    x = np.concatenate([nope_v, synth.bf16_bits_to_f32(rope_bits)], axis=1)
    nope, sc, rope = oracle.quantize_kv_mixed(x, rd)
    assert np.array_equal(nope, codes) and np.all(sc == 1.0) and np.array_equal(rope, rope_bits)
    back = oracle.dequant_kv_mixed(nope, sc, rope)
    assert np.array_equal(synth.bf16_bits_to_f32(back), x), "round trip"


def pin_kv_mixed_scale_and_bound():
    """Scaling the part without RoPE by 2^k scales the entry's scale by 2^k and keeps its codes;
    the dequantized channels are within half an E4M3 step (plus the bf16 rounding) of the
    fp32 entry; an entry whose part without RoPE is zero has scale 1 and zero codes."""
    rng = _rng(72)
    rows, dim, rd = 5, 512, 64
    x = (rng.standard_normal((rows, dim)) * rng.uniform(0.01, 50, (rows, 1))).astype(np.float32)
    x[2, : dim - rd] = 0.0
    nope, sc, rope = oracle.quantize_kv_mixed(x, rd)
    assert sc[2] == 1.0 and not np.any(nope[2])
    x2 = x.copy()
    x2[:, : dim - rd] *= 8.0
    nope2, sc2, rope2 = oracle.quantize_kv_mixed(x2, rd)
    assert np.array_equal(nope2, nope) and np.array_equal(rope2, rope)
    assert np.array_equal(sc2[[0, 1, 3, 4]], 8.0 * sc[[0, 1, 3, 4]])
    back = synth.bf16_bits_to_f32(oracle.dequant_kv_mixed(nope, sc, rope)).astype(np.float64)
    xn = x[:, : dim - rd].astype(np.float64)
    # E4M3 spacing at |x| / scale: 2^(e - 3) for |x| / scale in [2^e, 2^(e+1)), e >= -6
    e = np.maximum(np.floor(np.log2(np.maximum(np.abs(xn) / sc[:, None], 2.0 ** -6))), -6)
    step = np.exp2(e - 3)
    bound = 0.5 * step * sc[:, None] + 2.0 ** -8 * np.abs(xn) + 1e-30
    assert np.all(np.abs(back[:, : dim - rd] - xn) <= bound * (1 + 1e-6)), "dequant bound"
    assert np.array_equal(back[:, dim - rd:], synth.bf16_bits_to_f32(_bf(x[:, dim - rd:])).astype(np.float64))


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
