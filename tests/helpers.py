"""Shared test helpers: host/device conversion and the parity rules.

Parity rules (the build's stated tolerances):
  * bf16 outputs (compressed entries, attention outputs): |gpu - oracle| <= 2e-2 + 1e-2 |oracle|
    elementwise, the oracle in fp64 (fp32 accumulation on the GPU).
  * top-k indices: bit-exact, except where the oracle's k-th and (k+1)-th scores differ by
    less than 1e-5 relative; there a swap is allowed only between indices whose oracle scores
    lie within 1e-5 relative of the k-th score.
  * gathered rows and any integer output: bit-exact.
"""
from __future__ import annotations

import numpy as np

from compressed_sparse_attention_08_gb300 import synth

ATOL = 2e-2
RTOL = 1e-2
TOPK_REL = 1e-5


def dev_bf16(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bf16(t):
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(bits):
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def assert_bf16_close(gpu_bits, ref_f64, what="", atol=ATOL, rtol=RTOL):
    g = bf16_to_f64(gpu_bits)
    r = np.asarray(ref_f64, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    err = np.abs(g - r)
    bad = err > atol + rtol * np.abs(r)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(r))), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst at {i}: "
                             f"gpu {g[i]!r} oracle {r[i]!r}; max abs err {err.max():.3e}")
    return float(err.max())


def check_topk_row(gpu_idx, oracle_idx, oracle_scores, n_vis, k, what=""):
    """Apply the top-k parity rule to one row. Returns the number of tolerated swaps."""
    gpu_idx = np.asarray(gpu_idx)
    oracle_idx = np.asarray(oracle_idx)
    t = min(k, n_vis)
    # structure: ascending valid indices then -1 padding
    sel = gpu_idx[:t]
    assert np.all(gpu_idx[t:] == -1), f"{what}: padding"
    assert np.all(sel >= 0) and np.all(sel < n_vis), f"{what}: range"
    assert np.all(np.diff(sel) > 0), f"{what}: not ascending / duplicates"
    if np.array_equal(gpu_idx, oracle_idx):
        return 0
    s = np.asarray(oracle_scores[:n_vis], np.float64)
    order = np.lexsort((np.arange(n_vis), -s))
    sk = s[order[t - 1]]
    gap_ok = t < n_vis and abs(s[order[t - 1]] - s[order[t]]) < TOPK_REL * max(abs(sk), 1e-30)
    diff = np.setxor1d(sel, oracle_idx[:t])
    near = np.abs(s[diff] - sk) <= TOPK_REL * max(abs(sk), 1e-30)
    assert gap_ok and near.all(), (
        f"{what}: top-k differs at {len(diff)} indices; k-th gap "
        f"{abs(s[order[t - 1]] - s[order[t]]) if t < n_vis else 0:.3e}; "
        f"far ones {diff[~near][:8]} with scores {s[diff[~near]][:8]} vs k-th {sk}")
    return len(diff) // 2


def topk_valid_for_scores(gpu_idx, scores_f32, n_vis, k, what=""):
    """The GPU's selection is exactly the top-k of the GPU's own fp32 scores under the tie
    rule (-0 == +0, lower index first): a property check, independent of the oracle."""
    s = np.asarray(scores_f32[:n_vis], np.float32).astype(np.float64)
    t = min(k, n_vis)
    want = np.sort(np.lexsort((np.arange(n_vis), -s))[:t])
    got = np.asarray(gpu_idx[:t])
    assert np.array_equal(got, want), f"{what}: selection is not the top-k of its own scores"
