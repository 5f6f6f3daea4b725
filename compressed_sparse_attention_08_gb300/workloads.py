"""The five synthetic workloads of the CSA step, with their sizes and input recipes.

Sizes follow the workloads the pages' design targets: DeepSeek-V4 CSA layers with
ratio 4, top-k 512..2048, a 128-token sliding window, 64 indexer heads x 128 dims,
64 attention heads x 512 dims; the HCA layer with ratio 128; and a 1M-token context.
Every tensor is drawn by :mod:`synth` from its own (seed, tensor id) stream. This
module holds sizes and distributions only, none of the method's arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import synth

# Fixed stream ids, one per tensor, so every tensor is reproducible on its own.
TID = {
    "C": 1, "Z": 2, "bias": 3, "gamma": 4,           # main compressor
    "C_I": 5, "Z_I": 6, "bias_I": 7, "gamma_I": 8,   # indexer-key compressor
    "q_I": 9, "w": 10, "swa": 11, "q": 12, "sink": 13,
    "comp_kv": 14, "keys": 15, "win_raw": 16, "idx": 17, "scores": 18,
}


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    batch: int
    context: int             # tokens already in the context (decode) or before the chunk
    ratio: int
    head_dim: int            # D: compressed-entry width = attention head dim
    heads: int               # H: attention query heads
    idx_heads: int           # Hi: indexer heads (0: no indexer, HCA)
    idx_dim: int = 128       # Di
    top_k: int = 0
    window: int = 128
    rope_dim: int = 64
    new_tokens: int = 1      # query tokens per sequence this step (n_q)
    pregen_cache: bool = False   # compressed cache drawn directly instead of compressed
    extra: dict = field(default_factory=dict)

    @property
    def n_comp(self) -> int:
        """Compressed entries in the cache once this step's tokens are in."""
        return (self.context + (self.new_tokens if self.new_tokens > 1 else 0)) // self.ratio

    @property
    def max_comp(self) -> int:
        return self.n_comp

    @property
    def dense(self) -> bool:
        return self.idx_heads == 0

    @property
    def slots(self) -> int:
        """Rows per query in the gather buffer: top_k (max_comp when dense) + window."""
        return (self.max_comp if self.dense else self.top_k) + self.window


WORKLOADS = {
    0: Workload("csa_tiny_ctx1024_b1", seed=0, batch=1, context=1024, ratio=4, head_dim=128,
                heads=8, idx_heads=8, top_k=32),
    1: Workload("csa_decode_ctx8192_b16", seed=1, batch=16, context=8192, ratio=4, head_dim=512,
                heads=64, idx_heads=64, top_k=512),
    2: Workload("hca_decode_ctx8192_b64", seed=2, batch=64, context=8192, ratio=128, head_dim=512,
                heads=64, idx_heads=0, top_k=0),
    3: Workload("csa_decode_ctx1048576_b4", seed=3, batch=4, context=1048576, ratio=4,
                head_dim=512, heads=64, idx_heads=64, top_k=2048, pregen_cache=True),
    4: Workload("csa_prefill_ctx65536_chunk2048_b1", seed=4, batch=1, context=65536, ratio=4,
                head_dim=512, heads=64, idx_heads=64, top_k=1024, new_tokens=2048,
                pregen_cache=True),
}


def _bf16(wl, name, shape, mean=0.0, std=1.0):
    return synth.normal_bf16(wl.seed, TID[name], shape, mean, std)


def _f32_bf16_valued(wl, name, shape, mean=0.0, std=1.0):
    """fp32 array whose values are bf16-representable (checkpoint-style weights)."""
    return synth.bf16_bits_to_f32(_bf16(wl, name, shape, mean, std))


def make_inputs(wl: Workload, batch: int | None = None) -> dict:
    """All inputs of one step of workload ``wl`` as numpy arrays (bf16 as uint16 bits).

    ``batch`` (<= wl.batch) draws only the first sequences of every batched tensor; the
    values of those sequences are identical to the full draw.  Keys:

    * compressor: ``C, Z`` [B, T, D], ``bias`` [r, D], ``gamma`` [D], ``pos0`` [B];
      indexer-key compressor ``C_I, Z_I`` [B, T, Di], ``bias_I`` [r, Di], ``gamma_I`` [Di]
      (T = tokens compressed this step: the whole context, or the newest block / chunk).
    * caches: ``comp_kv`` [B, max_comp, D], ``keys`` [B, max_comp, Di] (pre-generated
      workloads only; otherwise the compressor produces them), ``n_comp`` [B].
    * indexer: ``q_I`` [B, n_q, Hi, Di], ``w`` [B, n_q, Hi], ``q_pos`` [B, n_q] or None.
    * attention: ``q`` [B, n_q, H, D], ``sink`` [H], window ``win`` [B, rows, D], ``win_len`` [B].
    """
    B = wl.batch if batch is None else batch
    D, Di, r, n_q = wl.head_dim, wl.idx_dim, wl.ratio, wl.new_tokens
    x = {}
    full = wl.batch

    def batched(name, per_seq_shape, mean=0.0, std=1.0):
        a = _bf16(wl, name, (full,) + tuple(per_seq_shape), mean, std) if B == full else \
            _bf16_prefix(wl, name, full, B, per_seq_shape, mean, std)
        return a

    if wl.pregen_cache:
        if n_q > 1:
            T = n_q                      # prefill: the new chunk is compressed this step
            old = wl.context // r
        else:
            T = r                        # decode: the newest block only
            old = wl.n_comp - 1
        x["pos0"] = np.full(B, wl.context - (r if n_q == 1 else 0), np.int64)
        x["comp_kv"] = batched("comp_kv", (wl.max_comp, D))
        x["keys"] = batched("keys", (wl.max_comp, Di))
        x["append_row"] = np.full(B, old, np.int32)
    else:
        T = wl.context
        x["pos0"] = np.zeros(B, np.int64)
        x["append_row"] = np.zeros(B, np.int32)
    x["T"] = T
    x["C"] = batched("C", (T, D))
    x["Z"] = batched("Z", (T, D))
    x["bias"] = _f32_bf16_valued(wl, "bias", (r, D), 0.0, 0.5)
    x["gamma"] = _f32_bf16_valued(wl, "gamma", (D,), 1.0, 0.1)
    if not wl.dense:
        x["C_I"] = batched("C_I", (T, Di))
        x["Z_I"] = batched("Z_I", (T, Di))
        x["bias_I"] = _f32_bf16_valued(wl, "bias_I", (r, Di), 0.0, 0.5)
        x["gamma_I"] = _f32_bf16_valued(wl, "gamma_I", (Di,), 1.0, 0.1)
        x["q_I"] = batched("q_I", (n_q, wl.idx_heads, Di))
        w = synth.normal_f32(wl.seed, TID["w"], (full, n_q, wl.idx_heads), 0.0,
                             1.0 / np.sqrt(wl.idx_heads))
        x["w"] = np.ascontiguousarray(w[:B])
    x["n_comp"] = np.full(B, wl.n_comp, np.int32)
    x["q"] = batched("q", (n_q, wl.heads, D))
    x["sink"] = synth.normal_f32(wl.seed, TID["sink"], (wl.heads,))
    if n_q > 1:
        # raw per-token KV of the window-1 tokens before the chunk and of the chunk itself
        rows = wl.window + n_q
        x["win"] = batched("win_raw", (rows, D))
        x["win_len"] = np.full(B, rows, np.int32)
        x["q_pos"] = np.tile(np.arange(wl.context, wl.context + n_q, dtype=np.int64), (B, 1))
    else:
        x["win"] = batched("swa", (wl.window, D))
        x["win_len"] = np.full(B, wl.window, np.int32)
        x["q_pos"] = None
    return x


# Seeds of the extra per-step input sets of step_inputs: wl.seed + VARIANT_SEED_STRIDE * j.
VARIANT_SEED_STRIDE = 1000


def step_inputs(wl: Workload, variant: int) -> dict:
    """The inputs that change from one decode step to the next (indexer queries ``q_I``, head
    weights ``w``, attention queries ``q`` and the newest block's ``C, Z, C_I, Z_I``), full
    batch, for a decode workload (one query per sequence) with pre-generated caches. Variant 0
    is exactly make_inputs' draw; variant j > 0 draws the same shapes and distributions from
    seed wl.seed + VARIANT_SEED_STRIDE * j. Replaying a step over several variants makes
    consecutive steps select different cache rows, as successive decode tokens do."""
    assert wl.pregen_cache and wl.new_tokens == 1 and not wl.dense
    seed = wl.seed + VARIANT_SEED_STRIDE * variant
    B, D, Di, r = wl.batch, wl.head_dim, wl.idx_dim, wl.ratio

    def bf(name, shape):
        return synth.normal_bf16(seed, TID[name], (B,) + shape)

    x = {"C": bf("C", (r, D)), "Z": bf("Z", (r, D)), "C_I": bf("C_I", (r, Di)), "Z_I": bf("Z_I", (r, Di)),
         "q_I": bf("q_I", (1, wl.idx_heads, Di)), "q": bf("q", (1, wl.heads, D))}
    x["w"] = synth.normal_f32(seed, TID["w"], (B, 1, wl.idx_heads), 0.0, 1.0 / np.sqrt(wl.idx_heads))
    return x


def _bf16_prefix(wl, name, full, B, per_seq_shape, mean, std):
    """First B sequences of a [full, ...] draw, without drawing the rest."""
    n_per = int(np.prod(per_seq_shape))
    key_shape = (B,) + tuple(per_seq_shape)
    # elements of the first B sequences are the first B * n_per elements of the stream
    flat = synth.normal_bf16(wl.seed, TID[name], (B * n_per,), mean, std)
    return flat.reshape(key_shape)
