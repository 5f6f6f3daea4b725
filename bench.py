#!/usr/bin/env python
"""Benchmark of the CSA decode step at 1M-token context (batch 4 per GPU), one JSON line.

A step is one pass of the whole hot path over one batch: compress the newest 4-token block
of the main KV and of the indexer keys into the caches, score all 262,144 compressed keys
with 64 indexer heads, select the top 2048 per sequence, gather those rows plus the
128-token window into the gather buffer and run 64-head sink attention over them. The step
is captured once in a CUDA graph and replayed; inputs stay resident in HBM (256 MiB of
keys and 1 GiB of compressed KV: larger than L2, so every step streams the keys from HBM).

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Under torchrun each rank runs its own batch (weak scaling, no data-path collective); rank 0
prints the line with the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CSA decode tokens/s per layer @1M ctx; indexer+gather HBM GB/s vs ~8 TB/s"
CFG = 3


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the chunked-prefill indexer scoring (tensor-core bound)")
    ap.add_argument("--fp8-only", action="store_true",
                    help="time only the decode step with the FP8 index-key cache")
    ap.add_argument("--decode-workload", type=int, choices=[1, 2], default=None,
                    help="time only the decode step of workload 1 (8K context, batch 16) or 2 (HCA)")
    ap.add_argument("--headline-only", action="store_true",
                    help="time only the headline step (no end-to-end, scorer, prefill, FP8 or other "
                         "workloads): a short run for profilers")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value, world, device="cpu"):
    """The largest per-rank value over all ranks (the value itself at world size 1)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank, world, ms_per_step):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


def step_bytes(wl):
    """Algorithmic bytes of one step: index keys scanned + gathered KV rows + outputs."""
    keys = wl.batch * wl.n_comp * wl.idx_dim * 2
    gathered = wl.batch * (wl.top_k + wl.window) * wl.head_dim * 2
    outputs = wl.batch * wl.heads * wl.head_dim * 2
    return keys, gathered, outputs


def scorer_bytes(wl):
    """Algorithmic bytes of one scoring launch (the index-key scan): every visible key (256 B)
    read once. Returns (scan bytes, side bytes): the side traffic, listed but not credited, is
    one fp32 score written per key plus the queries and head weights."""
    scan = wl.batch * wl.n_comp * wl.idx_dim * 2
    side = wl.batch * wl.n_comp * 4 + wl.batch * wl.idx_heads * (wl.idx_dim * 2 + 4)
    return scan, side


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return float(json.load(fh)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def prefill_scoring(m, steps):
    """The chunked-prefill indexer scoring alone: 2048 new query tokens x 64 heads x 128 dims
    against the 16,896 compressed keys with the causal block mask. A dense contraction, so
    it is reported in TFLOP/s against the measured bf16 tensor peak; flops count only the
    visible (query, key) pairs, 64 heads x 128 dims x 2 each."""
    import numpy as np
    import torch
    from compressed_sparse_attention_08_gb300.workloads import WORKLOADS, make_inputs
    wl = WORKLOADS[4]
    x = make_inputs(wl)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)

    q, keys = bf(x["q_I"]), bf(x["keys"])
    w = torch.from_numpy(np.ascontiguousarray(x["w"])).cuda()
    n_comp = torch.from_numpy(x["n_comp"]).cuda()
    q_pos = torch.from_numpy(x["q_pos"]).cuda()
    scores = torch.empty(1, wl.new_tokens, wl.max_comp, dtype=torch.float32, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def run():
        m.dsv4_index_score(q, w, keys, n_comp, scores, ws, ratio=wl.ratio, q_pos=q_pos, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            run()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(max(1, min(steps, 50)))]
        for a, b in evs:
            a.record(stream)
            run()
            b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    vis = np.minimum(x["n_comp"][0], (x["q_pos"][0] + 1) // wl.ratio)
    flops = float(vis.sum()) * wl.idx_heads * wl.idx_dim * 2
    peak, kind = measured_bf16_peak()
    achieved = flops / (ms * 1e-3) / 1e12
    return {"workload": wl.name, "bound": "tensor", "kernel": "index_score_kernel",
            "flops_per_launch": flops, "ms_per_launch": ms, "achieved": achieved, "peak": peak,
            "peak_kind": kind, "unit": "TFLOP/s", "frac": achieved / peak}


def fp8_keys_step(m, _abi, t, variants, wl, steps, stream, peak, mixed_kv=False):
    """The same decode step with the index-key cache in FP8 E4M3 (codes + one fp32 scale per
    key): the compressor writes the newest key in FP8, the scorer reads 128 + 4 bytes per key
    instead of 256. The query quantization runs inside the step. mixed_kv: the KV cache too in
    the pages' mixed storage (E4M3 codes of the 448 channels without RoPE, one fp32 scale,
    bf16 RoPE part: 580 bytes per gathered row instead of 1024). Replayed over the same
    rotating input sets as the headline. Reported beside the bf16 headline, not as it."""
    import torch
    B = wl.batch
    keys8 = torch.empty(B, wl.max_comp, wl.idx_dim, dtype=torch.uint8, device="cuda")
    kscale = torch.empty(B, wl.max_comp, dtype=torch.float32, device="cuda")
    q8 = torch.empty(t["q_I"].shape, dtype=torch.uint8, device="cuda")
    qscale = torch.empty(t["q_I"].shape[:-1], dtype=torch.float32, device="cuda")
    with torch.cuda.stream(stream):
        m.dsv4_quantize_rows_fp8(t["keys"], keys8, kscale, stream=stream)
    stream.synchronize()
    rd, D = wl.rope_dim, wl.head_dim
    if mixed_kv:
        # the cache's rows in the mixed storage (input preparation on the device, untimed)
        kvf = t["kv"].float()
        amax = kvf[..., : D - rd].abs().amax(dim=-1)
        kv_scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).contiguous()
        kv_nope = (kvf[..., : D - rd] / kv_scale[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
        kv_rope = t["kv"][..., D - rd:].contiguous()
        del kvf
    structs = []
    for v in variants:
        cq = _abi.compress_args(v["C_I"], v["Z_I"], t["bias_I"], t["gamma_I"], t["pos0"], keys8,
                                ratio=wl.ratio, out_row0=t["append_row"], out_scale=kscale)
        if mixed_kv:
            ck = _abi.compress_args(v["C"], v["Z"], t["bias"], t["gamma"], t["pos0"], kv_nope, ratio=wl.ratio,
                                    out_row0=t["append_row"], out_scale=kv_scale, out_rope=kv_rope)
            aa = _abi.attn_args(v["q"], t["sink"], None, t["n_comp"], t["win"], t["win_len"], t["out"],
                                idx=t["idx"], window=wl.window, ratio=wl.ratio, gather=t["gather"],
                                kv_nope=kv_nope, kv_scale=kv_scale, kv_rope=kv_rope)
        else:
            ck = _abi.compress_args(v["C"], v["Z"], t["bias"], t["gamma"], t["pos0"], t["kv"], ratio=wl.ratio,
                                    out_row0=t["append_row"])
            aa = _abi.attn_args(v["q"], t["sink"], t["kv"], t["n_comp"], t["win"], t["win_len"], t["out"],
                                idx=t["idx"], window=wl.window, ratio=wl.ratio, gather=t["gather"])
        ia = _abi.index_args(q8, v["w"], keys8, t["n_comp"], t["idx"], ratio=wl.ratio, q_scale=qscale,
                             key_scale=kscale)
        structs.append((v["q_I"], ck, cq, ia, aa))
    nbytes = m.dsv4_csa_decode_workspace_size(attn=structs[0][4], index=structs[0][3], compress_kv=structs[0][1],
                                              compress_keys=structs[0][2])
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")

    def step(s, j):
        q_I, ck, cq, ia, aa = structs[j]
        m.dsv4_quantize_rows_fp8(q_I, q8, qscale, stream=s)
        launches = m.dsv4_last_launch_count()
        m.dsv4_csa_decode(ws, attn=aa, index=ia, compress_kv=ck, compress_keys=cq, stream=s)
        return launches + m.dsv4_last_launch_count()

    with torch.cuda.stream(stream):
        for j in range(len(structs)):
            launches = step(stream, j)
    stream.synchronize()
    st, ew = m.dsv4_read_error_word(ws, stream)
    if ew:
        raise SystemExit(f"device error word {ew:#x} in the FP8-key step")
    graphs = []
    for j in range(len(structs)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                step(stream, j)
        graphs.append(g)
    # timed like the headline: one graph holds one step per input set
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_all, stream=stream):
            for j in range(len(structs)):
                step(stream, j)
    stream.synchronize()
    with torch.cuda.stream(stream):
        for i in range(10):
            graphs[i % len(graphs)].replay()
        g_all.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps // len(graphs)):
            g_all.replay()
        for i in range(steps % len(graphs)):
            graphs[i].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # the scorer alone on the FP8 cache
    score_ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    kw = dict(ratio=wl.ratio, stream=stream, q_scale=qscale, key_scale=kscale)
    with torch.cuda.stream(stream):
        for _ in range(3):
            m.dsv4_index_score(q8, t["w"], keys8, t["n_comp"], t["scores"], score_ws, **kw)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            a.record(stream)
            m.dsv4_index_score(q8, t["w"], keys8, t["n_comp"], t["scores"], score_ws, **kw)
            b.record(stream)
    torch.cuda.synchronize()
    score_ms_isolated = statistics.mean(a.elapsed_time(b) for a, b in evs)
    with torch.cuda.stream(stream):                   # back to back, as for the bf16 scorer
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(steps):
            m.dsv4_index_score(q8, t["w"], keys8, t["n_comp"], t["scores"], score_ws, **kw)
        c1.record(stream)
    torch.cuda.synchronize()
    score_ms = c0.elapsed_time(c1) / steps
    # algorithmic bytes of the scan: every key's code row and scale read once
    sb = B * wl.n_comp * (wl.idx_dim + 4)
    side = B * wl.n_comp * 4 + B * wl.idx_heads * (wl.idx_dim + 4 + 4)
    gbs = sb / (score_ms * 1e-3) / 1e9
    # the step's algorithmic bytes: keys (codes + scale) scanned, gathered rows, outputs
    row_b = (D - rd) + 4 + rd * 2 if mixed_kv else D * 2
    step_b = (B * wl.n_comp * (wl.idx_dim + 4) + B * wl.top_k * row_b + B * wl.window * D * 2 +
              B * wl.heads * D * 2)
    return {"value": B / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "launches_per_step": launches,
            "dtype": "fp8 e4m3 index keys, " + ("mixed fp8/bf16 KV" if mixed_kv else "bf16 KV"),
            "input_sets": len(structs),
            "timing": "one CUDA graph holding one step per input set, as for the headline",
            "step_bytes": step_b, "step_frac": step_b / (ms * 1e-3) / 1e9 / peak,
            "scorer": {"kernel": "index_score_kernel<FP8>", "bytes_per_launch": sb,
                       "side_bytes_per_launch": side,
                       "ms_per_launch": score_ms, "ms_per_launch_isolated": score_ms_isolated,
                       "achieved": gbs, "peak": peak, "unit": "GB/s",
                       "frac": gbs / peak,
                       "traffic": profile_traffic("index_score_kernel_fp8_csa_decode_ctx1048576_b4.md")}}


def decode_step_at(m, _abi, cfg, steps, peak):
    """The fused decode step of another decode workload (the 8K-context batch-16 CSA layer,
    the 8K-context batch-64 HCA layer), timed like the headline: the caches are filled once
    by compressing the whole context, then each step compresses the newest block into the
    last cache row and runs the rest of the step; one CUDA graph per step. Algorithmic
    bytes per step as for the headline (keys scanned + gathered rows + outputs)."""
    import numpy as np
    import torch
    from compressed_sparse_attention_08_gb300.workloads import WORKLOADS, make_inputs
    wl = WORKLOADS[cfg]
    x = make_inputs(wl)
    B, D, Di, r, T = wl.batch, wl.head_dim, wl.idx_dim, wl.ratio, wl.context

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)

    def dv(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    t = {k: bf(x[k]) for k in ("C", "Z", "q", "win")}
    t.update({k: dv(x[k]) for k in ("bias", "gamma", "pos0", "n_comp", "sink", "win_len")})
    t["kv"] = torch.zeros(B, wl.max_comp, D, dtype=torch.bfloat16, device="cuda")
    m.dsv4_compress(t["C"], t["Z"], t["bias"], t["gamma"], t["pos0"], t["kv"], ratio=r)
    t["pos_n"] = torch.full((B,), T - r, dtype=torch.int64, device="cuda")
    t["row_n"] = torch.full((B,), wl.n_comp - 1, dtype=torch.int32, device="cuda")
    t["Cn"], t["Zn"] = t["C"][:, T - r:].contiguous(), t["Z"][:, T - r:].contiguous()
    ck = _abi.compress_args(t["Cn"], t["Zn"], t["bias"], t["gamma"], t["pos_n"], t["kv"], ratio=r,
                            out_row0=t["row_n"])
    cq = ia = None
    k = wl.max_comp if wl.dense else wl.top_k
    t["out"] = torch.empty(B, 1, wl.heads, D, dtype=torch.bfloat16, device="cuda")
    t["gather"] = torch.empty(B, 1, k + wl.window, D, dtype=torch.bfloat16, device="cuda")
    if not wl.dense:
        t.update({kk: bf(x[kk]) for kk in ("C_I", "Z_I", "q_I")})
        t.update({kk: dv(x[kk]) for kk in ("bias_I", "gamma_I", "w")})
        t["keys"] = torch.zeros(B, wl.max_comp, Di, dtype=torch.bfloat16, device="cuda")
        m.dsv4_compress(t["C_I"], t["Z_I"], t["bias_I"], t["gamma_I"], t["pos0"], t["keys"], ratio=r)
        t["CIn"], t["ZIn"] = t["C_I"][:, T - r:].contiguous(), t["Z_I"][:, T - r:].contiguous()
        cq = _abi.compress_args(t["CIn"], t["ZIn"], t["bias_I"], t["gamma_I"], t["pos_n"], t["keys"], ratio=r,
                                out_row0=t["row_n"])
        t["idx"] = torch.empty(B, 1, k, dtype=torch.int32, device="cuda")
        ia = _abi.index_args(t["q_I"], t["w"], t["keys"], t["n_comp"], t["idx"], ratio=r)
    aa = _abi.attn_args(t["q"], t["sink"], t["kv"], t["n_comp"], t["win"], t["win_len"], t["out"],
                        idx=t.get("idx"), top_k=k, window=wl.window, ratio=r, gather=t["gather"])
    ws = torch.empty(max(m.dsv4_csa_decode_workspace_size(attn=aa, index=ia, compress_kv=ck, compress_keys=cq),
                         256), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def step(s):
        m.dsv4_csa_decode(ws, attn=aa, index=ia, compress_kv=ck, compress_keys=cq, stream=s)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step(stream)
    stream.synchronize()
    launches = m.dsv4_last_launch_count()
    st, ew = m.dsv4_read_error_word(ws, stream)
    if ew:
        raise SystemExit(f"device error word {ew:#x} in the {wl.name} step")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            step(stream)
    stream.synchronize()
    # the workload fits in L2: every timed replay starts from a flushed L2 (a 256 MiB write
    # between replays, outside the timed events)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(5):
            graph.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            graph.replay()
            b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    keys = 0 if wl.dense else B * wl.n_comp * Di * 2
    nbytes = keys + B * (k + wl.window) * D * 2 + B * wl.heads * D * 2
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": wl.name, "value": B / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms,
            "launches_per_step": launches, "bytes_per_step": nbytes, "achieved": gbs, "peak": peak,
            "unit_bw": "GB/s", "frac": gbs / peak, "l2": "flushed before every timed replay"}


def compressor_time(m, t, wl, steps, stream):
    """The compressor alone at the headline workload: the newest block of the KV cache and of
    the key cache, one dsv4_compress call each (in the fused step they share one launch),
    captured in a CUDA graph so the host does not pace it. A latency-bound reduction:
    microseconds per pair of calls."""
    import torch

    def run():
        m.dsv4_compress(t["C"], t["Z"], t["bias"], t["gamma"], t["pos0"], t["kv"], ratio=wl.ratio,
                        out_row0=t["append_row"], stream=stream)
        m.dsv4_compress(t["C_I"], t["Z_I"], t["bias_I"], t["gamma_I"], t["pos0"], t["keys"], ratio=wl.ratio,
                        out_row0=t["append_row"], stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            run()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            run()
    stream.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(5):
            g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps * 1000.0


def device_arena(specs):
    """One device buffer holding tensors of the given (name, shape, dtype), each at a
    256-byte aligned offset: returns the buffer (bytes) and a name -> view dict."""
    import math
    import torch
    offs, total = [], 0
    for _, shape, dt in specs:
        n = math.prod(shape) * torch.empty((), dtype=dt).element_size()
        offs.append(total)
        total += (n + 255) // 256 * 256
    buf = torch.zeros(total, dtype=torch.uint8, device="cuda")
    views = {}
    for (name, shape, dt), off in zip(specs, offs):
        n = math.prod(shape) * torch.empty((), dtype=dt).element_size()
        views[name] = buf[off:off + n].view(dt).view(*shape)
    return buf, views


def prefill_attention(m, steps):
    """The chunked-prefill attention alone: 2048 queries x 64 heads x 512 dims, each over its
    1024 selected compressed entries and its own 128-token window (causal), no gather buffer.
    Reported in TFLOP/s (QK and PV, 4 flops per head, slot and dim) against the measured bf16
    tensor peak."""
    import numpy as np
    import torch
    from compressed_sparse_attention_08_gb300 import synth
    from compressed_sparse_attention_08_gb300.workloads import WORKLOADS, make_inputs
    wl = WORKLOADS[4]
    x = make_inputs(wl)
    n_q = wl.new_tokens

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)

    def dv(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    nvis = np.minimum(x["n_comp"][0], (x["q_pos"][0] + 1) // wl.ratio).astype(np.int32)
    idx = synth.uniform_index_sets(wl.seed, 17, n_q, nvis, wl.top_k).reshape(1, n_q, wl.top_k)
    q, sink, kv = bf(x["q"]), dv(x["sink"]), bf(x["comp_kv"])
    n_comp, win, win_len, q_pos = dv(x["n_comp"]), bf(x["win"]), dv(x["win_len"]), dv(x["q_pos"])
    idx_d = dv(idx)
    out = torch.empty(1, n_q, wl.heads, wl.head_dim, dtype=torch.bfloat16, device="cuda")
    kw = dict(idx=idx_d, top_k=wl.top_k, window=wl.window, ratio=wl.ratio, q_pos=q_pos)
    ws = torch.empty(max(m.dsv4_sparse_attn_workspace_size(q, sink, kv, n_comp, win, win_len, out, **kw), 256),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()

    def run():
        m.dsv4_sparse_attn_decode(q, sink, kv, n_comp, win, win_len, out, ws, stream=stream, **kw)

    with torch.cuda.stream(stream):
        for _ in range(3):
            run()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(max(1, min(steps, 20)))]
        for a, b in evs:
            a.record(stream)
            run()
            b.record(stream)
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    flops = float(n_q) * wl.heads * (wl.top_k + wl.window) * wl.head_dim * 4
    peak, kind = measured_bf16_peak()
    achieved = flops / (ms * 1e-3) / 1e12
    return {"workload": wl.name, "bound": "tensor", "flops_per_call": flops, "ms_per_call": ms,
            "achieved": achieved, "peak": peak, "peak_kind": kind, "unit": "TFLOP/s", "frac": achieved / peak}


def profile_traffic(name="index_score_kernel_csa_decode_ctx1048576_b4.md"):
    """dram bytes per scoring launch from the committed ncu summary, if the kernel source
    still matches the hash recorded there; else None."""
    path = os.path.join(ROOT, "profiles", name)
    src = os.path.join(ROOT, "compressed_sparse_attention_08_gb300", "csrc", "indexer.cu")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m1 = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m2 = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not (m1 and m2):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != m1.group(1):
        return None
    return int(m2.group(1))


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while the GPU is under load."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        busy = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline(wl, x0, seconds_hint=None):
    """The oracle (single thread, fp64) on one sequence's step: newest-block compression of
    the KV and the keys, the 262,144-key indexer scan, top-2048, 2,176-row sink attention."""
    import numpy as np
    import oracle
    oracle.build()
    t0 = time.perf_counter()
    kv_bits, _ = oracle.compress(x0["C"], x0["Z"], x0["bias"], x0["gamma"], x0["pos0"], wl.ratio)
    key_bits, _ = oracle.compress(x0["C_I"], x0["Z_I"], x0["bias_I"], x0["gamma_I"], x0["pos0"], wl.ratio)
    comp_kv = x0["comp_kv"]
    keys = x0["keys"]
    comp_kv[:, -1] = kv_bits[:, 0]
    keys[:, -1] = key_bits[:, 0]
    s, nv = oracle.index_scores(x0["q_I"], x0["w"], keys, x0["n_comp"], wl.ratio)
    idx = oracle.topk(s, nv, wl.top_k)
    oracle.sparse_attn(x0["q"], x0["sink"], comp_kv, x0["n_comp"], idx, x0["win"], x0["win_len"],
                       wl.top_k, wl.window, wl.ratio)
    dt = time.perf_counter() - t0
    return {"value": 1.0 / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": "one sequence (1 token) of the 1M-context batch-4 decode step: newest-block "
                      "compression of KV and keys, 262,144-key indexer scan, top-2048, 2,176-row "
                      "sink attention; fp64, single thread",
            "seconds": dt, "cpu": _cpu_model(), "nproc": os.cpu_count()}


def _cpu_model():
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ----------------------------------------------------------------------------- shared config
N_INPUT_SETS = 8          # per-step input sets the timed replays rotate over


def workload_config(wl):
    """The workload as both arms report it (same keys, same values)."""
    return {"workload": wl.name, "batch_per_gpu": wl.batch, "context": wl.context,
            "n_comp": wl.n_comp, "top_k": wl.top_k, "window": wl.window,
            "idx_heads": wl.idx_heads, "heads": wl.heads, "head_dim": wl.head_dim,
            "input_sets": N_INPUT_SETS,
            "l2": "inputs larger than L2 (256 MiB of index keys scanned per step, 1 GiB KV cache); "
                  "consecutive steps rotate over the input sets, so each selects other cache rows"}


# ----------------------------------------------------------------------------- reference arm
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from compressed_sparse_attention_08_gb300.workloads import WORKLOADS, make_inputs
    wl = WORKLOADS[CFG]
    x0 = make_inputs(wl, batch=1)
    # a warm-up step only loads the oracle's library and touches the inputs: two suffice (each
    # step is ~2 s of one host core, and the whole run has to end within a few minutes)
    for _ in range(min(args.warmup, 2)):
        cpu_baseline(wl, dict(x0))
    times = []
    for _ in range(args.steps):
        times.append(cpu_baseline(wl, dict(x0))["seconds"])
    total = sum(times)
    value = args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl), "where": "host: the oracle on one core",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": "one sequence (1 token) of the 1M-context batch-4 decode step "
                                       "per timed step, fp64 oracle, single thread"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm
def run_ours(args):
    import numpy as np
    import torch
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    import __graft_entry__
    __graft_entry__.build()
    import compressed_sparse_attention_08_gb300 as m
    from compressed_sparse_attention_08_gb300 import _abi
    from compressed_sparse_attention_08_gb300.workloads import WORKLOADS, make_inputs, step_inputs

    wl = WORKLOADS[CFG]
    t0 = time.time()
    x = make_inputs(wl)
    log(f"[rank {rank}] inputs generated in {time.time() - t0:.1f}s")
    B, D, Di = wl.batch, wl.head_dim, wl.idx_dim

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).cuda().view(torch.bfloat16)

    def dv(a):
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()

    t = {}
    t["kv"], t["keys"] = bf(x["comp_kv"]), bf(x["keys"])
    for k in ("win",):
        t[k] = bf(x[k])
    for k in ("bias", "gamma", "bias_I", "gamma_I", "pos0", "append_row", "n_comp", "sink", "win_len"):
        t[k] = dv(x[k])
    # A step's inputs (queries, head weights, the newest block's C and Z for both caches) and
    # outputs (attention output, index list) each live in one device arena, so the host side
    # of a step is one copy in and one copy out. The timed replays rotate over N_INPUT_SETS
    # such input arenas (seeded variants of the same draw), so consecutive steps select
    # different cache rows and the gather does not find the previous step's rows in L2.
    per_step_in = [(k, x[k].shape, torch.bfloat16) for k in ("q_I", "q", "C", "Z", "C_I", "Z_I")]
    per_step_in.append(("w", x["w"].shape, torch.float32))
    arenas, variants = [], []
    for j in range(N_INPUT_SETS):
        xv = step_inputs(wl, j)
        arena_j, views_j = device_arena(per_step_in)
        for k, _, dt in per_step_in:
            views_j[k].copy_(bf(xv[k]) if dt == torch.bfloat16 else dv(xv[k]))
        arenas.append(arena_j)
        variants.append(views_j)
    t.update(variants[0])
    arena_out, oviews = device_arena([("out", (B, 1, wl.heads, D), torch.bfloat16),
                                      ("idx", (B, 1, wl.top_k), torch.int32)])
    t.update(oviews)
    t["gather"] = torch.empty(B, 1, wl.top_k + wl.window, D, dtype=torch.bfloat16, device="cuda")
    t["scores"] = torch.empty(B, 1, wl.max_comp, dtype=torch.float32, device="cuda")
    structs = []
    for v in variants:
        ck = _abi.compress_args(v["C"], v["Z"], t["bias"], t["gamma"], t["pos0"], t["kv"], ratio=wl.ratio,
                                out_row0=t["append_row"])
        cq = _abi.compress_args(v["C_I"], v["Z_I"], t["bias_I"], t["gamma_I"], t["pos0"], t["keys"],
                                ratio=wl.ratio, out_row0=t["append_row"])
        ia = _abi.index_args(v["q_I"], v["w"], t["keys"], t["n_comp"], t["idx"], ratio=wl.ratio)
        aa = _abi.attn_args(v["q"], t["sink"], t["kv"], t["n_comp"], t["win"], t["win_len"], t["out"],
                            idx=t["idx"], window=wl.window, ratio=wl.ratio, gather=t["gather"])
        structs.append((ck, cq, ia, aa))
    nbytes = m.dsv4_csa_decode_workspace_size(attn=structs[0][3], index=structs[0][2], compress_kv=structs[0][0],
                                              compress_keys=structs[0][1])
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    if args.fp8_only:
        peak, _ = measured_peaks()
        print(json.dumps({"fp8_keys": fp8_keys_step(m, _abi, t, variants, wl, args.steps, stream, peak)}),
              flush=True)
        return

    def step(s, j):
        ck, cq, ia, aa = structs[j]
        m.dsv4_csa_decode(ws, attn=aa, index=ia, compress_kv=ck, compress_keys=cq, stream=s)

    with torch.cuda.stream(stream):
        for i in range(max(3, args.warmup, N_INPUT_SETS)):
            step(stream, i % N_INPUT_SETS)
    stream.synchronize()
    launches = m.dsv4_last_launch_count()
    st, ew = m.dsv4_read_error_word(ws, stream)
    if ew:
        raise SystemExit(f"device error word {ew:#x} after warm-up")
    graphs = []
    for j in range(N_INPUT_SETS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                step(stream, j)
        graphs.append(g)
    # The timed steps: one graph holds one step per input set, in turn (a decode loop captures
    # many layer-steps in one graph, so no graph launch separates consecutive steps); K steps
    # are K // N_INPUT_SETS replays of it plus K % N_INPUT_SETS single-step graphs.
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g_all, stream=stream):
            for j in range(N_INPUT_SETS):
                step(stream, j)
    stream.synchronize()

    def run_steps(k):
        for _ in range(k // N_INPUT_SETS):
            g_all.replay()
        for i in range(k % N_INPUT_SETS):
            graphs[i].replay()

    clocks = ClockSampler(local)
    clocks.start()
    # soak: keep the GPU busy ~1 s so clocks settle and the sampler sees load
    with torch.cuda.stream(stream):
        t_end = time.time() + 1.0
        while time.time() < t_end:
            run_steps(48)
            stream.synchronize()
        run_steps(args.warmup)
    stream.synchronize()

    # ---- timed region: exactly K steps, each on the next input set
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        run_steps(args.steps)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, "cuda")
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    # the same K steps with one graph per step (a graph launch before every step), for reference
    with torch.cuda.stream(stream):
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(args.steps):
            graphs[i % N_INPUT_SETS].replay()
        f1.record(stream)
    torch.cuda.synchronize()
    ms_graph_per_step = max_over_ranks(f0.elapsed_time(f1) / args.steps, world, "cuda")
    if args.headline_only:
        clk = clocks.stop()
        if rank == 0:
            kb, gb, ob = step_bytes(wl)
            peak, _ = measured_peaks()
            print(json.dumps({"metric": METRIC, "value": job_throughput(B, world, ms), "unit": "tokens/s",
                              "ms_per_step": ms, "ms_per_step_one_graph_per_step": ms_graph_per_step,
                              "launches_per_step": launches, "config": workload_config(wl),
                              "step_frac": (kb + gb + ob) / (ms * 1e-3) / 1e9 / peak, "clocks": clk}), flush=True)
        return

    # ---- dominant kernel alone: the scoring launch, events on its stream
    score_ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(3):
            m.dsv4_index_score(t["q_I"], t["w"], t["keys"], t["n_comp"], t["scores"], score_ws,
                               ratio=wl.ratio, stream=stream)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for i, (a, b) in enumerate(evs):
            v = variants[i % N_INPUT_SETS]
            a.record(stream)
            m.dsv4_index_score(v["q_I"], v["w"], t["keys"], t["n_comp"], t["scores"], score_ws,
                               ratio=wl.ratio, stream=stream)
            b.record(stream)
    torch.cuda.synchronize()
    score_ms_isolated = statistics.mean(a.elapsed_time(b) for a, b in evs)
    # the launch's average duration over back-to-back calls (one event pair around all of them:
    # each call's launch overlaps the one before it, as in the step; each call still clears
    # its workspace header first)
    with torch.cuda.stream(stream):
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for i in range(args.steps):
            v = variants[i % N_INPUT_SETS]
            m.dsv4_index_score(v["q_I"], v["w"], t["keys"], t["n_comp"], t["scores"], score_ws,
                               ratio=wl.ratio, stream=stream)
        c1.record(stream)
    torch.cuda.synchronize()
    score_ms = c0.elapsed_time(c1) / args.steps

    # ---- end to end through the public API with host buffers (pinned), copies timed: each
    #      step's inputs from its pinned host arena (rotating over the input sets) into the
    #      device arena, and its outputs back into one pinned host arena, both by the library's
    #      copy kernel (dsv4_copy_async: the SMs load and store host memory over the
    #      chip-to-chip link; a copy-engine node for the 370 KB of inputs cost ~12 us a step)
    host_in = []
    for arena_j in arenas:
        h = torch.empty_like(arena_j, device="cpu").pin_memory()
        h.copy_(arena_j)
        host_in.append(h)
    host_out = torch.empty_like(arena_out, device="cpu").pin_memory()
    h2d = host_in[0].numel()
    d2h = host_out.numel()

    # the copies are captured with the step: one graph launch per step, copies included
    e2e_graphs = []
    for j in range(N_INPUT_SETS):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                m.dsv4_copy_async(arenas[0], host_in[j], stream=stream)
                step(stream, 0)
                m.dsv4_copy_async(host_out, arena_out, stream=stream)
        e2e_graphs.append(g)
    # as for the device-resident steps: one graph holds one step (copies included) per input set
    e2e_all = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(e2e_all, stream=stream):
            for j in range(N_INPUT_SETS):
                m.dsv4_copy_async(arenas[0], host_in[j], stream=stream)
                step(stream, 0)
                m.dsv4_copy_async(host_out, arena_out, stream=stream)
    stream.synchronize()

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_graphs[i % N_INPUT_SETS].replay()
        e2e_all.replay()
        stream.synchronize()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps // N_INPUT_SETS):
            e2e_all.replay()
        for i in range(args.steps % N_INPUT_SETS):
            e2e_graphs[i].replay()
        f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / args.steps, world, "cuda")
    if not torch.equal(host_out, arena_out.cpu()):
        raise SystemExit("the end-to-end step's host copy of the outputs differs from the device's")
    if not torch.equal(arenas[0].cpu(), host_in[(args.steps % N_INPUT_SETS or N_INPUT_SETS) - 1]):
        raise SystemExit("the end-to-end step's device copy of the inputs differs from the host's")
    clk = clocks.stop()
    # the end-to-end graphs wrote the last set's inputs into the first arena: put it back
    arenas[0].copy_(host_in[0])

    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    kb, gb, ob = step_bytes(wl)
    sb, side = scorer_bytes(wl)
    score_gbs = sb / (score_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": job_throughput(B, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl),
        "timing": ("one CUDA graph holding one step per input set (8 steps, the input sets in turn; no graph "
                   "launch between consecutive steps, as in a decode loop capturing many layer-steps), "
                   "replayed K // 8 times plus K % 8 single-step graphs; CUDA events around the K steps"),
        "ms_per_step_one_graph_per_step": ms_graph_per_step,
        "roofline": {"bound": "hbm", "kernel": "index_score_kernel",
                     "scope": "the step's dominant kernel alone (per-kernel figure; the whole step is "
                              "step_roofline)",
                     "achieved": score_gbs, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": score_gbs / peak, "traffic": profile_traffic(), "bytes_per_launch": sb,
                     "side_bytes_per_launch": side, "ms_per_launch": score_ms,
                     "timing": "CUDA events around K back-to-back launches (each with its header clear)",
                     "ms_per_launch_isolated": score_ms_isolated},
        "step_roofline": {"bytes": kb + gb + ob, "keys": kb, "gathered": gb, "outputs": ob,
                          "achieved": (kb + gb + ob) / (ms * 1e-3) / 1e9, "peak": peak,
                          "frac": (kb + gb + ob) / (ms * 1e-3) / 1e9 / peak, "unit": "GB/s"},
        "e2e": {"value": job_throughput(B, world, e2e_ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies": ("every step, in the step's stream and inside the timed region: its inputs from "
                           "pinned host memory into the device arena, the step, its outputs back into "
                           "pinned host memory, both copies by the library's copy kernel (dsv4_copy_async); "
                           "no overlap between steps")},
        "gpu_launches": launches * args.steps, "launches_per_step": launches,
        "clocks": clk,
    }
    if world == 1:
        line["prefill_scoring"] = prefill_scoring(m, args.steps)
        line["prefill_attention"] = prefill_attention(m, args.steps)
        line["fp8_keys"] = fp8_keys_step(m, _abi, t, variants, wl, args.steps, stream, peak)
        line["fp8_keys_mixed_kv"] = fp8_keys_step(m, _abi, t, variants, wl, args.steps, stream, peak,
                                                  mixed_kv=True)
        line["compressor_us"] = compressor_time(m, t, wl, args.steps, stream)
        line["other_decode_workloads"] = [decode_step_at(m, _abi, c, args.steps, peak) for c in (1, 2)]
    if world == 1 and not args.no_cpu_baseline:
        x0 = make_inputs(wl, batch=1)
        line["cpu_baseline"] = cpu_baseline(wl, x0)
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.decode_workload is not None:
        import torch
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA device")
        import __graft_entry__
        __graft_entry__.build()
        import compressed_sparse_attention_08_gb300 as m
        from compressed_sparse_attention_08_gb300 import _abi
        peak, _ = measured_peaks()
        print(json.dumps(decode_step_at(m, _abi, args.decode_workload, args.steps, peak)), flush=True)
    elif args.prefill_only:
        import torch
        if not torch.cuda.is_available():
            raise SystemExit("bench.py needs a CUDA device")
        import __graft_entry__
        __graft_entry__.build()
        import compressed_sparse_attention_08_gb300 as m
        print(json.dumps({"prefill_scoring": prefill_scoring(m, args.steps),
                          "prefill_attention": prefill_attention(m, args.steps)}), flush=True)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
