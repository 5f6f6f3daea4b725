"""Readings of the pages that a workload statement words differently, run both ways (CPU).

Causal visibility of compressed blocks in chunked prefill. The pages ("nvfp4-megamoe-kernel:
compare v0.1-e2e-working...v-c1-c2-c3-20260602", archived_plans/NEXT_STEPS.md "Issue 2") let
a query at position p see block j when the block's window ends at or before p:
(j + 1) r - 1 <= p, so (p + 1) // r blocks. The chunked-prefill workload's own wording ("a
query sees only blocks fully before its position") reads as (j + 1) r - 1 < p, so p // r
blocks. The library and the oracle take the pages' reading. This test runs the oracle both
ways on the chunked-prefill workload and states how many queries the other reading changes:
the two differ only for the block that ends exactly at p, i.e. for the queries with
(p + 1) % r == 0, one in r.
"""
from __future__ import annotations

import numpy as np

import oracle
from compressed_sparse_attention_08_gb300.workloads import WORKLOADS, make_inputs


def test_prefill_visibility_both_readings():
    wl = WORKLOADS[4]
    x = make_inputs(wl)
    p = x["q_pos"][0]
    n = int(x["n_comp"][0])
    pages = np.array([oracle.visible_entries(n, int(q), wl.ratio) for q in p])
    strict = np.minimum(n, p // wl.ratio)                 # blocks ending strictly before p
    assert np.array_equal(pages, np.minimum(n, (p + 1) // wl.ratio))
    differ = pages != strict
    assert differ.sum() == wl.new_tokens // wl.ratio == 512
    assert np.all((p[differ] + 1) % wl.ratio == 0) and np.all(pages[differ] == strict[differ] + 1)
    # the selections of a sample of those queries under both readings: the stricter reading is
    # the pages' reading at position p - 1 (p // r == ((p - 1) + 1) // r)
    sample = np.flatnonzero(differ)[::16]                 # 32 queries
    q_pos = x["q_pos"][:, sample]
    s_pages, nv_pages = oracle.index_scores(x["q_I"][:, sample], x["w"][:, sample], x["keys"], x["n_comp"],
                                            wl.ratio, q_pos=q_pos)
    s_strict, nv_strict = oracle.index_scores(x["q_I"][:, sample], x["w"][:, sample], x["keys"], x["n_comp"],
                                              wl.ratio, q_pos=q_pos - 1)
    assert np.array_equal(nv_pages[0], nv_strict[0] + 1)
    i_pages = oracle.topk(s_pages, nv_pages, wl.top_k)
    i_strict = oracle.topk(s_strict, nv_strict, wl.top_k)
    changed = 0
    for j in range(len(sample)):
        a, b = i_pages[0, j], i_strict[0, j]
        newest = nv_pages[0, j] - 1                        # the one extra block
        if not np.array_equal(a, b):
            changed += 1
            # the only possible change: the extra block enters and the k-th key of the
            # stricter reading leaves
            assert newest in a and newest not in b
            assert len(np.setxor1d(a, b)) == 2
    # printed for the record (pytest -s); the count is data-dependent, the structure is not
    print(f"prefill visibility: {differ.sum()} of {len(p)} queries see one more block under the "
          f"pages' reading; {changed} of {len(sample)} sampled such queries select differently")
