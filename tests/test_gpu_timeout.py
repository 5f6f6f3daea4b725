"""The bounded-wait path of the kernels, run on purpose and without any fault.

Every wait of a kernel on an asynchronous copy is bounded in time; when the limit runs out
the kernel records DSV4_EWORD_TIMEOUT, lets its own copies land, frees its tensor memory and
returns, so the call reports DSV4_ERR_TIMEOUT and the context stays usable. The library's
test control (dsv4_test_wait_fault) leaves one copy of the named kernel unissued and sets a
1 ms limit, so the wait for that copy runs out: a flag that nothing sets, no trap, no bad
address. After each such call, a normal call on the same workspace must return the oracle's
results: that also shows the timed-out launch released its tensor memory (a CTA that kept it
would leave the next kernel's allocation on that SM waiting).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from compressed_sparse_attention_08_gb300 import synth
from helpers import assert_bf16_close, dev, dev_bf16, host_bf16

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_sparse_attention_08_gb300 import _build
    _build.build()


@pytest.fixture
def m():
    import compressed_sparse_attention_08_gb300 as mod
    yield mod
    mod.dsv4_test_wait_fault(mod.DSV4_WAIT_FAULT_NONE, 0)


def test_wait_fault_control_rejects_bad_arguments(m):
    for which, us in ((3, 1000), (-1, 0), (1, 2000001)):
        with pytest.raises(m.Dsv4Error) as e:
            m.dsv4_test_wait_fault(which, us)
        assert e.value.status == m.DSV4_ERR_INVALID_ARG


def test_scorer_wait_times_out_then_recovers(m):
    """2 rows x 1,024 keys: every scoring CTA's first key stage is never loaded; the call
    ends with the timeout bit set, and the next normal call gives the oracle's top-k."""
    rng = np.random.default_rng(71)
    B, H, N, k = 2, 64, 1024, 64
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, 1, H, 128)).astype(np.float32))
    keys = synth.f32_to_bf16_bits(rng.standard_normal((B, N, 128)).astype(np.float32))
    w = (rng.standard_normal((B, 1, H)) / 8).astype(np.float32)
    n_comp = np.array([N, N - 100], np.int32)
    qd, wd, kd, nd = dev_bf16(q), dev(w), dev_bf16(keys), dev(n_comp)
    idx = torch.full((B, 1, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(m.dsv4_indexer_topk_workspace_size(qd, wd, kd, nd, idx, ratio=4), 256),
                     dtype=torch.uint8, device="cuda")
    m.dsv4_test_wait_fault(m.DSV4_WAIT_FAULT_SCORER_STAGE, 1000)
    m.dsv4_indexer_topk(qd, wd, kd, nd, idx, ws, ratio=4)
    m.dsv4_test_wait_fault(m.DSV4_WAIT_FAULT_NONE, 0)
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    assert ew & m.DSV4_EWORD_TIMEOUT, f"error word {ew:#x}: the wait did not run out"
    assert st == m.DSV4_ERR_TIMEOUT
    # the same workspace, a normal call: exact again
    m.dsv4_indexer_topk(qd, wd, kd, nd, idx, ws, ratio=4)
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    assert ew == 0 and st == m.DSV4_OK
    ref_s, nv = oracle.index_scores(q, w, keys, n_comp, 4)
    assert np.array_equal(idx.cpu().numpy(), oracle.topk(ref_s, nv, k))


def test_attention_wait_times_out_then_recovers(m):
    """The split-form attention (2 rows, 16 heads x 128 dims, 100 selected rows + a 28-row
    window): its query tile is never loaded; the call ends with the timeout bit set, and the
    next normal call matches the oracle."""
    rng = np.random.default_rng(72)
    B, H, D, N, k, W = 2, 16, 128, 300, 100, 28
    q = synth.f32_to_bf16_bits(rng.standard_normal((B, 1, H, D)).astype(np.float32))
    kv = synth.f32_to_bf16_bits(rng.standard_normal((B, N, D)).astype(np.float32))
    win = synth.f32_to_bf16_bits(rng.standard_normal((B, W, D)).astype(np.float32))
    sink = rng.standard_normal(H).astype(np.float32)
    n_comp = np.array([N, 250], np.int32)
    win_len = np.array([W, W], np.int32)
    idx = np.stack([np.sort(rng.choice(int(n), k, replace=False)) for n in n_comp]).astype(np.int32)
    idx = idx.reshape(B, 1, k)
    out = torch.empty(B, 1, H, D, dtype=torch.bfloat16, device="cuda")
    args = (dev_bf16(q), dev(sink), dev_bf16(kv), dev(n_comp), dev_bf16(win), dev(win_len), out)
    kw = dict(idx=dev(idx), window=W, ratio=4)
    ws = torch.empty(max(m.dsv4_sparse_attn_workspace_size(*args, **kw), 256), dtype=torch.uint8, device="cuda")
    m.dsv4_test_wait_fault(m.DSV4_WAIT_FAULT_ATTN_QUERY, 1000)
    m.dsv4_sparse_attn_decode(*args, ws, **kw)
    m.dsv4_test_wait_fault(m.DSV4_WAIT_FAULT_NONE, 0)
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    assert ew & m.DSV4_EWORD_TIMEOUT, f"error word {ew:#x}: the wait did not run out"
    assert st == m.DSV4_ERR_TIMEOUT
    m.dsv4_sparse_attn_decode(*args, ws, **kw)
    torch.cuda.synchronize()
    st, ew = m.dsv4_read_error_word(ws)
    assert ew == 0 and st == m.DSV4_OK
    _, ref, _ = oracle.sparse_attn(q, sink, kv, n_comp, idx, win, win_len, k, W, 4)
    assert_bf16_close(host_bf16(out), ref, "attention after a timed-out call")
