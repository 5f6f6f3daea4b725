"""dsv4_topk_noalloc: the top-k stage for callers that cannot allocate device memory.

Such callers (allocator hooks, serving loops that forbid cudaMalloc after start-up, plug-ins
handed only their buffers) get their scratch from a fixed per-GPU array inside the library.
This file runs last so that a failure here cannot hide the other tests of a run that stops
at the first failure. It compares the variant with the oracle's top-k (the definition: ties
to the lower index, ascending order, -1 padding) and with dsv4_topk, which uses a caller
workspace: the indices must be identical (integer output, bit-exact), on two calls in a
row with different scores, since the shared array keeps the previous call's contents.
"""
import numpy as np
import pytest

import oracle
from compressed_sparse_attention_08_gb300 import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_sparse_attention_08_gb300 import _build
    _build.build()


def _with_workspace(m, s, nv, k):
    idx = torch.empty(s.shape[0], k, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(m.dsv4_topk_workspace_size(s, nv, idx), 256), dtype=torch.uint8, device="cuda")
    m.dsv4_topk(s, nv, idx, ws)
    return idx


def test_noalloc_topk_matches_workspace_variant_twice():
    import compressed_sparse_attention_08_gb300 as m
    rows, max_comp, k = 4, 262144, 2048          # the long-row path: the scratch is really used
    for call, seed in enumerate((21, 22)):
        s_np = synth.normal_f32(seed, 18, (rows, max_comp), 0.0, 8.0)
        s_np[1] = np.round(s_np[1] * 2) / 2      # many ties
        n_np = np.array([max_comp, max_comp - 5, 100000, 1000 + call], np.int32)
        s = torch.from_numpy(s_np).cuda()
        nv = torch.from_numpy(n_np).cuda()
        want = _with_workspace(m, s, nv, k)
        got = torch.full((rows, k), 7, dtype=torch.int32, device="cuda")
        m.dsv4_topk_noalloc(s, nv, got)
        torch.cuda.synchronize()
        ref = oracle.topk(s_np, n_np, k)
        assert np.array_equal(got.cpu().numpy(), ref), f"call {call}: indices differ from the oracle's top-k"
        assert torch.equal(got, want), f"call {call}: indices differ from dsv4_topk"


def test_noalloc_topk_rejects_sizes_beyond_its_scratch():
    import compressed_sparse_attention_08_gb300 as m
    rows = 600                                    # 600 long rows need 33 KiB each: > 16 MiB
    s = torch.zeros(rows, 32769, dtype=torch.float32, device="cuda")
    nv = torch.full((rows,), 32769, dtype=torch.int32, device="cuda")
    idx = torch.empty(rows, 64, dtype=torch.int32, device="cuda")
    assert m.dsv4_topk_workspace_size(s, nv, idx) > (16 << 20)
    with pytest.raises(m.Dsv4Error) as e:
        m.dsv4_topk_noalloc(s, nv, idx)
    assert e.value.status == m.DSV4_ERR_INVALID_ARG
