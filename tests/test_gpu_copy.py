"""dsv4_copy_async: the SM copy between device memory and pinned host memory (GPU).

The copies must be byte-exact in every direction, must run after the kernel enqueued before
them on the stream (their source may be that kernel's output), and the library must refuse
memory the GPU cannot address (pageable host memory) with DSV4_ERR_INVALID_ARG.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from compressed_sparse_attention_08_gb300 import _build
    _build.build()


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, 294912, 3 << 20])
def test_copy_device_host_device(nbytes):
    import compressed_sparse_attention_08_gb300 as m
    g = torch.Generator().manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g)
    d0 = src.cuda()
    h = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    d1 = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    m.dsv4_copy_async(h, d0, stream=s)          # device -> pinned host
    m.dsv4_copy_async(d1, h, stream=s)          # pinned host -> device
    s.synchronize()
    assert torch.equal(h, src)
    assert torch.equal(d1.cpu(), src)


def test_copy_after_the_kernel_before_it():
    """The copy waits for the kernel before it: the top-k's indices, read back at once."""
    import compressed_sparse_attention_08_gb300 as m
    rows, n, k = 8, 3000, 64
    s_np = np.random.default_rng(5).standard_normal((rows, n)).astype(np.float32)
    sc = torch.from_numpy(s_np).cuda()
    nv = torch.full((rows,), n, dtype=torch.int32, device="cuda")
    idx = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(m.dsv4_topk_workspace_size(sc, nv, idx), 256), dtype=torch.uint8, device="cuda")
    host = torch.zeros(rows, k, dtype=torch.int32).pin_memory()
    st = torch.cuda.Stream()
    for _ in range(3):
        host.zero_()
        idx.fill_(-7)
        with torch.cuda.stream(st):
            m.dsv4_topk(sc, nv, idx, ws, stream=st)
            m.dsv4_copy_async(host, idx, stream=st)
        st.synchronize()
        want = np.sort(np.argsort(-s_np, axis=1, kind="stable")[:, :k], axis=1)
        assert np.array_equal(host.numpy(), want)


def test_copy_refuses_pageable_host_memory():
    import compressed_sparse_attention_08_gb300 as m
    from compressed_sparse_attention_08_gb300 import _abi
    buf = np.zeros(4096 + 16, np.uint8)
    off = (-buf.ctypes.data) % 16                  # a 16-byte aligned pageable address
    d = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    rc = _abi.library().dsv4_copy_async(ctypes.c_void_p(d.data_ptr()), ctypes.c_void_p(buf.ctypes.data + off), 4096,
                                        None)
    assert rc == m.DSV4_ERR_INVALID_ARG


def test_copy_captured_in_a_graph():
    """The copy captured in a CUDA graph after a kernel (the end-to-end step's form): each
    replay carries that replay's result to the pinned host buffer."""
    import compressed_sparse_attention_08_gb300 as m
    rows, n, k = 4, 2048, 32
    sc = torch.empty(rows, n, dtype=torch.float32, device="cuda")
    nv = torch.full((rows,), n, dtype=torch.int32, device="cuda")
    idx = torch.empty(rows, k, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(m.dsv4_topk_workspace_size(sc, nv, idx), 256), dtype=torch.uint8, device="cuda")
    host = torch.zeros(rows, k, dtype=torch.int32).pin_memory()
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    sc.copy_(torch.randn(rows, n, device="cuda"))
    with torch.cuda.stream(st):
        m.dsv4_topk(sc, nv, idx, ws, stream=st)              # (first call outside the capture)
        st.synchronize()
        with torch.cuda.graph(g, stream=st):
            m.dsv4_topk(sc, nv, idx, ws, stream=st)
            m.dsv4_copy_async(host, idx, stream=st)
    st.synchronize()
    for seed in range(3):
        s_np = np.random.default_rng(100 + seed).standard_normal((rows, n)).astype(np.float32)
        sc.copy_(torch.from_numpy(s_np).cuda())
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        want = np.sort(np.argsort(-s_np, axis=1, kind="stable")[:, :k], axis=1)
        assert np.array_equal(host.numpy(), want), f"replay {seed}"
