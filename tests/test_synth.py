"""The seeded input generator: both implementations give the same bits, draws are
reproducible, prefix-consistent and have the requested mean and spread (CPU only)."""
import numpy as np

from compressed_sparse_attention_08_gb300 import synth
from compressed_sparse_attention_08_gb300.workloads import WORKLOADS, make_inputs


def test_c_and_numpy_streams_identical():
    for seed, tid, n in ((0, 1, 4097), (3, 15, 1 << 18), (4, 9, 3)):
        assert np.array_equal(synth.normal_bf16(seed, tid, (n,)), synth.normal_bf16_numpy(seed, tid, (n,)))
    assert np.array_equal(synth.normal_f32(1, 10, (999,), 0.0, 0.125),
                          synth.normal_f32_numpy(1, 10, (999,), 0.0, 0.125))


def test_streams_distinct_and_moments():
    a = synth.bf16_bits_to_f32(synth.normal_bf16(2, 3, (1 << 20,), 1.0, 0.1)).astype(np.float64)
    assert abs(a.mean() - 1.0) < 1e-3 and abs(a.std() - 0.1) < 1e-3
    b = synth.normal_bf16(2, 4, (1000,))
    c = synth.normal_bf16(3, 3, (1000,))
    assert not np.array_equal(b, c)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 65504.0], np.float32)
    assert list(synth.f32_to_bf16_bits(x)) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x4780]


def test_workload_batch_prefix_consistent():
    wl = WORKLOADS[0]
    x = make_inputs(wl)
    assert x["C"].shape == (1, 1024, 128) and x["q_I"].shape == (1, 1, 8, 128)
    assert x["n_comp"][0] == 256 and x["win"].shape == (1, 128, 128)
    wl1 = WORKLOADS[1]
    full = synth.normal_bf16(wl1.seed, 12, (16, 1, 64, 512))
    part = make_inputs(wl1, batch=2)["q"]
    assert np.array_equal(full[:2], part)


def test_uniform_index_sets():
    idx = synth.uniform_index_sets(1, 17, 3, [10, 3, 0], 5)
    assert list(idx[1]) == sorted(idx[1][:3].tolist()) + [-1, -1]
    assert list(idx[2]) == [-1] * 5
    assert len(set(idx[0].tolist())) == 5 and idx[0].max() < 10


def test_step_input_variants():
    """The benchmark's rotating per-step inputs: variant 0 is the workload's own draw, other
    variants are different draws of the same shapes."""
    from compressed_sparse_attention_08_gb300.workloads import WORKLOADS, make_inputs, step_inputs
    wl = WORKLOADS[3]
    x = make_inputs(wl, batch=1)          # the first sequence of the full draw
    v0, v1 = step_inputs(wl, 0), step_inputs(wl, 1)
    for k, a in v0.items():
        assert np.array_equal(a[:1], x[k]), k
        assert v1[k].shape == a.shape and v1[k].dtype == a.dtype
        assert not np.array_equal(v1[k], a), k
