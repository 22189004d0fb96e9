"""The seeded generator: published splitmix64 values, determinism that does
not depend on the thread count, and the distributions the workloads ask for."""
import os

import numpy as np

import synth
from synth import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_outputs():
    vals = [int(l, 16) for l in open(os.path.join(GOLDEN, "splitmix64_seed0.txt"))
            if l.strip() and not l.startswith("#")]
    gamma = 0x9E3779B97F4A7C15
    assert [synth.splitmix64((k * gamma) & (2 ** 64 - 1)) for k in range(3)] == vals


def test_normal_is_deterministic_and_thread_independent():
    lib = synth.lib()
    a = np.empty(300_000, np.uint16)
    b = np.empty(300_000, np.uint16)
    lib.synth_normal_bf16(5, 77, a.size, 0.0, 1.0, a.ctypes.data, 1)
    lib.synth_normal_bf16(5, 77, b.size, 0.0, 1.0, b.ctypes.data, 7)
    assert np.array_equal(a, b)
    c = synth.normal_bf16(6, 77, 1000)
    assert not np.array_equal(a[:1000], c)


def test_normal_moments():
    x = synth.bf16_to_f32(synth.normal_bf16(0, 3, 400_000, 0.0, 0.02)).astype(np.float64)
    assert abs(x.mean()) < 2e-4 and abs(x.std() - 0.02) < 2e-4
    g = synth.bf16_to_f32(synth.normal_bf16(0, 4, 100_000, 1.0, 0.02)).astype(np.float64)
    assert abs(g.mean() - 1.0) < 1e-3


def test_kv_prefill_zero_beyond_context():
    ctx = np.array([3, 7], np.int32)
    kv = synth.kv_bf16(1, 9, 2, 2, 3, 8, 16, ctx)
    for b in range(2):
        assert not kv[:, b, :, ctx[b]:].any()
        assert np.count_nonzero(kv[:, b, :, :ctx[b]]) > 0.9 * kv[:, b, :, :ctx[b]].size


def test_uniform_range_and_ragged_contexts():
    u = synth.uniform_i32(0, 11, 50_000, 128, 4096)
    assert u.min() >= 128 and u.max() <= 4096 and len(set(u.tolist())) > 3000
    ctx = workloads.contexts("llama1b_b8_ragged")
    assert ctx.shape == (8,) and ctx.min() >= 128 and ctx.max() <= 4096
    assert workloads.max_ctx("llama1b_ctx1024") == 1152


def test_bf16_helpers_round_trip():
    x = np.array([1.0, -2.5, 3.140625, 1.00390625], np.float32)
    assert np.array_equal(synth.bf16_to_f32(synth.f32_to_bf16(x))[:3], x[:3])
    assert synth.f32_to_bf16(x)[3] == 0x3F80
