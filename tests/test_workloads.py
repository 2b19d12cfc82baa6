"""The seeded input generator: determinism, shapes, dtype round trips (no GPU)."""
import numpy as np

import workloads


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.005859375, -2.5, 3.0e-3, 65504.0], np.float32)
    b = workloads.f32_to_bf16_bits(x)
    back = workloads.bf16_bits_to_f32(b)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: rounds to even (1.0)
    assert back[1] == 1.0
    # 1 + 1.5 * 2^-8 rounds up to 1 + 2^-7
    assert back[2] == np.float32(1.0078125)
    assert back[3] == -2.5
    np.testing.assert_allclose(back, x, rtol=2 ** -8)


def test_tiny_workload_shapes_and_determinism():
    a = workloads.workload("tiny_gdn")
    b = workloads.workload("tiny_gdn")
    assert a.q.shape == (64, 1, 16) and a.v.shape == (64, 1, 16)
    assert a.g.shape == (64, 1) and a.pool.shape == (1, 1, 16, 16)
    assert a.chunk == 16 and a.qkv_dtype == "f32"
    for x, y in [(a.q, b.q), (a.k, b.k), (a.v, b.v), (a.beta, b.beta), (a.g, b.g)]:
        np.testing.assert_array_equal(x, y)
    assert np.all(a.g <= 0) and np.all((a.beta > 0) & (a.beta < 1))
    np.testing.assert_allclose(np.linalg.norm(a.k[:, 0], axis=-1), 1.0, rtol=1e-6)
    assert not np.any(a.pool)


def test_ragged_workload_lengths_and_slots():
    p = workloads.workload("ragged_gqa_kda")
    L = p.lengths
    assert len(L) == 8 and L.min() >= 64 and L.max() <= 8192
    assert len(set(p.slot_idx.tolist())) == 8 and p.slot_idx.max() < 64
    assert p.num_k_heads == 16 and p.num_v_heads == 32 and p.state_dtype == "bf16"
    assert p.pool.dtype == np.uint16 and p.pool.shape == (64, 32, 128, 128)
    assert p.g.shape == (p.total_tokens, 32, 128)


def test_subset_heads_keeps_groups():
    p = workloads.make_problem("t", num_seqs=2, lengths=[3, 4], num_k_heads=2, num_v_heads=4,
                               d=8, qkv_dtype="bf16", state_dtype="f32",
                               decay_kind="per_channel", chunk=16, zero_state=False, seed=3)
    s = workloads.subset_heads(p, [3])
    assert s.num_k_heads == 1 and s.num_v_heads == 2
    np.testing.assert_array_equal(s.v[:, 1], p.v[:, 3])
    np.testing.assert_array_equal(s.k[:, 0], p.k[:, 1])
