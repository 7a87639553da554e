"""The seeded input generators: shapes, determinism, page assignment, poison."""

import numpy as np

import workloads as wl


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38, 1e-40], dtype=np.float32)
    bits = wl.f32_to_bf16_bits(x)
    back = wl.bf16_bits_to_f32(bits)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7: ties to even -> 1.0
    assert back[0] == 1.0 and back[1] == 1.0
    # 1 + 3*2^-8 is halfway between 1+2^-7 and 1+2^-6: ties to even -> 1 + 2^-6
    assert back[2] == np.float32(1.015625)
    assert back[3] == -2.5
    assert np.isfinite(back[4])


def test_tiny_shapes_and_contiguous_pages():
    w = wl.tiny()
    assert w.q.shape == (2, 4, 128) and w.q.dtype == np.uint16
    assert list(w.num_blocks) == [8, 6]
    assert list(w.block_table[0, :8]) == list(range(8))
    assert list(w.block_table[1, :6]) == list(range(8, 14))
    assert w.index_k_bytes == (1000 + 700) * 128 * 2 == 435200


def test_generators_are_deterministic():
    a, b = wl.decode_point(), wl.decode_point()
    for x, y in [(a.q, b.q), (a.pool, b.pool), (a.block_table, b.block_table)]:
        np.testing.assert_array_equal(x, y)
    assert a.index_k_bytes == 35635200


def test_pages_are_not_shared_and_in_range():
    for w in (wl.decode_point(), wl.ragged(), wl.ragged(permute_rows=True)):
        used = []
        for b, nb in enumerate(w.num_blocks):
            row = w.block_table[b, :nb]
            assert np.all((row >= 0) & (row < w.num_pages))
            assert np.all(w.block_table[b, nb:] == -1)
            used.extend(row.tolist())
        assert len(used) == len(set(used))


def test_ragged_lengths():
    w = wl.ragged()
    assert list(w.seq_lens[:3]) == [131072, 0, 129]
    assert list(w.num_blocks[:3]) == [1024, 0, 2]
    assert w.index_k_bytes == 36995328


def test_partial_pages_are_poisoned():
    w = wl.decode_point()
    page = int(w.block_table[0, 67])
    tail = w.pool[page, 8700 % 128:]
    assert np.all(tail[0::2] == wl.BF16_NAN) and np.all(tail[1::2] == wl.BF16_BIG)


def test_adversarial_values_are_small_integers():
    w = wl.adversarial(batch=2)
    kv = wl.bf16_bits_to_f32(w.pool)
    assert np.all(kv == np.round(kv)) and kv.min() >= -9 and kv.max() <= 9
    qv = wl.bf16_bits_to_f32(w.q)
    assert set(np.unique(qv).tolist()) <= {-1.0, 0.0, 1.0}
    assert w.notes["biased_blocks"] == (64, 104)
