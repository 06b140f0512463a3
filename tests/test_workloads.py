"""The seeded generators produce the stated shapes, rates and structure."""
import numpy as np

import workloads as W


def test_insert_v41_1024():
    c = W.insert_v41_1024()
    assert c.kv.shape == (1024, 512) and c.kv.dtype == np.uint16
    assert c.record == 528 and c.block_size == 64 and c.num_pages == 32
    assert c.csc.shape == (4096, 64) and c.csc.dtype == np.float32
    assert (c.slots == -1).sum() == 51
    v = c.slots[c.slots >= 0]
    assert len(set(v.tolist())) == v.size and v.max() < 2048
    assert c.positions.min() >= 0 and c.positions.max() < 4096
    # deterministic
    d = W.insert_v41_1024()
    assert np.array_equal(c.kv, d.kv) and np.array_equal(c.slots, d.slots)


def test_roundtrip_v41_16384():
    c = W.roundtrip_v41_16384()
    assert c.kv.shape == (16384, 512) and c.num_pages == 512
    assert (c.slots == -1).sum() == 1311
    assert np.array_equal(c.indices, c.slots.astype(np.int32))


def test_cos_sin_table_rows():
    t = W.cos_sin_table(8)
    assert np.array_equal(t[0, :32], np.ones(32, np.float32))
    assert np.array_equal(t[0, 32:], np.zeros(32, np.float32))
    assert np.allclose(t[:, :32] ** 2 + t[:, 32:] ** 2, 1.0, atol=1e-6)


def test_small_gather_sparse_structure():
    c = W.gather_v41_sparse(cache_tokens=1 << 16, queries=4, topk=256, min_ctx=1024)
    assert c.indices.shape == (4, 256) and c.indices.dtype == np.int32
    for q in range(4):
        v = c.indices[q][c.indices[q] >= 0]
        assert len(set(v.tolist())) == v.size
        assert v.max() < c.meta["context_lengths"][q]
    assert (c.indices == -1).sum() == round(0.03 * 1024)
    assert np.array_equal(c.slots, np.arange(1 << 16))


def test_compressed_insert_structure():
    c = W.compressed_insert("c", 3, 100, 4, skip_rate=0.0, nan_rate=0.01, inf_rate=0.01)
    assert c.kv.shape == (300, 512) and c.meta["compress_ratio"] == 4
    assert np.array_equal(c.positions, np.tile(np.arange(100), 3))
    # 25 groups per sequence, every token carries its group's slot
    assert np.array_equal(c.slots[:100], np.arange(100) // 4)
    assert c.slots.max() == 3 * 25 - 1 and c.num_pages == 2
    bits = c.kv.reshape(-1)
    exp, man = (bits >> 7) & 0xFF, bits & 0x7F
    assert ((exp == 0xFF) & (man != 0)).sum() == round(0.01 * bits.size)   # NaN
    assert ((exp == 0xFF) & (man == 0)).sum() == round(0.01 * bits.size)   # +-inf
    d = W.compressed_insert("d", 2, 50, 1, inf_rate=0.02, nonfinite_dims=448)
    exp = (d.kv >> 7) & 0xFF
    assert (exp[:, 448:] != 0xFF).all() and (exp[:, :448] == 0xFF).sum() == round(0.02 * d.kv.size)
    big = W.compressed_v41_r4_262144
    assert big.__doc__ and "65536" in big.__doc__
