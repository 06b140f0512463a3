"""CPU pins of the oracle's sparse decode logits (the dequant-gather fused into its
consumer): the oracle's gather (pinned on its own) followed by a float64 matrix product;
hand-built records give closed-form sums, one-hot queries reduce the logits to the
gather's values, invalid entries give -inf."""
from __future__ import annotations

import numpy as np
import torch

import workloads as W
from test_oracle_qside import bf16_bits


def _one_record_cache(record=528, bs=32, pages=2):
    ps = {528: bs * 528, 584: -(-bs * 584 // 576) * 576}[record]
    return np.zeros(pages * ps, np.uint8), ps


def test_logits_hand_built_records(oracle_mod):
    """Hand-built V4.1 records: slot 1 holds code 0x38 (1.0) in every dim with scale byte
    127 (x1), slot 2 code 0x40 (2.0) with byte 126 (x0.5), slot 3 code 0x38 in dims 0..31
    with byte 130 (x8) and 0xB8 (-1.0) elsewhere with byte 127.  A query of all 0.5
    (one head) then gives 0.5 * 512 = 256 for slots 1 and 2, and
    0.5 * (32 * 8 - 480 * 1) = -112 for slot 3; with sm_scale 0.25, a quarter of that."""
    cache, ps = _one_record_cache()
    bs = 32

    def put(slot, codes, scales):
        page, row = divmod(slot, bs)
        cache[page * ps + row * 512: page * ps + row * 512 + 512] = codes
        cache[page * ps + bs * 512 + row * 16: page * ps + bs * 512 + row * 16 + 16] = scales
    put(1, 0x38, 127)
    put(2, 0x40, 126)
    codes = np.full(512, 0xB8, np.uint8)
    codes[:32] = 0x38
    scales = np.full(16, 127, np.uint8)
    scales[0] = 130
    put(3, codes, scales)
    q = bf16_bits(np.full((1, 1, 512), 0.5))
    idx = np.array([[1, 2, 3, -1]], np.int32)
    logits, bound, err = oracle_mod.sparse_logits(q, cache, 528, bs, 2, ps, idx, 0.25)
    assert err == 0
    assert logits.tolist() == [[[64.0, 64.0, -28.0, -np.inf]]]
    assert bound[0, 0, :3].tolist() == [64.0, 64.0, 0.25 * 0.5 * (32 * 8 + 480)]


def test_logits_one_hot_queries_are_the_gather(oracle_mod):
    """Head h of a one-hot query (1 at dim d_h) reads dim d_h of every gathered row: the
    logits are the gather's values themselves (times sm_scale = 1)."""
    c = W.random_insert("lg", 300, 584, 64, 8, 512, 0.1, seed=3)
    ps = oracle_mod.page_stride(584, 64)
    cache = np.zeros(8 * ps, np.uint8)
    oracle_mod.insert(c.kv, cache, 584, 64, 8, ps, c.slots, c.positions, c.csc)
    dims = [0, 63, 64, 447, 448, 449, 511]
    q = np.zeros((2, len(dims), 512), np.float32)
    for h, d in enumerate(dims):
        q[:, h, d] = 1.0
    idx = np.stack([c.slots[:40], c.slots[40:80]]).astype(np.int32)
    idx[0, 5] = 8 * 64 + 3                                   # past the cache
    logits, _, err = oracle_mod.sparse_logits(bf16_bits(q), cache, 584, 64, 8, ps, idx, 1.0)
    assert err == oracle_mod.ERR_INDEX
    rows, _ = oracle_mod.gather(cache, 584, 64, 8, ps, idx.reshape(-1))
    vals = oracle_mod.bf16_to_float(rows).reshape(2, 40, 512)
    ok = (idx >= 0) & (idx < 8 * 64)
    for h, d in enumerate(dims):
        assert np.array_equal(logits[:, h, :][ok], vals[:, :, d][ok])
        assert np.isneginf(logits[:, h, :][~ok]).all()


def test_logits_bf16_values_and_linearity(oracle_mod):
    """bf16_to_float is the bf16 definition (against torch); doubling the query or
    sm_scale doubles the logits exactly."""
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    v = oracle_mod.bf16_to_float(bits)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(np.isnan(v), np.isnan(t)) and np.array_equal(v[~np.isnan(v)], t[~np.isnan(t)])
    c = W.random_insert("lg2", 100, 528, 32, 8, 64, 0.0, seed=4)
    ps = oracle_mod.page_stride(528, 32)
    cache = np.zeros(8 * ps, np.uint8)
    oracle_mod.insert(c.kv, cache, 528, 32, 8, ps, c.slots, c.positions, c.csc)
    rng = np.random.default_rng(5)
    qf = rng.standard_normal((1, 3, 512)).astype(np.float32)
    idx = c.slots[None, :20].astype(np.int32)
    a, _, _ = oracle_mod.sparse_logits(bf16_bits(qf), cache, 528, 32, 8, ps, idx, 0.7)
    b, _, _ = oracle_mod.sparse_logits(bf16_bits(2 * qf), cache, 528, 32, 8, ps, idx, 0.7)
    s, _, _ = oracle_mod.sparse_logits(bf16_bits(qf), cache, 528, 32, 8, ps, idx, 1.4)
    assert np.array_equal(b, 2 * a) and np.array_equal(s, 2 * a)
