"""Pins of the oracle's compressed-KV insert (compress ratio, NaN sanitising) that do
not go through its own compressed code path:

  * a compressed insert writes exactly the records a plain insert writes for the
    group-boundary tokens alone, each placed at the group's first position (the
    pages' kernel text: write when (pos + 1) % R == 0, rotate with row pos // R * R);
  * sanitising changes nothing on NaN-free input;
  * a NaN in a NoPE dim is stored as a +0 there (plain insert of the same row with
    +0); a NaN in a RoPE pair zeroes both rotated values, which for non-negative
    cos/sin is the plain insert of the pair (0, 0);
  * the clamped scale rule on an infinite maximum (byte 254) and the saturating
    e4m3 cast of infinities.
The hand-derived records of tests/golden/worked_compressed.txt pin the rest.
"""
from __future__ import annotations

import itertools

import numpy as np
import pytest

import workloads as W

SENTINEL = 0xA5


def _cache(oracle_mod, record, bs, pages):
    ps = oracle_mod.page_stride(record, bs)
    return np.full(pages * ps, SENTINEL, np.uint8), ps


def _insert(oracle_mod, kv, record, bs, pages, slots, pos, csc, **kw):
    cache, ps = _cache(oracle_mod, record, bs, pages)
    err = oracle_mod.insert(kv, cache, record, bs, pages, ps, slots, pos, csc, **kw)
    return cache, err


@pytest.mark.parametrize("record", [528, 584])
@pytest.mark.parametrize("ratio", [1, 2, 3, 4, 128])
def test_compressed_is_plain_insert_of_boundary_tokens(oracle_mod, record, ratio):
    T, bs, pages, max_pos = 600, 32, 24, 700
    case = W.random_insert("cmp", T, record, bs, pages, max_pos, 0.1, seed=ratio,
                           outlier_rate=0.01)
    got, err = _insert(oracle_mod, case.kv, record, bs, pages, case.slots, case.positions,
                       case.csc, compress_ratio=ratio)
    assert err == 0
    boundary = (case.positions + 1) % ratio == 0
    group_row = case.positions - (ratio - 1)          # = pos // R * R at a boundary
    keep = boundary & (case.slots >= 0)
    ref, err2 = _insert(oracle_mod, case.kv[keep], record, bs, pages, case.slots[keep],
                        group_row[keep], case.csc)
    assert err2 == 0
    assert np.array_equal(got, ref)
    if ratio > 1:
        assert keep.sum() < (case.slots >= 0).sum()


@pytest.mark.parametrize("record", [528, 584])
def test_compressed_tiny_brute_force(oracle_mod, record):
    """Every ratio 1..3 over every position pattern of 3 tokens in [0, 6)."""
    bs, pages = 32, 2
    csc = W.cos_sin_table(6)
    rng = np.random.default_rng(7)
    kv = W.to_bf16_bits(rng.standard_normal((3, 512)).astype(np.float32))
    slots = np.array([1, 40, 17], np.int64)
    for ratio in (1, 2, 3):
        for pos in itertools.product(range(6), repeat=3):
            pos = np.array(pos, np.int64)
            got, err = _insert(oracle_mod, kv, record, bs, pages, slots, pos, csc,
                               compress_ratio=ratio)
            assert err == 0
            ref, _ = _insert(oracle_mod, kv, record, bs, pages, slots, pos, csc)  # plain
            ps = oracle_mod.page_stride(record, bs)
            D, S = oracle_mod.record_rows(record)
            for t in range(3):
                page, row = divmod(int(slots[t]), bs)
                dr = slice(page * ps + row * D, page * ps + row * D + D)
                sr = slice(page * ps + bs * D + row * S, page * ps + bs * D + row * S + S)
                if (pos[t] + 1) % ratio:
                    assert (got[dr] == SENTINEL).all() and (got[sr] == SENTINEL).all()
                else:
                    d, s = oracle_mod.encode(record, kv[t], csc[pos[t] // ratio * ratio])
                    assert np.array_equal(got[dr], d) and np.array_equal(got[sr], s)
                    if ratio == 1:
                        assert np.array_equal(got[dr], ref[dr])


def test_compressed_error_order(oracle_mod):
    bs, pages, record = 32, 2, 528
    csc = W.cos_sin_table(8)
    kv = np.full((5, 512), 0x3F80, np.uint16)
    slots = np.array([64, 3, 4, 5, 6], np.int64)
    pos = np.array([5, -1, 11, 5, 9], np.int64)   # R = 4: boundary at 3, 7, 11, ...
    _, err = _insert(oracle_mod, kv, record, bs, pages, slots, pos, csc, compress_ratio=4)
    # slot 64 is past the cache (1); pos -1 is negative (2); pos 11 is a boundary whose
    # row 8 is past the 8-row table (2); pos 5 and 9 are not boundaries
    assert err == 3
    _, err = _insert(oracle_mod, kv[3:], record, bs, pages, slots[3:], pos[3:], csc,
                     compress_ratio=4)
    assert err == 0
    with pytest.raises(ValueError):
        _insert(oracle_mod, kv, record, bs, pages, slots, pos, csc, compress_ratio=0)


@pytest.mark.parametrize("record", [528, 584])
def test_sanitize_is_identity_without_nan(oracle_mod, record):
    case = W.random_insert("san", 400, record, 32, 16, 300, 0.05, seed=3, dist="student_t3")
    a, _ = _insert(oracle_mod, case.kv, record, 32, 16, case.slots, case.positions, case.csc)
    b, _ = _insert(oracle_mod, case.kv, record, 32, 16, case.slots, case.positions, case.csc,
                   sanitize_nans=True)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("record", [528, 584])
def test_sanitize_nan_in_nope_dim_is_zero(oracle_mod, record):
    rng = np.random.default_rng(5)
    T = 64
    x = rng.standard_normal((T, 512)).astype(np.float32)
    zeroed = x.copy()
    for t in range(T):
        for d in rng.choice(448, size=1 + t % 5, replace=False):
            x[t, d] = np.nan
            zeroed[t, d] = 0.0
    csc = W.cos_sin_table(128)
    slots = np.arange(T, dtype=np.int64) * 3 % (16 * 32)
    pos = rng.integers(0, 128, T)
    a, _ = _insert(oracle_mod, W.to_bf16_bits(x), record, 32, 16, slots, pos, csc,
                   sanitize_nans=True)
    b, _ = _insert(oracle_mod, W.to_bf16_bits(zeroed), record, 32, 16, slots, pos, csc)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("record", [528, 584])
def test_sanitize_nan_in_rope_pair_zeroes_the_pair(oracle_mod, record):
    rng = np.random.default_rng(6)
    T = 64
    x = rng.standard_normal((T, 512)).astype(np.float32)
    zeroed = x.copy()
    for t in range(T):
        j = int(rng.integers(0, 32))
        x[t, 448 + 2 * j + (t & 1)] = np.nan      # even or odd member of the pair
        zeroed[t, 448 + 2 * j: 450 + 2 * j] = 0.0
    csc = rng.uniform(0.0, 1.0, (32, 64)).astype(np.float32)   # cos, sin >= 0
    slots = np.arange(T, dtype=np.int64)
    pos = rng.integers(0, 32, T)
    a, _ = _insert(oracle_mod, W.to_bf16_bits(x), record, 32, 4, slots, pos, csc,
                   sanitize_nans=True)
    b, _ = _insert(oracle_mod, W.to_bf16_bits(zeroed), record, 32, 4, slots, pos, csc)
    assert np.array_equal(a, b)


def test_infinite_maximum_and_saturation(oracle_mod):
    # ceil(log2(inf / 448)) = inf, clamped to 127 -> byte 254 (never the UE8M0 NaN 255)
    assert oracle_mod.ue8m0_byte(float("inf")) == 254
    assert oracle_mod.ue8m0_byte(3.3e38) == 247       # largest finite maxima stay at 247
    # the saturating cast maps +-inf to +-448
    assert oracle_mod.e4m3_encode(float("inf")) == 0x7E
    assert oracle_mod.e4m3_encode(float("-inf")) == 0xFE
