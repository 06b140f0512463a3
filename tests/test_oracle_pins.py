"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each check is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, an off-by-one exponent, a wrong
rounding direction, a misplaced row) fails at least one of them:
  * number formats against torch's float8_e4m3fn / bfloat16 casts;
  * the UE8M0 exponent rule against exact rational arithmetic (fractions);
  * RoPE against exact hand-computed cases and special angles;
  * whole records and their placement against the hand-derived golden file;
  * the gather against an exhaustive code x scale table decoded by torch;
  * brute force over tiny caches; closed-form error bounds; byte identities.
"""
from __future__ import annotations

import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from golden_parse import GOLDEN, load_worked, worked_inputs

SENTINEL = 0xA5


# --------------------------------------------------------------------------------
# number formats
# --------------------------------------------------------------------------------

def test_e4m3_decode_all_codes_match_torch(oracle_mod):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_mod.e4m3_value(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan], got[~nan])
    # signed zero
    assert math.copysign(1.0, got[0x80]) == -1.0


def _e4m3_probe_values() -> np.ndarray:
    pos = torch.arange(0, 0x7F, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    v = pos.to(torch.float64).numpy()                   # all finite non-negative values
    mids = (v[:-1] + v[1:]) / 2                         # every rounding boundary (exact)
    f32 = np.float32
    around = np.concatenate([np.nextafter(mids.astype(f32), f32(np.inf)),
                             np.nextafter(mids.astype(f32), f32(-np.inf))])
    rng = np.random.default_rng(1)
    rand = rng.uniform(0, 448, 20000).astype(np.float32)
    tiny = np.array([2.0 ** -10, 2.0 ** -11, 1e-30, 1e-40, 0.0], np.float32)
    allv = np.concatenate([v, mids, around, rand, tiny]).astype(np.float32)
    allv = allv[allv <= 448]
    return np.concatenate([allv, -allv]).astype(np.float32)


def test_e4m3_encode_matches_torch_at_every_boundary(oracle_mod):
    vals = _e4m3_probe_values()
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle_mod.e4m3_encode(float(x)) for x in vals], np.uint8)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(vals[i]), hex(ref[i]), hex(got[i])) for i in bad[:10]]


def test_e4m3_encode_saturates_and_keeps_sign(oracle_mod):
    # satfinite: anything at or beyond the largest finite value maps to +-448
    for y in (448.0, 449.0, 464.0, 480.0, 1e6, 3.0e38):
        assert oracle_mod.e4m3_encode(y) == 0x7E
        assert oracle_mod.e4m3_encode(-y) == 0xFE
    assert oracle_mod.e4m3_encode(-0.0) == 0x80
    assert oracle_mod.e4m3_encode(-1e-30) == 0x80
    assert oracle_mod.e4m3_encode(0.0) == 0x00


def test_bf16_decode_all_patterns_match_torch(oracle_mod):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_mod.bf16_value(b) for b in range(65536)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])


def test_bf16_encode_matches_torch(oracle_mod):
    rng = np.random.default_rng(2)
    raw = rng.integers(0, 2 ** 32, 40000, dtype=np.uint64).astype(np.uint32)
    vals = raw.view(np.float32)
    vals = vals[np.isfinite(vals)]
    # exact ties: bf16 value + half an ulp, in normal and subnormal ranges
    ties = (np.arange(0x0001, 0x7F7F, 97, dtype=np.uint32) << 16 | 0x8000).view(np.float32)
    extra = np.array([0.0, -0.0, 1e-45, -1e-45, 1e-39, 3.39e38, 3.4e38], np.float32)
    vals = np.concatenate([vals, ties, -ties, extra])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.bf16_encode(float(x)) for x in vals], np.uint16)
    bad = np.nonzero(ref != got)[0]
    assert bad.size == 0, [(float(vals[i]), hex(ref[i]), hex(got[i])) for i in bad[:10]]
    assert oracle_mod.bf16_encode(float("nan")) == 0x7FC0
    assert oracle_mod.bf16_encode(float("inf")) == 0x7F80


# --------------------------------------------------------------------------------
# UE8M0 exponent: ceil(log2(amax / 448)) clamped to [-127, 127], + 127
# --------------------------------------------------------------------------------

def _exact_scale_byte(a: float) -> int:
    if a == 0:
        return 0
    r = Fraction(a) / 448
    e = r.numerator.bit_length() - r.denominator.bit_length()
    while Fraction(2) ** e < r:
        e += 1
    while Fraction(2) ** (e - 1) >= r:
        e -= 1
    return min(max(e, -127), 127) + 127


def test_scale_byte_exhaustive_over_bf16_amax(oracle_mod):
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # all non-negative finite bf16
    vals = (bits << 16).view(np.float32)
    got = [oracle_mod.ue8m0_byte(float(v)) for v in vals]
    ref = [_exact_scale_byte(float(v)) for v in vals]
    bad = [(float(v), r, g) for v, r, g in zip(vals, ref, got) if r != g]
    assert not bad, bad[:10]


def test_scale_byte_random_fp32_and_boundaries(oracle_mod):
    rng = np.random.default_rng(3)
    raw = rng.integers(0, 0x7F800000, 20000, dtype=np.uint64).astype(np.uint32)
    vals = list(raw.view(np.float32))
    # boundaries 448 * 2^k and their fp32 neighbours
    for k in range(-140, 120):           # 448 * 2^119 = 1.75 * 2^127 is the largest in fp32
        b = np.float32(448.0 * 2.0 ** k)
        vals += [b, np.nextafter(b, np.float32(0)), np.nextafter(b, np.float32(np.inf))]
    for v in vals:
        assert oracle_mod.ue8m0_byte(float(v)) == _exact_scale_byte(float(v)), float(v)
    # closed-form spot values
    assert oracle_mod.ue8m0_byte(448.0) == 127
    assert oracle_mod.ue8m0_byte(450.0) == 128
    assert oracle_mod.ue8m0_byte(1.0) == 119
    assert oracle_mod.ue8m0_byte(0.0) == 0
    assert oracle_mod.ue8m0_byte(1e-40) == 0
    assert oracle_mod.ue8m0_byte(3.3e38) == 247


# --------------------------------------------------------------------------------
# RoPE pair
# --------------------------------------------------------------------------------

def test_rope_special_angles(oracle_mod):
    rng = np.random.default_rng(4)
    for e, o in rng.standard_normal((200, 2)).astype(np.float32):
        assert oracle_mod.rope_pair(e, o, 1.0, 0.0) == (e, o)          # identity
        eo, oo = oracle_mod.rope_pair(e, o, 0.0, 1.0)                  # quarter turn
        assert (eo, oo) == (-o, e)
        eo, oo = oracle_mod.rope_pair(e, o, -1.0, 0.0)                 # half turn
        assert (eo, oo) == (-e, -o)


def test_rope_hand_computed():
    import oracle
    assert oracle.rope_pair(3.0, 5.0, 0.5, 0.75) == (-2.25, 4.75)
    # each product rounded to fp32 before the sum (no fused multiply-add):
    # e*c = 1 + 2^-11 + 2^-24 rounds (tie, even) to 1 + 2^-11; minus 1 -> 2^-11.
    # A fused e*c - o*s would keep the 2^-24 term.
    e = 1.0 + 2.0 ** -12
    eo, oo = oracle.rope_pair(e, 1.0, e, 1.0)
    assert eo == 2.0 ** -11
    assert oo == 2.0 + 2.0 ** -11


def test_rope_matches_float32_evaluation(oracle_mod):
    rng = np.random.default_rng(5)
    v = rng.standard_normal((2000, 4)).astype(np.float32)
    for e, o, c, s in v:
        f = np.float32
        ref_e = f(f(e * c) - f(o * s))
        ref_o = f(f(o * c) + f(e * s))
        assert oracle_mod.rope_pair(e, o, c, s) == (ref_e, ref_o)


# --------------------------------------------------------------------------------
# byte identities and page geometry
# --------------------------------------------------------------------------------

def test_record_identities(oracle_mod):
    assert sum(oracle_mod.record_rows(528)) == 528 == 512 + 16
    assert sum(oracle_mod.record_rows(584)) == 584 == 448 + 128 + 8
    assert oracle_mod.page_stride(528, 64) == 33792 == 66 * 512
    assert oracle_mod.page_stride(584, 64) == 37440 == 65 * 576
    for bs in range(32, 1025, 32):
        assert oracle_mod.page_stride(528, bs) % 512 == 0
        assert oracle_mod.page_stride(528, bs) == bs * 528   # no padding when bs % 32 == 0
        assert oracle_mod.page_stride(584, bs) % 576 == 0
        assert 0 <= oracle_mod.page_stride(584, bs) - bs * 584 < 576


# --------------------------------------------------------------------------------
# hand-derived golden records
# --------------------------------------------------------------------------------

def _check_golden_insert(oracle_mod, w, record):
    kv, slots, pos, csc = worked_inputs(w)
    ps, expects = w.records[record]
    cache = np.full(w.num_pages * ps, SENTINEL, np.uint8)
    err = oracle_mod.insert(kv, cache, record, w.block_size, w.num_pages, ps, slots, pos, csc,
                            compress_ratio=w.compress_ratio, sanitize_nans=w.sanitize,
                            fp8_scale=w.fp8_scale.get(record))
    assert err == w.errors
    touched = np.zeros(cache.size, bool)
    for e in expects:
        D, S = e.data.size, e.scale.size
        got_d = cache[e.data_offset:e.data_offset + D]
        got_s = cache[e.scale_offset:e.scale_offset + S]
        assert np.array_equal(got_d, e.data), (record, e.token, np.nonzero(got_d != e.data))
        assert np.array_equal(got_s, e.scale), (record, e.token, got_s)
        touched[e.data_offset:e.data_offset + D] = True
        touched[e.scale_offset:e.scale_offset + S] = True
    assert (cache[~touched] == SENTINEL).all()


@pytest.mark.parametrize("record", [528, 584])
def test_golden_worked_records(oracle_mod, record):
    _check_golden_insert(oracle_mod, load_worked(), record)


@pytest.mark.parametrize("record", [528, 584])
def test_golden_compressed_records(oracle_mod, record):
    """Compress ratio 4 with NaN sanitising: group boundaries, the group's first
    cos/sin row (decoy rows at the tokens' own positions), NaN -> 0, infinite block
    maxima (byte 254, +-inf -> +-448), error bits."""
    w = load_worked(GOLDEN / "worked_compressed.txt")
    assert w.compress_ratio == 4 and w.sanitize
    _check_golden_insert(oracle_mod, w, record)


@pytest.mark.parametrize("record", [1024, 512])
def test_golden_full_cache_rows(oracle_mod, record):
    """bf16 and fp8 (scale 0.5) cache rows and their gathers, derived by hand."""
    w = load_worked(GOLDEN / "worked_full_caches.txt")
    _check_golden_insert(oracle_mod, w, record)
    kv, slots, pos, csc = worked_inputs(w)
    ps, _ = w.records[record]
    cache = np.full(w.num_pages * ps, SENTINEL, np.uint8)
    oracle_mod.insert(kv, cache, record, w.block_size, w.num_pages, ps, slots, pos, csc,
                      fp8_scale=w.fp8_scale.get(record))
    idx, expect = w.gathers[record]
    out, err = oracle_mod.gather(cache, record, w.block_size, w.num_pages, ps, idx,
                                 fp8_scale=w.fp8_scale.get(record))
    assert err == 0
    assert np.array_equal(out.astype(np.int64), expect)


@pytest.mark.parametrize("record", [528, 584])
def test_golden_gather(oracle_mod, record):
    w = load_worked()
    kv, slots, pos, csc = worked_inputs(w)
    ps, _ = w.records[record]
    cache = np.full(w.num_pages * ps, SENTINEL, np.uint8)
    oracle_mod.insert(kv, cache, record, w.block_size, w.num_pages, ps, slots, pos, csc)
    idx, expect = w.gathers[record]
    out, err = oracle_mod.gather(cache, record, w.block_size, w.num_pages, ps, idx)
    assert err == 0
    assert np.array_equal(out.astype(np.int64), expect)


def test_golden_all_ones_row(oracle_mod):
    # all-ones row at an identity angle: amax 1 -> byte 0x77, 1 * 2^8 = 256 -> 0x78
    kv = np.full(512, 0x3F80, np.uint16)
    csc = np.zeros(64, np.float32)
    csc[:32] = 1.0
    d, s = oracle_mod.encode(528, kv, csc)
    assert (d == 0x78).all() and (s == 0x77).all()
    d, s = oracle_mod.encode(584, kv, csc)
    assert (d[:448] == 0x78).all()
    assert (d[448:].reshape(-1, 2) == [0x80, 0x3F]).all()
    assert list(s) == [0x77] * 7 + [0x00]


# --------------------------------------------------------------------------------
# gather: exhaustive (code, scale) table
# --------------------------------------------------------------------------------

def _torch_decode(codes: np.ndarray, scale_bytes: np.ndarray) -> np.ndarray:
    """bf16 bits of e4m3(code) * 2^(byte - 127), computed with torch casts.
    The product is exact in fp32 (4 significant bits, exponent >= -136), so a
    single fp32 -> bf16 rounding gives the correctly rounded result."""
    v = torch.from_numpy(codes.astype(np.uint8)).view(torch.float8_e4m3fn).to(torch.float64)
    sc = torch.pow(torch.tensor(2.0, dtype=torch.float64),
                   torch.from_numpy(scale_bytes.astype(np.float64)) - 127)
    sc[torch.from_numpy(scale_bytes == 255)] = float("nan")
    p = (v * sc).to(torch.float32)
    out = p.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    out[np.isnan(p.numpy())] = 0x7FC0
    return out


def exhaustive_v41_cache():
    """128 records (bs 64, 2 pages): block k = 16*r + b has scale byte k % 256 and
    codes 32*(k // 256) + 0..31, so every (code, scale) pair occurs once."""
    bs, P = 64, 2
    ps = 64 * 528
    cache = np.zeros(P * ps, np.uint8)
    for r in range(128):
        page, row = divmod(r, bs)
        base = page * ps
        for b in range(16):
            k = 16 * r + b
            cache[base + row * 512 + 32 * b: base + row * 512 + 32 * b + 32] = \
                np.arange(32) + 32 * (k // 256)
            cache[base + bs * 512 + row * 16 + b] = k % 256
    return cache, bs, P, ps


def test_gather_exhaustive_code_scale_table(oracle_mod):
    cache, bs, P, ps = exhaustive_v41_cache()
    idx = np.arange(128, dtype=np.int32)
    out, err = oracle_mod.gather(cache, 528, bs, P, ps, idx)
    assert err == 0
    codes = np.zeros((128, 512), np.uint8)
    scales = np.zeros((128, 512), np.uint8)
    for r in range(128):
        for b in range(16):
            k = 16 * r + b
            codes[r, 32 * b:32 * b + 32] = np.arange(32) + 32 * (k // 256)
            scales[r, 32 * b:32 * b + 32] = k % 256
    ref = _torch_decode(codes, scales)
    bad = np.nonzero(ref != out)
    assert bad[0].size == 0, list(zip(codes[bad][:8], scales[bad][:8], ref[bad][:8], out[bad][:8]))
    pairs = set(zip(codes.reshape(-1).tolist(), scales.reshape(-1).tolist()))
    assert len(pairs) == 65536


def test_gather_invalid_and_out_of_range(oracle_mod):
    cache, bs, P, ps = exhaustive_v41_cache()
    idx = np.array([-1, 128, -5, 0], np.int32)
    out, err = oracle_mod.gather(cache, 528, bs, P, ps, idx)
    assert err == oracle_mod.ERR_INDEX
    assert (out[:3] == 0).all()
    assert (out[3] != 0).any()


# --------------------------------------------------------------------------------
# brute force over tiny caches
# --------------------------------------------------------------------------------

@pytest.mark.parametrize("record", [528, 584])
def test_bruteforce_tiny_slot_patterns(oracle_mod, record):
    bs, P = 32, 2
    ps = oracle_mod.page_stride(record, bs)
    D, S = oracle_mod.record_rows(record)
    rng = np.random.default_rng(6)
    max_pos = 16
    csc = rng.standard_normal((max_pos, 64)).astype(np.float32)
    choices = [-1, 0, 1, 31, 32, 63]
    n = 0
    for T in (1, 2, 3):
        for slots in itertools.product(choices, repeat=T):
            valid = [s for s in slots if s >= 0]
            if len(set(valid)) != len(valid):
                continue                   # duplicate slots are out of contract
            kv = (rng.standard_normal((T, 512)).astype(np.float32))
            kvb = torch.from_numpy(kv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            pos = rng.integers(0, max_pos, T)
            cache = np.full(P * ps, SENTINEL, np.uint8)
            err = oracle_mod.insert(kvb, cache, record, bs, P, ps, np.array(slots), pos, csc)
            assert err == 0
            expect = np.full(P * ps, SENTINEL, np.uint8)
            for t, s in enumerate(slots):
                if s < 0:
                    continue
                d, sc = oracle_mod.encode(record, kvb[t], csc[pos[t]])
                page, row = divmod(s, bs)
                expect[page * ps + row * D: page * ps + row * D + D] = d
                expect[page * ps + bs * D + row * S: page * ps + bs * D + row * S + S] = sc
            assert np.array_equal(cache, expect), (T, slots)
            n += 1
    assert n > 100


def test_insert_out_of_range_sets_error_and_writes_nothing(oracle_mod):
    bs, P = 32, 2
    ps = oracle_mod.page_stride(528, bs)
    csc = np.ones((4, 64), np.float32)
    kv = np.full((3, 512), 0x3F80, np.uint16)
    cache = np.full(P * ps, SENTINEL, np.uint8)
    err = oracle_mod.insert(kv, cache, 528, bs, P, ps, np.array([64, 5, -1]),
                            np.array([0, 4, 0]), csc)
    assert err == oracle_mod.ERR_SLOT | oracle_mod.ERR_POS
    assert (cache == SENTINEL).all()


# --------------------------------------------------------------------------------
# round-trip error bound (closed form)
# --------------------------------------------------------------------------------

@pytest.mark.parametrize("record", [528, 584])
def test_roundtrip_error_bound(oracle_mod, record):
    rng = np.random.default_rng(7)
    T = 64
    x = (rng.standard_t(3, (T, 512)) * rng.uniform(1e-3, 1e3, (T, 1))).astype(np.float32)
    kv = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xf = torch.from_numpy(kv.view(np.int16)).view(torch.bfloat16).double().numpy()
    csc = np.zeros((1, 64), np.float32)
    ang = rng.uniform(0, 2 * np.pi, 32)
    csc[0, :32], csc[0, 32:] = np.cos(ang), np.sin(ang)
    blk = 32 if record == 528 else 64
    nq = 512 if record == 528 else 448
    for t in range(T):
        d, s = oracle_mod.encode(record, kv[t], csc[0])
        back = oracle_mod.decode(record, d, s)
        xb = torch.from_numpy(back.view(np.int16)).view(torch.bfloat16).double().numpy()
        # rotated reference: the fp32 rotation (pinned above) of the bf16 input
        xr = xf[t].astype(np.float32).copy()
        for j in range(32):
            xr[448 + 2 * j], xr[449 + 2 * j] = oracle_mod.rope_pair(
                xr[448 + 2 * j], xr[449 + 2 * j], csc[0, j], csc[0, 32 + j])
        xr = xr.astype(np.float64)
        for b in range(nq // blk):
            seg = slice(b * blk, (b + 1) * blk)
            amax = np.abs(xr[seg]).max()
            e = int(s[b]) - 127
            err = np.abs(xr[seg] - xb[seg]).max()
            assert err <= 2.0 ** -3 * amax
            assert err <= 16 * 2.0 ** e          # half an e4m3 step in the top binade
        if record == 584:
            tail = torch.from_numpy(xr[448:].astype(np.float32)).to(torch.bfloat16).double().numpy()
            assert np.array_equal(xb[448:], tail)
