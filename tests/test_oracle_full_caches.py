"""Pins of the oracle's two plain KV-only cache formats (bf16 rows, fp8 e4m3 rows with
one fp32 scale) against library routines and hand values:

  * the rotation restated with numpy float32 (each product and sum separately
    rounded; numpy does not contract) then cast with torch: .to(bfloat16) for the
    bf16 cache, fp32 division by the scale then .to(float8_e4m3fn) for the fp8 cache
    (inputs kept inside +-448, where torch's cast is round-to-nearest-even);
  * the fp8 gather against torch: float8_e4m3fn -> fp32, fp32 product, -> bfloat16;
  * hand values for a scale that is not a power of two, saturation, and the scale
    checks (not a positive finite number -> nothing written, ERR_SCALE).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W

SENTINEL = 0xA5


def _rotate_f32(x: np.ndarray, csc_rows: np.ndarray) -> np.ndarray:
    x = x.astype(np.float32).copy()
    e, o = x[:, 448::2].copy(), x[:, 449::2].copy()
    c, s = csc_rows[:, :32], csc_rows[:, 32:]
    x[:, 448::2] = e * c - o * s
    x[:, 449::2] = o * c + e * s
    return x


def _case(T=200, seed=0, sigma=1.0):
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((T, 512)) * sigma).astype(np.float32)
    kv = W.to_bf16_bits(x)
    xf = torch.from_numpy(kv.view(np.int16)).view(torch.bfloat16).float().numpy()
    csc = W.cos_sin_table(512)
    pos = rng.integers(0, 512, T)
    slots = rng.permutation(8 * 32)[:T].astype(np.int64)
    return kv, xf, csc, pos, slots


def _rows(cache, record, ps, slots, bs=32):
    page, row = slots // bs, slots % bs
    start = page * ps + row * record
    return np.stack([cache[s:s + record] for s in start])


def test_bf16_cache_rows_match_torch_casts(oracle_mod):
    kv, xf, csc, pos, slots = _case()
    ps = oracle_mod.page_stride(1024, 32)
    cache = np.full(8 * ps, SENTINEL, np.uint8)
    assert oracle_mod.insert(kv, cache, 1024, 32, 8, ps, slots, pos, csc) == 0
    got = _rows(cache, 1024, ps, slots).view(np.uint16)
    ref = torch.from_numpy(_rotate_f32(xf, csc[pos])).to(torch.bfloat16).view(torch.int16)
    assert np.array_equal(got, ref.numpy().view(np.uint16))
    assert np.array_equal(got[:, :448], kv[:, :448])          # NoPE dims unchanged


@pytest.mark.parametrize("scale", [0.0078125, 0.37, 3.0, 1.0 / 3.0])
def test_fp8_cache_rows_match_torch_casts(oracle_mod, scale):
    kv, xf, csc, pos, slots = _case(sigma=0.7)
    xr = _rotate_f32(xf, csc[pos])
    # keep |x / scale| inside the finite e4m3 range: torch's cast does not saturate
    keep = np.abs(xr).max(axis=1) / scale < 440
    kv, xr, pos, slots = kv[keep], xr[keep], pos[keep], slots[keep]
    assert keep.sum() > 50
    ps = oracle_mod.page_stride(512, 32)
    cache = np.full(8 * ps, SENTINEL, np.uint8)
    assert oracle_mod.insert(kv, cache, 512, 32, 8, ps, slots, pos, csc,
                             fp8_scale=np.float32(scale)) == 0
    got = _rows(cache, 512, ps, slots)
    q = (torch.from_numpy(xr) / torch.tensor(np.float32(scale))).to(torch.float8_e4m3fn)
    assert np.array_equal(got, q.view(torch.uint8).numpy())


@pytest.mark.parametrize("scale", [0.5, 0.37, 3.0, 1e-3])
def test_fp8_gather_matches_torch(oracle_mod, scale):
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes & 0x7F) != 0x7F]                    # NaN codes checked below
    rows = np.resize(codes, (4, 512))
    ps = oracle_mod.page_stride(512, 32)
    cache = np.zeros(ps, np.uint8)
    cache[:4 * 512] = rows.reshape(-1)
    out, err = oracle_mod.gather(cache, 512, 32, 1, ps, np.array([0, 1, 2, 3, -1], np.int32),
                                 fp8_scale=np.float32(scale))
    assert err == 0
    v = torch.from_numpy(rows).view(torch.float8_e4m3fn).float() * torch.tensor(np.float32(scale))
    ref = v.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out[:4], ref)
    assert (out[4] == 0).all()
    cache[:2] = [0x7F, 0xFF]
    out, _ = oracle_mod.gather(cache, 512, 32, 1, ps, np.array([0], np.int32), fp8_scale=1.0)
    assert list(out[0, :2]) == [0x7FC0, 0x7FC0]


def test_fp8_hand_values(oracle_mod):
    """Scale 3: x = 1 -> fl32(1/3) = 0.3333333432...; e4m3 spacing 2^-5 in [0.25, 0.5)
    gives 10.67 steps -> 11 -> 0.34375 = 1.375*2^-2 -> E 5, M 3 -> 0x2B; read back
    0.34375 * 3 = 1.03125 (exact) -> bf16 0x3F84.  x = 1500 -> 500 -> saturates to
    448 = 0x7E; x = -1500 -> 0xFE."""
    kv = np.zeros((3, 512), np.uint16)
    kv[0, 0] = 0x3F80                                     # 1.0
    kv[1, 0] = W.to_bf16_bits(np.float32([1500.0]))[0]    # 1500 (exact in bf16)
    kv[2, 0] = W.to_bf16_bits(np.float32([-1500.0]))[0]
    csc = W.cos_sin_table(1)
    ps = oracle_mod.page_stride(512, 32)
    cache = np.zeros(ps, np.uint8)
    oracle_mod.insert(kv, cache, 512, 32, 1, ps, np.array([0, 1, 2]), np.zeros(3, np.int64),
                      csc, fp8_scale=3.0)
    assert cache[0] == 0x2B and cache[512] == 0x7E and cache[1024] == 0xFE
    out, _ = oracle_mod.gather(cache, 512, 32, 1, ps, np.array([0], np.int32), fp8_scale=3.0)
    assert out[0, 0] == 0x3F84


@pytest.mark.parametrize("scale", [0.0, -1.0, float("inf"), float("nan")])
def test_fp8_bad_scale_writes_nothing(oracle_mod, scale):
    kv, _, csc, pos, slots = _case(T=20)
    ps = oracle_mod.page_stride(512, 32)
    cache = np.full(8 * ps, SENTINEL, np.uint8)
    err = oracle_mod.insert(kv, cache, 512, 32, 8, ps, slots, pos, csc, fp8_scale=scale)
    assert err == oracle_mod.ERR_SCALE and (cache == SENTINEL).all()
    out, err = oracle_mod.gather(cache, 512, 32, 8, ps, slots[:4].astype(np.int32),
                                 fp8_scale=scale)
    assert err == oracle_mod.ERR_SCALE and (out == 0).all()


def test_full_cache_page_strides(oracle_mod):
    for bs in (16, 32, 48, 64):
        assert oracle_mod.page_stride(1024, bs) == bs * 1024
        assert oracle_mod.page_stride(512, bs) == bs * 512
