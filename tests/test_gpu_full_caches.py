"""GPU parity for the two plain KV-only caches (bf16 rows, fp8 e4m3 rows with one fp32
scale): kv_insert and kv_gather through the C ABI vs the CPU oracle, byte for byte over
the whole sentinel-filled backing buffer, with both insert kernels."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from golden_parse import GOLDEN, load_worked, worked_inputs
from helpers import (SENTINEL, assert_distinct_slots, bf16_from_bits, device_inputs,
                     first_mismatch, oracle_full_cache)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(params=["short", "staged", "stream"], autouse=True)
def insert_kernel_choice(request, gkr):
    """Run every insert test with each of the three insert kernels (register loads,
    shared-memory staging, streaming ring) regardless of the token count."""
    big = 1 << 62
    staged_min, stream_min = {"short": (big, big), "staged": (0, big),
                              "stream": (big, 0)}[request.param]
    with gkr.launch_policy(insert_staged_min=staged_min, insert_stream_min=stream_min):
        yield request.param


def _scale_t(scale):
    return None if scale is None else torch.tensor([scale], dtype=torch.float32, device=DEV)


def _insert(gkr, oracle_mod, case, record, scale=None, pad_units=0):
    """GPU and oracle insert of `case` into a `record` cache; returns (got, ref, errs)."""
    assert_distinct_slots(case.slots)
    ps = oracle_mod.page_stride(record, case.block_size) + 512 * pad_units
    kv, slots, pos, csc = device_inputs(case, DEV)
    cache = gkr.alloc_cache(case.num_pages, case.block_size, record, DEV, page_stride_bytes=ps,
                            fill=SENTINEL)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    gkr.kv_insert(kv, cache, slots, pos, csc, case.block_size, record, err_flag=err,
                  fp8_scale=_scale_t(scale))
    ref = np.full(case.num_pages * ps, SENTINEL, np.uint8)
    ref_err = oracle_mod.insert(case.kv, ref, record, case.block_size, case.num_pages, ps,
                                case.slots, case.positions, case.csc, fp8_scale=scale)
    return cache, gkr.cache_bytes(cache).cpu().numpy(), ref, int(err.item()), ref_err, ps


def _case(T, bs, seed, sigma=1.0, inf_rate=0.0):
    pages = max(2, -(-2 * T // bs))
    c = W.compressed_insert(f"plain_{T}", 1, T, 1, 528, block_size=bs, skip_rate=0.1,
                            seed=seed, sigma=sigma, dist="student_t3", inf_rate=inf_rate,
                            nonfinite_dims=448)
    c.positions = np.random.default_rng(seed).integers(0, c.csc.shape[0], T)
    # distinct random slots over twice the needed pages
    slots = np.random.default_rng(seed + 1).permutation(pages * bs)[:T].astype(np.int64)
    c.slots = np.where(c.slots >= 0, slots, -1)
    c.num_pages = pages
    return c


@pytest.mark.parametrize("record", [1024, 512])
def test_plain_cache_golden(gkr, record):
    w = load_worked(GOLDEN / "worked_full_caches.txt")
    kv_bits, slots, pos, csc = worked_inputs(w)
    ps, expects = w.records[record]
    cache = gkr.alloc_cache(w.num_pages, w.block_size, record, DEV, page_stride_bytes=ps,
                            fill=SENTINEL)
    scale = _scale_t(w.fp8_scale.get(record))
    gkr.kv_insert(bf16_from_bits(kv_bits, DEV), cache, torch.from_numpy(slots).to(DEV),
                  torch.from_numpy(pos).to(DEV), torch.from_numpy(csc).to(DEV), w.block_size,
                  record, fp8_scale=scale)
    got = gkr.cache_bytes(cache).cpu().numpy()
    touched = np.zeros(got.size, bool)
    for e in expects:
        assert np.array_equal(got[e.data_offset:e.data_offset + e.data.size], e.data), e.token
        touched[e.data_offset:e.data_offset + e.data.size] = True
    assert (got[~touched] == SENTINEL).all()
    idx, expect = w.gathers[record]
    out = torch.empty(idx.size, 512, dtype=torch.bfloat16, device=DEV)
    gkr.kv_gather(cache, torch.from_numpy(idx).to(DEV), out, fp8_scale=scale)
    got_out = out.cpu().view(torch.int16).numpy().view(np.uint16).astype(np.int64)
    assert np.array_equal(got_out, expect)


@pytest.mark.parametrize("record,scale", [(1024, None), (512, 0.0078125), (512, 0.37),
                                          (512, 3.0), (512, 1.0 / 3.0)])
@pytest.mark.parametrize("T,bs", [(1, 16), (17, 48), (1023, 64), (4099, 64)])
def test_plain_cache_insert_and_gather_match_oracle(gkr, oracle_mod, record, scale, T, bs):
    case = _case(T, bs, seed=T + bs, sigma=2.0, inf_rate=0.0005)
    cache, got, ref, err, ref_err, ps = _insert(gkr, oracle_mod, case, record, scale,
                                                pad_units=1)
    n, first = first_mismatch(got, ref)
    assert n == 0, f"{record} scale={scale}: {n} bytes differ, first {first}"
    assert err == ref_err == 0
    idx = np.concatenate([case.slots, [-1, 0, case.num_pages * bs - 1]]).astype(np.int32)
    out = torch.empty(idx.size, 512, dtype=torch.bfloat16, device=DEV)
    gkr.kv_gather(cache, torch.from_numpy(idx).to(DEV), out, fp8_scale=_scale_t(scale))
    ref_out, _ = oracle_mod.gather(ref, record, bs, case.num_pages, ps, idx, fp8_scale=scale)
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), ref_out)


@pytest.mark.parametrize("scale", [0.0, -1.0, float("inf"), float("nan")])
def test_fp8_bad_scale(gkr, oracle_mod, scale):
    case = _case(300, 32, seed=3)
    cache, got, ref, err, ref_err, ps = _insert(gkr, oracle_mod, case, 512, scale)
    assert err == ref_err == 8 and (got == SENTINEL).all() and (ref == SENTINEL).all()
    idx = torch.from_numpy(case.slots.astype(np.int32)).to(DEV)
    out = torch.full((idx.numel(), 512), 1.0, dtype=torch.bfloat16, device=DEV)
    e = torch.zeros(1, dtype=torch.int32, device=DEV)
    gkr.kv_gather(cache, idx, out, err_flag=e, fp8_scale=_scale_t(scale))
    assert int(e.item()) == 8 and (out.view(torch.int16) == 0).all()


@pytest.mark.parametrize("record", [1024, 512])
def test_plain_cache_error_bits(gkr, oracle_mod, record):
    case = _case(64, 32, seed=8)
    case.slots[3] = case.num_pages * 32
    case.positions[9] = case.csc.shape[0]
    _, got, ref, err, ref_err, _ = _insert(gkr, oracle_mod, case, record,
                                           0.5 if record == 512 else None)
    assert err == ref_err == 3
    assert first_mismatch(got, ref)[0] == 0


def test_fp8_scale_is_read_on_the_device_at_replay(gkr, oracle_mod):
    """The scale lives in device memory: a captured insert picks up a new value."""
    case = _case(512, 64, seed=11)
    ps = oracle_mod.page_stride(512, 64)
    kv, slots, pos, csc = device_inputs(case, DEV)
    cache = gkr.alloc_cache(case.num_pages, 64, 512, DEV, fill=SENTINEL)
    scale = torch.tensor([1.0], dtype=torch.float32, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gkr.kv_insert(kv, cache, slots, pos, csc, 64, 512, fp8_scale=scale)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gkr.kv_insert(kv, cache, slots, pos, csc, 64, 512, fp8_scale=scale)
    for value in (0.25, 3.0):
        scale.fill_(value)
        g.replay()
        torch.cuda.synchronize()
        ref = np.full(case.num_pages * ps, SENTINEL, np.uint8)
        oracle_mod.insert(case.kv, ref, 512, 64, case.num_pages, ps, case.slots, case.positions,
                          case.csc, fp8_scale=value)
        assert first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)[0] == 0


@pytest.mark.slow
@pytest.mark.parametrize("record", [1024, 512])
def test_plain_cache_full_size(gkr, oracle_mod, record):
    """262144 tokens in 8 contiguous sequences (the large-insert layout) into a plain
    cache: every byte of the cache against the oracle's (fp8 at scale 0.01)."""
    case = W.insert_v41_262144()
    scale = 0.01 if record == 512 else None
    kw = {} if scale is None else {"fp8_scale": scale}
    ref, ref_err, ps = oracle_full_cache(oracle_mod, case, record=record, **kw)
    kv, slots, pos, csc = device_inputs(case, DEV)
    cache = gkr.alloc_cache(case.num_pages, 64, record, DEV, page_stride_bytes=ps, fill=SENTINEL)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    gkr.kv_insert(kv, cache, slots, pos, csc, 64, record, err_flag=err, fp8_scale=_scale_t(scale))
    n, first = first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)
    assert n == 0, f"{n} bytes differ, first {first}"
    assert int(err.item()) == ref_err == 0


def _e4m3_midpoints() -> np.ndarray:
    """The 126 midpoints between consecutive finite non-negative e4m3 values."""
    v = np.array([0.0] + [m * 2.0 ** -9 for m in range(1, 8)] +
                 [(1 + m / 8) * 2.0 ** (e - 7) for e in range(1, 16) for m in range(8)
                  if not (e == 15 and m == 7)])
    return (v[:-1] + v[1:]) / 2


@pytest.mark.parametrize("scale", [3.0, 0.37, 2.0 ** -7, 1.0])
def test_fp8_signed_zeros_ties_and_overflow(gkr, oracle_mod, scale):
    """Values whose codes hinge on the quotient's sign handling and on its non-finite
    fallback: +-0 (two whole rows and scattered entries), quotients that underflow to a
    signed zero, exact e4m3 midpoints times the scale (ties to even; exact in bf16 at
    scales 3, 2^-7 and 1), products x / scale that overflow fp32 (+-3e38), and +-inf in
    dims 0..447; byte for byte against the oracle at general and power-of-two scales."""
    T = 600
    case = _case(T, 64, seed=31)
    rng = np.random.default_rng(32)
    s32 = float(np.float32(scale))
    x = (rng.standard_normal((T, 512)) * 20 * s32).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    flat = x.reshape(-1)
    nope = np.flatnonzero(np.arange(flat.size) % 512 < 448)
    nope = nope[nope >= 2 * 512]
    cut = rng.permutation(nope)
    sign = lambda k: np.where(rng.integers(0, 2, k) == 1, -1.0, 1.0)
    mids = _e4m3_midpoints()
    groups = [(1500, lambda k: sign(k) * 0.0),
              (1500, lambda k: sign(k) * s32 * 2.0 ** -12),
              (6000, lambda k: sign(k) * rng.choice(mids, k) * s32),
              (300, lambda k: sign(k) * 3e38),
              (200, lambda k: sign(k) * np.inf)]
    at = 0
    for k, make in groups:
        flat[cut[at:at + k]] = make(k).astype(np.float32)
        at += k
    rope = np.flatnonzero(np.arange(flat.size) % 512 >= 448)   # zeros and huge values there too
    cut = rng.permutation(rope[rope >= 2 * 512])
    flat[cut[:500]] = (sign(500) * 0.0).astype(np.float32)
    flat[cut[500:600]] = (sign(100) * 3e38).astype(np.float32)
    case.kv = W.to_bf16_bits(x)
    assert int((case.kv == 0x8000).sum()) > 1000 and int((case.kv == 0xFF80).sum()) > 50
    cache, got, ref, err, ref_err, ps = _insert(gkr, oracle_mod, case, 512, s32)
    n, first = first_mismatch(got, ref)
    assert n == 0 and err == ref_err == 0, f"scale={scale}: {n} bytes differ, first {first}"


@pytest.mark.parametrize("scale", [1e-30, 2.0 ** -64, float(np.nextafter(np.float32(2.0 ** -64), 0)),
                                   2.0 ** 64, float(np.nextafter(np.float32(2.0 ** 64), np.inf)),
                                   1e30, 7.0 / 3.0, 1.0, 2.0 ** -126, 2.0 ** 126, 2.0 ** 127,
                                   2.0 ** -127])
def test_fp8_scales_across_the_quotient_paths(gkr, oracle_mod, scale):
    """Powers of two in [2^-126, 2^126] take the single exact product, other scales inside
    [2^-64, 2^64] the corrected-reciprocal quotient, the rest (2^127, the subnormal 2^-127,
    1e-30, 1e30) the IEEE division: all must give the oracle's bytes.  kv is drawn around
    50 * scale (at most 1e36) so the quotients land inside the e4m3 range (saturating
    tails included)."""
    s32 = float(np.float32(scale))
    case = _case(2000, 64, seed=21)
    rng = np.random.default_rng(22)
    case.kv = W.to_bf16_bits((rng.standard_t(3, (2000, 512)) * min(50.0 * s32, 1e36))
                             .astype(np.float32))
    cache, got, ref, err, ref_err, ps = _insert(gkr, oracle_mod, case, 512, s32)
    n, first = first_mismatch(got, ref)
    assert n == 0 and err == ref_err == 0, first
    idx = case.slots.astype(np.int32)
    out = torch.empty(idx.size, 512, dtype=torch.bfloat16, device=DEV)
    gkr.kv_gather(cache, torch.from_numpy(idx).to(DEV), out, fp8_scale=_scale_t(s32))
    ref_out, _ = oracle_mod.gather(ref, 512, 64, case.num_pages, ps, idx, fp8_scale=s32)
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), ref_out)
