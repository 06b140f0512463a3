"""GPU parity of the fused attention write (qnorm_rope_kv_insert through the C ABI):
the KV records byte for byte against the oracle over the whole sentinel-filled cache,
every query value one of the oracle's two faithful bf16 roundings of the exact result
(and nearly always the nearest), padded heads zero, the error bits equal."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from helpers import SENTINEL, bf16_from_bits, bits_of, device_inputs, first_mismatch
from test_oracle_qside import _parse_cases, bf16_bits, csc_row

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _q_case(T, H, record=528, bs=64, seed=0, sigma=2.0, skip=0.1, max_pos=4096):
    pages = max(2, -(-2 * T // bs))
    c = W.random_insert(f"q{T}_{H}", T, record, bs, pages, max_pos, skip, seed)
    rng = np.random.default_rng(seed + 7)
    q = bf16_bits(rng.standard_normal((T, H, 512)).astype(np.float32) * np.float32(sigma))
    return c, q


def _run(gkr, oracle_mod, c, q, Hp, eps, norm, record, scale=None, in_place=False, **kw):
    ps = oracle_mod.page_stride(record, c.block_size)
    kv, slots, pos, csc = device_inputs(c, DEV)
    cache = gkr.alloc_cache(c.num_pages, c.block_size, record, DEV, fill=SENTINEL)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    qt = bf16_from_bits(q, DEV)
    sc = None if scale is None else torch.tensor([scale], dtype=torch.float32, device=DEV)
    q_out = qt if in_place else torch.full((c.num_tokens, Hp, 512), float("nan"),
                                           dtype=torch.bfloat16, device=DEV)
    gkr.qnorm_rope_kv_insert(qt, kv, cache, slots, pos, csc, Hp, eps, c.block_size, norm,
                             q_out=q_out, record=record, err_flag=err, fp8_scale=sc, **kw)
    torch.cuda.synchronize()
    ref = np.full(c.num_pages * ps, SENTINEL, np.uint8)
    rn, lo, hi, ref_err = _oracle(oracle_mod, q, Hp, eps, norm, c, ref, record, ps, scale)
    return gkr.cache_bytes(cache).cpu().numpy(), ref, bits_of(q_out), rn, (lo, hi), \
        int(err.item()), ref_err


def _oracle(oracle_mod, q, Hp, eps, norm, c, ref, record, ps, scale=None):
    rn, _, lo, hi, err = oracle_mod.qnorm_rope_kv_insert(q, Hp, eps, norm, c.kv, ref, record,
                                                         c.block_size, c.num_pages, ps, c.slots,
                                                         c.positions, c.csc, fp8_scale=scale)
    return rn, lo, hi, err


def _value(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .float().numpy()


def _assert_faithful(got, rn, bounds, min_nearest=0.999):
    """Every value inside the oracle's fp32-evaluation range (lo .. hi), nearly all equal
    to the nearest bf16 of the exact value."""
    lo, hi = bounds
    g = _value(got)
    ok = (_value(lo) <= g) & (g <= _value(hi))
    bad = np.nonzero(~ok)
    assert bad[0].size == 0, (f"{bad[0].size} query values outside the fp32 range; first "
                              f"{list(zip(*bad))[:4]} got {got[bad][:4]} rn {rn[bad][:4]} "
                              f"lo {lo[bad][:4]} hi {hi[bad][:4]}")
    if got.size:
        assert np.mean(got == rn) >= min_nearest


@pytest.mark.parametrize("case", _parse_cases(), ids=lambda c: c["name"])
def test_golden_heads(gkr, case):
    """The hand-derived heads through the whole op (one token, slot -1: no KV write)."""
    q = bf16_bits(case["x"]).reshape(1, 1, 512)
    kv = torch.zeros(1, 512, dtype=torch.bfloat16, device=DEV)
    cache = gkr.alloc_cache(2, 32, 528, DEV, fill=SENTINEL)
    csc = torch.from_numpy(csc_row(case["cos"], case["sin"]).reshape(1, 64)).to(DEV)
    out = gkr.qnorm_rope_kv_insert(bf16_from_bits(q, DEV), kv, cache,
                                   torch.tensor([-1], device=DEV), torch.tensor([0], device=DEV),
                                   csc, 1, case["eps"], 32, case["norm"])
    got = bits_of(out).reshape(-1)
    ok = (got == case["rn"]) | (got == case["alt"])
    assert ok.all(), np.nonzero(~ok)
    assert (gkr.cache_bytes(cache).cpu().numpy() == SENTINEL).all()


@pytest.mark.parametrize("record", [528, 584, 512, 1024])
@pytest.mark.parametrize("T,H,Hp", [(1, 1, 1), (37, 3, 8), (300, 16, 16), (1000, 5, 64)])
@pytest.mark.parametrize("norm", [True, False])
def test_matches_oracle(gkr, oracle_mod, record, T, H, Hp, norm):
    c, q = _q_case(T, H, seed=T + H + record)
    scale = 0.05 if record == 512 else None
    got, ref, qo, rn, bounds, err, ref_err = _run(gkr, oracle_mod, c, q, Hp, 1e-6, norm, record,
                                               scale=scale)
    n, first = first_mismatch(got, ref)
    assert n == 0, f"cache: {n} bytes differ, first {first}"
    assert err == ref_err == 0
    _assert_faithful(qo, rn, bounds)
    assert (qo[:, H:] == 0).all()


@pytest.mark.parametrize("eps", [0.0, 0.5, 30.0])
@pytest.mark.parametrize("sigma", [1e-12, 1.0, 1e12])
def test_eps_and_magnitudes(gkr, oracle_mod, eps, sigma):
    """eps 0 (a pure RMS norm), eps of the data's size, eps dominating; heads from
    1e-12 to 1e12 (the sum of squares stays inside fp32's normal range)."""
    c, q = _q_case(200, 4, seed=3, sigma=sigma)
    got, ref, qo, rn, bounds, err, ref_err = _run(gkr, oracle_mod, c, q, 4, eps, True, 528)
    assert first_mismatch(got, ref)[0] == 0 and err == ref_err == 0
    _assert_faithful(qo, rn, bounds)


@pytest.mark.parametrize("record", [528, 584])
def test_zero_heads_is_kv_insert(gkr, oracle_mod, record):
    """num_heads_padded = 0: exactly gkr_kv_insert (the KV-only op of the pages)."""
    c, _ = _q_case(3000, 0, record=record, seed=11)
    kv, slots, pos, csc = device_inputs(c, DEV)
    a = gkr.alloc_cache(c.num_pages, 64, record, DEV, fill=SENTINEL)
    b = gkr.alloc_cache(c.num_pages, 64, record, DEV, fill=SENTINEL)
    q = torch.empty(c.num_tokens, 0, 512, dtype=torch.bfloat16, device=DEV)
    gkr.qnorm_rope_kv_insert(q, kv, a, slots, pos, csc, 0, 1e-6, 64, True, record=record)
    gkr.kv_insert(kv, b, slots, pos, csc, 64, record)
    torch.cuda.synchronize()
    assert torch.equal(gkr.cache_bytes(a), gkr.cache_bytes(b))


def test_padded_heads_without_query_heads(gkr, oracle_mod):
    """H = 0, Hp = 4: every q_out head is +0, the KV rows as kv_insert."""
    c, q = _q_case(50, 0, seed=12)
    got, ref, qo, rn, bounds, err, ref_err = _run(gkr, oracle_mod, c, q, 4, 1e-6, True, 528)
    assert first_mismatch(got, ref)[0] == 0 and err == ref_err == 0
    assert (qo == 0).all()


def test_in_place(gkr, oracle_mod):
    """q_out = q (num_heads_padded == num_heads): the heads are replaced by the result."""
    c, q = _q_case(777, 8, seed=13)
    got, ref, qo, rn, bounds, err, ref_err = _run(gkr, oracle_mod, c, q, 8, 1e-6, True, 528,
                                               in_place=True)
    assert first_mismatch(got, ref)[0] == 0
    _assert_faithful(qo, rn, bounds)


def test_bad_positions_zero_the_heads_and_flag(gkr, oracle_mod):
    c, q = _q_case(120, 3, seed=14)
    c.positions[[5, 50]] = [c.csc.shape[0], -3]
    c.slots[5] = -1                       # the query side flags it even without a KV write
    got, ref, qo, rn, bounds, err, ref_err = _run(gkr, oracle_mod, c, q, 6, 1e-6, True, 584)
    assert first_mismatch(got, ref)[0] == 0
    assert err == ref_err == oracle_mod.ERR_POS
    assert (qo[[5, 50]] == 0).all()
    _assert_faithful(qo, rn, bounds)


def test_bad_fp8_scale_skips_only_the_kv_rows(gkr, oracle_mod):
    c, q = _q_case(90, 2, seed=15)
    got, ref, qo, rn, bounds, err, ref_err = _run(gkr, oracle_mod, c, q, 2, 1e-6, True, 512,
                                               scale=float("nan"))
    assert (got == SENTINEL).all() and first_mismatch(got, ref)[0] == 0
    assert err == ref_err == oracle_mod.ERR_SCALE
    _assert_faithful(qo, rn, bounds)


@pytest.mark.parametrize("opts", [dict(pdl=False), dict(early_metadata=True)])
def test_launch_options(gkr, oracle_mod, opts):
    c, q = _q_case(400, 4, seed=16)
    got, ref, qo, rn, bounds, err, ref_err = _run(gkr, oracle_mod, c, q, 8, 1e-6, True, 528,
                                               launch_opts=gkr.LaunchOpts(**opts))
    assert first_mismatch(got, ref)[0] == 0
    _assert_faithful(qo, rn, bounds)


def test_cuda_graph_replay(gkr, oracle_mod):
    """Captured once, replayed over new queries / KV rows / slots copied into the captured
    buffers (the last round with every slot -1)."""
    T, H, Hp = 500, 4, 8
    c0, q0 = _q_case(T, H, seed=20)
    kv, slots, pos, csc = device_inputs(c0, DEV)
    qt = bf16_from_bits(q0, DEV)
    cache = gkr.alloc_cache(c0.num_pages, 64, 528, DEV, fill=SENTINEL)
    out = torch.empty(T, Hp, 512, dtype=torch.bfloat16, device=DEV)
    fn = lambda: gkr.qnorm_rope_kv_insert(qt, kv, cache, slots, pos, csc, Hp, 1e-6, 64, True,
                                          q_out=out)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    ps = oracle_mod.page_stride(528, 64)
    for r in range(3):
        c, q = _q_case(T, H, seed=21 + r)
        if r == 2:
            c.slots[:] = -1
        cache_bytes = gkr.cache_bytes(cache)
        cache_bytes.fill_(SENTINEL)
        kv.copy_(bf16_from_bits(c.kv, DEV))
        slots.copy_(torch.from_numpy(c.slots))
        pos.copy_(torch.from_numpy(c.positions))
        qt.copy_(bf16_from_bits(q, DEV))
        g.replay()
        torch.cuda.synchronize()
        ref = np.full(c.num_pages * ps, SENTINEL, np.uint8)
        rn, lo, hi, _ = _oracle(oracle_mod, q, Hp, 1e-6, True, c, ref, 528, ps)
        assert first_mismatch(cache_bytes.cpu().numpy(), ref)[0] == 0, r
        _assert_faithful(bits_of(out), rn, (lo, hi))


# ---------------------------------------------------------------- e4m3 query output

def _e4m3_value(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn) \
        .double().numpy()


def _run_fp8q(gkr, oracle_mod, c, q, Hp, eps, norm, record, q_scale, fp8_scale=None):
    ps = oracle_mod.page_stride(record, c.block_size)
    kv, slots, pos, csc = device_inputs(c, DEV)
    cache = gkr.alloc_cache(c.num_pages, c.block_size, record, DEV, fill=SENTINEL)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    sc = None if fp8_scale is None else torch.tensor([fp8_scale], dtype=torch.float32, device=DEV)
    qs = torch.tensor([q_scale], dtype=torch.float32, device=DEV)
    q_out = torch.full((c.num_tokens, Hp, 512), 0x5A, dtype=torch.uint8, device=DEV)
    gkr.qnorm_rope_kv_insert(bf16_from_bits(q, DEV), kv, cache, slots, pos, csc, Hp, eps,
                             c.block_size, norm, q_out=q_out, record=record, err_flag=err,
                             fp8_scale=sc, q_scale=qs)
    torch.cuda.synchronize()
    ref = np.full(c.num_pages * ps, SENTINEL, np.uint8)
    kv_err = oracle_mod.insert(c.kv, ref, record, c.block_size, c.num_pages, ps, c.slots,
                               c.positions, c.csc,
                               fp8_scale=None if fp8_scale is None else np.float32(fp8_scale))
    rn, lo, hi, q_err = oracle_mod.qnorm_rope_fp8q(q, Hp, eps, norm, np.float32(q_scale),
                                                   c.positions, c.csc)
    return (gkr.cache_bytes(cache).cpu().numpy(), ref, q_out.cpu().numpy(), rn, lo, hi,
            int(err.item()), kv_err | q_err)


def _assert_codes(got, rn, lo, hi, min_nearest=0.999):
    """Every code between the codes of the oracle's fp32-evaluation range (by value),
    nearly all equal to the code of the nearest fp32."""
    g, vl, vh = _e4m3_value(got), _e4m3_value(lo), _e4m3_value(hi)
    bad = np.nonzero(~((vl <= g) & (g <= vh)))
    assert bad[0].size == 0, (f"{bad[0].size} codes outside the range; first "
                              f"{list(zip(*bad))[:4]} got {got[bad][:4]} rn {rn[bad][:4]}")
    if got.size:
        assert np.mean(got == rn) >= min_nearest


@pytest.mark.parametrize("record", [528, 512])
@pytest.mark.parametrize("T,H,Hp", [(1, 1, 1), (37, 3, 8), (300, 16, 16), (700, 5, 64)])
@pytest.mark.parametrize("norm", [True, False])
def test_fp8_q_matches_oracle(gkr, oracle_mod, record, T, H, Hp, norm):
    c, q = _q_case(T, H, seed=T + H + 11 * record)
    fp8 = 0.05 if record == 512 else None
    got, ref, qo, rn, lo, hi, err, ref_err = _run_fp8q(gkr, oracle_mod, c, q, Hp, 1e-6, norm,
                                                       record, 0.03, fp8_scale=fp8)
    n, first = first_mismatch(got, ref)
    assert n == 0, f"cache: {n} bytes differ, first {first}"
    assert err == ref_err == 0
    _assert_codes(qo, rn, lo, hi)
    assert (qo[:, H:] == 0).all()


@pytest.mark.parametrize("q_scale", [1.0, 2.0 ** -7, 7.3e-4, 1e-30, 3e25])
def test_fp8_q_scale_paths(gkr, oracle_mod, q_scale):
    """Powers of two (one product per value), a general scale (the corrected quotient),
    scales outside [2^-64, 2^64] (IEEE division): saturation at 1e-30, all-zero codes and
    underflow at 3e25."""
    c, q = _q_case(120, 4, seed=21, sigma=3.0)
    got, ref, qo, rn, lo, hi, err, ref_err = _run_fp8q(gkr, oracle_mod, c, q, 4, 1e-6, True,
                                                       528, q_scale)
    assert first_mismatch(got, ref)[0] == 0 and err == ref_err == 0
    _assert_codes(qo, rn, lo, hi)


@pytest.mark.parametrize("bad", [0.0, -2.0, float("inf"), float("nan")])
def test_fp8_q_bad_scale_zeroes_the_heads(gkr, oracle_mod, bad):
    """A query scale that is not a positive finite number: every query head +0 and
    GKR_ERR_SCALE; the KV records are inserted as ever."""
    c, q = _q_case(64, 3, seed=22)
    got, ref, qo, rn, lo, hi, err, ref_err = _run_fp8q(gkr, oracle_mod, c, q, 4, 1e-6, True,
                                                       528, bad)
    assert first_mismatch(got, ref)[0] == 0
    assert (qo == 0).all() and err == ref_err == gkr.ERR_SCALE


@pytest.mark.parametrize("fp8q", [False, True])
@pytest.mark.parametrize("T,H,Hp", [(37, 3, 8), (33, 0, 5), (129, 7, 23)])
def test_padded_heads_stay_inside_q_out(gkr, oracle_mod, fp8q, T, H, Hp):
    """The padded heads are written in 512-byte pieces, 16 per warp, across token
    boundaries: every padded head of q_out is +0, the query heads match the oracle, and
    the rows just before and after q_out (q_out is a view into a larger buffer) keep their
    fill."""
    c, q = _q_case(T, H, seed=T + H + Hp)
    kv, slots, pos, csc = device_inputs(c, DEV)
    cache = gkr.alloc_cache(c.num_pages, c.block_size, 528, DEV, fill=SENTINEL)
    dtype = torch.uint8 if fp8q else torch.int16
    fill = 0x5A if fp8q else 0x5A5A
    big = torch.full((T + 2, Hp, 512), fill, dtype=dtype, device=DEV)
    q_out = big[1:T + 1] if fp8q else big[1:T + 1].view(torch.bfloat16)
    qs = torch.tensor([0.03], dtype=torch.float32, device=DEV) if fp8q else None
    gkr.qnorm_rope_kv_insert(bf16_from_bits(q, DEV), kv, cache, slots, pos, csc, Hp, 1e-6,
                             c.block_size, True, q_out=q_out, record=528, q_scale=qs)
    torch.cuda.synchronize()
    b = big.cpu()
    assert (b[0] == fill).all() and (b[T + 1] == fill).all()
    got = b[1:T + 1].numpy()
    assert (got[:, H:] == 0).all()
    if fp8q:
        rn, lo, hi, _ = oracle_mod.qnorm_rope_fp8q(q, Hp, 1e-6, True, np.float32(0.03),
                                                   c.positions, c.csc)
        _assert_codes(got, rn, lo, hi)
    else:
        ref = np.full(c.num_pages * oracle_mod.page_stride(528, c.block_size), SENTINEL, np.uint8)
        rn, lo, hi, _ = _oracle(oracle_mod, q, Hp, 1e-6, True, c, ref, 528,
                                oracle_mod.page_stride(528, c.block_size))
        _assert_faithful(got.view(np.uint16), rn, (lo, hi))


@pytest.mark.parametrize("norm", [False, True])
@pytest.mark.parametrize("q_scale", [0.03, 0.25])
def test_fp8_q_signed_zeros(gkr, oracle_mod, norm, q_scale):
    """Query heads with exact +0 and -0 entries and whole zero heads, cast to e4m3 at a
    general and a power-of-two scale: the codes keep the sign of zero (0x00 / 0x80), which
    the two-wide quotient gets by flipping the sign bit of codes computed with -1/scale."""
    c, q = _q_case(96, 4, seed=41)
    rng = np.random.default_rng(42)
    flat = q.reshape(-1)
    pick = rng.permutation(flat.size)[:4000]
    flat[pick[:2000]] = 0x8000          # -0
    flat[pick[2000:]] = 0x0000          # +0
    q[5, 1] = 0x8000                    # a whole head of -0
    q[9, 2] = 0x0000                    # and of +0
    got, ref, qo, rn, lo, hi, err, ref_err = _run_fp8q(gkr, oracle_mod, c, q, 6, 1e-6, norm,
                                                       528, q_scale)
    assert first_mismatch(got, ref)[0] == 0 and err == ref_err == 0
    _assert_codes(qo, rn, lo, hi)
    zero = (lo == hi) & ((rn & 0x7F) == 0)
    assert zero.sum() > 1000
    assert np.array_equal(qo[zero], rn[zero])
    assert (qo[5, 1] == rn[5, 1]).all() and (qo[:, 4:] == 0).all()


@pytest.mark.parametrize("seed", range(32))
def test_random_configurations(gkr, oracle_mod, seed):
    """32 seeded draws over the record formats, token counts, head counts and padding
    (including none and query-free tokens), the norm on or off, eps, head magnitudes, the
    fp8 cache's scale and the query output (bf16, or e4m3 at a random scale)."""
    rng = np.random.default_rng(9000 + seed)
    record = int(rng.choice([528, 584, 512, 1024]))
    T = int(rng.choice([1, 17, 300, 1500]))
    H = int(rng.choice([0, 1, 4, 16, 33]))
    Hp = H + int(rng.choice([0, 0, 1, 7, 48]))
    if Hp == 0:
        Hp = 1
    norm = bool(rng.random() < 0.7)
    eps = float(rng.choice([0.0, 1e-6, 0.5])) if H > 0 else 1e-6
    c, q = _q_case(T, H, record=record, seed=seed, sigma=float(rng.choice([0.01, 1.0, 50.0])))
    if norm and eps == 0.0:
        q[..., 0] = 0x3F80                    # dim 0 = 1.0: no all-zero head when eps is 0
    fp8 = float(np.float32(2.0 ** rng.uniform(-6, 3))) if record == 512 else None
    if rng.random() < 0.5:
        qs = float(np.float32(2.0 ** rng.uniform(-8, 4)))
        got, ref, qo, rn, lo, hi, err, ref_err = _run_fp8q(gkr, oracle_mod, c, q, Hp, eps, norm,
                                                           record, qs, fp8_scale=fp8)
        _assert_codes(qo, rn, lo, hi)
    else:
        got, ref, qo, rn, bounds, err, ref_err = _run(gkr, oracle_mod, c, q, Hp, eps, norm, record,
                                                   scale=fp8)
        _assert_faithful(qo, rn, bounds)
    n, first = first_mismatch(got, ref)
    assert n == 0, f"cache: {n} bytes differ, first {first}"
    assert err == ref_err
    assert (qo[:, H:] == 0).all()
