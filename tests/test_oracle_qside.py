"""CPU pins of the oracle's query side (the fused attention write: q norm, q rotation,
bf16 q out, padded heads, beside the KV insert).

The pages give the op and its arguments (q, padded head count, eps, apply_q_norm) but
not the norm's formula; the reading (an RMS norm over each head's 512 dims, no weight,
eps inside the square root) is pinned here against closed forms and invariants that
any slip in it (a sum instead of a mean, eps outside the root, a wrong rotation dim or
sign, norm skipped) breaks.  Which norm the pages' kernel applies stays unpinned."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads as W
from golden_parse import GOLDEN, parse_value

HEAD = 512


def bf16_bits(values) -> np.ndarray:
    t = torch.tensor(np.asarray(values, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def csc_row(cos: float, sin: float) -> np.ndarray:
    return np.array([cos] * 32 + [sin] * 32, np.float32)


# ---------------------------------------------------------------- golden heads

def _parse_cases():
    cases, cur = [], None
    for raw in (GOLDEN / "worked_qnorm.txt").read_text().splitlines():
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        tok = line.split()
        if tok[0] == "case":
            kv = dict(t.split("=") for t in tok[2:])
            cur = dict(name=tok[1], eps=float(kv["eps"]), norm=kv["norm"] == "1",
                       cos=float(kv["cos"]), sin=float(kv["sin"]),
                       x=np.zeros(HEAD, np.float64), rn=np.full(HEAD, -1, np.int64),
                       alt=np.full(HEAD, -1, np.int64))
            cases.append(cur)
        elif tok[0] == "x":
            vals = [parse_value(v) for v in tok[2:]]
            a, b = (tok[1].split("..") + [None])[:2]
            if b is None:
                cur["x"][int(a):int(a) + len(vals)] = vals
            else:
                cur["x"][int(a):int(b) + 1] = np.tile(vals, (int(b) - int(a) + 1) // len(vals))
        elif tok[0] == "expect":
            pairs = [(int(v.split("/")[0], 16), int(v.split("/")[-1], 16)) for v in tok[2:]]
            a, b = (tok[1].split("..") + [None])[:2]
            idx = range(int(a), int(a) + len(pairs)) if b is None else range(int(a), int(b) + 1)
            for k, d in enumerate(idx):
                rn, alt = pairs[k if b is None else k % len(pairs)]
                cur["rn"][d], cur["alt"][d] = rn, alt
    return cases


@pytest.mark.parametrize("case", _parse_cases(), ids=lambda c: c["name"])
def test_golden_heads(oracle_mod, case):
    assert (case["rn"] >= 0).all(), "every dim has a hand-derived value"
    exact, rn, alt = oracle_mod.q_head(bf16_bits(case["x"]), csc_row(case["cos"], case["sin"]),
                                       case["eps"], case["norm"])
    assert np.array_equal(rn, case["rn"].astype(np.uint16)), np.nonzero(rn != case["rn"])
    assert np.array_equal(alt, case["alt"].astype(np.uint16)), np.nonzero(alt != case["alt"])


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("c", [0.5, -3.0, 1e-3, 250.0, 2.0 ** -20])
@pytest.mark.parametrize("eps", [0.0, 1e-6, 0.25, 5.0])
def test_constant_row_closed_form(oracle_mod, c, eps):
    """A constant row c (a bf16 value) has mean(x^2) = c^2, so every output is
    c / sqrt(c^2 + eps) (identity rotation); eps = 0 gives sign(c) exactly."""
    x = bf16_bits(np.full(HEAD, c))
    cb = float(torch.tensor(c, dtype=torch.float32).to(torch.bfloat16).float())
    exact, rn, _ = oracle_mod.q_head(x, csc_row(1.0, 0.0), eps, True)
    want = cb / math.sqrt(cb * cb + eps)
    assert np.allclose(exact, want, rtol=1e-15, atol=0)
    if eps == 0.0:
        assert (exact == math.copysign(1.0, cb)).all()
    assert (rn == bf16_bits(np.float32(want))[()]).all()   # want is far from a bf16 midpoint


def _random_head(rng, scale=1.0):
    return bf16_bits(rng.standard_normal(HEAD).astype(np.float32) * np.float32(scale))


def _value(bits: np.ndarray) -> np.ndarray:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def test_unit_rms_without_eps(oracle_mod):
    """With eps = 0 the normed head has mean(y^2) = 1 (the rotation preserves it)."""
    rng = np.random.default_rng(0)
    csc = W.cos_sin_table(4096)
    for k in range(20):
        exact, _, _ = oracle_mod.q_head(_random_head(rng, 10.0 ** rng.uniform(-3, 3)),
                                        csc[rng.integers(0, 4096)], 0.0, True)
        assert abs(np.mean(exact ** 2) - 1.0) < 1e-6      # cos^2 + sin^2 = 1 to fp32 rounding


def test_eps_shrinks_the_rms(oracle_mod):
    """mean(y^2) = m / (m + eps) for m = mean(x^2): eps enters inside the square root."""
    rng = np.random.default_rng(1)
    q = _random_head(rng)
    m = float(np.mean(_value(q) ** 2))
    for eps in (1e-3, 0.5, 3.0):
        exact, _, _ = oracle_mod.q_head(q, csc_row(1.0, 0.0), eps, True)
        assert abs(np.mean(exact ** 2) - m / (m + eps)) < 1e-12


def test_scale_invariance_without_eps(oracle_mod):
    """eps = 0: scaling the head by 2^k changes nothing (exact), by 3 nothing beyond
    rounding of the input."""
    rng = np.random.default_rng(2)
    csc = W.cos_sin_table(64)
    q = _random_head(rng)
    base, rn0, _ = oracle_mod.q_head(q, csc[17], 0.0, True)
    for k in (-40, -3, 5, 60):
        scaled = bf16_bits(_value(q) * 2.0 ** k)
        e2, rn2, _ = oracle_mod.q_head(scaled, csc[17], 0.0, True)
        assert np.array_equal(e2, base) and np.array_equal(rn2, rn0)


def test_norm_off_is_the_rotation_alone(oracle_mod):
    """apply_q_norm off: dims 0..447 come back unchanged; each rotated pair keeps its
    length (cos^2 + sin^2 = 1 to fp32 rounding); a quarter turn maps (e, o) to (-o, e)."""
    rng = np.random.default_rng(3)
    q = _random_head(rng)
    x = _value(q)
    exact, rn, _ = oracle_mod.q_head(q, csc_row(1.0, 0.0), 0.0, False)
    assert np.array_equal(exact, x) and np.array_equal(rn, q)
    exact, _, _ = oracle_mod.q_head(q, csc_row(0.0, 1.0), 0.0, False)
    assert np.array_equal(exact[448::2], -x[449::2]) and np.array_equal(exact[449::2], x[448::2])
    csc = W.cos_sin_table(1000)
    exact, _, _ = oracle_mod.q_head(q, csc[999], 0.0, False)
    assert np.array_equal(exact[:448], x[:448])
    before = x[448::2] ** 2 + x[449::2] ** 2
    after = exact[448::2] ** 2 + exact[449::2] ** 2
    assert np.allclose(after, before, rtol=1e-6, atol=0)
    # the rotation angle is the table's: pair j turns by atan2(sin_j, cos_j)
    j = 5
    z = complex(x[448 + 2 * j], x[449 + 2 * j]) * complex(csc[999][j], csc[999][32 + j])
    assert abs(exact[448 + 2 * j] - z.real) < 1e-12 and abs(exact[449 + 2 * j] - z.imag) < 1e-12


def test_faithful_pair_brackets_the_exact_value(oracle_mod):
    """rn is the nearest bf16 of the exact value, alt the bf16 on its other side (equal
    when the value is a bf16): they are adjacent and enclose the exact value."""
    rng = np.random.default_rng(4)
    csc = W.cos_sin_table(4096)
    for k in range(10):
        exact, rn, alt = oracle_mod.q_head(_random_head(rng), csc[rng.integers(0, 4096)],
                                           1e-6, True)
        vr, va = _value(rn), _value(alt)
        lo, hi = np.minimum(vr, va), np.maximum(vr, va)
        assert ((lo <= exact) & (exact <= hi)).all()
        assert (np.abs(vr - exact) <= np.abs(va - exact)).all()
        same = rn == alt
        assert (vr[same] == exact[same]).all()
        # adjacent: no bf16 strictly between them (one step in the bit pattern's magnitude)
        nz = ~same
        step = np.abs(vr[nz] - va[nz])
        assert (step <= np.spacing(np.abs(exact[nz]).astype(np.float32)).astype(np.float64) * 2 ** 16).all()
        assert torch.equal(torch.from_numpy(_value(rn)).to(torch.bfloat16).double(),
                           torch.from_numpy(exact).to(torch.bfloat16).double())


# ---------------------------------------------------------------- the whole op

def _op_case(T=40, H=3, seed=5, record=528, bs=32, bad_pos=False):
    c = W.random_insert("qside", T, record, bs, 4, 256, 0.2, seed)
    rng = np.random.default_rng(seed + 100)
    q = bf16_bits(rng.standard_normal((T, H, HEAD)).astype(np.float32) * 4)
    if bad_pos:
        c.positions[3] = 256            # past the table
        c.positions[7] = -1
    return c, q


@pytest.mark.parametrize("record", [528, 584, 1024])
def test_zero_heads_is_the_kv_insert(oracle_mod, record):
    c, _ = _op_case(record=record)
    ps = oracle_mod.page_stride(record, c.block_size)
    a = np.full(c.num_pages * ps, 0xA5, np.uint8)
    b = a.copy()
    rn, alt, _, _, err = oracle_mod.qnorm_rope_kv_insert(np.zeros((c.num_tokens, 0, HEAD), np.uint16),
                                                   0, 1e-6, True, c.kv, a, record, c.block_size,
                                                   c.num_pages, ps, c.slots, c.positions, c.csc)
    assert rn.shape == (c.num_tokens, 0, HEAD)
    assert err == oracle_mod.insert(c.kv, b, record, c.block_size, c.num_pages, ps, c.slots,
                                    c.positions, c.csc) == 0
    assert np.array_equal(a, b)


def test_heads_padded_and_kv_untouched_by_q(oracle_mod):
    c, q = _op_case()
    ps = oracle_mod.page_stride(528, c.block_size)
    a = np.full(c.num_pages * ps, 0xA5, np.uint8)
    b = a.copy()
    rn, alt, lo, hi, err = oracle_mod.qnorm_rope_kv_insert(q, 8, 1e-6, True, c.kv, a, 528, c.block_size,
                                                   c.num_pages, ps, c.slots, c.positions, c.csc)
    oracle_mod.insert(c.kv, b, 528, c.block_size, c.num_pages, ps, c.slots, c.positions, c.csc)
    assert err == 0 and np.array_equal(a, b)
    assert rn.shape == (c.num_tokens, 8, HEAD)
    assert (rn[:, 3:] == 0).all() and (alt[:, 3:] == 0).all()
    assert (lo[:, 3:] == 0).all() and (hi[:, 3:] == 0).all()
    # every token's heads (skipped slots too) are the per-head oracle at its position
    for t in (0, 1, c.num_tokens - 1):
        for h in range(3):
            _, r1, a1 = oracle_mod.q_head(q[t, h], c.csc[c.positions[t]], 1e-6, True)
            assert np.array_equal(rn[t, h], r1) and np.array_equal(alt[t, h], a1)
    assert (c.slots < 0).any()


def test_bad_position_zeroes_the_heads_and_flags(oracle_mod):
    c, q = _op_case(bad_pos=True)
    ps = oracle_mod.page_stride(528, c.block_size)
    a = np.full(c.num_pages * ps, 0xA5, np.uint8)
    rn, alt, lo, hi, err = oracle_mod.qnorm_rope_kv_insert(q, 3, 1e-6, False, c.kv, a, 528, c.block_size,
                                                   c.num_pages, ps, c.slots, c.positions, c.csc)
    assert err == oracle_mod.ERR_POS
    assert (rn[[3, 7]] == 0).all() and (alt[[3, 7]] == 0).all() and (hi[[3, 7]] == 0).all()
    assert (rn[[0, 1, 2, 4]] != 0).any()



def test_fp32_evaluation_range(oracle_mod):
    """lo .. hi (the bf16 values an fp32 evaluation may give) contain the faithful pair;
    for dims 0..447 they are exactly that pair (2^-19 |y| is far inside half a bf16
    step); for a rotated pair whose terms cancel the range follows the size of the
    products; a slip in the rotation (the sine's sign flipped) leaves it."""
    rng = np.random.default_rng(6)
    csc = W.cos_sin_table(4096)
    q = _random_head(rng)
    row = csc[1234]
    exact, rn, alt, lo, hi = oracle_mod.q_head(q, row, 1e-6, True, bounds=True)
    vl, vh, vr, va = _value(lo), _value(hi), _value(rn), _value(alt)
    assert (vl <= np.minimum(vr, va)).all() and (np.maximum(vr, va) <= vh).all()
    assert np.array_equal(np.minimum(vr, va)[:448], vl[:448])
    assert np.array_equal(np.maximum(vr, va)[:448], vh[:448])
    # a pair that cancels: (e, o) = (1, 1) turned by 45 degrees: e c - o s = 0 exactly in
    # real arithmetic but not for the fp32 cos/sin of 45 degrees
    x = np.zeros(HEAD, np.float32)
    x[448], x[449] = 1.0, 1.0
    c45 = np.float32(np.cos(np.pi / 4))
    s45 = np.float32(np.sin(np.pi / 4))
    e2, _, _, lo2, hi2 = oracle_mod.q_head(bf16_bits(x), csc_row(c45, s45), 0.0, False,
                                           bounds=True)
    assert abs(e2[448]) < 1e-7 and _value(hi2)[448] - _value(lo2)[448] >= 2 * 2.0 ** -19
    # the same head with the sine's sign flipped lands outside the range
    wrong, _, _ = oracle_mod.q_head(q, np.concatenate([row[:32], -row[32:]]), 1e-6, True)
    outside = (wrong[448:] < vl[448:]) | (wrong[448:] > vh[448:])
    assert outside.mean() > 0.9


# ---------------------------------------------------------------- e4m3 query output

def _e4m3_value(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(torch.float8_e4m3fn) \
        .double().numpy()


@pytest.mark.parametrize("c,s,code", [(0.5, 0.25, 0x48), (3.0, 1.0, 0x38), (-7.0, 2.0, 0xB0),
                                      (250.0, 1e-3, 0x7E), (-1e-3, 1e-3, 0xFE)])
def test_fp8_q_constant_row_closed_form(oracle_mod, c, s, code):
    """eps = 0: a constant row normalises to sign(c) exactly, so every code is that of
    sign(c) / s: 1/0.25 = 4 = 1.0 * 2^2 (exponent field 9: 0x48), 1.0 (0x38), -0.5 (sign
    bit, exponent field 6: 0xB0), and 1/1e-3 = 1000 saturating to 448 (0x7E, or 0xFE
    negative); the three codes agree."""
    rn, lo, hi = oracle_mod.q_head_fp8(bf16_bits(np.full(HEAD, c)), csc_row(1.0, 0.0), 0.0, s)
    assert (rn == code).all() and (lo == code).all() and (hi == code).all()


def test_fp8_q_without_norm_is_the_fp8_cache_row(oracle_mod):
    """apply_q_norm off: a query head is rotated like a KV row, and the fp8 cache encodes
    e4m3(RN32(x / scale)) of that row with one fp32 evaluation of the rotation, so the
    cache row's codes lie in the query range (and equal the nearest codes on the
    unrotated dims 0..447, where x is the bf16 input itself)."""
    rng = np.random.default_rng(11)
    csc = W.cos_sin_table(512)
    for k in range(6):
        row = bf16_bits(rng.standard_normal(HEAD).astype(np.float32) * np.float32(3.0))
        pos, s = int(rng.integers(0, 512)), float(np.float32(10.0 ** rng.uniform(-2, 1)))
        ps = oracle_mod.page_stride(512, 32)
        cache = np.zeros(ps, np.uint8)
        assert oracle_mod.insert(row.reshape(1, HEAD), cache, 512, 32, 1, ps,
                                 np.array([5]), np.array([pos]), csc, fp8_scale=np.float32(s)) == 0
        cache_row = cache[5 * 512:6 * 512]
        rn, lo, hi = oracle_mod.q_head_fp8(row, csc[pos], 0.0, s, apply_norm=False)
        v, vl, vh = _e4m3_value(cache_row), _e4m3_value(lo), _e4m3_value(hi)
        assert ((vl <= v) & (v <= vh)).all()
        assert np.array_equal(cache_row[:448], rn[:448])


def test_fp8_q_range_and_planted_slip(oracle_mod):
    """The nearest codes lie within lo .. hi; on the unrotated dims the range is almost
    always one code (2^-19 of the value is far inside an e4m3 step); multiplying by the
    scale instead of dividing lands outside the range."""
    rng = np.random.default_rng(12)
    csc = W.cos_sin_table(4096)
    q = _random_head(rng, 2.0)
    s = 0.0625
    rn, lo, hi = oracle_mod.q_head_fp8(q, csc[77], 1e-6, s)
    v, vl, vh = _e4m3_value(rn), _e4m3_value(lo), _e4m3_value(hi)
    assert ((vl <= v) & (v <= vh)).all()
    assert (lo[:448] == hi[:448]).mean() > 0.99
    exact, _, _ = oracle_mod.q_head(q, csc[77], 1e-6, True)
    wrong = np.array([oracle_mod.e4m3_encode(x * s) for x in exact], np.uint8)
    vw = _e4m3_value(wrong)
    assert ((vw < vl) | (vw > vh)).mean() > 0.9


def test_fp8_q_op_padding_positions_and_bad_scale(oracle_mod):
    """Padded heads and the heads of a token whose position is outside the table are +0
    (code 0) with ORACLE_ERR_POS for the latter; a scale that is not a positive finite
    number writes every head as +0 with ORACLE_ERR_SCALE; otherwise each head is
    q_head_fp8's."""
    c, q = _op_case(T=12, H=3, bad_pos=True)
    rn, lo, hi, err = oracle_mod.qnorm_rope_fp8q(q, 5, 1e-6, True, 0.5, c.positions, c.csc)
    assert rn.shape == (12, 5, HEAD) and err == oracle_mod.ERR_POS
    assert (rn[:, 3:] == 0).all() and (rn[3] == 0).all() and (rn[7] == 0).all()
    r1, l1, h1 = oracle_mod.q_head_fp8(q[0, 1], c.csc[c.positions[0]], 1e-6, 0.5)
    assert np.array_equal(rn[0, 1], r1) and np.array_equal(lo[0, 1], l1) and np.array_equal(hi[0, 1], h1)
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        rn, lo, hi, err = oracle_mod.qnorm_rope_fp8q(q, 5, 1e-6, True, bad, c.positions, c.csc)
        assert err & oracle_mod.ERR_SCALE and (rn == 0).all() and (lo == 0).all() and (hi == 0).all()
    # no head to cast (padded heads only, or every position outside the table): no scale
    # is read, so no scale error
    empty = np.zeros((12, 0, HEAD), np.uint16)
    assert oracle_mod.qnorm_rope_fp8q(empty, 4, 1e-6, True, 0.0, c.positions, c.csc)[3] == 0
    far = np.full(12, 10 ** 6, np.int64)
    assert oracle_mod.qnorm_rope_fp8q(q, 5, 1e-6, True, 0.0, far, c.csc)[3] == oracle_mod.ERR_POS
