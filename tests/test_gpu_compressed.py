"""GPU parity: the compressed-KV insert (rope_quant_insert) through the C ABI vs the
CPU oracle, byte for byte over the whole sentinel-filled backing buffer."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from golden_parse import GOLDEN, load_worked, worked_inputs
from helpers import SENTINEL, bf16_from_bits, case_page_stride, device_inputs, first_mismatch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _gpu(gkr, case, ps, ratio, sanitize, err=None):
    kv, slots, pos, csc = device_inputs(case, DEV)
    cache = gkr.alloc_cache(case.num_pages, case.block_size, case.record, DEV,
                            page_stride_bytes=ps, fill=SENTINEL)
    gkr.rope_quant_insert(kv, cache, slots, pos, csc, case.block_size, ratio, sanitize,
                          case.record, err_flag=err)
    return gkr.cache_bytes(cache).cpu().numpy(), kv


def _oracle(oracle_mod, case, ps, ratio, sanitize):
    ref = np.full(case.num_pages * ps, SENTINEL, np.uint8)
    err = oracle_mod.insert(case.kv, ref, case.record, case.block_size, case.num_pages, ps,
                            case.slots, case.positions, case.csc, compress_ratio=ratio,
                            sanitize_nans=sanitize)
    return ref, err


def _compare(gkr, oracle_mod, case, ratio, sanitize, pad_units=0):
    ps = case_page_stride(case, oracle_mod, pad_units)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kv_before = case.kv.copy()
    got, kv = _gpu(gkr, case, ps, ratio, sanitize, err)
    ref, ref_err = _oracle(oracle_mod, case, ps, ratio, sanitize)
    n, first = first_mismatch(got, ref)
    assert n == 0, f"{case.name} R={ratio} sanitize={sanitize}: {n} bytes differ, first {first}"
    assert int(err.item()) == ref_err
    assert np.array_equal(kv.cpu().view(torch.int16).numpy().view(np.uint16), kv_before)
    return ref


@pytest.mark.parametrize("record", [528, 584])
def test_compressed_golden_worked_example(gkr, record):
    w = load_worked(GOLDEN / "worked_compressed.txt")
    kv_bits, slots, pos, csc = worked_inputs(w)
    ps, expects = w.records[record]
    cache = gkr.alloc_cache(w.num_pages, w.block_size, record, DEV, page_stride_bytes=ps,
                            fill=SENTINEL)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    gkr.rope_quant_insert(bf16_from_bits(kv_bits, DEV), cache, torch.from_numpy(slots).to(DEV),
                          torch.from_numpy(pos).to(DEV), torch.from_numpy(csc).to(DEV),
                          w.block_size, w.compress_ratio, w.sanitize, record, err_flag=err)
    got = gkr.cache_bytes(cache).cpu().numpy()
    touched = np.zeros(got.size, bool)
    for e in expects:
        D, S = e.data.size, e.scale.size
        assert np.array_equal(got[e.data_offset:e.data_offset + D], e.data), e.token
        assert np.array_equal(got[e.scale_offset:e.scale_offset + S], e.scale), e.token
        touched[e.data_offset:e.data_offset + D] = True
        touched[e.scale_offset:e.scale_offset + S] = True
    assert (got[~touched] == SENTINEL).all()
    assert int(err.item()) == w.errors


@pytest.mark.parametrize("record", [528, 584])
@pytest.mark.parametrize("ratio", [1, 2, 3, 4, 15, 16, 128])
@pytest.mark.parametrize("sanitize", [False, True])
def test_compressed_sequences_match_oracle(gkr, oracle_mod, record, ratio, sanitize):
    """Contiguous sequences (the compressor's layout), ragged lengths, skips, +-inf
    entries; with sanitising also NaN entries, and non-finite values in every dim
    (without it only in the NoPE dims: an infinite RoPE input can rotate into NaN)."""
    case = W.compressed_insert(f"seq_{record}", 5, 613, ratio, record, block_size=32,
                               skip_rate=0.05, seed=ratio, dist="student_t3",
                               nan_rate=0.002 if sanitize else 0.0, inf_rate=0.001,
                               nonfinite_dims=512 if sanitize else 448)
    _compare(gkr, oracle_mod, case, ratio, sanitize)


@pytest.mark.parametrize("record", [528, 584])
@pytest.mark.parametrize("ratio", [1, 4, 128])
@pytest.mark.parametrize("T", [1, 17, 1023, 4099])
def test_compressed_random_positions_match_oracle(gkr, oracle_mod, record, ratio, T):
    bs = 64 if T > 64 else 32
    pages = max(2, -(-2 * T // bs))
    case = W.random_insert(f"rnd_{record}_{T}", T, record, bs, pages, 700, 0.1, seed=T,
                           outlier_rate=0.01)
    _compare(gkr, oracle_mod, case, ratio, True, pad_units=1)


@pytest.mark.parametrize("record", [528, 584])
def test_ratio_one_without_sanitising_is_kv_insert(gkr, oracle_mod, record):
    case = W.random_insert("r1", 2000, record, 64, 64, 512, 0.05, seed=2)
    ps = case_page_stride(case, oracle_mod)
    got, _ = _gpu(gkr, case, ps, 1, False)
    kv, slots, pos, csc = device_inputs(case, DEV)
    cache = gkr.alloc_cache(case.num_pages, case.block_size, record, DEV, page_stride_bytes=ps,
                            fill=SENTINEL)
    gkr.kv_insert(kv, cache, slots, pos, csc, case.block_size, record)
    assert np.array_equal(got, gkr.cache_bytes(cache).cpu().numpy())


@pytest.mark.parametrize("record", [528, 584])
def test_compressed_error_bits(gkr, oracle_mod, record):
    case = W.compressed_insert("err", 2, 64, 4, record, block_size=32, skip_rate=0.0, seed=9)
    case.slots[3] = case.num_pages * 32          # boundary token, slot past the cache
    case.slots[5] = 10 ** 9                      # non-boundary token, slot past the cache
    case.positions[10] = -4                      # negative position
    case.positions[70] = 67                      # boundary; row 64 is past the 64-row table
    _compare(gkr, oracle_mod, case, 4, True)


@pytest.mark.parametrize("record", [528, 584])
@pytest.mark.parametrize("ratio", [2**31 - 1, 2**31 - 2])
def test_compressed_largest_ratios(gkr, oracle_mod, record, ratio):
    """Ratios near 2^31 with positions near 2^32: the boundary test takes its 64-bit
    form, a group-end position R - 1 maps to cos/sin row 0, and 2R - 1 to row R (past
    the table: error bit, nothing written)."""
    case = W.compressed_insert("bigR", 2, 64, 4, record, block_size=32, skip_rate=0.0, seed=11)
    rng = np.random.default_rng(12)
    case.positions = rng.integers(0, 4 * ratio, case.positions.size).astype(np.int64)
    case.positions[::7] = ratio - 1              # group ends, row 0
    case.positions[3::11] = 2 * ratio - 1        # group ends, row R: past the table
    case.positions[5::13] = 3 * ratio - 2        # ends no group
    ref = _compare(gkr, oracle_mod, case, ratio, True)
    assert (ref != SENTINEL).any()               # some records were written


@pytest.mark.parametrize("record", [528, 584])
def test_compressed_cuda_graph_replay(gkr, oracle_mod, record):
    T, bs, ratio = 1024, 32, 4
    cases = [W.compressed_insert("graph", 4, 256, ratio, record, block_size=bs, seed=30 + r,
                                 nan_rate=0.001) for r in range(3)]
    cases[2].slots[:] = -1
    P = cases[0].num_pages
    ps = case_page_stride(cases[0], oracle_mod)
    kv = torch.empty(T, 512, dtype=torch.bfloat16, device=DEV)
    slots = torch.full((T,), -1, dtype=torch.int64, device=DEV)
    pos = torch.zeros(T, dtype=torch.int64, device=DEV)
    csc = torch.from_numpy(cases[0].csc).to(DEV)
    cache = gkr.alloc_cache(P, bs, record, DEV, fill=SENTINEL)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gkr.rope_quant_insert(kv, cache, slots, pos, csc, bs, ratio, True, record)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gkr.rope_quant_insert(kv, cache, slots, pos, csc, bs, ratio, True, record)
    ref = np.full(P * ps, SENTINEL, np.uint8)
    for c in cases:
        kv.copy_(bf16_from_bits(c.kv, DEV))
        slots.copy_(torch.from_numpy(c.slots))
        pos.copy_(torch.from_numpy(c.positions))
        g.replay()
        oracle_mod.insert(c.kv, ref, record, bs, P, ps, c.slots, c.positions, c.csc,
                          compress_ratio=ratio, sanitize_nans=True)
        torch.cuda.synchronize()
        n, first = first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)
        assert n == 0, first


def test_compressed_then_gather_round_trip(gkr, oracle_mod):
    """Gather the compressed cache back: bit-exact against the oracle's gather of the
    oracle's cache."""
    case = W.compressed_insert("rt", 4, 1000, 4, 528, block_size=64, seed=4, nan_rate=0.001,
                               inf_rate=0.0005)
    ps = case_page_stride(case, oracle_mod)
    kv, slots, pos, csc = device_inputs(case, DEV)
    cache = gkr.alloc_cache(case.num_pages, 64, 528, DEV, fill=SENTINEL)
    gkr.rope_quant_insert(kv, cache, slots, pos, csc, 64, 4, True)
    ref, _ = _oracle(oracle_mod, case, ps, 4, True)
    written = np.unique(case.slots[(case.slots >= 0) & ((case.positions + 1) % 4 == 0)])
    idx = np.concatenate([written, [-1]]).astype(np.int32)
    out = torch.empty(idx.size, 512, dtype=torch.bfloat16, device=DEV)
    gkr.kv_gather(cache, torch.from_numpy(idx).to(DEV), out)
    ref_out, _ = oracle_mod.gather(ref, 528, 64, case.num_pages, ps, idx)
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), ref_out)


@pytest.mark.parametrize("name", ["compressed_v41_r4_262144", "compressed_v41_r128_262144"])
def test_compressed_full_size(gkr, oracle_mod, name):
    case = W.WORKLOADS[name]()
    _compare(gkr, oracle_mod, case, case.meta["compress_ratio"], True)


def test_compressed_rejects_bad_ratio(gkr):
    kv = torch.zeros(4, 512, dtype=torch.bfloat16, device=DEV)
    cache = gkr.alloc_cache(2, 32, 528, DEV)
    e = torch.zeros(4, dtype=torch.int64, device=DEV)
    csc = torch.zeros(4, 64, device=DEV)
    with pytest.raises(ValueError, match="compress_ratio"):
        gkr.rope_quant_insert(kv, cache, e, e, csc, 32, 0)
