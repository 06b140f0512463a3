"""GPU parity: kv_insert through the C ABI vs the CPU oracle, byte for byte.

The whole backing buffer (records, other rows, page padding) starts as the
sentinel 0xA5 on both sides and must match exactly after the insert.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from golden_parse import load_worked, worked_inputs
from helpers import (SENTINEL, bf16_from_bits, case_page_stride, first_mismatch, gpu_insert,
                     oracle_full_cache, oracle_insert)

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


def _compare_whole_cache(gkr, oracle_mod, case, pad_units=0):
    ps = case_page_stride(case, oracle_mod, pad_units)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cache, kv = gpu_insert(gkr, case, DEV, ps, err=err)
    kv_before = case.kv.copy()
    ref, ref_err = oracle_insert(oracle_mod, case, ps)
    got = gkr.cache_bytes(cache).cpu().numpy()
    n, first = first_mismatch(got, ref)
    assert n == 0, f"{case.name}: {n} bytes differ, first {first}"
    assert int(err.item()) == ref_err == 0
    # kv is read only
    assert np.array_equal(kv.cpu().view(torch.int16).numpy().view(np.uint16), kv_before)


@pytest.mark.parametrize("record", [528, 584])
@pytest.mark.parametrize("T", [1, 17, 1023, 1024, 4099])
def test_insert_small_matches_oracle(gkr, oracle_mod, record, T):
    bs = 64 if T > 64 else 32
    pages = max(2, -(-2 * T // bs))
    case = W.random_insert(f"small_{record}_{T}", T, record, bs, pages, 512, 0.1, seed=T,
                           outlier_rate=0.01)
    _compare_whole_cache(gkr, oracle_mod, case)


@pytest.mark.parametrize("record", [528, 584])
@pytest.mark.parametrize("bs,pad", [(32, 1), (64, 3), (96, 2), (128, 0)])
def test_insert_padded_page_strides(gkr, oracle_mod, record, bs, pad):
    case = W.random_insert("padded", 700, record, bs, 24, 300, 0.05, seed=bs + pad,
                           dist="student_t3")
    _compare_whole_cache(gkr, oracle_mod, case, pad_units=pad)


def test_insert_value_extremes(gkr, oracle_mod):
    """Zero rows, subnormal bf16, huge magnitudes, exact scale boundaries."""
    rng = np.random.default_rng(11)
    T = 256
    x = rng.standard_normal((T, 512)).astype(np.float32)
    x[0] = 0.0                                        # amax 0 -> byte 0
    x[1] = 1e-39                                      # bf16 subnormals
    x[2] = 1.0e38 * np.sign(x[2])                     # large (rotation stays finite)
    x[3, :32] = 448.0                                 # amax exactly 448 * 2^0
    x[4] = np.float32(448.0 * 2.0 ** -20)             # exact boundary at a small scale
    x[5] = -0.0
    x[6] = x[6] * 2.0 ** -130
    x[7::2] *= rng.uniform(1e-30, 1e30, (T - 7 + 1) // 2)[:, None].astype(np.float32)
    kv = W.to_bf16_bits(x)
    csc = W.cos_sin_table(64)
    for record in (528, 584):
        case = W.InsertCase("extremes", record, 32, 16, kv, np.arange(T, dtype=np.int64) * 2,
                            rng.integers(0, 64, T), csc)
        _compare_whole_cache(gkr, oracle_mod, case)


@pytest.mark.parametrize("record", [528, 584])
def test_insert_infinities(gkr, oracle_mod, record):
    """+-inf entries in the NoPE dims: a block whose maximum is infinite gets byte 254
    (the exponent clamp at 127) and +-inf is stored as +-448."""
    case = W.compressed_insert(f"inf_{record}", 3, 700, 1, record, block_size=32,
                               skip_rate=0.05, seed=12, inf_rate=0.003, nonfinite_dims=448)
    _compare_whole_cache(gkr, oracle_mod, case)


@pytest.mark.parametrize("record", [528, 584])
def test_insert_golden_worked_example(gkr, record):
    w = load_worked()
    kv_bits, slots, pos, csc = worked_inputs(w)
    ps, expects = w.records[record]
    cache = gkr.alloc_cache(w.num_pages, w.block_size, record, DEV, page_stride_bytes=ps,
                            fill=SENTINEL)
    gkr.kv_insert(bf16_from_bits(kv_bits, DEV), cache, torch.from_numpy(slots).to(DEV),
                  torch.from_numpy(pos).to(DEV), torch.from_numpy(csc).to(DEV), w.block_size,
                  record)
    got = gkr.cache_bytes(cache).cpu().numpy()
    touched = np.zeros(got.size, bool)
    for e in expects:
        D, S = e.data.size, e.scale.size
        assert np.array_equal(got[e.data_offset:e.data_offset + D], e.data), e.token
        assert np.array_equal(got[e.scale_offset:e.scale_offset + S], e.scale), e.token
        touched[e.data_offset:e.data_offset + D] = True
        touched[e.scale_offset:e.scale_offset + S] = True
    assert (got[~touched] == SENTINEL).all()


@pytest.mark.parametrize("record", [528, 584])
def test_insert_all_skipped_writes_nothing(gkr, oracle_mod, record):
    case = W.random_insert("skip", 512, record, 64, 16, 128, 0.0, seed=3)
    case.slots[:] = -1
    ps = case_page_stride(case, oracle_mod)
    cache, _ = gpu_insert(gkr, case, DEV, ps)
    assert (gkr.cache_bytes(cache).cpu().numpy() == SENTINEL).all()


def test_insert_zero_tokens_is_noop(gkr):
    cache = gkr.alloc_cache(2, 32, 528, DEV, fill=SENTINEL)
    e = torch.empty(0, dtype=torch.int64, device=DEV)
    gkr.kv_insert(torch.empty(0, 512, dtype=torch.bfloat16, device=DEV), cache, e, e,
                  torch.ones(4, 64, device=DEV), 32)
    assert (gkr.cache_bytes(cache).cpu().numpy() == SENTINEL).all()


@pytest.mark.parametrize("record", [528, 584])
def test_insert_out_of_range_sets_error_bits(gkr, oracle_mod, record):
    case = W.random_insert("oob", 64, record, 32, 4, 16, 0.0, seed=5)
    case.slots[3] = 4 * 32          # one past the cache
    case.slots[7] = 10 ** 9
    case.positions[9] = 16          # one past the table
    case.positions[11] = -2
    ps = case_page_stride(case, oracle_mod)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cache, _ = gpu_insert(gkr, case, DEV, ps, err=err)
    ref, ref_err = oracle_insert(oracle_mod, case, ps)
    assert ref_err == 3 and int(err.item()) == 3
    n, first = first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)
    assert n == 0, first


@pytest.mark.parametrize("record", [528, 584])
def test_insert_cuda_graph_replay(gkr, oracle_mod, record):
    """Capture one insert in a CUDA graph, then replay it on three rounds of new
    inputs copied into the captured buffers (the last round all -1)."""
    T, bs, P = 1024, 64, 40
    ps = oracle_mod.page_stride(record, bs)
    cases = [W.random_insert("graph", T, record, bs, P, 256, 0.1, seed=20 + r) for r in range(3)]
    cases[2].slots[:] = -1
    kv = torch.empty(T, 512, dtype=torch.bfloat16, device=DEV)
    slots = torch.empty(T, dtype=torch.int64, device=DEV)
    pos = torch.empty(T, dtype=torch.int64, device=DEV)
    csc = torch.from_numpy(cases[0].csc).to(DEV)
    cache = gkr.alloc_cache(P, bs, record, DEV, fill=SENTINEL)
    slots.fill_(-1)
    pos.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gkr.kv_insert(kv, cache, slots, pos, csc, bs, record)   # warm-up (all -1)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gkr.kv_insert(kv, cache, slots, pos, csc, bs, record)
    ref = np.full(P * ps, SENTINEL, np.uint8)
    for c in cases:
        kv.copy_(bf16_from_bits(c.kv, DEV))
        slots.copy_(torch.from_numpy(c.slots))
        pos.copy_(torch.from_numpy(c.positions))
        g.replay()
        oracle_mod.insert(c.kv, ref, record, bs, P, ps, c.slots, c.positions, c.csc)
        torch.cuda.synchronize()
        n, first = first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)
        assert n == 0, first


# ---------------------------------------------------------------- full-size workloads

def test_insert_v41_1024_full(gkr, oracle_mod):
    _compare_whole_cache(gkr, oracle_mod, W.insert_v41_1024())


def test_roundtrip_v41_16384_insert_full(gkr, oracle_mod):
    _compare_whole_cache(gkr, oracle_mod, W.roundtrip_v41_16384())


@pytest.mark.slow
def test_insert_v4_65536_full(gkr, oracle_mod):
    _compare_whole_cache(gkr, oracle_mod, W.insert_v4_65536())


@pytest.mark.slow
def test_insert_v41_262144_full(gkr, oracle_mod):
    """262144 tokens in 8 contiguous sequences: every byte of the 277 MB cache against
    the oracle's (computed once, split over host threads), under each insert kernel."""
    case = W.insert_v41_262144()
    ref, ref_err, ps = oracle_full_cache(oracle_mod, case)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    cache, kv = gpu_insert(gkr, case, DEV, ps, err=err)
    n, first = first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)
    assert n == 0, f"{n} bytes differ, first {first}"
    assert int(err.item()) == ref_err == 0
