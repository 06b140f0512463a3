"""GPU parity: kv_gather through the C ABI vs the CPU oracle, bit for bit.

Gather inputs are caches built by the oracle (or by the generators), never
by the CUDA insert, so no expected value comes from the CUDA path.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from golden_parse import load_worked, worked_inputs
from helpers import (SENTINEL, bits_of, case_page_stride, first_mismatch, oracle_full_cache,
                     oracle_gather_parallel, oracle_insert)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _cache_from_host(gkr, flat: np.ndarray, num_pages, bs, record, ps):
    cache = gkr.alloc_cache(num_pages, bs, record, DEV, page_stride_bytes=ps)
    gkr.cache_bytes(cache).copy_(torch.from_numpy(flat))
    return cache


def _gather(gkr, cache, idx: np.ndarray, err=None):
    ti = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to(DEV)
    out = torch.full(tuple(idx.shape) + (512,), float("nan"), dtype=torch.bfloat16, device=DEV)
    gkr.kv_gather(cache, ti, out, err_flag=err)
    return bits_of(out)


def _assert_bits_equal(got, ref):
    bad = np.nonzero(got != ref)
    assert bad[0].size == 0, f"{bad[0].size} values differ; first {list(zip(*bad))[:5]} " \
                             f"got {got[bad][:5]} ref {ref[bad][:5]}"


def _exhaustive_cache(record: int):
    """Every (e4m3 code, scale byte) pair once.  V4.1: 128 records of 16 blocks x 32
    codes; V4: records of 7 blocks x 64 codes plus a bf16 tail of all 65536 patterns
    spread over the records."""
    bs = 64
    if record == 528:
        n_rec, nb, blk, D, S = 128, 16, 32, 512, 16
    else:
        n_rec, nb, blk, D, S = 147, 7, 64, 576, 8      # 147 * 7 = 1029 >= 1024 blocks
    P = -(-n_rec // bs)
    ps = bs * record if record == 528 else -(-bs * 584 // 576) * 576
    flat = np.zeros(P * ps, np.uint8)
    tail_pattern = np.arange(65536, dtype=np.uint32)
    for r in range(n_rec):
        page, row = divmod(r, bs)
        b0 = page * ps
        for b in range(nb):
            k = nb * r + b
            codes = (np.arange(blk) + blk * (k // 256)) % 256
            flat[b0 + row * D + blk * b: b0 + row * D + blk * b + blk] = codes
            flat[b0 + bs * D + row * S + b] = k % 256
        if record == 584:
            t = tail_pattern[(64 * r + np.arange(64)) % 65536].astype(np.uint16)
            flat[b0 + row * D + 448: b0 + row * D + 576] = t.view(np.uint8)
            flat[b0 + bs * D + row * S + 7] = 0
    return flat, bs, P, ps, n_rec


@pytest.mark.parametrize("record", [528, 584])
def test_gather_exhaustive_code_scale_table(gkr, oracle_mod, record):
    flat, bs, P, ps, n_rec = _exhaustive_cache(record)
    cache = _cache_from_host(gkr, flat, P, bs, record, ps)
    idx = np.arange(n_rec, dtype=np.int32)
    ref, ref_err = oracle_mod.gather(flat, record, bs, P, ps, idx)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _gather(gkr, cache, idx, err)
    assert ref_err == 0 and int(err.item()) == 0
    _assert_bits_equal(got, ref)


@pytest.mark.parametrize("record", [528, 584])
def test_gather_golden_worked_example(gkr, record):
    w = load_worked()
    kv_bits, slots, pos, csc = worked_inputs(w)
    ps, _ = w.records[record]
    import oracle
    flat = np.full(w.num_pages * ps, SENTINEL, np.uint8)
    oracle.insert(kv_bits, flat, record, w.block_size, w.num_pages, ps, slots, pos, csc)
    cache = _cache_from_host(gkr, flat, w.num_pages, w.block_size, record, ps)
    idx, expect = w.gathers[record]
    got = _gather(gkr, cache, idx)
    assert np.array_equal(got.astype(np.int64), expect)


@pytest.mark.parametrize("record", [528, 584])
@pytest.mark.parametrize("N", [1, 33, 1000, 4097])
def test_gather_random_matches_oracle(gkr, oracle_mod, record, N):
    case = W.random_insert("g", 2048, record, 64, 40, 512, 0.0, seed=N, outlier_rate=0.01)
    ps = case_page_stride(case, oracle_mod)
    flat, _ = oracle_insert(oracle_mod, case, ps)
    cache = _cache_from_host(gkr, flat, case.num_pages, 64, record, ps)
    rng = np.random.default_rng(N)
    idx = rng.integers(-1, 40 * 64, N).astype(np.int32)     # includes -1 and unwritten slots
    ref, _ = oracle_mod.gather(flat, record, 64, case.num_pages, ps, idx)
    _assert_bits_equal(_gather(gkr, cache, idx), ref)


@pytest.mark.parametrize("record", [528, 584])
def test_gather_invalid_indices_zero_and_flag(gkr, oracle_mod, record):
    flat, bs, P, ps, n_rec = _exhaustive_cache(record)
    cache = _cache_from_host(gkr, flat, P, bs, record, ps)
    idx = np.array([[-1, 5, P * bs, -7], [2 ** 31 - 1, -1, 0, -2 ** 31]], np.int32)
    ref, ref_err = oracle_mod.gather(flat, record, bs, P, ps, idx)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    got = _gather(gkr, cache, idx, err)
    assert ref_err == 4 and int(err.item()) == 4
    _assert_bits_equal(got, ref)
    assert (got[0, 0] == 0).all() and (got[0, 2] == 0).all()


def test_gather_zero_indices_is_noop(gkr):
    cache = gkr.alloc_cache(2, 32, 528, DEV, fill=0)
    out = torch.empty(0, 512, dtype=torch.bfloat16, device=DEV)
    gkr.kv_gather(cache, torch.empty(0, dtype=torch.int32, device=DEV), out)


def test_roundtrip_v41_16384_gather_full(gkr, oracle_mod):
    """The round-trip workload: gather every slot of the insert (incl. the -1 slots)."""
    case = W.roundtrip_v41_16384()
    ps = case_page_stride(case, oracle_mod)
    flat, _ = oracle_insert(oracle_mod, case, ps)
    cache = _cache_from_host(gkr, flat, case.num_pages, case.block_size, 528, ps)
    ref, ref_err = oracle_mod.gather(flat, 528, case.block_size, case.num_pages, ps, case.indices)
    got = _gather(gkr, cache, case.indices)
    assert ref_err == 0
    _assert_bits_equal(got, ref)
    # round-trip bound on the non-rotated dims, |x - x_hat| <= 2^-3 * block amax
    x = torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).float()
    xh = torch.from_numpy(got.view(np.int16)).view(torch.bfloat16).float()
    v = torch.from_numpy(case.slots >= 0)
    xb = x[v, :448].reshape(-1, 14, 32)
    err = (xb - xh[v, :448].reshape(-1, 14, 32)).abs().amax(-1)
    assert (err <= xb.abs().amax(-1) / 8).all()
    assert (xh[~v] == 0).all()


@pytest.mark.slow
def test_gather_v41_sparse_full(gkr, oracle_mod):
    """The sparse decode workload at full size: the CUDA insert fills a 1,048,576-token
    cache, compared byte for byte (553 MB) with the oracle's fill; then the 128 x 2048
    gathered rows, every value, against the oracle's gather of the oracle's cache."""
    case = W.gather_v41_sparse()
    ref, ref_err, ps = oracle_full_cache(oracle_mod, case)
    assert ref_err == 0
    kv = torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).to(DEV)
    cache = gkr.alloc_cache(case.num_pages, 64, 528, DEV, fill=SENTINEL)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    gkr.kv_insert(kv, cache, torch.from_numpy(case.slots).to(DEV),
                  torch.from_numpy(case.positions).to(DEV), torch.from_numpy(case.csc).to(DEV),
                  64, 528, err_flag=err)
    del kv
    out = torch.empty(128, 2048, 512, dtype=torch.bfloat16, device=DEV)
    ti = torch.from_numpy(case.indices).to(DEV)
    gkr.kv_gather(cache, ti, out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    n, first = first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)
    assert n == 0, f"fill: {n} bytes differ, first {first}"
    ref_out, gerr = oracle_gather_parallel(oracle_mod, ref, 528, 64, case.num_pages, ps,
                                           case.indices)
    assert gerr == 0
    _assert_bits_equal(bits_of(out), ref_out)


@pytest.mark.parametrize("pdl", [True, False])
@pytest.mark.parametrize("record", [528, 584])
def test_insert_then_gather_same_stream(gkr, oracle_mod, record, pdl):
    """Back-to-back insert -> gather -> insert -> ... on one stream: every gather must
    see the insert queued before it (the programmatic-launch wait keeps stream order)."""
    with gkr.launch_policy(pdl=pdl):
        bs, P = 64, 64
        ps = oracle_mod.page_stride(record, bs)
        cache = gkr.alloc_cache(P, bs, record, DEV, fill=0)
        ref = np.zeros(P * ps, np.uint8)
        outs, refs = [], []
        for r in range(6):
            case = W.random_insert("chain", 2048, record, bs, P, 256, 0.05, seed=40 + r)
            kv = torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).to(DEV)
            gkr.kv_insert(kv, cache, torch.from_numpy(case.slots).to(DEV),
                          torch.from_numpy(case.positions).to(DEV),
                          torch.from_numpy(case.csc).to(DEV), bs, record)
            idx = np.random.default_rng(r).integers(-1, P * bs, 3000).astype(np.int32)
            out = torch.empty(3000, 512, dtype=torch.bfloat16, device=DEV)
            gkr.kv_gather(cache, torch.from_numpy(idx).to(DEV), out)
            outs.append(out)
            oracle_mod.insert(case.kv, ref, record, bs, P, ps, case.slots, case.positions, case.csc)
            refs.append(oracle_mod.gather(ref, record, bs, P, ps, idx)[0])
        torch.cuda.synchronize()
        for out, r in zip(outs, refs):
            _assert_bits_equal(bits_of(out), r)


@pytest.mark.parametrize("record", [528, 584, 512, 1024])
def test_gather_cuda_graph_replay(gkr, oracle_mod, record):
    """Capture one gather in a CUDA graph, then replay it over three rounds of new
    indices copied into the captured buffer (the last round all -1); for the fp8 cache a
    new scale is also written between replays (it is read on the device)."""
    bs, P, N = 64, 40, 1500
    case = W.random_insert("ggraph", 2000, 528, bs, P, 512, 0.0, seed=record)
    ps = oracle_mod.page_stride(record, bs)
    scale0 = 0.05
    sc = torch.tensor([scale0], dtype=torch.float32, device=DEV) if record == 512 else None
    cache = gkr.alloc_cache(P, bs, record, DEV, fill=SENTINEL)
    kv, slots, pos, csc = (torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).to(DEV),
                           torch.from_numpy(case.slots).to(DEV),
                           torch.from_numpy(case.positions).to(DEV),
                           torch.from_numpy(case.csc).to(DEV))
    gkr.kv_insert(kv, cache, slots, pos, csc, bs, record, fp8_scale=sc)
    ref = np.full(P * ps, SENTINEL, np.uint8)
    oracle_mod.insert(case.kv, ref, record, bs, P, ps, case.slots, case.positions, case.csc,
                      fp8_scale=scale0 if record == 512 else None)
    idx = torch.full((N,), -1, dtype=torch.int32, device=DEV)
    out = torch.empty(N, 512, dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gkr.kv_gather(cache, idx, out, fp8_scale=sc)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        gkr.kv_gather(cache, idx, out, fp8_scale=sc)
    rng = np.random.default_rng(record)
    for r, scale in enumerate([scale0, 0.5, 2.0]):
        ind = rng.integers(-1, P * bs, N).astype(np.int32)
        if r == 2:
            ind[:] = -1
        idx.copy_(torch.from_numpy(ind))
        if sc is not None:
            sc.fill_(scale)
        g.replay()
        torch.cuda.synchronize()
        want, _ = oracle_mod.gather(ref, record, bs, P, ps, ind,
                                    fp8_scale=scale if record == 512 else None)
        got = out.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(got, want), (record, r)
