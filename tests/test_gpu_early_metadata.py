"""GPU parity with early metadata reads on (the early_metadata launch option): inserts of every
format through the register-load and staged kernels, the compressed insert, gathers and
the benchmark's round-trip graph give the oracle's bytes, and data the kernel just ahead
in the stream writes (kv, the cache) is still read after the wait.  The metadata itself
(slots, positions, indices) is never written by the kernel ahead of its reader here, as
the setting requires."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
import workloads as W
from helpers import (SENTINEL, assert_distinct_slots, bf16_from_bits, bits_of, device_inputs,
                     first_mismatch)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(autouse=True)
def early_metadata(gkr):
    assert gkr.get_pdl()
    with gkr.launch_policy(early_metadata=True):
        yield


@pytest.mark.parametrize("record", [528, 584, 512, 1024])
@pytest.mark.parametrize("T", [17, 1024, 30000])
def test_insert_and_gather_match_oracle(gkr, oracle_mod, record, T):
    bs = 64
    P = max(2, -(-2 * T // bs))
    case = W.random_insert(f"early{record}_{T}", T, 528, bs, P, 4096, 0.08, seed=T + record,
                           outlier_rate=0.01)
    assert_distinct_slots(case.slots)
    scale = 0.05 if record == 512 else None
    sc = None if scale is None else torch.tensor([scale], dtype=torch.float32, device=DEV)
    ps = oracle_mod.page_stride(record, bs)
    kv, slots, pos, csc = device_inputs(case, DEV)
    cache = gkr.alloc_cache(P, bs, record, DEV, fill=SENTINEL)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    gkr.kv_insert(kv, cache, slots, pos, csc, bs, record, err_flag=err, fp8_scale=sc)
    idx = np.concatenate([case.slots, [-1, 0]]).astype(np.int32)
    out = torch.empty(idx.size, 512, dtype=torch.bfloat16, device=DEV)
    gkr.kv_gather(cache, torch.from_numpy(idx).to(DEV), out, err_flag=err, fp8_scale=sc)
    ref = np.full(P * ps, SENTINEL, np.uint8)
    assert oracle_mod.insert(case.kv, ref, record, bs, P, ps, case.slots, case.positions,
                             case.csc, fp8_scale=scale) == 0
    n, first = first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)
    assert n == 0, first
    ref_out, _ = oracle_mod.gather(ref, record, bs, P, ps, idx, fp8_scale=scale)
    assert np.array_equal(bits_of(out), ref_out)
    assert int(err.item()) == 0


def test_compressed_insert_matches_oracle(gkr, oracle_mod):
    case = W.compressed_insert("early_c", 4, 3000, 4, 528, block_size=64, seed=3,
                               nan_rate=0.001)
    ps = oracle_mod.page_stride(528, 64)
    kv, slots, pos, csc = device_inputs(case, DEV)
    cache = gkr.alloc_cache(case.num_pages, 64, 528, DEV, fill=SENTINEL)
    gkr.rope_quant_insert(kv, cache, slots, pos, csc, 64, 4, True, 528)
    ref = np.full(case.num_pages * ps, SENTINEL, np.uint8)
    assert oracle_mod.insert(case.kv, ref, 528, 64, case.num_pages, ps, case.slots,
                             case.positions, case.csc, compress_ratio=4, sanitize_nans=True) == 0
    assert first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)[0] == 0


def test_roundtrip_graph_matches_oracle(gkr, oracle_mod):
    case = W.roundtrip_v41_16384()
    sets = bench.device_sets(case, DEV, bench.ROTATE)
    g = bench.roundtrip_graph(torch, gkr, case, sets, DEV)
    g.replay()
    torch.cuda.synchronize()
    ps = oracle_mod.page_stride(528, 64)
    ref = np.zeros(case.num_pages * ps, np.uint8)
    oracle_mod.insert(case.kv, ref, 528, 64, case.num_pages, ps, case.slots, case.positions,
                      case.csc)
    ref_out, _ = oracle_mod.gather(ref, 528, 64, case.num_pages, ps, case.indices)
    for s in sets:
        assert first_mismatch(gkr.cache_bytes(s["cache"]).cpu().numpy(), ref)[0] == 0
        assert np.array_equal(bits_of(s["out"]), ref_out)


@pytest.mark.parametrize("record", [528, 584])
def test_data_written_just_ahead_is_read_after_the_wait(gkr, oracle_mod, record):
    """Each round a torch kernel rewrites kv right before the insert, and the gather
    reads the cache the insert just wrote; both must see the new data.  Slots, positions
    and indices are written by host copies, never by the kernel just ahead."""
    T, bs, P = 4096, 64, 160
    ps = oracle_mod.page_stride(record, bs)
    rounds = [W.random_insert(f"ahead{r}", T, 528, bs, P, 4096, 0.05, seed=40 + r)
              for r in range(3)]
    kv = torch.empty(T, 512, dtype=torch.bfloat16, device=DEV)
    slots = torch.empty(T, dtype=torch.int64, device=DEV)
    pos = torch.empty(T, dtype=torch.int64, device=DEV)
    idx = torch.empty(T, dtype=torch.int32, device=DEV)
    csc = torch.from_numpy(rounds[0].csc).to(DEV)
    cache = gkr.alloc_cache(P, bs, record, DEV, fill=SENTINEL)
    out = torch.empty(T, 512, dtype=torch.bfloat16, device=DEV)
    ref = np.full(P * ps, SENTINEL, np.uint8)
    for c in rounds:
        slots.copy_(torch.from_numpy(c.slots))
        pos.copy_(torch.from_numpy(c.positions))
        idx.copy_(torch.from_numpy(c.slots.astype(np.int32)))
        src = bf16_from_bits(c.kv, DEV)
        torch.cuda.synchronize()
        torch.mul(src, 1, out=kv)                       # the kernel just ahead writes kv
        gkr.kv_insert(kv, cache, slots, pos, csc, bs, record)
        gkr.kv_gather(cache, idx, out)
        oracle_mod.insert(c.kv, ref, record, bs, P, ps, c.slots, c.positions, c.csc)
        torch.cuda.synchronize()
        assert first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)[0] == 0
        ref_out, _ = oracle_mod.gather(ref, record, bs, P, ps, c.slots.astype(np.int32))
        assert np.array_equal(bits_of(out), ref_out)
