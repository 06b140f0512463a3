"""GPU parity in the launch configurations the benchmark times: the round-trip step
(insert 16384 tokens, gather the same slot ids) captured GRAPH_STEPS times over the
rotating input sets in one CUDA graph; the V4 65536-token insert, the ratio-4 compressed
insert, the 262144-token insert and the 1M-token sparse gather captured back to back as
the sweep launches them.  After the replays, every byte of every cache and every row of
every gather output is compared with the oracle's; the full-size references are computed
by the oracle on host threads over disjoint token ranges."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
import workloads as W
from helpers import bits_of, first_mismatch, oracle_full_cache, oracle_gather_parallel

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _distinct_buffers(sets, keys):
    for key in keys:
        ptrs = [s[key].data_ptr() for s in sets]
        assert len(set(ptrs)) == len(ptrs), key


def test_timed_roundtrip_graph_matches_oracle(gkr, oracle_mod):
    case = W.roundtrip_v41_16384()
    sets = bench.device_sets(case, DEV, bench.ROTATE)
    _distinct_buffers(sets, ("kv", "slots", "pos", "idx", "cache", "out"))   # no set shares L2 lines
    g = bench.roundtrip_graph(torch, gkr, case, sets, DEV)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    ps = oracle_mod.page_stride(528, case.block_size)
    ref = np.zeros(case.num_pages * ps, np.uint8)            # device_sets fills caches with 0
    assert oracle_mod.insert(case.kv, ref, 528, case.block_size, case.num_pages, ps, case.slots,
                             case.positions, case.csc) == 0
    ref_out, ref_err = oracle_mod.gather(ref, 528, case.block_size, case.num_pages, ps,
                                         case.indices)
    assert ref_err == 0
    for k, s in enumerate(sets):
        n, first = first_mismatch(gkr.cache_bytes(s["cache"]).cpu().numpy(), ref)
        assert n == 0, f"set {k}: {n} cache bytes differ, first {first}"
        got = bits_of(s["out"])
        assert np.array_equal(got, ref_out), f"set {k}: gather output differs"


@pytest.mark.slow
def test_sweep_v4_65536_graph_matches_oracle(gkr, oracle_mod):
    case = W.insert_v4_65536()
    sets = bench.device_sets(case, DEV, 3)
    _distinct_buffers(sets, ("kv", "cache"))
    g = bench.capture_steps(torch, DEV, lambda k: gkr.kv_insert(
        sets[k % 3]["kv"], sets[k % 3]["cache"], sets[k % 3]["slots"], sets[k % 3]["pos"],
        sets[k % 3]["csc"], case.block_size, case.record), 12)
    g.replay()
    torch.cuda.synchronize()
    ps = oracle_mod.page_stride(584, case.block_size)
    ref = np.zeros(case.num_pages * ps, np.uint8)
    assert oracle_mod.insert(case.kv, ref, 584, case.block_size, case.num_pages, ps, case.slots,
                             case.positions, case.csc) == 0
    for k, s in enumerate(sets):
        n, first = first_mismatch(gkr.cache_bytes(s["cache"]).cpu().numpy(), ref)
        assert n == 0, f"set {k}: {n} cache bytes differ, first {first}"


@pytest.mark.slow
def test_sweep_compressed_r4_graph_matches_oracle(gkr, oracle_mod):
    """The compressed insert as the sweep launches it: input sets reading kv through
    shifted windows of one buffer, 12 launches back to back in a CUDA graph."""
    case = W.compressed_v41_r4_262144()
    R, T = case.meta["compress_ratio"], case.num_tokens
    sets = bench.compressed_sets(case, DEV, bench.compressed_insert_bytes(
        case.slots, case.positions, R, case.record))
    n = len(sets)
    assert n > 1
    _distinct_buffers(sets, ("kv", "slots", "cache"))
    g = bench.capture_steps(torch, DEV, lambda k: gkr.rope_quant_insert(
        sets[k % n]["kv"], sets[k % n]["cache"], sets[k % n]["slots"], sets[k % n]["pos"],
        sets[k % n]["csc"], case.block_size, R, True, case.record), 12)
    g.replay()
    torch.cuda.synchronize()
    ps = oracle_mod.page_stride(case.record, case.block_size)
    kv_all = np.concatenate([case.kv, case.kv[:n]])
    for k in (0, n - 1):
        ref = np.zeros(case.num_pages * ps, np.uint8)
        assert oracle_mod.insert(kv_all[k:k + T], ref, case.record, case.block_size,
                                 case.num_pages, ps, case.slots, case.positions, case.csc,
                                 compress_ratio=R, sanitize_nans=True) == 0
        n_bad, first = first_mismatch(gkr.cache_bytes(sets[k]["cache"]).cpu().numpy(), ref)
        assert n_bad == 0, f"set {k}: {n_bad} cache bytes differ, first {first}"


@pytest.mark.slow
def test_sweep_insert_v41_262144_graph_matches_oracle(gkr, oracle_mod):
    """The 262144-token insert as the sweep launches it: 12 launches back to back in a
    CUDA graph into the same cache; every byte of the cache against the oracle's."""
    case = W.insert_v41_262144()
    s = bench.device_sets(case, DEV, 1)[0]
    g = bench.capture_steps(torch, DEV, lambda k: gkr.kv_insert(
        s["kv"], s["cache"], s["slots"], s["pos"], s["csc"], case.block_size, case.record), 12)
    g.replay()
    torch.cuda.synchronize()
    ref, ref_err, ps = oracle_full_cache(oracle_mod, case, fill=0)   # device_sets fills 0
    assert ref_err == 0
    n, first = first_mismatch(gkr.cache_bytes(s["cache"]).cpu().numpy(), ref)
    assert n == 0, f"{n} cache bytes differ, first {first}"


@pytest.mark.slow
def test_sweep_sparse_gather_graph_matches_oracle(gkr, oracle_mod):
    """The 1M-token sparse gather as the sweep launches it: a cache filled by the insert,
    then 12 gathers of the 128 x 2048 indices back to back in a CUDA graph, alternating
    between two output buffers; the fill byte for byte and every row of both outputs
    against the oracle (its fill, then its gather)."""
    case = W.gather_v41_sparse()
    kv = torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).to(DEV)
    cache = gkr.alloc_cache(case.num_pages, 64, 528, DEV, fill=0)
    gkr.kv_insert(kv, cache, torch.from_numpy(case.slots).to(DEV),
                  torch.from_numpy(case.positions).to(DEV), torch.from_numpy(case.csc).to(DEV),
                  64, 528)
    del kv
    idx = torch.from_numpy(case.indices).to(DEV)
    outs = [torch.empty(case.indices.shape + (512,), dtype=torch.bfloat16, device=DEV)
            for _ in range(2)]
    g = bench.capture_steps(torch, DEV, lambda k: gkr.kv_gather(cache, idx, outs[k % 2]), 12)
    g.replay()
    torch.cuda.synchronize()
    ref, ref_err, ps = oracle_full_cache(oracle_mod, case)
    assert ref_err == 0
    # every slot of the cache is written and V4.1 pages at block 64 have no padding, so
    # the fill value of either side never shows
    n, first = first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)
    assert n == 0, f"fill: {n} cache bytes differ, first {first}"
    ref_out, gerr = oracle_gather_parallel(oracle_mod, ref, 528, 64, case.num_pages, ps,
                                           case.indices)
    assert gerr == 0
    for k, o in enumerate(outs):
        assert np.array_equal(bits_of(o), ref_out), f"output {k} differs"
