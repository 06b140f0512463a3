"""GPU parity in the launch configurations the benchmark times: the round-trip step
(insert 16384 tokens, gather the same slot ids) captured GRAPH_STEPS times over the
rotating input sets in one CUDA graph; the V4 65536-token insert, the ratio-4 compressed
insert, the 262144-token insert and the 1M-token sparse gather captured back to back as
the sweep launches them.  Caches and gather outputs are compared with the oracle after the
replays: in full, or on sampled records and rows at the largest sizes."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bench
import workloads as W
from helpers import bits_of, first_mismatch

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
def test_sweep_insert_v41_262144_graph_matches_oracle_sampled(gkr, oracle_mod):
    """The 262144-token insert as the sweep launches it: 12 launches back to back in a
    CUDA graph into the same cache; sampled records against the oracle's encoding."""
    case = W.insert_v41_262144()
    s = bench.device_sets(case, DEV, 1)[0]
    g = bench.capture_steps(torch, DEV, lambda k: gkr.kv_insert(
        s["kv"], s["cache"], s["slots"], s["pos"], s["csc"], case.block_size, case.record), 12)
    g.replay()
    torch.cuda.synchronize()
    got = gkr.cache_bytes(s["cache"]).cpu().numpy()
    ps, bs = oracle_mod.page_stride(528, case.block_size), case.block_size
    rng = np.random.default_rng(5)
    valid = np.nonzero(case.slots >= 0)[0]
    for t in np.concatenate([valid[:4], valid[-4:], rng.choice(valid, 1500, replace=False)]):
        d, sc = oracle_mod.encode(528, case.kv[t], case.csc[case.positions[t]])
        page, row = divmod(int(case.slots[t]), bs)
        b = page * ps
        assert np.array_equal(got[b + row * 512: b + row * 512 + 512], d), t
        assert np.array_equal(got[b + bs * 512 + row * 16: b + bs * 512 + row * 16 + 16], sc), t


@pytest.mark.slow
def test_sweep_sparse_gather_graph_matches_oracle_sampled(gkr, oracle_mod):
    """The 1M-token sparse gather as the sweep launches it: a cache filled by the insert,
    then 12 gathers of the 128 x 2048 indices back to back in a CUDA graph, alternating
    between two output buffers; sampled rows of both against the oracle's decode of its
    own encoding (and zeros for -1)."""
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
    flat = case.indices.reshape(-1)
    rng = np.random.default_rng(6)
    pick = np.concatenate([rng.choice(flat.size, 1500, replace=False),
                           np.nonzero(flat == -1)[0][:32]])
    for o in outs:
        got = bits_of(o).reshape(-1, 512)
        for i in pick:
            sl = int(flat[i])
            if sl < 0:
                assert (got[i] == 0).all(), i
                continue
            d, sc = oracle_mod.encode(528, case.kv[sl], case.csc[case.positions[sl]])
            assert np.array_equal(got[i], oracle_mod.decode(528, d, sc)), i
