"""The KV-only insert test matrix of the pages' test design ("PR #56441 [Perf][DSpark]
KV-only context insertion across V4.1 cache formats", section "实现拆解" item 4), over this
library's four formats: cache format x tokens {1, 17, 1023, 1024} x CUDA graph {off, on}.
Each case runs three rounds with new kv, positions and slots (the third with every slot
-1) into a padded-stride, sentinel-filled cache, compares the whole backing buffer with
the oracle's byte for byte after every round, and checks kv is never modified."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from helpers import SENTINEL, assert_distinct_slots, bf16_from_bits, first_mismatch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.mark.parametrize("record", [528, 584, 512, 1024])
@pytest.mark.parametrize("T", [1, 17, 1023, 1024])
@pytest.mark.parametrize("graph", [False, True])
def test_insert_matrix(gkr, oracle_mod, record, T, graph):
    bs = 64
    P = max(2, -(-2 * T // bs))
    align = 576 if record == 584 else 512
    ps = oracle_mod.page_stride(record, bs) + 2 * align                 # padded pages
    scale = 0.02 if record == 512 else None
    rounds = [W.random_insert(f"m{record}_{T}_{r}", T, 528, bs, P, 300, 0.1, seed=100 * T + r,
                              outlier_rate=0.01) for r in range(3)]
    rounds[2].slots[:] = -1
    kv = torch.empty(T, 512, dtype=torch.bfloat16, device=DEV)
    slots = torch.full((T,), -1, dtype=torch.int64, device=DEV)
    pos = torch.zeros(T, dtype=torch.int64, device=DEV)
    csc = torch.from_numpy(rounds[0].csc).to(DEV)
    sc = None if scale is None else torch.tensor([scale], dtype=torch.float32, device=DEV)
    cache = gkr.alloc_cache(P, bs, record, DEV, page_stride_bytes=ps, fill=SENTINEL)

    def insert():
        gkr.kv_insert(kv, cache, slots, pos, csc, bs, record, fp8_scale=sc)

    g = None
    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            insert()                                   # warm-up with every slot -1
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            insert()
    ref = np.full(P * ps, SENTINEL, np.uint8)
    for c in rounds:
        assert_distinct_slots(c.slots)
        kv_in = bf16_from_bits(c.kv, DEV)
        kv.copy_(kv_in)
        slots.copy_(torch.from_numpy(c.slots))
        pos.copy_(torch.from_numpy(c.positions))
        if g is not None:
            g.replay()
        else:
            insert()
        oracle_mod.insert(c.kv, ref, record, bs, P, ps, c.slots, c.positions, c.csc,
                          fp8_scale=scale)
        torch.cuda.synchronize()
        n, first = first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)
        assert n == 0, f"round {c.name}: {n} bytes differ, first {first}"
        assert torch.equal(kv.view(torch.int16), kv_in.view(torch.int16))  # kv unmodified
