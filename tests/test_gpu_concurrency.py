"""Concurrent use: several host threads, each with its own CUDA stream, cache and inputs,
insert and gather at the same time (the library's only shared state is the launch policy,
a mutex-guarded occupancy cache and a thread-local last error).  Every result must equal
the oracle's."""
from __future__ import annotations

import threading

import numpy as np
import pytest
import torch

import workloads as W
from helpers import SENTINEL, device_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def test_threads_on_separate_streams(gkr, oracle_mod):
    jobs = []
    for k, (record, T) in enumerate([(528, 3000), (584, 700), (1024, 40000), (512, 20000),
                                     (528, 150000), (584, 33000)]):
        case = W.random_insert(f"conc{k}", T, 528, 64, -(-2 * T // 64), 4096, 0.05, seed=k)
        jobs.append((record, case, 0.05 if record == 512 else None))
    results = [None] * len(jobs)
    errors = []
    barrier = threading.Barrier(len(jobs))

    def work(i):
        try:
            record, case, scale = jobs[i]
            stream = torch.cuda.Stream(DEV)
            with torch.cuda.stream(stream):
                kv, slots, pos, csc = device_inputs(case, DEV)
                cache = gkr.alloc_cache(case.num_pages, 64, record, DEV, fill=SENTINEL)
                sc = None if scale is None else torch.tensor([scale], device=DEV)
                idx = torch.from_numpy(case.slots.astype(np.int32)).to(DEV)
                out = torch.empty(case.num_tokens, 512, dtype=torch.bfloat16, device=DEV)
                barrier.wait()
                for _ in range(3):
                    gkr.kv_insert(kv, cache, slots, pos, csc, 64, record, fp8_scale=sc)
                    gkr.kv_gather(cache, idx, out, fp8_scale=sc)
            stream.synchronize()
            results[i] = (gkr.cache_bytes(cache).cpu().numpy(),
                          out.cpu().view(torch.int16).numpy().view(np.uint16))
        except Exception as e:            # reported after the join
            errors.append((i, repr(e)))

    threads = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    for (record, case, scale), (got, got_out) in zip(jobs, results):
        ps = oracle_mod.page_stride(record, 64)
        ref = np.full(case.num_pages * ps, SENTINEL, np.uint8)
        oracle_mod.insert(case.kv, ref, record, 64, case.num_pages, ps, case.slots,
                          case.positions, case.csc, fp8_scale=scale)
        assert np.array_equal(got, ref), record
        ref_out, _ = oracle_mod.gather(ref, record, 64, case.num_pages, ps,
                                       case.slots.astype(np.int32), fp8_scale=scale)
        assert np.array_equal(got_out, ref_out), record
