"""Concurrent use: several host threads, each with its own CUDA stream, cache and inputs,
insert and gather at the same time (the library's only shared state is the process-wide
default launch policy, a mutex-guarded occupancy cache and a thread-local last error), with
the defaults or each with its own per-call launch options.  Every result must equal the
oracle's."""
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


def test_threads_with_different_launch_policies(gkr, oracle_mod):
    """Per-call launch options: threads insert and gather at the same time, each under
    its own policy (kernel choice, programmatic dependent launch, early metadata reads),
    with no process-wide setting changed; each thread's results equal the oracle's and
    the process defaults are untouched afterwards."""
    big = 1 << 62
    policies = [dict(insert_staged_min=big, insert_stream_min=big, pdl=True),
                dict(insert_staged_min=0, insert_stream_min=big, pdl=False),
                dict(insert_staged_min=big, insert_stream_min=0, early_metadata=True),
                dict(insert_staged_min=0, insert_stream_min=big, early_metadata=True, pdl=True),
                dict(insert_staged_min=big, insert_stream_min=0, pdl=False)]
    defaults = (gkr.get_pdl(), gkr.get_early_metadata(), gkr.get_insert_staged_min(),
                gkr.get_insert_stream_min())
    jobs = [(528 if k % 2 == 0 else 584,
             W.random_insert(f"pol{k}", 5000 + 700 * k, 528, 64, 200, 4096, 0.05, seed=50 + k))
            for k in range(len(policies))]
    results = [None] * len(jobs)
    kernels = [None] * len(jobs)
    errors = []
    barrier = threading.Barrier(len(jobs))

    def work(i):
        try:
            record, case = jobs[i]
            stream = torch.cuda.Stream(DEV)
            with gkr.launch_policy(**policies[i]), torch.cuda.stream(stream):
                kernels[i] = gkr.insert_kernel_for(case.num_tokens)
                kv, slots, pos, csc = device_inputs(case, DEV)
                cache = gkr.alloc_cache(case.num_pages, 64, record, DEV, fill=SENTINEL)
                idx = torch.from_numpy(case.slots.astype(np.int32)).to(DEV)
                out = torch.empty(case.num_tokens, 512, dtype=torch.bfloat16, device=DEV)
                barrier.wait()
                for _ in range(4):
                    gkr.kv_insert(kv, cache, slots, pos, csc, 64, record)
                    gkr.kv_gather(cache, idx, out)
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
    assert kernels == ["insert_short_kernel", "insert_staged_kernel", "insert_kernel",
                       "insert_staged_kernel", "insert_kernel"]
    assert (gkr.get_pdl(), gkr.get_early_metadata(), gkr.get_insert_staged_min(),
            gkr.get_insert_stream_min()) == defaults
    for (record, case), (got, got_out) in zip(jobs, results):
        ps = oracle_mod.page_stride(record, 64)
        ref = np.full(case.num_pages * ps, SENTINEL, np.uint8)
        oracle_mod.insert(case.kv, ref, record, 64, case.num_pages, ps, case.slots,
                          case.positions, case.csc)
        assert np.array_equal(got, ref), record
        ref_out, _ = oracle_mod.gather(ref, record, 64, case.num_pages, ps,
                                       case.slots.astype(np.int32))
        assert np.array_equal(got_out, ref_out), record
