"""Shared helpers for the GPU parity tests (CUDA path vs oracle on the same inputs)."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

SENTINEL = 0xA5


def bf16_from_bits(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def case_page_stride(case, oracle_mod, pad_units: int = 0) -> int:
    align = 512 if case.record == 528 else 576
    base = case.page_stride or oracle_mod.page_stride(case.record, case.block_size)
    return base + pad_units * align


def device_inputs(case, device, tokens: slice | None = None):
    sl = tokens or slice(None)
    kv = bf16_from_bits(case.kv[sl], device)
    slots = torch.from_numpy(np.ascontiguousarray(case.slots[sl])).to(device)
    pos = torch.from_numpy(np.ascontiguousarray(case.positions[sl])).to(device)
    csc = torch.from_numpy(case.csc).to(device)
    return kv, slots, pos, csc


def gpu_insert(gkr, case, device, page_stride: int, fill: int = SENTINEL, err=None):
    """Insert the whole case on the GPU into a sentinel-filled cache; returns the cache view."""
    kv, slots, pos, csc = device_inputs(case, device)
    cache = gkr.alloc_cache(case.num_pages, case.block_size, case.record, device,
                            page_stride_bytes=page_stride, fill=fill)
    gkr.kv_insert(kv, cache, slots, pos, csc, case.block_size, case.record, err_flag=err)
    return cache, kv


def assert_distinct_slots(slots: np.ndarray) -> None:
    """Valid slots must be distinct: two tokens writing one row race (outside the
    contract), so a test built that way would compare an arbitrary winner."""
    v = np.asarray(slots)
    v = v[(v >= 0)]
    assert len(np.unique(v)) == v.size, "test input writes one slot twice"


def oracle_insert(oracle_mod, case, page_stride: int, fill: int = SENTINEL):
    assert_distinct_slots(case.slots)
    cache = np.full(case.num_pages * page_stride, fill, np.uint8)
    err = oracle_mod.insert(case.kv, cache, case.record, case.block_size, case.num_pages,
                            page_stride, case.slots, case.positions, case.csc)
    return cache, err


def first_mismatch(a: np.ndarray, b: np.ndarray, n: int = 8):
    d = np.nonzero(a != b)[0]
    return d.size, [(int(i), int(a[i]), int(b[i])) for i in d[:n]]


# ---------------------------------------------------------------- the oracle at full size
#
# The C oracle runs without the GIL (ctypes releases it for the call), so a full-size
# reference is computed by host threads on disjoint token (index) ranges.  Valid slots are
# distinct, so the ranges write disjoint records of the one shared host cache.

def _ranges(n: int, parts: int):
    edges = np.linspace(0, n, parts + 1).astype(np.int64)
    return [(int(a), int(b)) for a, b in zip(edges[:-1], edges[1:]) if b > a]


def _threads() -> int:
    return max(1, os.cpu_count() or 1)


def oracle_insert_parallel(oracle_mod, kv, cache, record, bs, num_pages, ps, slots, positions,
                           csc, **kw) -> int:
    """oracle_mod.insert over every token, split over host threads; returns the OR of the
    error bits.  kw: compress_ratio, sanitize_nans, fp8_scale."""
    if kw.get("compress_ratio", 1) == 1:
        assert_distinct_slots(slots)      # distinct records: the ranges never overlap
    oracle_mod.e4m3_encode(1.0)        # the oracle fills its e4m3 value table on first use

    def run(r):
        a, b = r
        return oracle_mod.insert(kv[a:b], cache, record, bs, num_pages, ps, slots[a:b],
                                 positions[a:b], csc, **kw)
    n = _threads()
    with ThreadPoolExecutor(n) as ex:
        errs = list(ex.map(run, _ranges(len(slots), 4 * n)))
    err = 0
    for e in errs:
        err |= e
    return err


def oracle_gather_parallel(oracle_mod, cache, record, bs, num_pages, ps, indices, **kw):
    """oracle_mod.gather over every index, split over host threads: (bf16 bits
    [*indices.shape, 512] as uint16, error bits).  kw: fp8_scale."""
    flat = np.ascontiguousarray(indices, dtype=np.int32).reshape(-1)
    out = np.empty((flat.size, 512), np.uint16)

    def run(r):
        a, b = r
        o, e = oracle_mod.gather(cache, record, bs, num_pages, ps, flat[a:b], **kw)
        out[a:b] = o
        return e
    n = _threads()
    with ThreadPoolExecutor(n) as ex:
        errs = list(ex.map(run, _ranges(flat.size, 4 * n)))
    err = 0
    for e in errs:
        err |= e
    return out.reshape(tuple(indices.shape) + (512,)), err


_REFERENCE_CACHES = {}


def oracle_full_cache(oracle_mod, case, record=None, fill=SENTINEL, **kw):
    """The oracle's whole cache for a workload (flat uint8, every byte; kept for the
    session, so the tests that run a workload under several kernels or launch shapes
    compute it once): (cache, error bits, page stride)."""
    record = case.record if record is None else record
    key = (case.name, case.num_tokens, record, fill, tuple(sorted(kw.items())))
    if key not in _REFERENCE_CACHES:
        if len(_REFERENCE_CACHES) >= 2:
            _REFERENCE_CACHES.clear()
        ps = oracle_mod.page_stride(record, case.block_size)
        ref = np.full(case.num_pages * ps, fill, np.uint8)
        err = oracle_insert_parallel(oracle_mod, case.kv, ref, record, case.block_size,
                                     case.num_pages, ps, case.slots, case.positions, case.csc,
                                     **kw)
        _REFERENCE_CACHES[key] = (ref, err, ps)
    return _REFERENCE_CACHES[key]
