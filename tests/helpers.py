"""Shared helpers for the GPU parity tests (CUDA path vs oracle on the same inputs)."""
from __future__ import annotations

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


def written_mask(case, page_stride: int) -> np.ndarray:
    """Bytes of the flat cache covered by the records of the valid slots."""
    D, S = (512, 16) if case.record == 528 else (576, 8)
    bs = case.block_size
    m = np.zeros(case.num_pages * page_stride, bool)
    v = case.slots[case.slots >= 0]
    page, row = v // bs, v % bs
    d0 = page * page_stride + row * D
    s0 = page * page_stride + bs * D + row * S
    for off, n in ((d0, D), (s0, S)):
        idx = (off[:, None] + np.arange(n)[None, :]).reshape(-1)
        m[idx] = True
    return m
