"""GPU parity at the limits of the cache geometry: page strides just under 2^31 bytes, so
record offsets pass 2^32 and every address is 64-bit; slots up to the last row of the last
page; a gather of the last slot.  Whole 6.4 GB backing buffers are compared with the
oracle's byte for byte."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from helpers import SENTINEL, assert_distinct_slots, device_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = torch.device("cuda:0")
STRIDE = (1 << 31) - 512          # a multiple of 512, above every record's page size


@pytest.mark.parametrize("record", [528, 1024])
def test_page_stride_near_two_gigabytes(gkr, oracle_mod, record):
    bs, P, T = 32, 3, 80
    case = W.random_insert("max", T, 528, bs, P, 256, 0.0, seed=record)
    last = P * bs - 1                                            # last row of the last page
    perm = np.random.default_rng(1).permutation(P * bs)
    case.slots[:] = np.concatenate([[last], perm[perm != last]])[:T]   # distinct slots
    assert_distinct_slots(case.slots)
    kv, slots, pos, csc = device_inputs(case, DEV)
    cache = gkr.alloc_cache(P, bs, record, DEV, page_stride_bytes=STRIDE, fill=SENTINEL)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    gkr.kv_insert(kv, cache, slots, pos, csc, bs, record, err_flag=err)
    got = gkr.cache_bytes(cache).cpu().numpy()
    ref = np.full(P * STRIDE, SENTINEL, np.uint8)
    assert oracle_mod.insert(case.kv, ref, record, bs, P, STRIDE, case.slots, case.positions,
                             case.csc) == 0
    assert int(err.item()) == 0
    assert got.size == ref.size and np.array_equal(got, ref)
    idx = torch.tensor([P * bs - 1, -1, int(case.slots[5])], dtype=torch.int32, device=DEV)
    out = torch.empty(3, 512, dtype=torch.bfloat16, device=DEV)
    gkr.kv_gather(cache, idx, out)
    ref_out, _ = oracle_mod.gather(ref, record, bs, P, STRIDE, idx.cpu().numpy())
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), ref_out)
    del cache, got, ref
    torch.cuda.empty_cache()
