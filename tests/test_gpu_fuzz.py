"""Randomised GPU parity: 48 seeded configurations drawn across every format (528, 584,
fp8 rows, bf16 rows), every insert kernel (register loads, shared-memory staging,
streaming ring), the compressed insert (ratios 1-8 and 128, with and without NaN
sanitising), padded page strides, block sizes, skip rates, value distributions and fp8
scales, with early metadata reads on or off; each insert is compared byte for byte with
the oracle over the whole sentinel-filled backing buffer, then a gather of random indices
(valid, -1 and out of range) bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from helpers import SENTINEL, assert_distinct_slots, device_inputs, first_mismatch

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BIG = 1 << 62


def _config(seed: int) -> dict:
    rng = np.random.default_rng(1000 + seed)
    record = int(rng.choice([528, 584, 512, 1024]))
    packed = record in (528, 584)
    bs = int(rng.choice([32, 64, 96])) if packed else int(rng.choice([16, 48, 64, 80]))
    T = int(rng.choice([1, 7, 33, 500, 1777, 3000]))
    pages = max(2, int(np.ceil(T * rng.uniform(1.05, 3.0) / bs)))
    compressed = packed and rng.random() < 0.4
    return dict(
        record=record, bs=bs, T=T, pages=pages, pad=int(rng.integers(0, 3)),
        skip=float(rng.choice([0.0, 0.05, 0.5])), dist=str(rng.choice(["normal", "student_t3"])),
        outliers=float(rng.choice([0.0, 0.01])), mode=str(rng.choice(["short", "staged", "stream"])),
        compressed=compressed, ratio=int(rng.choice([1, 2, 3, 4, 8, 128])) if compressed else 1,
        sanitize=bool(rng.random() < 0.5) if compressed else False,
        scale=float(np.float32(2.0 ** rng.uniform(-10, 10))) if record == 512 else None,
        max_pos=int(rng.choice([64, 1000, 5000])),
        early=bool(rng.random() < 0.5))      # drawn last: the earlier draws are unchanged


@pytest.mark.parametrize("seed", range(48))
def test_random_configuration_matches_oracle(gkr, oracle_mod, seed):
    c = _config(seed)
    staged_min, stream_min = {"short": (BIG, BIG), "staged": (0, BIG), "stream": (BIG, 0)}[c["mode"]]
    with gkr.launch_policy(insert_staged_min=staged_min, insert_stream_min=stream_min,
                           early_metadata=c["early"]):
        case = W.random_insert(f"fuzz{seed}", c["T"], 528, c["bs"], c["pages"], c["max_pos"],
                               c["skip"], seed=seed, dist=c["dist"], outlier_rate=c["outliers"])
        record, bs, P = c["record"], c["bs"], c["pages"]
        assert_distinct_slots(case.slots)
        align = 576 if record == 584 else 512
        ps = oracle_mod.page_stride(record, bs) + c["pad"] * align
        kv, slots, pos, csc = device_inputs(case, DEV)
        cache = gkr.alloc_cache(P, bs, record, DEV, page_stride_bytes=ps, fill=SENTINEL)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        scale_t = None if c["scale"] is None else torch.tensor([c["scale"]], device=DEV)
        if c["compressed"]:
            gkr.rope_quant_insert(kv, cache, slots, pos, csc, bs, c["ratio"], c["sanitize"],
                                  record, err_flag=err)
        else:
            gkr.kv_insert(kv, cache, slots, pos, csc, bs, record, err_flag=err, fp8_scale=scale_t)
        ref = np.full(P * ps, SENTINEL, np.uint8)
        ref_err = oracle_mod.insert(case.kv, ref, record, bs, P, ps, case.slots, case.positions,
                                    case.csc, compress_ratio=c["ratio"],
                                    sanitize_nans=c["sanitize"], fp8_scale=c["scale"])
        got = gkr.cache_bytes(cache).cpu().numpy()
        n, first = first_mismatch(got, ref)
        assert n == 0, f"{c}: {n} bytes differ, first {first}"
        assert int(err.item()) == ref_err, c

        rng = np.random.default_rng(2000 + seed)
        N = int(rng.integers(1, 2000))
        idx = rng.integers(-1, P * bs, N).astype(np.int32)
        idx[rng.random(N) < 0.02] = P * bs + 5                   # past the cache
        out = torch.empty(N, 512, dtype=torch.bfloat16, device=DEV)
        gerr = torch.zeros(1, dtype=torch.int32, device=DEV)
        gkr.kv_gather(cache, torch.from_numpy(idx).to(DEV), out, err_flag=gerr, fp8_scale=scale_t)
        ref_out, ref_gerr = oracle_mod.gather(ref, record, bs, P, ps, idx, fp8_scale=c["scale"])
        got_out = out.cpu().view(torch.int16).numpy().view(np.uint16)
        n, first = first_mismatch(got_out.reshape(-1), ref_out.reshape(-1))
        assert n == 0, f"{c}: gather differs at {n} values, first {first}"
        assert int(gerr.item()) == ref_gerr
