"""GPU parity of the sparse decode logits (sparse_logits through the C ABI: the top-k
records gathered and dequantised on chip, the products on the tensor cores) against the
oracle: -inf exactly at the invalid entries, every other value within the fp32
accumulation bound 2^-13 * |sm_scale| * sum_d |q_d K_d| of the oracle's float64 value.
Caches are built by the oracle (or, at full size, by the CUDA insert compared with the
oracle's byte for byte first), so no expected value comes from the CUDA path."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads as W
from helpers import first_mismatch, oracle_full_cache, oracle_gather_parallel
from test_oracle_qside import bf16_bits

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
REL = 2.0 ** -13     # fp32 accumulation of 512 exact products: 512 * 2^-23 = 2^-14, x2 margin


def _host_cache(oracle_mod, record, T, bs, pages, seed, scale=None):
    c = W.random_insert(f"lg{record}_{T}", T, 528, bs, pages, 4096, 0.0, seed=seed)
    ps = oracle_mod.page_stride(record, bs)
    flat = np.zeros(pages * ps, np.uint8)
    oracle_mod.insert(c.kv, flat, record, bs, pages, ps, c.slots, c.positions, c.csc,
                      fp8_scale=scale)
    return c, flat, ps


def _to_device_cache(gkr, flat, pages, bs, record, ps):
    cache = gkr.alloc_cache(pages, bs, record, DEV, page_stride_bytes=ps)
    gkr.cache_bytes(cache).copy_(torch.from_numpy(flat))
    return cache


def _indices(rng, Q, topk, slots, bad_rate=0.0, skip_rate=0.05, num_slots=None):
    idx = np.stack([rng.choice(slots, topk, replace=False) for _ in range(Q)]).astype(np.int32)
    idx[rng.random(idx.shape) < skip_rate] = -1
    if bad_rate:
        idx[rng.random(idx.shape) < bad_rate] = num_slots + 7
    return idx


def _check(got: np.ndarray, exact: np.ndarray, bound: np.ndarray):
    inf = np.isneginf(exact)
    assert np.array_equal(np.isneginf(got), inf), "the -inf entries differ"
    err = np.abs(got[~inf] - exact[~inf])
    tol = REL * bound[~inf] + 1e-30
    worst = float(np.max(err / np.maximum(bound[~inf], 1e-30))) if err.size else 0.0
    assert (err <= tol).all(), f"{int((err > tol).sum())} logits outside the bound; " \
                               f"worst error / sum|q k| = {worst:.3e}"
    return worst


@pytest.mark.parametrize("record", [528, 584, 512, 1024])
@pytest.mark.parametrize("Q,H,topk", [(1, 1, 4), (1, 128, 256), (3, 64, 260), (2, 7, 2048),
                                      (5, 128, 516)])
def test_matches_oracle(gkr, oracle_mod, record, Q, H, topk):
    bs, pages = 64, 48
    scale = 0.03 if record == 512 else None
    c, flat, ps = _host_cache(oracle_mod, record, pages * bs, bs, pages, seed=Q + H + topk,
                              scale=scale)
    rng = np.random.default_rng(topk + H)
    idx = _indices(rng, Q, topk, np.arange(pages * bs), bad_rate=0.01, num_slots=pages * bs)
    q = bf16_bits(rng.standard_normal((Q, H, 512)).astype(np.float32))
    cache = _to_device_cache(gkr, flat, pages, bs, record, ps)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    fp8 = None if scale is None else torch.tensor([scale], dtype=torch.float32, device=DEV)
    out = gkr.sparse_logits(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(DEV),
                            cache, torch.from_numpy(idx).to(DEV), 0.0625, err_flag=err,
                            fp8_scale=fp8)
    torch.cuda.synchronize()
    exact, bound, ref_err = oracle_mod.sparse_logits(q, flat, record, bs, pages, ps, idx, 0.0625,
                                                     fp8_scale=scale)
    _check(out.cpu().numpy(), exact, bound)
    assert int(err.item()) == ref_err == (oracle_mod.ERR_INDEX if (idx >= pages * bs).any() else 0)


def test_scales_and_magnitudes(gkr, oracle_mod):
    """Negative and tiny sm_scale, large and small query magnitudes."""
    bs, pages = 64, 16
    c, flat, ps = _host_cache(oracle_mod, 528, pages * bs, bs, pages, seed=7)
    cache = _to_device_cache(gkr, flat, pages, bs, 528, ps)
    rng = np.random.default_rng(8)
    idx = _indices(rng, 2, 512, np.arange(pages * bs))
    for sm, mag in ((-0.5, 1.0), (1e-6, 1e3), (3.0, 1e-3), (0.0, 1.0)):
        q = bf16_bits(rng.standard_normal((2, 96, 512)).astype(np.float32) * np.float32(mag))
        out = gkr.sparse_logits(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(DEV),
                                cache, torch.from_numpy(idx).to(DEV), sm)
        exact, bound, _ = oracle_mod.sparse_logits(q, flat, 528, bs, pages, ps, idx, sm)
        _check(out.cpu().numpy(), exact, bound)


def test_bad_fp8_scale_gives_minus_inf(gkr, oracle_mod):
    bs, pages = 64, 8
    c, flat, ps = _host_cache(oracle_mod, 512, pages * bs, bs, pages, seed=9, scale=0.5)
    cache = _to_device_cache(gkr, flat, pages, bs, 512, ps)
    idx = np.arange(64, dtype=np.int32).reshape(1, 64)
    q = torch.randn(1, 4, 512).to(torch.bfloat16).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gkr.sparse_logits(q, cache, torch.from_numpy(idx).to(DEV), 1.0, err_flag=err,
                            fp8_scale=torch.tensor([float("inf")], device=DEV))
    assert torch.isneginf(out).all() and int(err.item()) == gkr.ERR_SCALE


@pytest.mark.parametrize("record", [528, 584])
def test_many_queries_per_cta(gkr, oracle_mod, record):
    """400 queries of 132 entries: two items per query (the second one 4 entries long), so
    every CTA's run crosses several queries and reloads the query tile between products;
    40 heads leave the last head quarter partly empty."""
    bs, pages, Q, H, K = 64, 40, 400, 40, 132
    c, flat, ps = _host_cache(oracle_mod, record, pages * bs, bs, pages, seed=21)
    rng = np.random.default_rng(22)
    idx = _indices(rng, Q, K, np.arange(pages * bs), bad_rate=0.005, num_slots=pages * bs)
    q = bf16_bits(rng.standard_normal((Q, H, 512)).astype(np.float32))
    cache = _to_device_cache(gkr, flat, pages, bs, record, ps)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gkr.sparse_logits(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(DEV),
                            cache, torch.from_numpy(idx).to(DEV), -0.03, err_flag=err)
    torch.cuda.synchronize()
    exact, bound, ref_err = oracle_mod.sparse_logits(q, flat, record, bs, pages, ps, idx, -0.03)
    _check(out.cpu().numpy(), exact, bound)
    assert int(err.item()) == ref_err


@pytest.mark.parametrize("record", [528, 512])
def test_one_chunk_per_query(gkr, oracle_mod, record):
    """700 queries of 100 entries: one item per query, several per CTA, so every item
    starts a new query (the chunk count wraps at each item) and reloads the query tile."""
    bs, pages, Q, H, K = 64, 40, 700, 16, 100
    scale = 0.05 if record == 512 else None
    c, flat, ps = _host_cache(oracle_mod, record, pages * bs, bs, pages, seed=31, scale=scale)
    rng = np.random.default_rng(32)
    idx = _indices(rng, Q, K, np.arange(pages * bs), bad_rate=0.01, num_slots=pages * bs)
    q = bf16_bits(rng.standard_normal((Q, H, 512)).astype(np.float32))
    cache = _to_device_cache(gkr, flat, pages, bs, record, ps)
    kw = {} if scale is None else {"fp8_scale": torch.tensor([scale], dtype=torch.float32, device=DEV)}
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gkr.sparse_logits(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(DEV),
                            cache, torch.from_numpy(idx).to(DEV), 0.07, err_flag=err, **kw)
    torch.cuda.synchronize()
    exact, bound, ref_err = oracle_mod.sparse_logits(q, flat, record, bs, pages, ps, idx, 0.07,
                                                     fp8_scale=scale)
    _check(out.cpu().numpy(), exact, bound)
    assert int(err.item()) == ref_err


@pytest.mark.parametrize("seed", range(48))
def test_random_configurations(gkr, oracle_mod, seed):
    """48 seeded draws over the record formats, block sizes, cache sizes, query counts
    (runs within one query and across many), head counts (full and partial lane
    quarters), top-k (multiples of 4 from 4 to 700, one to six chunks), fp8 scales, query
    magnitudes, sm_scale signs and invalid-index rates."""
    rng = np.random.default_rng(7000 + seed)
    record = int(rng.choice([528, 584, 512, 1024]))
    bs = int(rng.choice([32, 64, 96])) if record in (528, 584) else int(rng.choice([16, 48, 64]))
    pages = int(rng.integers(4, 40))
    Q = int(rng.choice([1, 3, 40, 300]))
    H = int(rng.choice([1, 16, 33, 64, 100, 128]))
    K = int(rng.choice([4, 8, 100, 128, 132, 260, 700]))
    pages = max(pages, -(-K // bs) + 1)   # enough slots for K distinct indices
    scale = float(np.float32(2.0 ** rng.uniform(-8, 2))) if record == 512 else None
    sm = float(rng.choice([0.0625, -0.03, 1.0]))
    c, flat, ps = _host_cache(oracle_mod, record, pages * bs, bs, pages, seed=seed, scale=scale)
    idx = _indices(rng, Q, K, np.arange(pages * bs), bad_rate=float(rng.choice([0.0, 0.02])),
                   num_slots=pages * bs)
    q = bf16_bits((rng.standard_normal((Q, H, 512)) * rng.choice([0.1, 1.0, 30.0]))
                  .astype(np.float32))
    cache = _to_device_cache(gkr, flat, pages, bs, record, ps)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    kw = {} if scale is None else {"fp8_scale": torch.tensor([scale], dtype=torch.float32,
                                                             device=DEV)}
    out = gkr.sparse_logits(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(DEV),
                            cache, torch.from_numpy(idx).to(DEV), sm, err_flag=err, **kw)
    torch.cuda.synchronize()
    exact, bound, ref_err = oracle_mod.sparse_logits(q, flat, record, bs, pages, ps, idx, sm,
                                                     fp8_scale=scale)
    _check(out.cpu().numpy(), exact, bound)
    assert int(err.item()) == ref_err


def test_graph_replay_and_launch_options(gkr, oracle_mod):
    """Captured once (programmatic dependent launch off by option), replayed over new
    queries and indices copied into the captured buffers."""
    bs, pages, Q, H, K = 64, 32, 4, 128, 1024
    c, flat, ps = _host_cache(oracle_mod, 584, pages * bs, bs, pages, seed=10)
    cache = _to_device_cache(gkr, flat, pages, bs, 584, ps)
    qd = torch.empty(Q, H, 512, dtype=torch.bfloat16, device=DEV)
    idxd = torch.empty(Q, K, dtype=torch.int32, device=DEV)
    out = torch.empty(Q, H, K, dtype=torch.float32, device=DEV)
    qd.normal_()
    idxd.fill_(-1)
    fn = lambda: gkr.sparse_logits(qd, cache, idxd, 0.1, out=out,
                                   launch_opts=gkr.LaunchOpts(pdl=False))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    rng = np.random.default_rng(11)
    for r in range(2):
        q = bf16_bits(rng.standard_normal((Q, H, 512)).astype(np.float32))
        idx = _indices(rng, Q, K, np.arange(pages * bs))
        qd.copy_(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16))
        idxd.copy_(torch.from_numpy(idx))
        g.replay()
        torch.cuda.synchronize()
        exact, bound, _ = oracle_mod.sparse_logits(q, flat, 584, bs, pages, ps, idx, 0.1)
        _check(out.cpu().numpy(), exact, bound)


@pytest.mark.slow
def test_sparse_decode_full_size(gkr, oracle_mod):
    """The sparse decode workload at full size: 128 queries x 2048 indices over the
    1,048,576-token cache filled by the CUDA insert (checked byte for byte against the
    oracle's fill), 128 heads; every logit against the oracle's."""
    case = W.gather_v41_sparse()
    ref, ref_err, ps = oracle_full_cache(oracle_mod, case)
    kv = torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).to(DEV)
    cache = gkr.alloc_cache(case.num_pages, 64, 528, DEV, fill=0)
    gkr.kv_insert(kv, cache, torch.from_numpy(case.slots).to(DEV),
                  torch.from_numpy(case.positions).to(DEV), torch.from_numpy(case.csc).to(DEV),
                  64, 528)
    del kv
    q = W.decode_queries(case.indices.shape[0], 128)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = gkr.sparse_logits(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).to(DEV),
                            cache, torch.from_numpy(case.indices).to(DEV), 512 ** -0.5,
                            err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert first_mismatch(gkr.cache_bytes(cache).cpu().numpy(), ref)[0] == 0
    got = out.cpu().numpy()
    for a in range(0, 128, 32):        # the oracle in slices of 32 queries (memory)
        exact, bound, e = oracle_mod.sparse_logits(q[a:a + 32], ref, 528, 64, case.num_pages, ps,
                                                   case.indices[a:a + 32], 512 ** -0.5)
        assert e == 0
        _check(got[a:a + 32], exact, bound)
