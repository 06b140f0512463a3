"""The C ABI on the CPU: libgkr.so loads, exports every symbol include/gkr.h
declares, and its host-side checks return the documented status codes before
anything touches a GPU (no compute calls here)."""
from __future__ import annotations

import ctypes
import re
import subprocess
from pathlib import Path

import pytest
import torch

ROOT = Path(__file__).resolve().parents[1]
HEADER = ROOT / "include" / "gkr.h"


def declared_symbols() -> set[str]:
    text = HEADER.read_text()
    return set(re.findall(r"GKR_API\s+[\w\s\*]*?\b(gkr_\w+)\s*\(", text))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    assert {"gkr_kv_insert", "gkr_kv_gather", "gkr_page_stride", "gkr_record_rows",
            "gkr_status_string", "gkr_last_cuda_error", "gkr_version", "gkr_set_pdl",
            "gkr_get_pdl", "gkr_set_insert_stream_min", "gkr_get_insert_stream_min",
            "gkr_set_insert_staged_min", "gkr_get_insert_staged_min",
            "gkr_rope_quant_insert", "gkr_set_early_metadata", "gkr_get_early_metadata",
            "gkr_qnorm_rope_kv_insert", "gkr_sparse_logits"} <= syms


def test_library_exports_every_declared_symbol(gkr):
    lib = gkr.lib()
    for name in declared_symbols():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", str(gkr.library_path())],
                         capture_output=True, text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and "gkr_" in l}
    assert declared_symbols() <= exported
    # nothing else of ours leaks out of the library (hidden visibility)
    assert {s for s in exported if s.startswith("gkr")} == declared_symbols()


def test_page_stride_and_rows(gkr):
    assert gkr.page_stride(528, 64) == 33792
    assert gkr.page_stride(584, 64) == 37440
    assert gkr.page_stride(528, 32) == 16896
    assert gkr.page_stride(584, 32) == 19008
    assert gkr.page_stride(500, 64) == -1
    assert gkr.page_stride(528, 48) == -1
    assert gkr.page_stride(528, 0) == -1
    assert gkr.record_rows(528) == (512, 16, 512)
    assert gkr.record_rows(584) == (576, 8, 576)
    assert gkr.record_rows(512) == (512, 0, 512)          # fp8 e4m3 rows
    assert gkr.record_rows(1024) == (1024, 0, 512)        # bf16 rows
    assert gkr.page_stride(512, 48) == 48 * 512           # plain caches: any block size
    assert gkr.page_stride(1024, 1) == 1024
    assert gkr.page_stride(1024, 0) == -1
    with pytest.raises(ValueError):
        gkr.record_rows(500)
    assert gkr.lib().gkr_version() == 30200
    assert gkr.get_insert_stream_min() == 131072
    assert gkr.get_insert_staged_min() == 24576
    assert gkr.insert_kernel_for(16384) == "insert_short_kernel"
    assert gkr.insert_kernel_for(65536) == "insert_staged_kernel"
    assert gkr.insert_kernel_for(262144) == "insert_kernel"


def test_early_metadata_setting_round_trips(gkr):
    assert gkr.get_early_metadata() is False               # off by default
    try:
        gkr.set_early_metadata(True)
        assert gkr.get_early_metadata() is True
        gkr.lib().gkr_set_early_metadata(7)                # any non-zero value means on
        assert gkr.lib().gkr_get_early_metadata() == 1
    finally:
        gkr.set_early_metadata(False)
    assert gkr.get_early_metadata() is False
    gkr.set_insert_stream_min(5)
    gkr.set_insert_staged_min(3)
    assert gkr.get_insert_stream_min() == 5 and gkr.get_insert_staged_min() == 3
    assert gkr.insert_kernel_for(4) == "insert_staged_kernel"
    gkr.set_insert_stream_min(-1)
    gkr.set_insert_staged_min(-1)
    assert gkr.get_insert_stream_min() == 131072 and gkr.get_insert_staged_min() == 24576
    assert gkr.status_string(0) == "ok"


# --- host-side checks through the raw ABI (fake device pointers never reach a kernel:
# every call below fails a host check, or enqueues nothing, before any launch)

A16 = 0x10000          # 16-byte aligned fake pointers: checks must fail before any launch
A16b = 0x20000


def desc(gkr, record=528, bs=64, pages=4, ps=None):
    return gkr.CacheDesc(record, bs, pages, gkr.page_stride(record, bs) if ps is None else ps)


def _o(opts):
    return None if opts is None else ctypes.byref(opts)


def insert(gkr, d, T=8, kv=A16, cache=A16b, slots=A16, pos=A16, csc=A16, max_pos=16, err=None,
           scale=None, opts=None):
    return gkr.lib().gkr_kv_insert(kv, T, cache, None if d is None else ctypes.byref(d),
                                   slots, pos, csc, max_pos, scale, err, _o(opts), None)


def rq_insert(gkr, d, T=8, kv=A16, cache=A16b, slots=A16, pos=A16, csc=A16, max_pos=16,
              ratio=4, sanitize=1, err=None, opts=None):
    return gkr.lib().gkr_rope_quant_insert(kv, T, cache, None if d is None else ctypes.byref(d),
                                           slots, pos, csc, max_pos, ratio, sanitize, err,
                                           _o(opts), None)


def gather(gkr, d, N=8, cache=A16b, idx=A16, out=A16, err=None, scale=None, opts=None):
    return gkr.lib().gkr_kv_gather(cache, None if d is None else ctypes.byref(d), idx, N,
                                   out, scale, err, _o(opts), None)


def qinsert(gkr, d, T=8, q=A16b + 0x1000, H=2, Hp=4, qout=A16b + 0x2000, eps=1e-6, norm=1,
            kv=A16, cache=A16b, slots=A16, pos=A16, csc=A16, max_pos=16, err=None, scale=None,
            opts=None, qscale=None):
    return gkr.lib().gkr_qnorm_rope_kv_insert(q, H, Hp, qout, qscale, eps, norm, kv, T, cache,
                                              None if d is None else ctypes.byref(d), slots, pos,
                                              csc, max_pos, scale, err, _o(opts), None)


def logits(gkr, d, Q=2, H=8, topk=64, q=A16b + 0x1000, cache=A16b, idx=A16, out=A16,
           scale=1.0, fp8=None, err=None, opts=None):
    return gkr.lib().gkr_sparse_logits(q, H, cache, None if d is None else ctypes.byref(d), idx,
                                       Q, topk, scale, fp8, out, err, _o(opts), None)


@pytest.mark.parametrize("op", [insert, rq_insert, gather, qinsert, logits])
def test_geometry_checks(gkr, op):
    assert op(gkr, None) == 1                                        # null descriptor
    assert op(gkr, desc(gkr, record=500)) == 2                       # unsupported record
    assert op(gkr, desc(gkr, bs=48)) == 1                            # block size % 32
    assert op(gkr, desc(gkr, bs=0)) == 1
    assert op(gkr, desc(gkr, pages=0)) == 1
    assert op(gkr, desc(gkr, pages=2 ** 30)) == 1                    # slots >= 2^31
    assert op(gkr, desc(gkr, ps=33792 - 512)) == 3                   # stride too small
    assert op(gkr, desc(gkr, ps=33792 + 16)) == 3                    # not a multiple of 512
    assert op(gkr, desc(gkr, record=584, ps=37440 + 512)) == 3       # not a multiple of 576


def test_insert_argument_checks(gkr):
    d = desc(gkr)
    assert insert(gkr, d, T=-1) == 1
    assert insert(gkr, d, max_pos=0) == 1
    assert insert(gkr, d, T=0, kv=None, cache=None, slots=None, pos=None, csc=None) == 0
    # an empty call reads no cos/sin table: max_pos is not checked, the descriptor is
    assert insert(gkr, d, T=0, max_pos=0, kv=None, cache=None, slots=None, pos=None,
                  csc=None) == 0
    assert rq_insert(gkr, d, T=0, max_pos=0, kv=None, cache=None, slots=None, pos=None,
                     csc=None) == 0
    assert insert(gkr, desc(gkr, record=500), T=0, max_pos=0) == 2
    assert gather(gkr, desc(gkr, bs=48), N=0, cache=None, idx=None, out=None) == 1
    assert insert(gkr, d, kv=None) == 1
    assert insert(gkr, d, csc=None) == 1
    assert insert(gkr, d, kv=A16 + 8) == 4                           # kv not 16-aligned
    assert insert(gkr, d, cache=A16 + 4) == 4
    assert insert(gkr, d, csc=A16 + 8) == 4
    assert insert(gkr, d, slots=A16 + 4) == 4
    assert insert(gkr, d, err=A16 + 2) == 4


@pytest.mark.parametrize("op", [insert, gather])
def test_plain_cache_checks(gkr, op):
    assert op(gkr, desc(gkr, record=1024, bs=48, ps=48 * 1024 + 256)) == 3   # not % 512
    assert op(gkr, desc(gkr, record=1024, bs=48, ps=47 * 1024)) == 3
    assert op(gkr, desc(gkr, record=512, bs=0)) == 1
    assert op(gkr, desc(gkr, record=512)) == 1                        # fp8 without a scale
    assert op(gkr, desc(gkr, record=512), scale=A16 + 2) == 4         # misaligned scale


def test_compressed_insert_rejects_plain_caches(gkr):
    assert rq_insert(gkr, desc(gkr, record=1024)) == 2
    assert rq_insert(gkr, desc(gkr, record=512)) == 2


def test_insert_max_pos_bound(gkr):
    d = desc(gkr)
    assert insert(gkr, d, max_pos=2 ** 31) == 1                       # table rows < 2^31
    assert rq_insert(gkr, d, max_pos=2 ** 31) == 1


def test_rope_quant_insert_argument_checks(gkr):
    d = desc(gkr)
    assert rq_insert(gkr, d, ratio=0) == 1
    assert rq_insert(gkr, d, ratio=-3) == 1
    assert rq_insert(gkr, d, sanitize=2) == 1
    assert rq_insert(gkr, d, T=-1) == 1
    assert rq_insert(gkr, d, max_pos=0) == 1
    assert rq_insert(gkr, d, T=0, kv=None, cache=None, slots=None, pos=None, csc=None) == 0
    assert rq_insert(gkr, d, kv=None) == 1
    assert rq_insert(gkr, d, kv=A16 + 8) == 4
    assert rq_insert(gkr, d, csc=A16 + 8) == 4
    assert rq_insert(gkr, d, pos=A16 + 4) == 4
    assert rq_insert(gkr, desc(gkr, record=584, ps=37440 + 16)) == 3


def test_gather_argument_checks(gkr):
    d = desc(gkr)
    assert gather(gkr, d, N=-1) == 1
    assert gather(gkr, d, N=0, cache=None, idx=None, out=None) == 0
    assert gather(gkr, d, out=None) == 1
    assert gather(gkr, d, out=A16 + 8) == 4
    assert gather(gkr, d, idx=A16 + 2) == 4
    assert gather(gkr, d, cache=A16 + 8) == 4


def test_qnorm_rope_kv_insert_argument_checks(gkr):
    d = desc(gkr)
    assert qinsert(gkr, d, H=-1) == 1
    assert qinsert(gkr, d, H=4, Hp=3) == 1                            # padded below heads
    assert qinsert(gkr, d, Hp=4097) == 1
    assert qinsert(gkr, d, norm=2) == 1
    assert qinsert(gkr, d, eps=-1e-6) == 1
    assert qinsert(gkr, d, eps=float("nan")) == 1
    assert qinsert(gkr, d, eps=float("inf")) == 1
    assert qinsert(gkr, d, T=-1) == 1
    assert qinsert(gkr, d, T=0, q=None, qout=None, kv=None, cache=None, slots=None, pos=None,
                   csc=None, max_pos=0) == 0                           # nothing to do
    assert qinsert(gkr, d, q=None) == 1
    assert qinsert(gkr, d, qout=None) == 1
    assert qinsert(gkr, d, q=A16 + 8) == 4
    assert qinsert(gkr, d, qout=A16 + 8) == 4
    assert qinsert(gkr, d, kv=A16 + 8) == 4
    assert qinsert(gkr, d, kv=None) == 1
    assert qinsert(gkr, desc(gkr, record=512)) == 1                   # fp8 without a scale
    assert qinsert(gkr, desc(gkr, record=500)) == 2
    # an e4m3 query output: its scale 4-byte aligned, its 512-byte rows clear of q_in
    assert qinsert(gkr, d, qscale=A16 + 2) == 4
    assert qinsert(gkr, d, qscale=A16, qout=A16b + 0x2000) == 1       # inside q_in
    assert qinsert(gkr, d, qscale=A16, qout=A16b) == 1                # ends inside q_in


def test_sparse_logits_argument_checks(gkr):
    d = desc(gkr)
    assert logits(gkr, d, H=0) == 1
    assert logits(gkr, d, H=129) == 1                                 # heads beyond one tile
    assert logits(gkr, d, topk=6) == 1                                # not a multiple of 4
    assert logits(gkr, d, Q=-1) == 1
    assert logits(gkr, d, scale=float("inf")) == 1
    assert logits(gkr, d, scale=float("nan")) == 1
    assert logits(gkr, d, Q=0, q=None, cache=None, idx=None, out=None) == 0
    assert logits(gkr, d, topk=0, q=None, cache=None, idx=None, out=None) == 0
    assert logits(gkr, d, q=None) == 1
    assert logits(gkr, d, out=None) == 1
    assert logits(gkr, d, q=A16 + 8) == 4
    assert logits(gkr, d, out=A16 + 4) == 4
    assert logits(gkr, d, idx=A16 + 2) == 4
    assert logits(gkr, desc(gkr, record=512)) == 1                    # fp8 without a scale


@pytest.mark.parametrize("op", [insert, rq_insert, gather, qinsert, logits])
def test_launch_options_are_checked(gkr, op):
    """Per-call launch options: -1 takes the process default; other negative values and
    flags other than 0 / 1 are rejected before anything is enqueued."""
    O = gkr.LaunchOpts
    bad = [O(), O(), O(), O()]
    bad[0].pdl = 2
    bad[1].early_metadata = -2
    bad[2].insert_staged_min = -5
    bad[3].insert_stream_min = -2
    for o in bad:
        assert op(gkr, desc(gkr), opts=o) == 1
    # valid options reach the next check (a misaligned pointer here), not a launch
    misaligned = {insert: dict(kv=A16 + 8), rq_insert: dict(kv=A16 + 8),
                  gather: dict(out=A16 + 8), qinsert: dict(kv=A16 + 8),
                  logits: dict(out=A16 + 8)}[op]
    for o in (O(), O(pdl=False, early_metadata=True, insert_staged_min=0, insert_stream_min=7)):
        assert op(gkr, desc(gkr), opts=o, **misaligned) == 4


def test_launch_policy_is_context_local(gkr):
    """launch_policy sets the options of this thread's calls only (the process defaults
    stay as they are) and nests; an explicit LaunchOpts wins over it."""
    import threading
    assert gkr.insert_kernel_for(16384) == "insert_short_kernel"
    seen = {}
    with gkr.launch_policy(insert_staged_min=0):
        assert gkr.insert_kernel_for(16384) == "insert_staged_kernel"
        with gkr.launch_policy(insert_stream_min=100):
            assert gkr.insert_kernel_for(16384) == "insert_kernel"
            assert gkr.insert_kernel_for(50) == "insert_staged_kernel"
        t = threading.Thread(target=lambda: seen.update(k=gkr.insert_kernel_for(16384)))
        t.start()
        t.join()
        assert gkr.get_insert_staged_min() == 24576            # the process default is untouched
        eff = gkr._binding._opts(gkr.LaunchOpts(insert_staged_min=30000))._obj
        assert eff.insert_staged_min == 30000 and eff.insert_stream_min == -1
    assert seen["k"] == "insert_short_kernel"                   # the other thread saw defaults
    assert gkr.insert_kernel_for(16384) == "insert_short_kernel"
    assert gkr._binding._opts(None) is None


def test_status_strings(gkr):
    for s in range(6):
        assert gkr.status_string(s)
    assert "unknown" in gkr.status_string(99)


# --- Python binding checks (raise before calling into the library)

def _cpu_args(T=4, record=528, bs=32):
    kv = torch.zeros(T, 512, dtype=torch.bfloat16)
    cache = torch.as_strided(torch.zeros(2 * 16896, dtype=torch.uint8), (2, bs, record),
                             (16896, record, 1))
    slots = torch.zeros(T, dtype=torch.int64)
    pos = torch.zeros(T, dtype=torch.int64)
    csc = torch.zeros(8, 64, dtype=torch.float32)
    return kv, cache, slots, pos, csc


def test_binding_rejects_bad_tensors(gkr):
    kv, cache, slots, pos, csc = _cpu_args()
    with pytest.raises(ValueError, match="kv must be"):
        gkr.kv_insert(kv.float(), cache, slots, pos, csc, 32)
    with pytest.raises(ValueError, match="kv must be"):
        gkr.kv_insert(kv[:, :256], cache, slots, pos, csc, 32)
    with pytest.raises(ValueError, match="slot_mapping"):
        gkr.kv_insert(kv, cache, slots.int(), pos, csc, 32)
    with pytest.raises(ValueError, match="cos_sin_cache"):
        gkr.kv_insert(kv, cache, slots, pos, csc.double(), 32)
    with pytest.raises(ValueError, match="block_size"):
        gkr.kv_insert(kv, cache, slots, pos, csc, 64)
    with pytest.raises(ValueError, match="record"):
        gkr.kv_insert(kv, cache, slots, pos, csc, 32, record=584)
    with pytest.raises(ValueError, match="width"):
        bad = torch.zeros(2, 32, 512, dtype=torch.uint8)
        gkr.kv_insert(kv, bad, slots, pos, csc, 32)
    with pytest.raises(ValueError, match="positions must cover"):
        gkr.kv_insert(kv, cache, slots, pos[:2], csc, 32)
    with pytest.raises(ValueError, match="CUDA"):
        gkr.kv_insert(kv, cache, slots, pos, csc, 32)          # CPU tensors: no CPU path
    with pytest.raises(ValueError, match="compress_ratio"):
        gkr.rope_quant_insert(kv, cache, slots, pos, csc, 32, compress_ratio=0)
    with pytest.raises(ValueError, match="compress_ratio"):             # would wrap in int32
        gkr.rope_quant_insert(kv, cache, slots, pos, csc, 32, compress_ratio=2**32 + 4)
    with pytest.raises(ValueError, match="kv must be"):
        gkr.rope_quant_insert(kv.float(), cache, slots, pos, csc, 32, 4)
    with pytest.raises(ValueError, match="CUDA"):
        gkr.rope_quant_insert(kv, cache, slots, pos, csc, 32, 4, True)
    idx = torch.zeros(3, dtype=torch.int32)
    with pytest.raises(ValueError, match="out must be"):
        gkr.kv_gather(cache, idx, torch.zeros(3, 256, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="indices"):
        gkr.kv_gather(cache, idx.long(), torch.zeros(3, 512, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="CUDA"):
        gkr.kv_gather(cache, idx, torch.zeros(3, 512, dtype=torch.bfloat16))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    import gather_kv_rope_gb300._binding as b
    monkeypatch.setattr(b, "LIB", tmp_path / "nope.so")
    monkeypatch.setattr(b, "_lib", None)
    with pytest.raises(RuntimeError, match="no fallback"):
        b.lib()
