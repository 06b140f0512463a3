"""Parser for the hand-written golden fixtures tests/golden/worked_*.txt."""
from __future__ import annotations

from dataclasses import dataclass, field
from pathlib import Path

import numpy as np

GOLDEN = Path(__file__).resolve().parent / "golden"


def parse_value(s: str) -> float:
    if "*" in s:
        a, b = s.split("*", 1)
        return float(a) * parse_value(b)
    if "^" in s:
        base, exp = s.split("^", 1)
        return float(base) ** int(exp)
    return float(s)


def _span(tok: str) -> tuple[int, int | None]:
    if ".." in tok:
        a, b = tok.split("..")
        return int(a), int(b)
    return int(tok), None


def _fill(arr: np.ndarray, span_tok: str, values: list) -> None:
    start, end = _span(span_tok)
    if end is None:
        arr[start:start + len(values)] = values
    else:
        n = end - start + 1
        assert n % len(values) == 0, (span_tok, values)
        arr[start:end + 1] = np.tile(np.array(values, dtype=arr.dtype), n // len(values))


@dataclass
class Token:
    name: str
    slot: int
    pos: int
    x: np.ndarray = field(default_factory=lambda: np.zeros(512, np.float64))


@dataclass
class Expect:
    token: str
    data_offset: int
    scale_offset: int
    data: np.ndarray
    scale: np.ndarray


@dataclass
class Worked:
    block_size: int = 0
    num_pages: int = 0
    csc_rows: dict = field(default_factory=dict)
    tokens: list = field(default_factory=list)
    records: dict = field(default_factory=dict)   # record -> (page_stride, [Expect])
    fp8_scale: dict = field(default_factory=dict)  # record -> fp32 scale (fp8 rows)
    gathers: dict = field(default_factory=dict)   # record -> (indices, out uint16 [n,512])
    compress_ratio: int = 1
    sanitize: bool = False
    errors: int = 0                               # expected error bits of the insert


def load_worked(path: Path = GOLDEN / "worked_records.txt") -> Worked:
    w = Worked()
    cur_token = None
    cur_record = None
    cur_expect = None
    cur_gather = None
    for raw in path.read_text(encoding="utf-8").splitlines():
        line = raw.split("#", 1)[0].strip()
        if not line:
            continue
        f = line.split()
        kw = dict(p.split("=", 1) for p in f[1:] if "=" in p)
        if f[0] == "geometry":
            w.block_size = int(kw["block_size"])
            w.num_pages = int(kw["num_pages"])
        elif f[0] == "mode":
            w.compress_ratio = int(kw.get("compress_ratio", 1))
            w.sanitize = bool(int(kw.get("sanitize", 0)))
            w.errors = int(kw.get("errors", 0))
        elif f[0] == "csc_row":
            w.csc_rows[int(f[1])] = (float(kw["cos"]), float(kw["sin"]))
        elif f[0] == "token":
            cur_token = Token(f[1], int(kw["slot"]), int(kw["pos"]))
            w.tokens.append(cur_token)
        elif f[0] == "x":
            _fill(cur_token.x, f[1], [parse_value(v) for v in f[2:]])
        elif f[0] == "record":
            cur_record = int(f[1])
            w.records[cur_record] = (int(kw["page_stride"]), [])
            if "fp8_scale" in kw:
                w.fp8_scale[cur_record] = float(kw["fp8_scale"])
        elif f[0] == "expect":
            D, S = {528: (512, 16), 584: (576, 8), 512: (512, 0), 1024: (1024, 0)}[cur_record]
            cur_expect = Expect(f[1], int(kw["data_offset"]), int(kw.get("scale_offset", 0)),
                                np.full(D, -1, np.int32), np.full(S, -1, np.int32))
            w.records[cur_record][1].append(cur_expect)
        elif f[0] in ("data", "scale"):
            arr = cur_expect.data if f[0] == "data" else cur_expect.scale
            _fill(arr, f[1], [int(v, 16) for v in f[2:]])
        elif f[0] == "gather":
            rec = int(f[1])
            idx = np.array([int(v) for v in kw["indices"].split(",")], np.int32)
            cur_gather = np.full((len(idx), 512), -1, np.int64)
            w.gathers[rec] = (idx, cur_gather)
        elif f[0] == "out":
            _fill(cur_gather[int(f[1])], f[2], [int(v, 16) for v in f[3:]])
        else:
            raise ValueError(f"bad golden line: {raw!r}")
    for _, exps in w.records.values():
        for e in exps:
            assert (e.data >= 0).all() and (e.scale >= 0).all(), "golden record incomplete"
    for _, out in w.gathers.values():
        assert (out >= 0).all(), "golden gather incomplete"
    return w


def worked_inputs(w: Worked):
    """Inputs of the worked example as arrays: kv bf16 bits, slots, positions, csc."""
    import torch
    kv = np.stack([t.x for t in w.tokens]).astype(np.float32)
    kv_bits = torch.from_numpy(kv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # every value in the fixture is exact in bf16 (NaN included: any NaN is NaN)
    assert np.array_equal(torch.from_numpy(kv_bits.view(np.int16)).view(torch.bfloat16)
                          .float().numpy(), kv, equal_nan=True)
    slots = np.array([t.slot for t in w.tokens], np.int64)
    pos = np.array([t.pos for t in w.tokens], np.int64)
    csc = np.zeros((max(w.csc_rows) + 1, 64), np.float32)
    for r, (c, s) in w.csc_rows.items():
        csc[r, :32] = c
        csc[r, 32:] = s
    return kv_bits, slots, pos, csc
