"""CPU oracle for the paged KV insert / dequant-gather path.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the library in
``gather_kv_rope_gb300`` never does, and the two share no code.

The arithmetic lives in ``gkr_oracle.c`` (plain C, compiled with
``-O2 -ffp-contract=off -fno-fast-math``); this module only compiles it with
gcc and marshals numpy arrays through ctypes.  Every function cites the page
passage it follows in the C source.

Pinning status (what each function is checked against, on the CPU):
  e4m3 encode / decode  -- torch.float8_e4m3fn casts (all codes, all midpoints)
  bf16 encode / decode  -- torch.bfloat16 casts
  UE8M0 scale byte      -- exact rational ceil(log2(amax/448)), all bf16 amax
  RoPE pair             -- hand-computed exact cases, special angles
  record encoders       -- hand-written golden records (tests/golden)
  page placement        -- hand-computed byte offsets, brute-force tiny caches
  gather / decode       -- exhaustive code x scale table vs decode definition
  compressed insert     -- hand-written golden records (group boundaries, the
                           group's cos/sin row, NaN -> 0, infinite maxima)
  bf16 / fp8 caches     -- hand-written golden rows; torch bfloat16 / float8_e4m3fn
                           casts of the numpy-float32 rotation and fp32 quotient
  sparse logits         -- the pinned gather followed by a float64 matrix product (a
                           library routine); one-hot queries reduce it to the gather,
                           hand-built records give closed-form sums
  query side (q norm + q rotation) -- closed forms (constant rows, sqrt(2) cases),
                           unit RMS, scale invariance, rotation invariants, hand-written
                           golden heads; zero heads reduce to the KV insert.  The norm
                           formula itself is a reading of the pages (they print only the
                           op's name and arguments): parity unpinned against the pages
                           for the norm, pinned for everything else.
  e4m3 query output     -- closed-form codes of hand-built heads, the fp8 cache row
                           it reduces to without the norm, the scale's edge cases.
                           The scale's meaning (one fp32 divisor per call) is a
                           reading: parity unpinned against the pages for it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "gkr_oracle.c"
_OUT = _HERE / "_build" / "liboracle.so"

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-fvisibility=hidden", "-std=c11", "-Wall", "-Wextra"]

ERR_SLOT = 1
ERR_POS = 2
ERR_INDEX = 4
ERR_SCALE = 8


def build(force: bool = False) -> Path:
    """Compile the oracle with gcc (a second or so).  Returns the .so path."""
    if not force and _OUT.exists() and _OUT.stat().st_mtime >= _SRC.stat().st_mtime:
        return _OUT
    _OUT.parent.mkdir(parents=True, exist_ok=True)
    tmp = _OUT.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["gcc", *CFLAGS, "-o", str(tmp), str(_SRC), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _OUT)
    return _OUT


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(str(build()))
        u8, u16, i32, i64 = ctypes.c_uint8, ctypes.c_uint16, ctypes.c_int, ctypes.c_int64
        vp, f32, f64 = ctypes.c_void_p, ctypes.c_float, ctypes.c_double
        L.oracle_e4m3_value.argtypes, L.oracle_e4m3_value.restype = [u8], f64
        L.oracle_e4m3_encode.argtypes, L.oracle_e4m3_encode.restype = [f64], u8
        L.oracle_bf16_value.argtypes, L.oracle_bf16_value.restype = [u16], f64
        L.oracle_bf16_encode.argtypes, L.oracle_bf16_encode.restype = [f64], u16
        L.oracle_ue8m0_byte.argtypes, L.oracle_ue8m0_byte.restype = [f32], u8
        L.oracle_rope_pair.argtypes = [f32, f32, f32, f32, vp, vp]
        L.oracle_rope_pair.restype = None
        L.oracle_encode_v41.argtypes = [vp, vp, vp, vp]
        L.oracle_encode_v41.restype = None
        L.oracle_encode_v4.argtypes = [vp, vp, vp, vp]
        L.oracle_encode_v4.restype = None
        L.oracle_insert.argtypes = [vp, i64, vp, i32, i32, i64, i64, vp, vp, vp, i64]
        L.oracle_insert.restype = i32
        L.oracle_rope_quant_insert.argtypes = [vp, i64, vp, i32, i32, i64, i64, vp, vp, vp,
                                               i64, i64, i32]
        L.oracle_rope_quant_insert.restype = i32
        L.oracle_kv_insert.argtypes = [vp, i64, vp, i32, i32, i64, i64, vp, vp, vp, i64, f32]
        L.oracle_kv_insert.restype = i32
        L.oracle_kv_gather.argtypes = [vp, i32, i32, i64, i64, vp, i64, f32, vp]
        L.oracle_kv_gather.restype = i32
        L.oracle_decode.argtypes = [vp, vp, i32, vp]
        L.oracle_decode.restype = None
        L.oracle_gather.argtypes = [vp, i32, i32, i64, i64, vp, i64, vp]
        L.oracle_gather.restype = i32
        L.oracle_q_head.argtypes = [vp, vp, f64, i32, vp, vp, vp, vp, vp]
        L.oracle_q_head.restype = None
        L.oracle_qnorm_rope_kv_insert.argtypes = [vp, i32, i32, f64, i32, vp, vp, vp, vp, vp,
                                                  i64, vp, i32, i32, i64, i64, vp, vp, vp, i64,
                                                  f32]
        L.oracle_qnorm_rope_kv_insert.restype = i32
        L.oracle_q_head_fp8.argtypes = [vp, vp, f64, i32, f32, vp, vp, vp]
        L.oracle_q_head_fp8.restype = None
        L.oracle_qnorm_rope_fp8q.argtypes = [vp, i32, i32, f64, i32, f32, i64, vp, vp, i64,
                                             vp, vp, vp]
        L.oracle_qnorm_rope_fp8q.restype = i32
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


# --- scalar number-format helpers ------------------------------------------------

def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(code)


def e4m3_encode(y: float) -> int:
    return lib().oracle_e4m3_encode(float(y))


def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(bits)


def bf16_encode(y: float) -> int:
    return lib().oracle_bf16_encode(float(y))


def ue8m0_byte(amax: float) -> int:
    return lib().oracle_ue8m0_byte(float(amax))


def rope_pair(e: float, o: float, c: float, s: float) -> tuple[float, float]:
    eo, oo = ctypes.c_float(), ctypes.c_float()
    lib().oracle_rope_pair(e, o, c, s, ctypes.byref(eo), ctypes.byref(oo))
    return eo.value, oo.value


# --- records ----------------------------------------------------------------------

def record_rows(record: int) -> tuple[int, int]:
    """(data row bytes, scale row bytes) of a cache format, from its definition:
    528 / 584 packed MXFP8 records, 512 fp8 e4m3 rows, 1024 bf16 rows."""
    if record == 528:
        return 512, 16
    if record == 584:
        return 576, 8
    if record in (512, 1024):
        return record, 0
    raise ValueError(f"unknown record width {record}")


def encode(record: int, kv_row: np.ndarray, csc_row: np.ndarray):
    """Encode one token (bf16 bits [512], fp32 cos/sin row [64]) -> (data, scales)."""
    kv_row = np.ascontiguousarray(kv_row, dtype=np.uint16)
    csc_row = np.ascontiguousarray(csc_row, dtype=np.float32)
    assert kv_row.shape == (512,) and csc_row.shape == (64,)
    D, S = record_rows(record)
    data = np.zeros(D, np.uint8)
    scales = np.zeros(S, np.uint8)
    fn = lib().oracle_encode_v41 if record == 528 else lib().oracle_encode_v4
    fn(_ptr(kv_row), _ptr(csc_row), _ptr(data), _ptr(scales))
    return data, scales


def insert(kv: np.ndarray, cache: np.ndarray, record: int, block_size: int,
           num_pages: int, page_stride: int, slots: np.ndarray,
           positions: np.ndarray, csc: np.ndarray, compress_ratio: int = 1,
           sanitize_nans: bool = False, fp8_scale: float | None = None) -> int:
    """Insert into a flat uint8 host cache of num_pages * page_stride bytes, in place.
    compress_ratio > 1 or sanitize_nans selects the compressed-KV insert (a token is
    written only at a group boundary, rotated with the group's first cos/sin row;
    NaN -> 0 after rotation).  Records 512 (fp8 e4m3 rows, fp8_scale required) and
    1024 (bf16 rows) are the plain caches.  Returns the error bits."""
    kv = np.ascontiguousarray(kv, dtype=np.uint16).reshape(-1, 512)
    slots = np.ascontiguousarray(slots, dtype=np.int64).reshape(-1)
    positions = np.ascontiguousarray(positions, dtype=np.int64).reshape(-1)
    csc = np.ascontiguousarray(csc, dtype=np.float32).reshape(-1, 64)
    assert cache.dtype == np.uint8 and cache.flags["C_CONTIGUOUS"]
    assert cache.size >= num_pages * page_stride
    T = slots.shape[0]
    assert kv.shape[0] == T and positions.shape[0] == T
    if record in (512, 1024):
        assert compress_ratio == 1 and not sanitize_nans
        err = lib().oracle_kv_insert(_ptr(kv), T, _ptr(cache), record, block_size, num_pages,
                                     page_stride, _ptr(slots), _ptr(positions), _ptr(csc),
                                     csc.shape[0], 1.0 if fp8_scale is None else fp8_scale)
    elif compress_ratio == 1 and not sanitize_nans:
        err = lib().oracle_insert(_ptr(kv), T, _ptr(cache), record, block_size, num_pages,
                                  page_stride, _ptr(slots), _ptr(positions), _ptr(csc),
                                  csc.shape[0])
    else:
        err = lib().oracle_rope_quant_insert(_ptr(kv), T, _ptr(cache), record, block_size,
                                             num_pages, page_stride, _ptr(slots),
                                             _ptr(positions), _ptr(csc), csc.shape[0],
                                             int(compress_ratio), int(bool(sanitize_nans)))
    if err < 0:
        raise ValueError(f"unknown record width {record} or compress ratio {compress_ratio}")
    return err


def decode(record: int, data: np.ndarray, scales: np.ndarray) -> np.ndarray:
    data = np.ascontiguousarray(data, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    out = np.zeros(512, np.uint16)
    lib().oracle_decode(_ptr(data), _ptr(scales), record, _ptr(out))
    return out


def gather(cache: np.ndarray, record: int, block_size: int, num_pages: int,
           page_stride: int, indices: np.ndarray, fp8_scale: float | None = None):
    """Returns (bf16 bits [*indices.shape, 512] as uint16, error bits).  fp8_scale is
    required for record 512 (fp8 e4m3 rows)."""
    idx = np.ascontiguousarray(indices, dtype=np.int32)
    flat = idx.reshape(-1)
    out = np.zeros((flat.shape[0], 512), np.uint16)
    assert cache.dtype == np.uint8 and cache.flags["C_CONTIGUOUS"]
    if record in (512, 1024):
        err = lib().oracle_kv_gather(_ptr(cache), record, block_size, num_pages, page_stride,
                                     _ptr(flat), flat.shape[0],
                                     1.0 if fp8_scale is None else fp8_scale, _ptr(out))
    else:
        err = lib().oracle_gather(_ptr(cache), record, block_size, num_pages, page_stride,
                                  _ptr(flat), flat.shape[0], _ptr(out))
    if err < 0:
        raise ValueError(f"unknown record width {record}")
    return out.reshape(*idx.shape, 512), err


def page_stride(record: int, block_size: int) -> int:
    """Page stride for a record: block_size * record bytes rounded up to the page
    alignment (576 for the 584 B record, 512 for every other format)."""
    align = 576 if record == 584 else 512
    need = block_size * record
    return -(-need // align) * align


# --- fused query-side write ------------------------------------------------------

def q_head(q_row: np.ndarray, csc_row: np.ndarray, eps: float, apply_norm: bool = True,
           bounds: bool = False):
    """One query head (bf16 bits [512]) -> (exact values float64 [512], nearest-even bf16
    bits, the other faithful bf16 bits), plus with bounds=True the lowest and highest bf16
    (bits) an fp32 evaluation in any order may give."""
    q_row = np.ascontiguousarray(q_row, dtype=np.uint16)
    csc_row = np.ascontiguousarray(csc_row, dtype=np.float32)
    assert q_row.shape == (512,) and csc_row.shape == (64,)
    exact = np.zeros(512, np.float64)
    rn, alt, lo, hi = (np.zeros(512, np.uint16) for _ in range(4))
    lib().oracle_q_head(_ptr(q_row), _ptr(csc_row), float(eps), int(bool(apply_norm)),
                        _ptr(exact), _ptr(rn), _ptr(alt), _ptr(lo), _ptr(hi))
    return (exact, rn, alt, lo, hi) if bounds else (exact, rn, alt)


def qnorm_rope_kv_insert(q: np.ndarray, num_heads_padded: int, eps: float, apply_norm: bool,
                         kv: np.ndarray, cache: np.ndarray, record: int, block_size: int,
                         num_pages: int, page_stride: int, slots: np.ndarray,
                         positions: np.ndarray, csc: np.ndarray,
                         fp8_scale: float | None = None):
    """The fused op on the host: q bf16 bits [T, H, 512]; the KV rows go into the flat
    cache in place.  Returns (q_rn, q_alt, q_lo, q_hi, error bits): the nearest-even bf16
    query output [T, num_heads_padded, 512], the other faithful rounding of each value,
    and the lowest / highest bf16 an fp32 evaluation in any order may give."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    T = int(np.asarray(slots).shape[0])
    q = q.reshape(T, -1, 512)
    H = q.shape[1]
    assert num_heads_padded >= H
    kv = np.ascontiguousarray(kv, dtype=np.uint16).reshape(-1, 512)
    slots = np.ascontiguousarray(slots, dtype=np.int64).reshape(-1)
    positions = np.ascontiguousarray(positions, dtype=np.int64).reshape(-1)
    csc = np.ascontiguousarray(csc, dtype=np.float32).reshape(-1, 64)
    assert cache.dtype == np.uint8 and cache.flags["C_CONTIGUOUS"]
    assert kv.shape[0] == T and positions.shape[0] == T
    q_rn, q_alt, q_lo, q_hi = (np.zeros((T, num_heads_padded, 512), np.uint16)
                               for _ in range(4))
    err = lib().oracle_qnorm_rope_kv_insert(
        _ptr(q), H, int(num_heads_padded), float(eps), int(bool(apply_norm)), _ptr(q_rn),
        _ptr(q_alt), _ptr(q_lo), _ptr(q_hi), _ptr(kv), T, _ptr(cache), record, block_size,
        num_pages, page_stride, _ptr(slots), _ptr(positions), _ptr(csc), csc.shape[0],
        1.0 if fp8_scale is None else fp8_scale)
    if err < 0:
        raise ValueError(f"unknown record width {record}")
    return q_rn, q_alt, q_lo, q_hi, err


def q_head_fp8(q_row: np.ndarray, csc_row: np.ndarray, eps: float, q_scale: float,
               apply_norm: bool = True):
    """One query head (bf16 bits [512]) cast to e4m3 with the fp32 scale q_scale ->
    (nearest codes, lowest codes, highest codes) uint8 [512]: e4m3(RN32(x / q_scale)) for
    x = the fp32 nearest the exact value, and for the smallest / largest fp32 an fp32
    evaluation of the head in any order may give (lowest / highest by value)."""
    q_row = np.ascontiguousarray(q_row, dtype=np.uint16)
    csc_row = np.ascontiguousarray(csc_row, dtype=np.float32)
    assert q_row.shape == (512,) and csc_row.shape == (64,)
    rn, lo, hi = (np.zeros(512, np.uint8) for _ in range(3))
    lib().oracle_q_head_fp8(_ptr(q_row), _ptr(csc_row), float(eps), int(bool(apply_norm)),
                            float(q_scale), _ptr(rn), _ptr(lo), _ptr(hi))
    return rn, lo, hi


def qnorm_rope_fp8q(q: np.ndarray, num_heads_padded: int, eps: float, apply_norm: bool,
                    q_scale: float, positions: np.ndarray, csc: np.ndarray):
    """The query side of the fused op with an e4m3 output: q bf16 bits [T, H, 512] ->
    (codes_rn, codes_lo, codes_hi, error bits), codes uint8 [T, num_heads_padded, 512]
    (see q_head_fp8; padded heads, heads of a token with a position outside the table, and
    every head under a q_scale that is not a positive finite number are +0)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    positions = np.ascontiguousarray(positions, dtype=np.int64).reshape(-1)
    T = positions.shape[0]
    q = q.reshape(T, -1, 512)
    H = q.shape[1]
    assert num_heads_padded >= H
    csc = np.ascontiguousarray(csc, dtype=np.float32).reshape(-1, 64)
    rn, lo, hi = (np.zeros((T, num_heads_padded, 512), np.uint8) for _ in range(3))
    err = lib().oracle_qnorm_rope_fp8q(_ptr(q), H, int(num_heads_padded), float(eps),
                                       int(bool(apply_norm)), float(q_scale), T,
                                       _ptr(positions), _ptr(csc), csc.shape[0], _ptr(rn),
                                       _ptr(lo), _ptr(hi))
    return rn, lo, hi, err


# --- sparse decode logits (the gather fused into its consumer) --------------------

def bf16_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (a bf16 is the top half of an fp32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    with np.errstate(invalid="ignore"):          # NaN patterns stay NaN
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def sparse_logits(q: np.ndarray, cache: np.ndarray, record: int, block_size: int,
                  num_pages: int, page_stride: int, indices: np.ndarray, sm_scale: float,
                  fp8_scale: float | None = None):
    """FlashMLA overview page, DSA section: each query i attends to the entries its
    index row lists (-1 = invalid), the FP8 entries dequantised to bf16 before the
    product.  Here: logits[i, h, k] = sm_scale * sum_d q[i, h, d] * K[i, k, d], K the bf16
    rows of the oracle's gather, computed in float64 (every product of two bf16 values is
    exact there, and the 512-term sum is within 2^-44 of the exact value relative to the
    sum of |terms|).  An entry whose gather row is not a record (index -1 or outside the
    cache, or every entry of an fp8 cache with a bad scale) gives -inf.
    q: bf16 bits [Q, H, 512]; indices int32 [Q, K].  Returns (logits float64 [Q, H, K],
    bound float64 [Q, H, K] = |sm_scale| * sum_d |q d * K d|, error bits)."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    idx = np.ascontiguousarray(indices, dtype=np.int32)
    Q, H = q.shape[0], q.shape[1]
    rows, err = gather(cache, record, block_size, num_pages, page_stride, idx.reshape(-1),
                       fp8_scale=fp8_scale)
    keys = bf16_to_float(rows).reshape(Q, idx.shape[1], 512)
    qv = bf16_to_float(q)
    logits = np.matmul(qv, keys.transpose(0, 2, 1)) * float(sm_scale)
    bound = np.matmul(np.abs(qv), np.abs(keys).transpose(0, 2, 1)) * abs(float(sm_scale))
    valid = (idx >= 0) & (idx < num_pages * block_size)
    if record == 512 and not (fp8_scale is not None and np.isfinite(fp8_scale) and fp8_scale > 0):
        valid[:] = False
    logits = np.where(valid[:, None, :], logits, -np.inf)
    return logits, bound, err
