"""ctypes binding of libgkr.so: argument checks and marshalling only.

Every step of the hot path runs in the library's CUDA kernels; this module
only validates torch tensors, builds the cache descriptor and passes raw
device pointers plus torch's current CUDA stream.  There is no fallback: if
the library is not built, or a tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import contextlib
import contextvars
import ctypes
import threading
from pathlib import Path

import torch

from .build import LIB

GKR_OK = 0
GKR_EINVAL = 1
GKR_EUNSUPPORTED_RECORD = 2
GKR_EBAD_PAGE_GEOMETRY = 3
GKR_EALIGN = 4
GKR_ECUDA = 5

ERR_SLOT = 1
ERR_POS = 2
ERR_INDEX = 4
ERR_SCALE = 8
ERR_TIMEOUT = 16

# cache formats by record width (bytes a token occupies): the packed MXFP8 records
# (uint8 [pages, block, 528 | 584]) and the plain caches of 512 elements a row
# (float8_e4m3fn [pages, block, 512] -> record 512; bfloat16 [...] -> record 1024)
RECORDS = (528, 584, 512, 1024)
PACKED = (528, 584)
HEAD_DIM = 512


class GkrError(RuntimeError):
    """A non-OK status returned by the C ABI."""

    def __init__(self, status: int, message: str):
        super().__init__(f"gkr status {status}: {message}")
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("record", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("page_stride", ctypes.c_int64)]


class LaunchOpts(ctypes.Structure):
    """gkr_launch_opts: per-call launch options; -1 = the process-wide default."""
    _fields_ = [("pdl", ctypes.c_int32), ("early_metadata", ctypes.c_int32),
                ("insert_staged_min", ctypes.c_int64), ("insert_stream_min", ctypes.c_int64)]

    def __init__(self, pdl=None, early_metadata=None, insert_staged_min=None,
                 insert_stream_min=None):
        def flag(v):
            return -1 if v is None else int(bool(v))

        def count(v):
            return -1 if v is None else int(v)
        super().__init__(flag(pdl), flag(early_metadata), count(insert_staged_min),
                         count(insert_stream_min))

    def merged(self, other: "LaunchOpts | None") -> "LaunchOpts":
        """These options with every field that `other` sets taken from `other`."""
        out = LaunchOpts()
        for name, _ in self._fields_:
            v = getattr(other, name) if other is not None else -1
            setattr(out, name, v if v != -1 else getattr(self, name))
        return out


# Launch options of the calls made in the current thread / context (launch_policy), so
# that concurrent users of the library never change each other's launches.
_POLICY: contextvars.ContextVar = contextvars.ContextVar("gkr_launch_policy", default=None)


@contextlib.contextmanager
def launch_policy(**fields):
    """Within the block, calls from this thread (context) pass these launch options
    (pdl, early_metadata, insert_staged_min, insert_stream_min) to the library, on top
    of any enclosing launch_policy; an explicit launch_opts= argument wins over both."""
    cur = _POLICY.get()
    new = (cur or LaunchOpts()).merged(LaunchOpts(**fields))
    token = _POLICY.set(new)
    try:
        yield new
    finally:
        _POLICY.reset(token)


def _opts(launch_opts):
    """The options pointer of a call: launch_opts over the context's launch_policy."""
    cur = _POLICY.get()
    if launch_opts is not None and not isinstance(launch_opts, LaunchOpts):
        raise ValueError("launch_opts must be a LaunchOpts")
    eff = launch_opts if cur is None else cur.merged(launch_opts)
    return None if eff is None else ctypes.byref(eff)


_lib = None
_lock = threading.Lock()


def library_path() -> Path:
    return LIB


def lib() -> ctypes.CDLL:
    """Load libgkr.so (built in-tree by gather_kv_rope_gb300.build())."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not LIB.exists():
                    raise RuntimeError(f"{LIB} is missing: run gather_kv_rope_gb300.build() "
                                       "(the CUDA library is required; there is no fallback)")
                L = ctypes.CDLL(str(LIB))
                vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
                L.gkr_page_stride.argtypes, L.gkr_page_stride.restype = [i32, i32], i64
                L.gkr_record_rows.argtypes = [i32, vp, vp, vp]
                L.gkr_record_rows.restype = ctypes.c_int
                opt = ctypes.POINTER(LaunchOpts)
                # kv, T, k_cache, desc, slots, positions, csc, max_pos, fp8_scale, err, opts,
                # stream
                L.gkr_kv_insert.argtypes = [vp, i64, vp, ctypes.POINTER(CacheDesc), vp, vp, vp, i64,
                                            vp, vp, opt, vp]
                L.gkr_kv_insert.restype = ctypes.c_int
                L.gkr_rope_quant_insert.argtypes = [vp, i64, vp, ctypes.POINTER(CacheDesc), vp,
                                                    vp, vp, i64, i32, i32, vp, opt, vp]
                L.gkr_rope_quant_insert.restype = ctypes.c_int
                L.gkr_kv_gather.argtypes = [vp, ctypes.POINTER(CacheDesc), vp, i64, vp, vp, vp,
                                            opt, vp]
                L.gkr_kv_gather.restype = ctypes.c_int
                # q_in, H, Hp, q_out, q_scale, eps, apply_q_norm, then gkr_kv_insert's
                # arguments
                L.gkr_qnorm_rope_kv_insert.argtypes = [vp, i32, i32, vp, vp, ctypes.c_float, i32,
                                                       vp, i64, vp, ctypes.POINTER(CacheDesc), vp,
                                                       vp, vp, i64, vp, vp, opt, vp]
                L.gkr_qnorm_rope_kv_insert.restype = ctypes.c_int
                # q, H, k_cache, desc, indices, Q, topk, sm_scale, fp8_scale, out, err, opts,
                # stream
                L.gkr_sparse_logits.argtypes = [vp, i32, vp, ctypes.POINTER(CacheDesc), vp, i64,
                                                i64, ctypes.c_float, vp, vp, vp, opt, vp]
                L.gkr_sparse_logits.restype = ctypes.c_int
                L.gkr_status_string.argtypes, L.gkr_status_string.restype = [ctypes.c_int], \
                    ctypes.c_char_p
                L.gkr_last_cuda_error.argtypes, L.gkr_last_cuda_error.restype = [], i32
                L.gkr_version.argtypes, L.gkr_version.restype = [], i32
                L.gkr_set_pdl.argtypes, L.gkr_set_pdl.restype = [i32], None
                L.gkr_get_pdl.argtypes, L.gkr_get_pdl.restype = [], i32
                L.gkr_set_early_metadata.argtypes = [i32]
                L.gkr_set_early_metadata.restype = None
                L.gkr_get_early_metadata.argtypes, L.gkr_get_early_metadata.restype = [], i32
                L.gkr_set_insert_stream_min.argtypes = [i64]
                L.gkr_set_insert_stream_min.restype = None
                L.gkr_get_insert_stream_min.argtypes, L.gkr_get_insert_stream_min.restype = [], i64
                L.gkr_set_insert_staged_min.argtypes = [i64]
                L.gkr_set_insert_staged_min.restype = None
                L.gkr_get_insert_staged_min.argtypes, L.gkr_get_insert_staged_min.restype = [], i64
                _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().gkr_status_string(status).decode()


def _raise(status: int) -> None:
    if status == GKR_OK:
        return
    msg = status_string(status)
    if status == GKR_ECUDA:
        msg += f" (cudaError {lib().gkr_last_cuda_error()})"
        raise GkrError(status, msg)
    raise ValueError(f"gkr status {status}: {msg}")


def set_pdl(enable: bool) -> None:
    """Turn programmatic dependent launch on or off for later launches (process-wide)."""
    lib().gkr_set_pdl(1 if enable else 0)


def get_pdl() -> bool:
    return bool(lib().gkr_get_pdl())


def set_early_metadata(enable: bool) -> None:
    """Let later inserts read slot_mapping / positions, and gathers read indices, before
    waiting for the kernel ahead of them in the stream (process-wide, default off).  Only
    for streams where that kernel never writes those arrays."""
    lib().gkr_set_early_metadata(1 if enable else 0)


def get_early_metadata() -> bool:
    return bool(lib().gkr_get_early_metadata())


def set_insert_stream_min(tokens: int) -> None:
    """Token count from which inserts use the streaming kernel (negative = default)."""
    lib().gkr_set_insert_stream_min(int(tokens))


def get_insert_stream_min() -> int:
    return int(lib().gkr_get_insert_stream_min())


def set_insert_staged_min(tokens: int) -> None:
    """Token count from which inserts below the streaming threshold use the staged
    kernel (negative = default)."""
    lib().gkr_set_insert_staged_min(int(tokens))


def get_insert_staged_min() -> int:
    return int(lib().gkr_get_insert_staged_min())


def insert_kernel_for(num_tokens: int) -> str:
    """Name of the kernel kv_insert launches for `num_tokens` under the current policy
    (the process defaults, overridden by the context's launch_policy)."""
    cur = _POLICY.get()
    stream_min = get_insert_stream_min() if cur is None or cur.insert_stream_min < 0 \
        else cur.insert_stream_min
    staged_min = get_insert_staged_min() if cur is None or cur.insert_staged_min < 0 \
        else cur.insert_staged_min
    if num_tokens < stream_min:
        return "insert_short_kernel" if num_tokens < staged_min else "insert_staged_kernel"
    return "insert_kernel"


def page_stride(record: int, block_size: int) -> int:
    """Smallest valid page stride for a record and block size (-1 if unsupported)."""
    return int(lib().gkr_page_stride(record, block_size))


def record_rows(record: int) -> tuple[int, int, int]:
    """(data row bytes, scale row bytes, page alignment) of a record."""
    d, s, a = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _raise(lib().gkr_record_rows(record, ctypes.byref(d), ctypes.byref(s), ctypes.byref(a)))
    return d.value, s.value, a.value


def alloc_cache(num_pages: int, block_size: int, record: int, device="cuda",
                page_stride_bytes: int | None = None, fill: int | None = None) -> torch.Tensor:
    """Allocate a paged cache whose stride(0) is the page stride (padded to the
    record's alignment): uint8 [num_pages, block_size, record] for the packed records
    (inside a page the bytes are a data region then a scale region, not row by row),
    float8_e4m3fn [num_pages, block_size, 512] for record 512, bfloat16
    [num_pages, block_size, 512] for record 1024.  `fill` sets every byte."""
    ps = page_stride(record, block_size) if page_stride_bytes is None else int(page_stride_bytes)
    if ps <= 0:
        raise ValueError(f"unsupported record {record} / block_size {block_size}")
    flat = torch.empty(num_pages * ps, dtype=torch.uint8, device=device)
    if fill is not None:
        flat.fill_(fill)
    if record in PACKED:
        return torch.as_strided(flat, (num_pages, block_size, record), (ps, record, 1))
    dt, es = (torch.float8_e4m3fn, 1) if record == 512 else (torch.bfloat16, 2)
    if ps % es:
        raise ValueError("page stride must be a whole number of elements")
    return torch.as_strided(flat.view(dt), (num_pages, block_size, HEAD_DIM),
                            (ps // es, HEAD_DIM, 1))


def cache_bytes(k_cache: torch.Tensor) -> torch.Tensor:
    """The flat byte view (num_pages * page_stride) behind a paged cache view."""
    u8 = k_cache if k_cache.dtype == torch.uint8 else k_cache.view(torch.uint8)
    P = u8.shape[0]
    return torch.as_strided(u8, (P * u8.stride(0),), (1,), u8.storage_offset())


def _cache_desc(k_cache: torch.Tensor) -> CacheDesc:
    """The record width is the format selector: uint8 [pages, block, 528 | 584] are
    the packed MXFP8 records; float8_e4m3fn / bfloat16 [pages, block, 512] the plain
    caches (records 512 / 1024)."""
    if k_cache.dim() != 3:
        raise ValueError("k_cache must be a 3-D paged cache [num_pages, block_size, width]")
    P, bs, w = k_cache.shape
    if k_cache.dtype == torch.uint8:
        if w not in PACKED:
            raise ValueError(f"unsupported paged KV record width {w} (expected 528 or 584)")
        rec, es = w, 1
    elif k_cache.dtype in (torch.float8_e4m3fn, torch.bfloat16):
        if w != HEAD_DIM:
            raise ValueError(f"a {k_cache.dtype} cache must have width 512, not {w}")
        rec, es = (512, 1) if k_cache.dtype == torch.float8_e4m3fn else (1024, 2)
    else:
        raise ValueError("k_cache must be uint8 (packed records), float8_e4m3fn or bfloat16")
    if k_cache.stride(2) != 1 or k_cache.stride(1) != w:
        raise ValueError("k_cache must have stride(2) == 1 and stride(1) == its width")
    return CacheDesc(rec, bs, P, k_cache.stride(0) * es)


def _check(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _same_cuda_device(*ts: torch.Tensor) -> torch.device:
    dev = ts[0].device
    if dev.type != "cuda":
        raise ValueError("kv_insert / kv_gather need CUDA tensors (there is no CPU path)")
    for t in ts[1:]:
        if t is not None and t.device != dev:
            raise ValueError(f"all tensors must be on {dev}; got one on {t.device}")
    return dev


def _check_fp8_scale(desc: CacheDesc, fp8_scale):
    if desc.record == 512:
        _check(fp8_scale is not None and fp8_scale.dtype == torch.float32
               and fp8_scale.numel() == 1, "an fp8 cache needs fp8_scale: a float32 tensor "
               "with one element")
    else:
        _check(fp8_scale is None, "fp8_scale is only taken by an fp8 (float8_e4m3fn) cache")


def _check_err_flag(err_flag):
    if err_flag is not None:
        _check(err_flag.dtype == torch.int32 and err_flag.numel() >= 1 and err_flag.is_contiguous(),
               "err_flag must be a contiguous int32 tensor with at least one element")


def _insert_args(kv, k_cache, slot_mapping, positions, cos_sin_cache, block_size, record,
                 err_flag):
    desc = _cache_desc(k_cache)
    if record is not None:
        _check(int(record) == desc.record,
               f"record {record} does not match k_cache width {desc.record}")
    _check(int(block_size) == desc.block_size,
           f"block_size {block_size} != k_cache.size(1) {desc.block_size}")
    _check(kv.dtype == torch.bfloat16 and kv.dim() == 2 and kv.shape[1] == HEAD_DIM
           and kv.is_contiguous(), "kv must be a contiguous bf16 tensor [tokens, 512]")
    _check(slot_mapping.dtype == torch.int64 and slot_mapping.dim() == 1
           and slot_mapping.is_contiguous(), "slot_mapping must be a contiguous int64 [T] tensor")
    _check(positions.dtype == torch.int64 and positions.dim() == 1 and positions.is_contiguous(),
           "positions must be a contiguous int64 1-D tensor")
    T = slot_mapping.shape[0]
    _check(kv.shape[0] >= T, "kv has fewer rows than slot_mapping")
    _check(positions.shape[0] >= kv.shape[0], "positions must cover every kv row")
    _check(cos_sin_cache.dtype == torch.float32 and cos_sin_cache.dim() == 2
           and cos_sin_cache.shape[1] == 64 and cos_sin_cache.is_contiguous(),
           "cos_sin_cache must be a contiguous fp32 tensor [max_pos, 64]")
    _check_err_flag(err_flag)
    dev = _same_cuda_device(kv, k_cache, slot_mapping, positions, cos_sin_cache, err_flag)
    return desc, T, dev


def kv_insert(kv: torch.Tensor, k_cache: torch.Tensor, slot_mapping: torch.Tensor,
              positions: torch.Tensor, cos_sin_cache: torch.Tensor, block_size: int,
              record: int | None = None, err_flag: torch.Tensor | None = None,
              fp8_scale: torch.Tensor | None = None,
              launch_opts: LaunchOpts | None = None) -> None:
    """RoPE + MXFP8 quantise + paged insert, in place into k_cache.

    kv             bf16 [tokens, 512], contiguous; not modified.
    k_cache        uint8 [num_pages, block_size, record] (stride(0) = page stride), or a
                   plain float8_e4m3fn / bfloat16 [num_pages, block_size, 512] cache.
    slot_mapping   int64 [T] (T = number of tokens processed, <= tokens); -1 = skip.
    positions      int64, contiguous, covering every kv row.
    cos_sin_cache  fp32 [max_pos, 64], contiguous (cos 0..31 | sin 0..31).
    block_size     must equal k_cache.size(1).
    record         528 / 584, or None to take it from k_cache.size(2).
    err_flag       optional int32 device tensor; error bits are OR-ed into element 0.
    fp8_scale      float32 device tensor of one element: required for an fp8 cache
                   (stored codes are e4m3(x / scale)), None otherwise.
    launch_opts    this call's LaunchOpts (over the context's launch_policy), or None.
    """
    desc, T, dev = _insert_args(kv, k_cache, slot_mapping, positions, cos_sin_cache,
                                block_size, record, err_flag)
    _check_fp8_scale(desc, fp8_scale)
    if fp8_scale is not None:
        _same_cuda_device(kv, fp8_scale)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = lib().gkr_kv_insert(_ptr(kv), T, _ptr(k_cache), ctypes.byref(desc),
                                 _ptr(slot_mapping), _ptr(positions), _ptr(cos_sin_cache),
                                 cos_sin_cache.shape[0], _ptr(fp8_scale), _ptr(err_flag),
                                 _opts(launch_opts), stream)
    _raise(st)


def rope_quant_insert(kv: torch.Tensor, k_cache: torch.Tensor, slot_mapping: torch.Tensor,
                      positions: torch.Tensor, cos_sin_cache: torch.Tensor, block_size: int,
                      compress_ratio: int = 1, sanitize_nans: bool = False,
                      record: int | None = None, err_flag: torch.Tensor | None = None,
                      launch_opts: LaunchOpts | None = None) -> None:
    """Compressed-KV insert, in place into k_cache: a token is written only when
    (position + 1) % compress_ratio == 0, rotated with the cos/sin row of its group's
    first position (position // compress_ratio * compress_ratio); with sanitize_nans
    every NaN of the rotated row is stored as +0.  Arguments as for kv_insert."""
    _check(isinstance(compress_ratio, int) and 1 <= compress_ratio <= 0x7FFFFFFF,
           "compress_ratio must be an int in [1, 2^31 - 1]")
    desc, T, dev = _insert_args(kv, k_cache, slot_mapping, positions, cos_sin_cache,
                                block_size, record, err_flag)
    _check(desc.record in PACKED, "the compressed insert writes the packed 528 / 584 records")
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = lib().gkr_rope_quant_insert(_ptr(kv), T, _ptr(k_cache), ctypes.byref(desc),
                                         _ptr(slot_mapping), _ptr(positions),
                                         _ptr(cos_sin_cache), cos_sin_cache.shape[0],
                                         int(compress_ratio), 1 if sanitize_nans else 0,
                                         _ptr(err_flag), _opts(launch_opts), stream)
    _raise(st)


def kv_gather(k_cache: torch.Tensor, indices: torch.Tensor, out: torch.Tensor,
              err_flag: torch.Tensor | None = None,
              fp8_scale: torch.Tensor | None = None,
              launch_opts: LaunchOpts | None = None) -> torch.Tensor:
    """Dequantise the records at `indices` into `out` (bf16 [*indices.shape, 512]).
    An index of -1 writes zeros.  An fp8 cache needs its fp8_scale.  Returns out."""
    desc = _cache_desc(k_cache)
    _check_fp8_scale(desc, fp8_scale)
    _check(indices.dtype == torch.int32 and indices.is_contiguous(),
           "indices must be a contiguous int32 tensor")
    _check(out.dtype == torch.bfloat16 and out.is_contiguous()
           and tuple(out.shape) == tuple(indices.shape) + (HEAD_DIM,),
           "out must be a contiguous bf16 tensor of shape indices.shape + (512,)")
    _check_err_flag(err_flag)
    dev = _same_cuda_device(k_cache, indices, out, err_flag, fp8_scale)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = lib().gkr_kv_gather(_ptr(k_cache), ctypes.byref(desc), _ptr(indices),
                                 indices.numel(), _ptr(out), _ptr(fp8_scale), _ptr(err_flag),
                                 _opts(launch_opts), stream)
    _raise(st)
    return out


def qnorm_rope_kv_insert(q: torch.Tensor, kv: torch.Tensor, k_cache: torch.Tensor,
                         slot_mapping: torch.Tensor, positions: torch.Tensor,
                         cos_sin_cache: torch.Tensor, num_heads_padded: int, eps: float,
                         block_size: int, apply_q_norm: bool = True,
                         q_out: torch.Tensor | None = None, record: int | None = None,
                         err_flag: torch.Tensor | None = None,
                         fp8_scale: torch.Tensor | None = None,
                         q_scale: torch.Tensor | None = None,
                         launch_opts: LaunchOpts | None = None) -> torch.Tensor:
    """The fused attention write: each query head of q (bf16 [T, H, 512]) divided by
    sqrt(mean(q^2) + eps) when apply_q_norm, dims 448..511 rotated with the token's
    cos/sin row, written as bf16 to q_out [T, num_heads_padded, 512] (padded heads +0),
    and the KV rows inserted into k_cache exactly as kv_insert does, in one launch.
    q_out may be q itself when num_heads_padded == H.  With q_scale (a float32 CUDA
    tensor of one element) q_out holds e4m3 codes instead, e4m3(x / q_scale) of each fp32
    value (float8_e4m3fn or uint8, not overlapping q).  Returns q_out (allocated when
    None).  The other arguments are kv_insert's."""
    _check(q.dtype == torch.bfloat16 and q.dim() == 3 and q.shape[2] == HEAD_DIM
           and q.is_contiguous(), "q must be a contiguous bf16 tensor [tokens, heads, 512]")
    desc, T, dev = _insert_args(kv, k_cache, slot_mapping, positions, cos_sin_cache,
                                block_size, record, err_flag)
    _check_fp8_scale(desc, fp8_scale)
    H, Hp = int(q.shape[1]), int(num_heads_padded)
    _check(q.shape[0] >= T, "q has fewer tokens than slot_mapping")
    _check(Hp >= H, "num_heads_padded must be at least q.shape[1]")
    fp8_q = q_scale is not None
    if fp8_q:
        _check(q_scale.dtype == torch.float32 and q_scale.numel() == 1 and q_scale.is_cuda,
               "q_scale must be a float32 CUDA tensor of one element")
    out_types = (torch.float8_e4m3fn, torch.uint8) if fp8_q else (torch.bfloat16,)
    if q_out is None:
        q_out = torch.empty(T, Hp, HEAD_DIM, dtype=out_types[0], device=dev)
    _check(q_out.dtype in out_types and q_out.is_contiguous() and q_out.dim() == 3
           and q_out.shape[0] >= T and q_out.shape[1] == Hp and q_out.shape[2] == HEAD_DIM,
           "q_out must be a contiguous tensor [tokens, num_heads_padded, 512] of bf16 "
           "(e4m3 codes: float8_e4m3fn or uint8 with q_scale)")
    _same_cuda_device(kv, q, q_out, fp8_scale, q_scale)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = lib().gkr_qnorm_rope_kv_insert(_ptr(q), H, Hp, _ptr(q_out), _ptr(q_scale), float(eps),
                                            1 if apply_q_norm else 0, _ptr(kv), T, _ptr(k_cache),
                                            ctypes.byref(desc), _ptr(slot_mapping),
                                            _ptr(positions), _ptr(cos_sin_cache),
                                            cos_sin_cache.shape[0], _ptr(fp8_scale),
                                            _ptr(err_flag), _opts(launch_opts), stream)
    _raise(st)
    return q_out


def sparse_logits(q: torch.Tensor, k_cache: torch.Tensor, indices: torch.Tensor,
                  sm_scale: float, out: torch.Tensor | None = None,
                  err_flag: torch.Tensor | None = None, fp8_scale: torch.Tensor | None = None,
                  launch_opts: LaunchOpts | None = None) -> torch.Tensor:
    """Sparse decode logits with the dequant-gather fused in: for query i, head h and
    entry k, out[i, h, k] = sm_scale * q[i, h, :] . K, K the bf16 row kv_gather returns
    for indices[i, k] (-1, or an index outside the cache: -inf).  q bf16 [Q, H, 512]
    (H <= 128), indices int32 [Q, topk] (topk a multiple of 4), out fp32 [Q, H, topk]
    (allocated when None).  Returns out."""
    desc = _cache_desc(k_cache)
    _check_fp8_scale(desc, fp8_scale)
    _check(q.dtype == torch.bfloat16 and q.dim() == 3 and q.shape[2] == HEAD_DIM
           and q.is_contiguous(), "q must be a contiguous bf16 tensor [queries, heads, 512]")
    _check(indices.dtype == torch.int32 and indices.dim() == 2 and indices.is_contiguous()
           and indices.shape[0] == q.shape[0],
           "indices must be a contiguous int32 tensor [queries, topk]")
    Q, H, K = int(q.shape[0]), int(q.shape[1]), int(indices.shape[1])
    if out is None:
        out = torch.empty(Q, H, K, dtype=torch.float32, device=q.device)
    _check(out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (Q, H, K),
           "out must be a contiguous fp32 tensor [queries, heads, topk]")
    _check_err_flag(err_flag)
    dev = _same_cuda_device(q, k_cache, indices, out, err_flag, fp8_scale)
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev).cuda_stream
        st = lib().gkr_sparse_logits(_ptr(q), H, _ptr(k_cache), ctypes.byref(desc), _ptr(indices),
                                     Q, K, float(sm_scale), _ptr(fp8_scale), _ptr(out),
                                     _ptr(err_flag), _opts(launch_opts), stream)
    _raise(st)
    return out
