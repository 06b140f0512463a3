"""Seeded synthetic inputs for the paged KV insert / gather path.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark.  It only draws random numbers and lays out input arrays: it contains
none of the method's arithmetic (no rotation, quantisation or page addressing).

Every workload is drawn from ``numpy.random.default_rng(seed)`` in a fixed
order: kv values -> outlier mask -> positions -> slot permutation -> skip
(-1) mask -> (gather) context lengths -> indices -> invalid (-1) mask.  kv is
drawn in float32 and rounded to bfloat16 (round to nearest even) once; arrays
are returned as numpy, kv as raw bf16 bit patterns (uint16).

The cos/sin table is the usual rotary table for a 64-dim rotary slice:
row p = [cos(p * w_0) .. cos(p * w_31) | sin(p * w_0) .. sin(p * w_31)],
w_j = theta^(-2j/64), theta = 10000, computed in float64 and rounded to fp32.
The pages give only the row layout; the values are an input and do not affect
parity.

Workloads (named by what they are):
  insert_v41_1024       1024 tokens, 528 B record, bs 64, 32 pages
  roundtrip_v41_16384   16384 tokens insert + gather back, 528 B, 512 pages
  insert_v4_65536       65536 tokens, 584 B legacy record, 2048 pages
  insert_v41_262144     262144 tokens in 8 contiguous sequences, 8192 pages
  gather_v41_sparse     1,048,576-token cache; 128 queries x top-2048 indices
  compressed_v41_r4_262144    8 sequences x 32768 positions, one record per 4
  compressed_v41_r128_262144  the same with one record per 128 positions
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

ROTARY_THETA = 10000.0


@dataclass
class InsertCase:
    name: str
    record: int            # 528 (V4.1) or 584 (V4 legacy)
    block_size: int
    num_pages: int
    kv: np.ndarray         # uint16 [T, 512]: bf16 bit patterns
    slots: np.ndarray      # int64 [T]; -1 = skip
    positions: np.ndarray  # int64 [T]
    csc: np.ndarray        # float32 [max_pos, 64]
    page_stride: int | None = None   # None = the record's minimal aligned stride
    indices: np.ndarray | None = None  # int32 [...]: gather list, -1 = invalid
    meta: dict = field(default_factory=dict)

    @property
    def num_tokens(self) -> int:
        return int(self.slots.shape[0])


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest even (via torch's cast)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def cos_sin_table(max_pos: int, theta: float = ROTARY_THETA) -> np.ndarray:
    j = np.arange(32, dtype=np.float64)
    w = theta ** (-2.0 * j / 64.0)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * w[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def _skip_mask(rng, n: int, rate: float) -> np.ndarray:
    k = int(round(rate * n))
    m = np.zeros(n, bool)
    if k:
        m[rng.choice(n, size=k, replace=False)] = True
    return m


def _kv_values(rng, T: int, dist: str, outlier_rate: float = 0.0,
               outlier_scale: float = 50.0, sigma: float = 1.0) -> np.ndarray:
    if dist == "normal":
        x = rng.standard_normal((T, 512), dtype=np.float32) * np.float32(sigma)
    elif dist == "student_t3":
        x = rng.standard_t(3, size=(T, 512)).astype(np.float32)
    else:
        raise ValueError(dist)
    if outlier_rate:
        k = int(round(outlier_rate * x.size))
        if k:
            idx = rng.choice(x.size, size=k, replace=False)
            x.reshape(-1)[idx] *= np.float32(outlier_scale)
    return to_bf16_bits(x)


def random_insert(name: str, T: int, record: int, block_size: int, num_pages: int,
                  max_pos: int, skip_rate: float, seed: int = 0, dist: str = "normal",
                  outlier_rate: float = 0.0, page_stride: int | None = None,
                  sigma: float = 1.0) -> InsertCase:
    """T tokens with random positions in [0, max_pos) and distinct random slots
    (the first T entries of a permutation of all num_pages * block_size slots),
    a fraction skip_rate of them replaced by -1."""
    rng = np.random.default_rng(seed)
    n_slots = num_pages * block_size
    if T > n_slots:
        raise ValueError("more tokens than slots")
    kv = _kv_values(rng, T, dist, outlier_rate, sigma=sigma)
    positions = rng.integers(0, max_pos, size=T, dtype=np.int64)
    slots = rng.permutation(n_slots)[:T].astype(np.int64)
    slots[_skip_mask(rng, T, skip_rate)] = -1
    return InsertCase(name, record, block_size, num_pages, kv, slots, positions,
                      cos_sin_table(max_pos), page_stride)


def insert_v41_1024(seed: int = 0) -> InsertCase:
    """1024 tokens, N(0,1) with 1% of entries x50; positions U[0,4096);
    bs 64, 32 pages; slots from a permutation of the 2048 slots, 5% -> -1."""
    return random_insert("insert_v41_1024", 1024, 528, 64, 32, 4096, 0.05, seed,
                         outlier_rate=0.01)


def roundtrip_v41_16384(seed: int = 0) -> InsertCase:
    """16384 tokens, same distributions, 512 pages, 8% -> -1; the gather list is
    the slot list itself (int32), so -1 entries come back as zeros."""
    c = random_insert("roundtrip_v41_16384", 16384, 528, 64, 512, 4096, 0.08, seed,
                      outlier_rate=0.01)
    c.indices = c.slots.astype(np.int32)
    return c


def insert_v4_65536(seed: int = 0) -> InsertCase:
    """65536 tokens, 584 B legacy record, Student-t (nu=3) values, positions
    U[0,131072), bs 64, 2048 pages (stride 37440), 5% -> -1."""
    return random_insert("insert_v4_65536", 65536, 584, 64, 2048, 131072, 0.05, seed,
                         dist="student_t3")


def insert_v41_262144(seed: int = 0) -> InsertCase:
    """262144 tokens as 8 sequences of 32768: positions 0..32767 in each, sequence
    s writes slots s*65536 + [0, 32768); N(0, 0.5); bs 64, 8192 pages; 2% -> -1."""
    rng = np.random.default_rng(seed)
    S, L = 8, 32768
    T = S * L
    kv = _kv_values(rng, T, "normal", sigma=0.5)
    positions = np.tile(np.arange(L, dtype=np.int64), S)
    slots = (np.repeat(np.arange(S, dtype=np.int64) * 65536, L)
             + np.tile(np.arange(L, dtype=np.int64), S))
    slots[_skip_mask(rng, T, 0.02)] = -1
    return InsertCase("insert_v41_262144", 528, 64, 8192, kv, slots, positions,
                      cos_sin_table(L), None)


def gather_v41_sparse(seed: int = 0, cache_tokens: int = 1 << 20, queries: int = 128,
                      topk: int = 2048, min_ctx: int = 8192) -> InsertCase:
    """A cache of cache_tokens tokens (bs 64) filled in slot order from N(0,1)
    with position = token index; then `queries` index lists of `topk` distinct
    indices, each drawn uniformly from [0, L_q) with L_q ~ U[min_ctx, cache_tokens),
    3% of all indices -> -1.  indices: int32 [queries, topk]."""
    rng = np.random.default_rng(seed)
    T = cache_tokens
    kv = _kv_values(rng, T, "normal")
    positions = np.arange(T, dtype=np.int64)
    slots = np.arange(T, dtype=np.int64)
    ctx = rng.integers(min_ctx, cache_tokens, size=queries)
    indices = np.stack([rng.choice(int(L), size=topk, replace=False) for L in ctx])
    indices = indices.astype(np.int32)
    indices.reshape(-1)[_skip_mask(rng, indices.size, 0.03)] = -1
    c = InsertCase("gather_v41_sparse", 528, 64, T // 64, kv, slots, positions,
                   cos_sin_table(T), None, indices)
    c.meta["context_lengths"] = ctx
    return c


def insert_v41_131072(seed: int = 0) -> InsertCase:
    """Profiling-size contiguous insert: 4 sequences of 32768 tokens (positions
    0..32767 each), sequence s writes slots s*32768 + [0, 32768); N(0, 0.5); bs 64,
    2048 pages; 2% -> -1.  kv 134 MB + cache 69 MB, larger than L2."""
    rng = np.random.default_rng(seed)
    S, L = 4, 32768
    T = S * L
    kv = _kv_values(rng, T, "normal", sigma=0.5)
    positions = np.tile(np.arange(L, dtype=np.int64), S)
    slots = (np.repeat(np.arange(S, dtype=np.int64) * L, L) + np.tile(np.arange(L, dtype=np.int64), S))
    slots[_skip_mask(rng, T, 0.02)] = -1
    return InsertCase("insert_v41_131072", 528, 64, 2048, kv, slots, positions,
                      cos_sin_table(L), None)


def roundtrip_v41_65536(seed: int = 1) -> InsertCase:
    """65536 tokens with random slots (2048 pages, 5% -> -1) and positions U[0, 8192),
    N(0,1); the gather list is the slot list: the token count the pages time on GB300,
    for profiler captures of the insert and of the gather at >= 65536 items."""
    c = random_insert("roundtrip_v41_65536", 65536, 528, 64, 2048, 8192, 0.05, seed)
    c.indices = c.slots.astype(np.int32)
    return c


def decode_queries(queries: int, heads: int, seed: int = 5) -> np.ndarray:
    """Decode queries for the sparse logits: bf16 bit patterns [queries, heads, 512] drawn
    from N(0,1) (the queries' values; the keys come from a cache workload)."""
    rng = np.random.default_rng(seed)
    return to_bf16_bits(rng.standard_normal((queries, heads, 512), dtype=np.float32))


def gather_v41_sparse_262144(seed: int = 0) -> InsertCase:
    """Profiling-size sparse gather: a 262144-token cache (138 MB) and 32 queries x 2048."""
    c = gather_v41_sparse(seed, cache_tokens=1 << 18, queries=32, topk=2048, min_ctx=8192)
    c.name = "gather_v41_sparse_262144"
    return c


def compressed_insert(name: str, S: int, L: int, ratio: int, record: int = 528,
                      block_size: int = 64, skip_rate: float = 0.02, seed: int = 0,
                      sigma: float = 0.5, nan_rate: float = 0.0, inf_rate: float = 0.0,
                      dist: str = "normal", nonfinite_dims: int = 512) -> InsertCase:
    """Compressed-KV insert input: S sequences of L tokens, positions 0..L-1 in each;
    every token of sequence s carries the compressed slot s * ceil(L / ratio) +
    position // ratio (the slot of its group), so only the group-boundary tokens
    (position + 1) % ratio == 0 decide what is written.  A fraction skip_rate of the
    tokens get slot -1; disjoint fractions nan_rate / inf_rate of the kv entries (drawn
    after the skip mask, among dims [0, nonfinite_dims) of every row) are set to NaN /
    +-inf with random signs.  Pages: ceil(S * ceil(L / ratio) / block_size)."""
    rng = np.random.default_rng(seed)
    T = S * L
    kv = _kv_values(rng, T, dist, sigma=sigma)
    positions = np.tile(np.arange(L, dtype=np.int64), S)
    per_seq = -(-L // ratio)
    slots = np.repeat(np.arange(S, dtype=np.int64) * per_seq, L) + positions // ratio
    slots[_skip_mask(rng, T, skip_rate)] = -1
    k_nan, k_inf = int(round(nan_rate * kv.size)), int(round(inf_rate * kv.size))
    if k_nan + k_inf:
        pick = rng.choice(T * nonfinite_dims, size=k_nan + k_inf, replace=False)  # disjoint
        idx = pick // nonfinite_dims * 512 + pick % nonfinite_dims
        sign = rng.integers(0, 2, size=k_nan + k_inf).astype(bool)
        val = np.where(np.arange(k_nan + k_inf) < k_nan, np.nan, np.inf)
        kv.reshape(-1)[idx] = to_bf16_bits(np.where(sign, -val, val).astype(np.float32))
    pages = -(-S * per_seq // block_size)
    c = InsertCase(name, record, block_size, pages, kv, slots, positions, cos_sin_table(L), None)
    c.meta["compress_ratio"] = ratio
    return c


def compressed_v41_r4_262144(seed: int = 0) -> InsertCase:
    """262144 tokens (8 x 32768), ratio 4: 65536 boundary tokens into 1024 pages."""
    return compressed_insert("compressed_v41_r4_262144", 8, 32768, 4, seed=seed)


def compressed_v41_r128_262144(seed: int = 0) -> InsertCase:
    """262144 tokens (8 x 32768), ratio 128: 2048 boundary tokens into 32 pages."""
    return compressed_insert("compressed_v41_r128_262144", 8, 32768, 128, seed=seed)


WORKLOADS = {
    "insert_v41_1024": insert_v41_1024,
    "roundtrip_v41_16384": roundtrip_v41_16384,
    "insert_v4_65536": insert_v4_65536,
    "insert_v41_262144": insert_v41_262144,
    "gather_v41_sparse": gather_v41_sparse,
    "compressed_v41_r4_262144": compressed_v41_r4_262144,
    "compressed_v41_r128_262144": compressed_v41_r128_262144,
}

# smaller cases of the same kernels, sized for profiler captures
PROFILE_WORKLOADS = {
    "insert_v41_262144": insert_v41_262144,
    "gather_v41_sparse": gather_v41_sparse,
    "insert_v41_131072": insert_v41_131072,
    "insert_v4_65536": insert_v4_65536,
    "gather_v41_sparse_262144": gather_v41_sparse_262144,
    "roundtrip_v41_16384": roundtrip_v41_16384,
    "roundtrip_v41_65536": roundtrip_v41_65536,
    "compressed_v41_r4_262144": compressed_v41_r4_262144,
}
