"""Seeded synthetic inputs for absorbed-path MLA decode.

This module only draws random inputs and lays them out; it holds none of the
decode arithmetic.  Both sides consume what it produces: the CUDA library
(through the Python binding) and the fp64 oracle (``oracle/``).

Workload recipe (the five decode workloads of the benchmark, sizes verbatim):

  tiny       B=2,   H=16,  s_q=1, seqlens {64, 100}, pool = exactly the 3 pages needed,
             fp32 out.
  uniform4k  B=32,  H=128, s_q=1, every seqlen 4096, pool 2048 pages, bf16 out.
  ragged     B=64,  H=128, s_q=1, seqlens round(exp(U(ln 256, ln 32768))), pool of
             ceil(1.25 * pages needed), sequences take a random injective sample of it.
  long       B=4,   H=128, s_q=1, seqlens {131072, 65536, 100000, 8192}, pool 4763 pages.
  fp8_mtp2   B=128, H=128, s_q=2 (causal within the two new tokens), seqlens uniform
             in [2048, 16384], latent stored as FP8 E4M3 with one float32 scale per
             128-element tile per token, RoPE part bf16.

Common to all: page size 64; block tables map each sequence's logical pages to a
random set of physical pages; q~, q^R, c, k^R are N(0, 1) draws in float32 rounded
to bf16 (round-to-nearest-even); scale 1/sqrt(192).  The FP8 cache is quantised
from N(0, 1) float32 values: scale = amax/448 per tile (1 when amax = 0), code =
E4M3(x/scale) rounded to nearest even.  The seed defaults to the workload index;
draws use numpy's default_rng in a fixed order (seqlens, pages, q~, q^R, cache).
Block-table entries past a sequence's last page hold -1 and are never read.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE = 64
D_C = 512
D_R = 64
D_QK = D_C + D_R                     # 576 elements per cached token
FP8_ROW_BYTES = D_C + 4 * (D_C // 128) + 2 * D_R  # 656
BF16_ROW_BYTES = 2 * D_QK            # 1152
SCALE = 1.0 / math.sqrt(192.0)

WORKLOADS = ["tiny", "uniform4k", "ragged", "long", "fp8_mtp2"]


@dataclass
class Workload:
    name: str
    batch: int
    s_q: int
    num_heads: int
    causal: bool
    kv_dtype: str                  # "bf16" | "fp8"
    out_dtype: str                 # "f32" | "bf16"
    seqlens: np.ndarray            # int32 [B], includes the s_q new tokens
    block_table: np.ndarray        # int32 [B, max_pages]
    kv: np.ndarray                 # uint16 [pages, 64, 576] (bf16 bits) | uint8 [pages, 64, 656]
    q_nope: np.ndarray             # uint16 [B, s_q, H, 512] bf16 bits (absorbed query q~)
    q_rope: np.ndarray             # uint16 [B, s_q, H, 64] bf16 bits
    scale: float = SCALE
    page_size: int = PAGE
    meta: dict = field(default_factory=dict)

    @property
    def num_pages(self) -> int:
        return self.kv.shape[0]

    @property
    def tokens(self) -> int:
        return int(self.seqlens.astype(np.int64).sum())


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> raw bf16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def quantize_fp8_rows(c: np.ndarray, kr_bits: np.ndarray) -> np.ndarray:
    """Build 656-byte FP8 cache rows from float32 latents c [n, 512] and bf16 RoPE bits [n, 64]."""
    n = c.shape[0]
    tiles = c.reshape(n, D_C // 128, 128)
    amax = np.abs(tiles).max(axis=2)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    y = np.clip(tiles / scale[:, :, None], -448.0, 448.0).astype(np.float32)
    codes = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy().reshape(n, D_C)
    rows = np.empty((n, FP8_ROW_BYTES), np.uint8)
    rows[:, :D_C] = codes
    rows[:, D_C:D_C + 16] = scale.view(np.uint8).reshape(n, 16)
    rows[:, D_C + 16:] = kr_bits.view(np.uint8).reshape(n, 2 * D_R)
    return rows


def quantize_query_fp8(w) -> np.ndarray:
    """The workload's query in the FP8 row layout (as a cache row: absorbed query -> 512 codes and 4
    tile scales, RoPE query copied): uint8 [B, s_q, H, 656], the input of an FP8-QK decode."""
    lat = (w.q_nope.astype(np.uint32) << 16).view(np.float32).reshape(-1, D_C)
    rows = quantize_fp8_rows(lat, w.q_rope.reshape(-1, D_R))
    return rows.reshape(w.batch, w.s_q, w.num_heads, FP8_ROW_BYTES)


def _fill_pool(rng: np.random.Generator, num_pages: int, kv_dtype: str) -> np.ndarray:
    """N(0,1) page pool, generated in chunks of pages to bound host memory."""
    if kv_dtype == "bf16":
        pool = np.empty((num_pages, PAGE, D_QK), np.uint16)
    else:
        pool = np.empty((num_pages, PAGE, FP8_ROW_BYTES), np.uint8)
    chunk = 2048
    for p0 in range(0, num_pages, chunk):
        p1 = min(num_pages, p0 + chunk)
        x = rng.standard_normal((p1 - p0) * PAGE * D_QK, dtype=np.float32).reshape(-1, D_QK)
        if kv_dtype == "bf16":
            pool[p0:p1] = to_bf16_bits(x).reshape(p1 - p0, PAGE, D_QK)
        else:
            rows = quantize_fp8_rows(x[:, :D_C], to_bf16_bits(x[:, D_C:]))
            pool[p0:p1] = rows.reshape(p1 - p0, PAGE, FP8_ROW_BYTES)
    return pool


def make_custom(seqlens, num_heads: int = 128, s_q: int = 1, causal: bool = True, kv_dtype: str = "bf16",
                out_dtype: str = "bf16", pool_factor: float = 1.0, seed: int = 0, name: str = "custom",
                extra_pages: int = 0) -> Workload:
    """A workload with the given per-sequence lengths; pages scattered over a pool of
    ceil(pool_factor * pages needed) + extra_pages physical pages."""
    rng = np.random.default_rng(seed)
    seqlens = np.asarray(seqlens, dtype=np.int32)
    B = len(seqlens)
    need = [(int(L) + PAGE - 1) // PAGE for L in seqlens]
    total = sum(need)
    pool = max(1, int(math.ceil(pool_factor * total)) + extra_pages)
    perm = rng.permutation(pool).astype(np.int32)
    max_pages = max(1, max(need) if need else 1)
    bt = np.full((B, max_pages), -1, np.int32)
    o = 0
    for b, n in enumerate(need):
        bt[b, :n] = perm[o:o + n]
        o += n
    q_nope = to_bf16_bits(rng.standard_normal((B, s_q, num_heads, D_C), dtype=np.float32))
    q_rope = to_bf16_bits(rng.standard_normal((B, s_q, num_heads, D_R), dtype=np.float32))
    kv = _fill_pool(rng, pool, kv_dtype)
    return Workload(name=name, batch=B, s_q=s_q, num_heads=num_heads, causal=causal, kv_dtype=kv_dtype,
                    out_dtype=out_dtype, seqlens=seqlens, block_table=bt, kv=kv, q_nope=q_nope, q_rope=q_rope,
                    meta={"seed": seed, "pool_pages": pool, "pages_used": total})


def workload_seqlens(index: int, rng: np.random.Generator) -> np.ndarray:
    if index == 0:
        return np.array([64, 100], np.int32)
    if index == 1:
        return np.full(32, 4096, np.int32)
    if index == 2:
        return np.round(np.exp(rng.uniform(math.log(256), math.log(32768), size=64))).astype(np.int32)
    if index == 3:
        return np.array([131072, 65536, 100000, 8192], np.int32)
    if index == 4:
        return rng.integers(2048, 16385, size=128).astype(np.int32)
    raise ValueError(index)


def make_workload(index: int, seed: int | None = None) -> Workload:
    """The benchmark workload `index` (0..4, see the module docstring)."""
    seed = index if seed is None else seed
    rng = np.random.default_rng(seed)
    seqlens = workload_seqlens(index, rng)
    H = 16 if index == 0 else 128
    s_q = 2 if index == 4 else 1
    kv_dtype = "fp8" if index == 4 else "bf16"
    out_dtype = "f32" if index == 0 else "bf16"
    pool_factor = 1.25 if index == 2 else 1.0
    sub_seed = int(rng.integers(0, 2**31 - 1))
    w = make_custom(seqlens, num_heads=H, s_q=s_q, causal=True, kv_dtype=kv_dtype, out_dtype=out_dtype,
                    pool_factor=pool_factor, seed=sub_seed, name=WORKLOADS[index])
    w.meta["index"] = index
    w.meta["seed"] = seed
    return w


def first_sequences(w: Workload, batch: int) -> Workload:
    """The same workload cut to its first `batch` sequences (pages and cache pool unchanged)."""
    import dataclasses
    b = max(1, min(int(batch), w.batch))
    return dataclasses.replace(w, batch=b, seqlens=w.seqlens[:b].copy(), block_table=w.block_table[:b].copy(),
                               q_nope=w.q_nope[:b].copy(), q_rope=w.q_rope[:b].copy(),
                               meta=dict(w.meta, first_sequences=b))


@dataclass
class ExtendWorkload:
    """Inputs of an extend by the expand path: the paged bf16 cache of `cache` (its last s_q rows
    per sequence are the new tokens), the new tokens' non-absorbed queries and the per-head
    up-projections (bf16 bit patterns)."""
    cache: Workload
    s_q: int
    q_nope: np.ndarray   # uint16 [B, s_q, H, d_nope]
    q_rope: np.ndarray   # uint16 [B, s_q, H, 64]
    w_uk: np.ndarray     # uint16 [H, d_nope, 512]
    w_uv: np.ndarray     # uint16 [H, 512, d_v]
    scale: float


def make_extend(seqlens, s_q: int, num_heads: int = 128, seed: int = 0, d_nope: int = 128, d_v: int = 128,
                nan_tail: bool = True) -> ExtendWorkload:
    """Seeded N(0, 1) cache and queries; W_UK and W_UV N(0, 1/512) so that expanded keys and values
    are O(1).  nan_tail: cache rows past each sequence's end in its last page hold NaN."""
    cache = make_custom(seqlens, num_heads=num_heads, s_q=1, seed=seed)
    rng = np.random.default_rng(seed + 1)
    B = cache.batch
    if nan_tail:
        for b in range(B):
            L = int(cache.seqlens[b])
            if L % PAGE:
                cache.kv[cache.block_table[b, L // PAGE], L % PAGE:] = 0x7FC0
    sd = 1.0 / math.sqrt(D_C)
    return ExtendWorkload(
        cache=cache, s_q=s_q,
        q_nope=to_bf16_bits(rng.standard_normal((B, s_q, num_heads, d_nope), dtype=np.float32)),
        q_rope=to_bf16_bits(rng.standard_normal((B, s_q, num_heads, D_R), dtype=np.float32)),
        w_uk=to_bf16_bits((rng.standard_normal((num_heads, d_nope, D_C)) * sd).astype(np.float32)),
        w_uv=to_bf16_bits((rng.standard_normal((num_heads, D_C, d_v)) * sd).astype(np.float32)),
        scale=1.0 / math.sqrt(d_nope + D_R))
