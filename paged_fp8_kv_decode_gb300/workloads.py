"""Seeded synthetic decode batches (shared by the CUDA path's tests, the oracle's
tests and the benchmark).

This module only draws inputs: shapes, lengths, page assignments, tags and
bf16 K/V/q values.  It holds none of the method's arithmetic: no quantisation,
no attention, no tag checking.  Quantising the pool is the job of the library's
``kv_append`` (CUDA path) or of the oracle's ``kv_append`` (CPU reference); both
start from the same bf16 rows drawn here.

Workloads (Llama-3.1-8B-shaped stand-ins for the serving traffic the pages
measure, which is not available here):
  tiny     B=2, Hq=4, Hkv=2, D=64, lens {37, 100}, BF16, pool of 32 pages
  llama8b  B=32, Hq=32, Hkv=8, D=128, lens ~ U[512, 8192], FP8, 65,536 pages,
           one appended token per sequence, then attention over len+1 tokens
  long     B=4, Hq=32, Hkv=8, D=128, lens {128K, 256K, 384K, 512K}, FP8,
           split-KV chunks of 4096 tokens
  sweep    B in {1, 8, 16, 32, 64}, every len 32768, BF16 or FP8, pages drawn
           from a pool sized like an 80 GB cache
  evict    B=16, base len ~ U[4096, 32768], per-head length base // r with r
           per (request, kv head) from {1, 8, 64}, per-head tables, FP8, one in
           a thousand live units carries a stale tag

Value recipe: q ~ N(0, 1); K, V ~ N(0, 1) with each element multiplied by 20
with probability 0.01 (outliers); everything rounded to bf16.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

PAGE_SIZE = 16
BASE_SEED = 20261202


@dataclasses.dataclass
class Spec:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    kv_dtype: str                  # "bf16" or "fp8"
    num_pages: int
    lens: np.ndarray               # int32 [B] (shared tables) or [B][Hkv] (per-head)
    per_head: bool = False         # per-(request, kv head) block tables and lengths
    append: bool = False           # one token appended before attention
    tags: bool = True
    stale_per_mille: float = 0.0   # stale tags: round(live_units * x / 1000) units
    split_tokens: int = 0          # 0 = library's automatic split
    outlier_prob: float = 0.01
    outlier_mult: float = 20.0
    seed: int = BASE_SEED

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


# --------------------------------------------------------------------------
# workload specs
# --------------------------------------------------------------------------
def spec_tiny(seed: int = BASE_SEED + 1) -> Spec:
    return Spec("tiny", B=2, Hq=4, Hkv=2, D=64, kv_dtype="bf16", num_pages=32,
                lens=np.array([37, 100], dtype=np.int32), tags=True, outlier_prob=0.0,
                seed=seed)


def spec_llama8b(scale: str = "full", seed: int = BASE_SEED + 2) -> Spec:
    rng = _rng(seed)
    if scale == "full":
        B, lo, hi, NP = 32, 512, 8192, 65536
    elif scale == "small":
        B, lo, hi, NP = 4, 200, 1500, 1024
    else:
        raise ValueError(scale)
    lens = rng.integers(lo, hi, size=B, endpoint=True).astype(np.int32)
    return Spec("llama8b", B=B, Hq=32, Hkv=8, D=128, kv_dtype="fp8", num_pages=NP, lens=lens,
                append=True, tags=True, seed=seed)


def spec_long(scale: str = "full", seed: int = BASE_SEED + 3) -> Spec:
    if scale == "full":
        lens = np.array([131072, 262144, 393216, 524288], dtype=np.int32)
        NP, split = 131072, 4096
    elif scale == "small":
        lens = np.array([2500, 5203], dtype=np.int32)
        NP, split = 1024, 1024
    else:
        raise ValueError(scale)
    return Spec("long", B=len(lens), Hq=32, Hkv=8, D=128, kv_dtype="fp8", num_pages=NP,
                lens=lens, tags=True, split_tokens=split, seed=seed)


def sweep_pool_pages(kv_dtype: str, Hkv: int = 8, D: int = 128,
                     pool_bytes: float = 80e9) -> int:
    """Pages of an 80 GB (decimal) K+V pool: a page holds 16 tokens of every kv
    head, K and V; FP8 pages also carry two fp32 scales per kv head."""
    per_page = 2 * Hkv * PAGE_SIZE * D * (2 if kv_dtype == "bf16" else 1)
    if kv_dtype == "fp8":
        per_page += 2 * Hkv * 4
    return int(pool_bytes // per_page)


def spec_sweep(B: int, kv_dtype: str, scale: str = "full", seed: int = BASE_SEED + 4,
               num_pages: Optional[int] = None) -> Spec:
    L = 32768 if scale == "full" else 1000
    NP = num_pages if num_pages is not None else (
        sweep_pool_pages(kv_dtype) if scale == "full" else 4096)
    return Spec(f"sweep-{kv_dtype}-b{B}", B=B, Hq=32, Hkv=8, D=128, kv_dtype=kv_dtype,
                num_pages=NP, lens=np.full(B, L, dtype=np.int32), tags=True, seed=seed + B)


def spec_evict(scale: str = "full", seed: int = BASE_SEED + 5) -> Spec:
    rng = _rng(seed)
    if scale == "full":
        B, lo, hi, NP = 16, 4096, 32768, 65536
    elif scale == "small":
        B, lo, hi, NP = 6, 600, 3000, 2048
    else:
        raise ValueError(scale)
    Hkv = 8
    base = rng.integers(lo, hi, size=B, endpoint=True)
    r = rng.choice(np.array([1, 8, 64]), size=(B, Hkv))
    lens = (base[:, None] // r).astype(np.int32)
    return Spec("evict", B=B, Hq=32, Hkv=Hkv, D=128, kv_dtype="fp8", num_pages=NP, lens=lens,
                per_head=True, tags=True, stale_per_mille=1.0, seed=seed)


# --------------------------------------------------------------------------
# structure: tables, tags
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Batch:
    """Host arrays of one decode step (no pool contents: see module docstring)."""
    spec: Spec
    seq_lens: np.ndarray        # int32, [B] or [B][Hkv]: tokens attended
    fill_lens: np.ndarray       # int32, same shape: tokens already in the cache
    positions: np.ndarray       # int32, same shape: where the appended token goes
    len_strides: tuple          # (stride_b, stride_h) of the three arrays above
    block_tables: np.ndarray    # int32 [B][MP] or [B][Hkv][MP]
    bt_strides: tuple
    max_pages: int
    page_tags: np.ndarray       # uint32 [NP][Hkv] (tags as they are in the pool)
    expected_tags: np.ndarray   # uint32, shaped like block_tables
    stale_units: np.ndarray     # int64 [k][2] (phys, h) with a stale tag
    live_units: int

    def lens_bh(self, which: str = "seq") -> np.ndarray:
        a = self.seq_lens if which == "seq" else self.fill_lens
        if a.ndim == 1:
            return np.repeat(a[:, None], self.spec.Hkv, axis=1)
        return a

    def table_row(self, b: int, h: int) -> np.ndarray:
        if self.block_tables.ndim == 2:
            return self.block_tables[b]
        return self.block_tables[b, h]


def make_batch(spec: Spec) -> Batch:
    rng = _rng(spec.seed + 7919)
    B, Hkv, NP = spec.B, spec.Hkv, spec.num_pages
    fill = np.asarray(spec.lens, dtype=np.int32)
    seq = fill + 1 if spec.append else fill.copy()
    positions = fill.copy()
    if spec.per_head:
        assert fill.shape == (B, Hkv)
        len_strides = (Hkv, 1)
    else:
        assert fill.shape == (B,)
        len_strides = (1, 0)
    pages_needed = (seq.astype(np.int64) + PAGE_SIZE - 1) // PAGE_SIZE
    MP = int(max(1, pages_needed.max()))
    if spec.per_head:
        bt = np.full((B, Hkv, MP), -1, dtype=np.int32)
        for h in range(Hkv):
            need = int(pages_needed[:, h].sum())
            if need > NP:
                raise ValueError(f"{spec.name}: head {h} needs {need} pages > pool {NP}")
            perm = rng.permutation(NP)[:need].astype(np.int32)
            off = 0
            for b in range(B):
                k = int(pages_needed[b, h])
                bt[b, h, :k] = perm[off:off + k]
                off += k
        bt_strides = (Hkv * MP, MP)
    else:
        need = int(pages_needed.sum())
        if need > NP:
            raise ValueError(f"{spec.name}: needs {need} pages > pool {NP}")
        perm = rng.permutation(NP)[:need].astype(np.int32)
        bt = np.full((B, MP), -1, dtype=np.int32)
        off = 0
        for b in range(B):
            k = int(pages_needed[b])
            bt[b, :k] = perm[off:off + k]
            off += k
        bt_strides = (MP, 0)

    page_tags = rng.integers(0, 2 ** 32, size=(NP, Hkv), dtype=np.uint64).astype(np.uint32)
    # expected tags: what the server recorded at allocation time (entries past
    # a row's live length are padding and are never read)
    expected = np.zeros(bt.shape, dtype=np.uint32)
    live = []
    for b in range(B):
        for h in range(Hkv):
            k = int(pages_needed[b, h] if spec.per_head else pages_needed[b])
            if k == 0:
                continue
            if spec.per_head:
                rows = bt[b, h, :k]
                expected[b, h, :k] = page_tags[rows, h]
            elif h == 0:
                rows = bt[b, :k]
                expected[b, :k] = page_tags[rows, 0]
            for p in range(k):
                live.append((int(bt[b, h, p] if spec.per_head else bt[b, p]), h))
    if not spec.per_head:
        # one table shared by all heads: the server gives every head of a page
        # the same tag
        page_tags[:, 1:] = page_tags[:, :1]
    live = np.array(live, dtype=np.int64).reshape(-1, 2)
    n_stale = int(round(len(live) * spec.stale_per_mille / 1000.0)) if spec.tags else 0
    stale = live[rng.choice(len(live), size=n_stale, replace=False)] if n_stale else \
        np.zeros((0, 2), dtype=np.int64)
    for phys, h in stale:
        flip = np.uint32(rng.integers(1, 2 ** 32, dtype=np.uint64))
        if spec.per_head:
            page_tags[phys, h] ^= flip
        else:
            page_tags[phys, :] ^= flip
    return Batch(spec=spec, seq_lens=seq.astype(np.int32), fill_lens=fill, positions=positions,
                 len_strides=len_strides, block_tables=bt, bt_strides=bt_strides, max_pages=MP,
                 page_tags=page_tags, expected_tags=expected, stale_units=stale,
                 live_units=len(live))


# --------------------------------------------------------------------------
# values (bf16), drawn with torch so that large batches can be drawn on the GPU
# --------------------------------------------------------------------------
def draw_bf16(shape, seed: int, outlier_prob: float = 0.0, outlier_mult: float = 20.0,
              device="cpu"):
    """N(0,1) values, each multiplied by ``outlier_mult`` with probability
    ``outlier_prob``, rounded to bf16 (torch's round-to-nearest-even)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if outlier_prob > 0:
        u = torch.rand(*shape, generator=g, device=device, dtype=torch.float32)
        x = torch.where(u < outlier_prob, x * outlier_mult, x)
    return x.to(torch.bfloat16)


def draw_q(spec: Spec, device="cpu"):
    return draw_bf16((spec.B, spec.Hq, spec.D), spec.seed + 11, 0.0, device=device)


def draw_kv_rows(spec: Spec, T: int, which: str, device="cpu", head_slice=None):
    """bf16 K or V rows [B][Hkv][T][D] for the tokens already in the cache."""
    s = spec.seed + (101 if which == "k" else 202)
    shape = (spec.B, spec.Hkv, T, spec.D)
    return draw_bf16(shape, s, spec.outlier_prob, spec.outlier_mult, device=device)


def draw_new_token(spec: Spec, which: str, device="cpu"):
    """bf16 K or V of the token appended at this step, [B][Hkv][1][D]."""
    s = spec.seed + (303 if which == "k" else 404)
    return draw_bf16((spec.B, spec.Hkv, 1, spec.D), s, spec.outlier_prob, spec.outlier_mult,
                     device=device)


def bf16_bits(t) -> np.ndarray:
    """Host uint16 view of a bf16 torch tensor."""
    import torch
    if t.dtype != torch.bfloat16:
        raise TypeError(f"bf16_bits: expected a bfloat16 tensor, got {t.dtype}")
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
