"""Helpers that turn a ``workloads.Batch`` into the oracle's host arrays.

Used by the oracle pins and by the GPU parity tests: the oracle quantises the
pool itself, from the same bf16 rows the CUDA path receives.
"""
import numpy as np

import oracle
from paged_fp8_kv_decode_gb300 import workloads as W


def empty_pool(spec):
    NP, H, D = spec.num_pages, spec.Hkv, spec.D
    if spec.kv_dtype == "bf16":
        k = np.zeros((NP, H, W.PAGE_SIZE, D), dtype=np.uint16)
        v = np.zeros_like(k)
        ks = vs = None
    else:
        k = np.zeros((NP, H, W.PAGE_SIZE, D), dtype=np.uint8)
        v = np.zeros_like(k)
        ks = np.ones((NP, H), dtype=np.float32)
        vs = np.ones((NP, H), dtype=np.float32)
    return k, v, ks, vs


def cache_dict(spec, batch, k, v, ks, vs, tags=True):
    return dict(num_pages=spec.num_pages, num_kv_heads=spec.Hkv, head_dim=spec.D,
                dtype=0 if spec.kv_dtype == "bf16" else 1, k_pages=k, v_pages=v,
                k_scale=ks, v_scale=vs,
                page_tags=batch.page_tags if (tags and spec.tags) else None)


def pages_dict(spec, batch, lens, tags=True):
    return dict(batch=spec.B, max_pages=batch.max_pages, block_tables=batch.block_tables,
                bt_stride_b=batch.bt_strides[0], bt_stride_h=batch.bt_strides[1],
                seq_lens=lens, len_stride_b=batch.len_strides[0],
                len_stride_h=batch.len_strides[1],
                expected_tags=batch.expected_tags if (tags and spec.tags) else None)


def fill_pool(spec, batch, k_rows_bits, v_rows_bits, tags_during_fill=False):
    """Quantise/store the cached tokens (positions 0..fill_len-1) with the
    oracle's kv_append.  Tags are not checked during the fill (the stale tags
    model pages reallocated after the fill)."""
    k, v, ks, vs = empty_pool(spec)
    cache = cache_dict(spec, batch, k, v, ks, vs, tags=tags_during_fill)
    pages = pages_dict(spec, batch, batch.seq_lens, tags=tags_during_fill)
    zeros = np.zeros_like(batch.fill_lens)
    oracle.kv_append(cache, pages, zeros, k_rows_bits, v_rows_bits, new_lens=batch.fill_lens)
    return k, v, ks, vs


# --------------------------------------------------------------------------
# GPU-vs-oracle comparison helpers (used by the -m gpu tests)
# --------------------------------------------------------------------------
ATOL = 1e-2   # the contract: |gpu - ref| <= 1e-2 + 1e-2 * |ref| per element
RTOL = 1e-2


def host_pool(t):
    """Host numpy view of a device pool tensor (uint16 bits for bf16)."""
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def assert_outputs_close(gpu_out, ref, label=""):
    """Element-wise |gpu - ref| <= ATOL + RTOL*|ref|; returns (max_abs, max_rel)."""
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = np.argwhere(err > bound)
    assert bad.size == 0, (label, [(tuple(i), g[tuple(i)], ref[tuple(i)]) for i in bad[:8]])
    max_abs = float(err.max()) if err.size else 0.0
    max_rel = float((err / np.maximum(np.abs(ref), 1e-30)).max()) if err.size else 0.0
    return max_abs, max_rel


def oracle_reference(spec, batch, k_rows, v_rows, q, k_new=None, v_new=None,
                     split_check=None, tags=True):
    """Run the whole step on the oracle: fill, append (if the workload appends),
    attention.  Returns dict(k, v, ks, vs, append_flags, out, flags)."""
    k, v, ks, vs = fill_pool(spec, batch, W.bf16_bits(k_rows), W.bf16_bits(v_rows))
    res = dict(fill_k=k.copy(), fill_v=v.copy(),
               fill_ks=None if ks is None else ks.copy(),
               fill_vs=None if vs is None else vs.copy())
    cache = cache_dict(spec, batch, k, v, ks, vs, tags=tags)
    pages = pages_dict(spec, batch, batch.seq_lens, tags=tags)
    aflags = np.zeros(spec.B, dtype=np.uint8)
    if spec.append:
        oracle.kv_append(cache, pages, batch.positions, W.bf16_bits(k_new), W.bf16_bits(v_new),
                         flags=aflags)
    out, flags = oracle.paged_decode(cache, pages, W.bf16_bits(q), spec.Hq, spec.sm_scale,
                                     int(batch.seq_lens.max()))
    res.update(k=k, v=v, ks=ks, vs=vs, append_flags=aflags, out=out, flags=flags)
    return res
