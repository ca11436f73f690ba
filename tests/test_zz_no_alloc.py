"""pfkv_paged_decode_attn_noalloc: the attention entry point for callers that
cannot allocate device memory at decode time (an engine whose GPU memory is all
given to weights and the KV pool, a plugin whose host framework owns every
allocation, a loop that must not risk a synchronising cudaMalloc).  It uses a
fixed workspace inside the library instead of one the caller passes.

Checked through the C ABI against pfkv_paged_decode_attn with a caller
workspace and against the oracle, on calls in a row with different inputs:
the first leaves the shared array full of another batch's partial rows and
validation bits (a stale tag on request 0, longer sequences), so a second
call that read anything it did not write first would show it.  This file is
named to be collected last and builds what it needs, so it runs the same alone
in a fresh process or after the other tests.
"""
import dataclasses

import numpy as np
import pytest
import torch

from oracle_cases import ATOL, RTOL, assert_outputs_close, oracle_reference
from paged_fp8_kv_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_fp8_kv_decode_gb300 import build as pbuild
    pbuild.build()
    from paged_fp8_kv_decode_gb300 import binding
    binding.lib()
    return binding


def _close(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return bool(np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b)))


def _batch(spec, stale_request=None):
    """A batch without an appended token; with `stale_request`, one live page
    of that request carries a tag that no longer matches."""
    batch = W.make_batch(spec)
    if stale_request is not None:
        row = batch.table_row(stale_request, 0)
        n = int(batch.lens_bh("seq")[stale_request, 0])
        phys = int(row[(n - 1) // W.PAGE_SIZE // 2])
        heads = slice(0, 1) if batch.block_tables.ndim == 3 else slice(None)  # per-head tables
        batch.page_tags[phys, heads] ^= np.uint32(0x5A5A0001)
    return batch


def _check(B, db, spec, batch, ref):
    """One noalloc call on db: flags and output against the oracle (ref) and
    against the caller-workspace call."""
    out = torch.full_like(db.out, 7.0)
    flags = torch.full_like(db.flags, 0xEE)
    B.pfkv_paged_decode_attn_noalloc(db.cache, db.pages, db.q, spec.sm_scale, db.split_tokens,
                                     db.max_seq_len, out, flags)
    torch.cuda.synchronize()
    assert np.array_equal(flags.cpu().numpy()[:spec.B], ref["flags"]), spec.name
    assert_outputs_close(out, ref["out"], spec.name)
    ws_out = torch.empty_like(db.out)
    ws_flags = torch.zeros_like(db.flags)
    B.pfkv_paged_decode_attn(db.cache, db.pages, db.q, spec.sm_scale, db.split_tokens,
                             db.max_seq_len, db.workspace, ws_out, ws_flags)
    torch.cuda.synchronize()
    assert torch.equal(flags[:spec.B], ws_flags[:spec.B]), spec.name
    assert _close(out, ws_out), spec.name
    return flags.cpu().numpy()[:spec.B]


@pytest.mark.parametrize("kind", ["llama8b", "evict", "bf16"])
def test_noalloc_calls_in_a_row_with_different_inputs(B, kind):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    if kind == "llama8b":
        first = dataclasses.replace(W.spec_llama8b("small"), append=False, name="first")
        second = dataclasses.replace(W.spec_llama8b("small", seed=W.BASE_SEED + 77), append=False,
                                     lens=np.array([150, 33, 410], np.int32), B=3, name="second")
    elif kind == "evict":
        first = dataclasses.replace(W.spec_evict("small"), name="first")
        second = dataclasses.replace(W.spec_evict("small", seed=W.BASE_SEED + 78), stale_per_mille=0.0,
                                     name="second")
        second = dataclasses.replace(second, lens=np.maximum(second.lens // 3, 1))
    else:
        first = dataclasses.replace(W.spec_sweep(3, "bf16", scale="small"), name="first",
                                    lens=np.array([999, 700, 1000], np.int32))
        second = dataclasses.replace(W.spec_sweep(2, "bf16", scale="small"), name="second",
                                     lens=np.array([64, 300], np.int32))
    runs = []
    for spec, stale in ((first, 0), (second, None)):
        batch = _batch(spec, stale)
        db = DeviceBatch(batch, keep_rows=True)
        ref = oracle_reference(spec, batch, db.k_rows.cpu(), db.v_rows.cpu(), db.q.cpu())
        runs.append((spec, batch, db, ref))
    f1 = _check(B, *(runs[0][i] for i in (2, 0, 1, 3)))
    assert f1[0] & B.PFKV_FLAG_TAG_MISMATCH  # the first call leaves request 0 flagged
    f2 = _check(B, *(runs[1][i] for i in (2, 0, 1, 3)))
    assert not f2.any()                      # nothing of it carries over
    _check(B, *(runs[0][i] for i in (2, 0, 1, 3)))  # and back again


def test_noalloc_rejects_calls_beyond_its_workspace(B):
    """A call that would need more than the built-in workspace is refused
    with PFKV_ERR_WORKSPACE before anything runs; out is left untouched."""
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    spec = dataclasses.replace(W.spec_llama8b("small"), Hq=64)  # groups of 8 query heads
    db = DeviceBatch(W.make_batch(spec))
    # 16-token chunks of up to 2^20 tokens: the split kernel's tables fill up
    # (4,096 segments) and every partial row holds 8 heads: a large workspace
    split, max_len = 16, 1 << 20
    need = B.pfkv_decode_workspace_size(db.cache, db.pages, spec.Hq, split, max_len)
    assert need > B.PFKV_NOALLOC_WORKSPACE_BYTES
    out = torch.full_like(db.out, 3.0)
    with pytest.raises(B.PfkvError) as e:
        B.pfkv_paged_decode_attn_noalloc(db.cache, db.pages, db.q, spec.sm_scale, split, max_len,
                                         out, db.flags)
    assert e.value.status == B.PFKV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out.float() == 3.0).all())
