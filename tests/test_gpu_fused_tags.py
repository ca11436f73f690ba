"""The tag check fused into the attention kernel (pfkv_paged_decode_attn_fused_tags)
against the oracle, on every kernel path: the persistent tensor-core kernel
(head_dim 128 and 64, FP8 and BF16, with a coarsened split and in request
groups; the per-chunk kernel's fused check is in the multi-query tests).
Flags must equal the oracle's tag/bounds check bit for bit; outputs are within the contract tolerance (the fused call may split the
work differently from the two-kernel call, so the two are not compared bit for
bit with each other)."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle_cases import assert_outputs_close
from paged_fp8_kv_decode_gb300 import workloads as W
from test_gpu_parity import B, run_and_compare  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def test_evict_small_stale_tags_fused(B):
    db, ref, _ = run_and_compare(W.spec_evict("small"), label="evict fused", fused_tags=True)
    assert ref["flags"].any() and not ref["flags"].all()


@pytest.mark.parametrize("split", [0, 48])
def test_llama8b_small_with_stale_tags_fused(B, split):
    spec = dataclasses.replace(W.spec_llama8b("small"), split_tokens=split, stale_per_mille=1.0)
    db, ref, _ = run_and_compare(spec, label=f"llama fused split {split}", fused_tags=True)
    assert ref["flags"].any() and not ref["flags"].all()


@pytest.mark.parametrize("kv_dtype,D,G", [("bf16", 128, 4), ("fp8", 64, 2), ("fp8", 128, 8),
                                          ("bf16", 64, 1)])
def test_per_chunk_kernels_with_stale_tags_fused(B, kv_dtype, D, G):
    base = W.spec_sweep(6, kv_dtype, scale="small")
    spec = dataclasses.replace(base, D=D, Hkv=4, Hq=4 * G, stale_per_mille=10.0,
                               lens=np.array([1000, 37, 512, 999, 16, 700], np.int32))
    db, ref, _ = run_and_compare(spec, label=f"{kv_dtype} D{D} G{G} fused", fused_tags=True)
    assert ref["flags"].any() and not ref["flags"].all()


def test_without_tags_fused_equals_plain(B):
    """With the no-op tracker the fused entry is the plain call."""
    spec = W.spec_llama8b("small")
    db, ref, _ = run_and_compare(spec, tags=False, label="no tags fused", fused_tags=True)
    out_fused = db.out.clone()
    db.fused_tags = False
    db.attend()
    torch.cuda.synchronize()
    assert torch.equal(out_fused, db.out)


def test_bad_ids_and_stale_tags_fused(B):
    """Out-of-pool ids are BAD_PAGE, stale in-pool pages TAG_MISMATCH, both in the
    same request and apart, as the separate validation reports them."""
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    spec = dataclasses.replace(W.spec_evict("small"), stale_per_mille=0.0)
    batch = W.make_batch(spec)
    db = DeviceBatch(batch, fused_tags=True)
    lens = batch.lens_bh("seq")
    bt = db.block_tables.view(spec.B, spec.Hkv, -1)
    ex = db.expected_tags.view(spec.B, spec.Hkv, -1)
    bt[0, 1, 0] = spec.num_pages + 5            # request 0: bad id
    ex[1, 2, (int(lens[1, 2]) - 1) // 16] ^= 1   # request 1: stale tag on its last live page
    bt[2, 0, 0] = -7                             # request 2: bad id and a stale tag
    ex[2, 3, 0] ^= 1 << 4
    db.attend()
    torch.cuda.synchronize()
    flags = db.flags.cpu().numpy()[:spec.B]
    want = np.zeros(spec.B, np.uint8)
    want[0] = 2
    want[1] = 1
    want[2] = 3
    assert np.array_equal(flags, want), flags
    for b in range(3):
        assert not db.out[b].float().abs().sum().item()
    # the separate validation reports the same bits
    db.fused_tags = False
    db.attend()
    torch.cuda.synchronize()
    assert np.array_equal(db.flags.cpu().numpy()[:spec.B], want)


def test_many_segments_coarsened_fused(B):
    """More segments than the persistent kernel's tables at the caller's split
    size: a coarser split, with the tag check fused into the kernel."""
    lens = np.array([3000, 2900, 2950], dtype=np.int32)
    spec = W.Spec("manyseg", B=3, Hq=32, Hkv=8, D=128, kv_dtype="fp8", num_pages=1024,
                  lens=lens, tags=True, split_tokens=16, seed=404, stale_per_mille=0.5)
    db, ref, _ = run_and_compare(spec, label="many-segments fused", fused_tags=True)
    assert ref["flags"].any() and not ref["flags"].all()


def test_request_groups_fused(B):
    """520 requests x 8 kv heads: request groups, tag check fused."""
    rng = np.random.default_rng(909)
    lens = rng.integers(1, 80, size=520, endpoint=True).astype(np.int32)
    spec = W.Spec("groups-fused", B=520, Hq=32, Hkv=8, D=128, kv_dtype="fp8",
                  num_pages=int(((lens + 16) // 16).sum()) + 16, lens=lens, append=True, tags=True,
                  stale_per_mille=3.0, seed=909)
    db, ref, _ = run_and_compare(spec, label="request groups fused", fused_tags=True)
    assert ref["flags"].any()
