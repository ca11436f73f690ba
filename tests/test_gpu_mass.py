"""Attention mass (pfkv_paged_decode_attn_mass) against the oracle on every
kernel configuration: the persistent kernel (FP8 and BF16, head_dim 128 and
64, G up to 8, automatic and fixed splits, per-head tables, stale tags) and
its many-segment coarsening, with the separate and the fused tag check.

The accumulator starts from seeded non-zero values and has padded rows, so
the test sees accumulation, strides, and that entries past a head's length
and rows of flagged requests stay untouched.  Tolerance: |gpu - ref| <=
1e-6 + 1e-3 |ref| per entry (weights are fp32 2^(score - lse); the oracle is
fp64), and every head's masses sum to G within 1e-3."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle_cases import assert_outputs_close, cache_dict, oracle_reference, pages_dict
from paged_fp8_kv_decode_gb300 import workloads as W
from test_gpu_parity import B  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def _run(B, spec, fused=False, label=""):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    batch = W.make_batch(spec)
    db = DeviceBatch(batch, keep_rows=True)
    db.append_step()
    torch.cuda.synchronize()
    L = int(batch.seq_lens.max())
    ws = torch.empty(B.pfkv_decode_mass_workspace_size(db.cache, db.pages, spec.Hq,
                                                       spec.split_tokens, L),
                     dtype=torch.uint8, device="cuda")
    gen = torch.Generator().manual_seed(99)
    init = torch.rand((spec.B, spec.Hkv, L + 7), generator=gen, dtype=torch.float32)
    mass = init.cuda()
    B.pfkv_paged_decode_attn_mass(db.cache, db.pages, db.q, spec.sm_scale, spec.split_tokens, L,
                                  ws, db.out, db.flags, mass,
                                  B.PFKV_STAGE_FUSED_TAGS if fused else 0)
    torch.cuda.synchronize()
    ref = oracle_reference(spec, batch, db.k_rows.cpu(), db.v_rows.cpu(), db.q.cpu(),
                           None if db.k_new is None else db.k_new.cpu(),
                           None if db.v_new is None else db.v_new.cpu())
    flags = db.flags.cpu().numpy()[:spec.B]
    assert np.array_equal(flags, ref["flags"]), (label, flags, ref["flags"])
    assert_outputs_close(db.out, ref["out"], label)
    cache = cache_dict(spec, batch, ref["k"], ref["v"], ref["ks"], ref["vs"])
    pages = pages_dict(spec, batch, batch.seq_lens)
    want = oracle.attention_mass(cache, pages, W.bf16_bits(db.q), spec.Hq, spec.sm_scale, L,
                                 mass=init.numpy().astype(np.float64))
    got = mass.cpu().numpy().astype(np.float64)
    bad = np.argwhere(np.abs(got - want) > 1e-6 + 1e-3 * np.abs(want))
    assert bad.size == 0, (label, [(tuple(i), got[tuple(i)], want[tuple(i)]) for i in bad[:6]])
    lens = batch.lens_bh("seq")
    base = init.numpy().astype(np.float64)
    for b in range(spec.B):
        for h in range(spec.Hkv):
            n = int(lens[b, h])
            added = got[b, h] - base[b, h]
            if flags[b] or n == 0:
                assert np.array_equal(got[b, h], base[b, h]), (label, b, h)
            else:
                assert abs(added[:n].sum() - spec.G) < 1e-3, (label, b, h, added[:n].sum())
                assert np.array_equal(got[b, h, n:], base[b, h, n:]), (label, b, h)
    return flags


@pytest.mark.parametrize("split", [0, 48, 1024])
def test_llama8b_small(B, split):
    _run(B, dataclasses.replace(W.spec_llama8b("small"), split_tokens=split), label=f"llama {split}")


@pytest.mark.parametrize("fused", [False, True])
def test_evict_small_per_head_and_stale_tags(B, fused):
    flags = _run(B, W.spec_evict("small"), fused=fused, label=f"evict fused={fused}")
    assert flags.any() and not flags.all()


def test_long_small_split(B):
    _run(B, W.spec_long("small"), label="long")


@pytest.mark.parametrize("kv_dtype,D,G", [("bf16", 128, 4), ("fp8", 64, 2), ("fp8", 128, 8),
                                          ("bf16", 64, 1)])
def test_per_chunk_kernels(B, kv_dtype, D, G):
    base = W.spec_sweep(5, kv_dtype, scale="small")
    spec = dataclasses.replace(base, D=D, Hkv=4, Hq=4 * G,
                               lens=np.array([1000, 37, 512, 16, 700], np.int32))
    _run(B, spec, label=f"{kv_dtype} D{D} G{G}")


def test_many_segments_coarsened(B):
    lens = np.array([3000, 2900, 2950], dtype=np.int32)
    spec = W.Spec("manyseg", B=3, Hq=32, Hkv=8, D=128, kv_dtype="fp8", num_pages=1024,
                  lens=lens, tags=True, split_tokens=16, seed=404)
    _run(B, spec, label="many-segments")


def test_request_groups(B):
    """520 requests x 8 kv heads: request groups; the scores and final
    normalisers of every group meet in the one mass pass."""
    rng = np.random.default_rng(808)
    lens = rng.integers(1, 60, size=520, endpoint=True).astype(np.int32)
    spec = W.Spec("groups-mass", B=520, Hq=32, Hkv=8, D=128, kv_dtype="fp8",
                  num_pages=int(((lens + 16) // 16).sum()) + 16, lens=lens, tags=True,
                  stale_per_mille=3.0, seed=808)
    _run(B, spec, label="request groups")


def test_zero_length_heads(B):
    lens = np.array([[0, 40, 17, 0], [33, 0, 0, 5]], dtype=np.int32)
    spec = W.Spec("zeros", B=2, Hq=8, Hkv=4, D=128, kv_dtype="fp8", num_pages=64, lens=lens,
                  per_head=True, tags=True, seed=77)
    _run(B, spec, label="zero-length heads")
