"""Multi-query verify (pfkv_paged_decode_attn_multi) against the oracle: kq
candidate tokens per request, the last kq tokens of every head, query token i
attending to the first n - kq + 1 + i tokens.  Covers the persistent FP8
kernel (automatic and fixed splits, per-head tables, stale tags with the
separate and the fused check, BF16, head_dim 64, G = 8), a split coarsened to
fit, request groups, the per-chunk kernel (more query tokens x kv heads than
one persistent launch's tables hold), heads shorter than kq, and kq = 1 equal
to the plain call.  Outputs within the contract tolerance; flags bit for bit."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle_cases import assert_outputs_close, cache_dict, fill_pool, pages_dict
from paged_fp8_kv_decode_gb300 import workloads as W
from test_gpu_parity import B  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def _run(B, spec, kq, fused=False, label=""):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    batch = W.make_batch(spec)
    db = DeviceBatch(batch, keep_rows=True)
    g = torch.Generator(device="cuda").manual_seed(1234 + kq)
    q = torch.randn((spec.B, kq, spec.Hq, spec.D), generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    L = int(batch.seq_lens.max())
    ws = torch.empty(max(256, B.pfkv_decode_multi_workspace_size(db.cache, db.pages, spec.Hq, kq,
                                                                 spec.split_tokens, L)),
                     dtype=torch.uint8, device="cuda")
    B.pfkv_paged_decode_attn_multi(db.cache, db.pages, q, spec.sm_scale, spec.split_tokens, L,
                                   ws, out, db.flags, B.PFKV_STAGE_FUSED_TAGS if fused else 0)
    torch.cuda.synchronize()
    k, v, ks, vs = fill_pool(spec, batch, W.bf16_bits(db.k_rows), W.bf16_bits(db.v_rows))
    cache = cache_dict(spec, batch, k, v, ks, vs)
    pages = pages_dict(spec, batch, batch.seq_lens)
    ref, rflags = oracle.paged_decode_multi(cache, pages, W.bf16_bits(q), spec.Hq, kq,
                                            spec.sm_scale, L)
    flags = db.flags.cpu().numpy()[:spec.B]
    assert np.array_equal(flags, rflags), (label, flags, rflags)
    assert_outputs_close(out, ref, label)
    return db, q, out, flags, ws


@pytest.mark.parametrize("kq", [1, 2, 4, 7])
@pytest.mark.parametrize("split", [0, 48])
def test_llama8b_small(B, kq, split):
    spec = dataclasses.replace(W.spec_llama8b("small"), append=False, split_tokens=split)
    _run(B, spec, kq, label=f"llama kq={kq} split={split}")


@pytest.mark.parametrize("fused", [False, True])
def test_evict_small_per_head_and_stale_tags(B, fused):
    _, _, _, flags, _ = _run(B, W.spec_evict("small"), 3, fused=fused, label=f"evict fused={fused}")
    assert flags.any() and not flags.all()


@pytest.mark.parametrize("kv_dtype,D,G,kq", [("bf16", 128, 4, 3), ("fp8", 64, 2, 2),
                                             ("fp8", 128, 8, 4), ("bf16", 64, 1, 5),
                                             ("fp8", 64, 8, 3), ("bf16", 64, 4, 2)])
def test_dtypes_head_dims_and_groups(B, kv_dtype, D, G, kq):
    base = W.spec_sweep(5, kv_dtype, scale="small")
    spec = dataclasses.replace(base, D=D, Hkv=4, Hq=4 * G,
                               lens=np.array([1000, 37, 512, 16, 700], np.int32))
    _run(B, spec, kq, label=f"{kv_dtype} D{D} G{G} kq={kq}")


@pytest.mark.parametrize("kv_dtype,D,fused", [("fp8", 128, False), ("fp8", 128, True),
                                              ("bf16", 64, False), ("fp8", 64, True)])
def test_per_chunk_kernel_for_many_query_tokens(B, kv_dtype, D, fused):
    """520 query tokens x 8 kv heads = 4,160 virtual (request, kv head)
    pairs: more than one persistent launch holds even for one request, so
    the per-chunk kernel and its combine take the call (with the separate or
    the fused tag check; a stale tag flags a request)."""
    lens = np.array([700, 530], dtype=np.int32)
    spec = W.Spec(f"perchunk-{kv_dtype}-d{D}", B=2, Hq=16, Hkv=8, D=D, kv_dtype=kv_dtype,
                  num_pages=int(((lens + 16) // 16).sum()) + 8, lens=lens, tags=True,
                  stale_per_mille=30.0, split_tokens=0, seed=808 + D)
    _run(B, spec, 520, fused=fused, label=f"per-chunk {kv_dtype} D{D} fused={fused} kq=520")


def test_many_segments_coarsened(B):
    lens = np.array([3000, 2900, 2950], dtype=np.int32)
    spec = W.Spec("manyseg", B=3, Hq=32, Hkv=8, D=128, kv_dtype="fp8", num_pages=1024,
                  lens=lens, tags=True, split_tokens=16, seed=404)
    _run(B, spec, 2, label="many-segments kq=2")


def test_request_groups(B):
    """200 requests x 3 query tokens x 8 kv heads > 4,096 virtual (request,
    kv head) pairs: request groups whose virtual requests stay whole; stale
    tags flag some requests."""
    rng = np.random.default_rng(707)
    lens = rng.integers(3, 70, size=200, endpoint=True).astype(np.int32)
    spec = W.Spec("groups-kq3", B=200, Hq=32, Hkv=8, D=128, kv_dtype="fp8",
                  num_pages=int(((lens + 16) // 16).sum()) + 16, lens=lens, tags=True,
                  stale_per_mille=4.0, seed=707)
    _, _, _, flags, _ = _run(B, spec, 3, label="request groups kq=3")
    assert flags.any() and not flags.all()


def test_heads_shorter_than_the_candidates(B):
    lens = np.array([[2, 40, 1, 0], [33, 3, 0, 5]], dtype=np.int32)
    spec = W.Spec("short", B=2, Hq=8, Hkv=4, D=128, kv_dtype="fp8", num_pages=64, lens=lens,
                  per_head=True, tags=True, seed=78)
    _, _, out, _, _ = _run(B, spec, 4, label="short heads")
    assert not out[0, 0, 0:2].float().abs().sum().item()   # n = 2: queries 0, 1 see nothing
    assert not out[0, 1, 0:2].float().abs().sum().item()
    assert out[0, 2, 0:2].float().abs().sum().item()


def test_one_query_token_equals_the_plain_call(B):
    spec = dataclasses.replace(W.spec_llama8b("small"), append=False)
    db, q, out, _, _ = _run(B, spec, 1, label="kq=1")
    db.q.copy_(q[:, 0])
    db.attend()
    torch.cuda.synchronize()
    assert torch.equal(db.out, out[:, 0])


@pytest.mark.parametrize("kv_dtype,D", [("fp8", 128), ("bf16", 128), ("fp8", 64)])
def test_cuda_core_option_matches_the_oracle(B, kv_dtype, D):
    """PFKV_STAGE_CUDA_CORES runs the per-chunk CUDA-core kernels for a shape
    the tensor-core kernel would take; the result matches the oracle too."""
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    base = W.spec_sweep(5, kv_dtype, scale="small")
    spec = dataclasses.replace(base, D=D, Hkv=4, Hq=16, lens=np.array([1000, 37, 512, 16, 700], np.int32))
    batch = W.make_batch(spec)
    db = DeviceBatch(batch, keep_rows=True)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty_like(db.out)
    B.pfkv_paged_decode_attn_stages(db.cache, db.pages, db.q, spec.sm_scale, 0, db.max_seq_len, ws, out,
                                    db.flags, B.PFKV_STAGE_ALL | B.PFKV_STAGE_CUDA_CORES)
    torch.cuda.synchronize()
    k, v, ks, vs = fill_pool(spec, batch, W.bf16_bits(db.k_rows), W.bf16_bits(db.v_rows))
    cache = cache_dict(spec, batch, k, v, ks, vs)
    pages = pages_dict(spec, batch, batch.seq_lens)
    ref, rflags = oracle.paged_decode_multi(cache, pages, W.bf16_bits(db.q[:, None]), spec.Hq, 1,
                                            spec.sm_scale, db.max_seq_len)
    assert np.array_equal(db.flags.cpu().numpy()[:spec.B], rflags)
    assert_outputs_close(out, ref[:, 0], f"cuda cores {kv_dtype} D{D}")
