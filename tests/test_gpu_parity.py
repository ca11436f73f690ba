"""GPU path vs the oracle on the same seeded inputs (small sizes that still
span several units, chunks and a ragged tail).

Bit-exact: e4m3 bytes and fp32 scales written by kv_append (fill and the
decode-step append), append flags and attention flags.  Within the contract
tolerance |gpu - ref| <= 1e-2 + 1e-2 |ref|: bf16 attention outputs (both sides
read the same e4m3 bytes, each produced by its own quantiser).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle_cases import (assert_outputs_close, cache_dict, host_pool, oracle_reference,
                          pages_dict)
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


def _db(batch, **kw):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    return DeviceBatch(batch, keep_rows=True, **kw)


def run_and_compare(spec, tags=None, rows=None, q=None, label="", fused_tags=False,
                    max_seq_len=None):
    """Fill, append, attend on the GPU and on the oracle; compare everything."""
    batch = W.make_batch(spec)
    use_tags = spec.tags if tags is None else tags
    db = _db(batch, tags=use_tags, rows=rows, q=q, fused_tags=fused_tags, max_seq_len=max_seq_len)
    ref = oracle_reference(spec, batch, db.k_rows.cpu(), db.v_rows.cpu(), db.q.cpu(),
                           None if db.k_new is None else db.k_new.cpu(),
                           None if db.v_new is None else db.v_new.cpu(), tags=use_tags)
    # the fill: bytes and scales bit for bit
    assert np.array_equal(host_pool(db.cache.k_pages), ref["fill_k"]), label
    assert np.array_equal(host_pool(db.cache.v_pages), ref["fill_v"]), label
    if spec.kv_dtype == "fp8":
        assert np.array_equal(db.cache.k_scale.cpu().numpy(), ref["fill_ks"]), label
        assert np.array_equal(db.cache.v_scale.cpu().numpy(), ref["fill_vs"]), label
    # the decode step
    db.append_step()
    db.attend()
    torch.cuda.synchronize()
    assert np.array_equal(host_pool(db.cache.k_pages), ref["k"]), label
    assert np.array_equal(host_pool(db.cache.v_pages), ref["v"]), label
    if spec.kv_dtype == "fp8":
        assert np.array_equal(db.cache.k_scale.cpu().numpy(), ref["ks"]), label
        assert np.array_equal(db.cache.v_scale.cpu().numpy(), ref["vs"]), label
    assert np.array_equal(db.append_flags.cpu().numpy()[:spec.B], ref["append_flags"]), label
    flags = db.flags.cpu().numpy()[:spec.B]
    assert np.array_equal(flags, ref["flags"]), (label, flags, ref["flags"])
    errs = assert_outputs_close(db.out, ref["out"], label)
    # flagged requests are all zero
    for b in np.nonzero(flags)[0]:
        assert not db.out[b].float().abs().sum().item()
    return db, ref, errs


# --------------------------------------------------------------------------
# the workloads at reduced size
# --------------------------------------------------------------------------
def test_tiny_bf16(B):
    run_and_compare(W.spec_tiny(), label="tiny")


@pytest.mark.parametrize("split", [0, 16, 48, 256, 1024, 8192])
def test_llama8b_small_fp8_append(B, split):
    spec = dataclasses.replace(W.spec_llama8b("small"), split_tokens=split)
    run_and_compare(spec, label=f"llama8b-small split={split}")


@pytest.mark.parametrize("split", [0, 1024])
def test_twelve_worker_shape(B, split):
    """A large host-known length bound (4 requests x 8 kv heads x 8,192 units,
    above 8 x 64 units per SM) selects the split kernel's 12-worker shape,
    while the actual lengths stay small enough for the oracle."""
    spec = dataclasses.replace(W.spec_llama8b("small"), split_tokens=split)
    run_and_compare(spec, label=f"llama8b-small 12 workers split={split}", max_seq_len=131072)


@pytest.mark.parametrize("kv_dtype", ["fp8", "bf16"])
@pytest.mark.parametrize("bound", [None, 131072])
def test_groups_of_eight_heads(B, kv_dtype, bound):
    """64 query heads over 8 kv heads: groups of 8, so every MMA column is a
    real head; one segment per head.  The large length bound selects the
    12-worker shape."""
    spec = dataclasses.replace(W.spec_llama8b("small"), Hq=64, kv_dtype=kv_dtype, name="g8")
    run_and_compare(spec, label=f"g8 {kv_dtype} bound={bound}", max_seq_len=bound)


@pytest.mark.parametrize("Bn,G", [(1, 4), (5, 4), (9, 4), (20, 4), (1, 8), (3, 8), (5, 8), (10, 8)])
def test_combine_query_head_groups(B, Bn, G):
    """Many partial rows per kv head (64-token chunks): the combine splits each
    kv head's G query heads over 1, 2, 4 or 8 CTAs, as many as keep one wave
    over the SMs. On 152 SMs these batches take every split of G = 4 and
    G = 8; a stale tag flags some requests."""
    rng = np.random.default_rng(700 + 10 * Bn + G)
    lens = rng.integers(60, 700, size=Bn, endpoint=True).astype(np.int32)
    spec = W.Spec(f"comb{Bn}x{G}", B=Bn, Hq=8 * G, Hkv=8, D=128, kv_dtype="fp8",
                  num_pages=int(((lens + 16) // 16 + 1).sum()) + 8, lens=lens, append=True,
                  stale_per_mille=2.0 if Bn >= 5 else 0.0, split_tokens=64, seed=7000 + Bn)
    run_and_compare(spec, label=f"combine groups B={Bn} G={G}")


def test_long_small_split(B):
    run_and_compare(W.spec_long("small"), label="long-small")


def test_evict_small_per_head_tables_and_stale_tags(B):
    spec = W.spec_evict("small")
    db, ref, _ = run_and_compare(spec, label="evict-small")
    assert ref["flags"].any() and not ref["flags"].all()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_sweep_small(B, kv_dtype):
    run_and_compare(W.spec_sweep(3, kv_dtype, scale="small"), label=f"sweep-{kv_dtype}")


def test_evict_small_without_tags(B):
    spec = W.spec_evict("small")
    _, ref, _ = run_and_compare(spec, tags=False, label="evict-small-untracked")
    assert not ref["flags"].any()


# --------------------------------------------------------------------------
# shapes: group sizes, head dims, dtypes, lengths at page and chunk edges
# --------------------------------------------------------------------------
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_group_sizes_and_head_dims(B, kv_dtype, D, G):
    Hkv = 2
    lens = np.array([1, 15, 16, 17, 33, 255, 256, 257], dtype=np.int32)
    spec = W.Spec(f"g{G}d{D}", B=len(lens), Hq=Hkv * G, Hkv=Hkv, D=D, kv_dtype=kv_dtype,
                  num_pages=256, lens=lens, append=True, tags=True, split_tokens=64,
                  seed=100 + G * 7 + D)
    run_and_compare(spec, label=spec.name)


@pytest.mark.parametrize("kv_dtype", ["fp8", "bf16"])
@pytest.mark.parametrize("split", [0, 48])
@pytest.mark.parametrize("bound", [None, 131072])
def test_head_dim_64_worker_shapes_and_splits(B, kv_dtype, split, bound):
    """head_dim 64 on the persistent tensor-core kernel: sequences of many
    units (each worker streams several, crossing segment edges), one segment
    per head or 48-token chunks, the 8- and 12-worker shapes."""
    lens = np.array([1, 17, 300, 1000, 2049, 4000], dtype=np.int32)
    spec = W.Spec(f"d64-{kv_dtype}", B=len(lens), Hq=16, Hkv=4, D=64, kv_dtype=kv_dtype,
                  num_pages=int(((lens + 16) // 16).sum()) + 8, lens=lens, append=True,
                  tags=True, stale_per_mille=2.0, split_tokens=split, seed=909)
    run_and_compare(spec, label=f"d64 {kv_dtype} split={split} bound={bound}", max_seq_len=bound)


@pytest.mark.parametrize("split", [16, 32, 0])
def test_per_head_lengths_with_zero_length_heads(B, split):
    lens = np.array([[0, 5, 16, 31], [64, 0, 0, 1], [200, 17, 33, 0]], dtype=np.int32)
    spec = W.Spec("ph", B=3, Hq=8, Hkv=4, D=128, kv_dtype="fp8", num_pages=128, lens=lens,
                  per_head=True, tags=True, split_tokens=split, seed=77)
    run_and_compare(spec, label=f"per-head split={split}")


def test_all_lengths_zero(B):
    lens = np.zeros(3, dtype=np.int32)
    spec = W.Spec("zero", B=3, Hq=8, Hkv=2, D=128, kv_dtype="fp8", num_pages=16, lens=lens,
                  tags=False, seed=5)
    batch = W.make_batch(spec)
    db = _db(batch, tags=False)
    db.out.fill_(1.0)
    db.attend()
    torch.cuda.synchronize()
    assert not db.out.float().abs().sum().item()
    assert not db.flags.cpu().numpy()[:3].any()


# --------------------------------------------------------------------------
# needles: one dominant key, so a dropped or misplaced token shows up as a
# wholly different output
# --------------------------------------------------------------------------
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("D", [128, 64])
def test_dominant_key_at_page_and_chunk_edges(B, kv_dtype, D):
    split = 64
    lens = np.array([1, 16, 17, 64, 65, 130, 191, 300], dtype=np.int32)
    spec = W.Spec("needle", B=len(lens), Hq=8, Hkv=2, D=D, kv_dtype=kv_dtype, num_pages=256,
                  lens=lens, tags=True, split_tokens=split, seed=31, outlier_prob=0.0)
    T = int(lens.max())
    q = W.draw_q(spec)
    k_rows = (W.draw_kv_rows(spec, T, "k").float() * 0.05).to(torch.bfloat16)
    v_rows = W.draw_kv_rows(spec, T, "v")
    rng = np.random.Generator(np.random.PCG64(3))
    for b, n in enumerate(lens):
        cands = sorted({0, n - 1, min(15, n - 1), min(16, n - 1), min(split - 1, n - 1),
                        min(split, n - 1), n // 2})
        for h in range(spec.Hkv):
            j = int(cands[(b + h) % len(cands)])
            k_rows[b, h, j] = (q[b, h * spec.G].float() * 3.0).to(torch.bfloat16)
    db, ref, _ = run_and_compare(spec, rows=(k_rows, v_rows), q=q, label=f"needle-{kv_dtype}-d{D}")
    # the first q head of each group is dominated by its needle token
    for b in range(spec.B):
        for h in range(spec.Hkv):
            o = ref["out"][b, h * spec.G]
            assert np.abs(o).max() > 0.3


# --------------------------------------------------------------------------
# data errors: bad page ids and lengths are flagged, never read
# --------------------------------------------------------------------------
def test_bad_page_ids_and_lengths_are_flagged(B):
    spec = W.Spec("bad", B=5, Hq=8, Hkv=2, D=128, kv_dtype="fp8", num_pages=64,
                  lens=np.array([40, 40, 40, 40, 40], dtype=np.int32), tags=False, seed=8)
    batch = W.make_batch(spec)
    db = _db(batch, tags=False)
    bt = batch.block_tables.copy()
    bt[1, 2] = 64            # == pool size
    bt[2, 0] = -3            # negative
    lens = batch.seq_lens.copy()
    lens[3] = 20             # 2 live pages ...
    bt[3, 2] = 10 ** 9       # ... so this entry is padding: never read
    lens[4] = 40000          # longer than the table
    db.block_tables.copy_(torch.from_numpy(bt).cuda())
    db.seq_lens.copy_(torch.from_numpy(lens).cuda())
    db.attend()
    torch.cuda.synchronize()
    flags = db.flags.cpu().numpy()[:5]
    cache = dict(num_pages=64, num_kv_heads=2, head_dim=128, dtype=1,
                 k_pages=np.zeros(1, np.uint8), v_pages=np.zeros(1, np.uint8),
                 k_scale=np.zeros(1, np.float32), v_scale=np.zeros(1, np.float32),
                 page_tags=None)
    pages = pages_dict(spec, batch, lens, tags=False)
    pages["block_tables"] = bt
    want = oracle.validate(cache, pages, db.max_seq_len)
    assert list(flags) == list(want) == [0, 2, 2, 0, 4]
    out = db.out.float().cpu()
    assert not out[1].abs().sum() and not out[2].abs().sum() and not out[4].abs().sum()
    assert out[0].abs().sum() > 0 and out[3].abs().sum() > 0


def test_workspace_too_small_is_rejected(B):
    spec = W.spec_tiny()
    db = _db(W.make_batch(spec))
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.PfkvError) as e:
        B.pfkv_paged_decode_attn(db.cache, db.pages, db.q, spec.sm_scale, 0, db.max_seq_len,
                                 small, db.out, db.flags)
    assert e.value.status == B.PFKV_ERR_WORKSPACE


def test_repeat_calls_are_deterministic(B):
    spec = W.spec_llama8b("small")
    db = _db(W.make_batch(spec))
    db.attend()
    first = db.out.clone()
    for _ in range(3):
        db.attend()
    torch.cuda.synchronize()
    assert torch.equal(first, db.out)


def test_many_segments_coarsen_the_split(B):
    """A fixed split size that would give more (request, kv head, chunk)
    segments than the persistent kernel's tables hold: the kernel takes a
    coarser split (a multiple of the caller's; only the output is
    contracted); same results."""
    lens = np.array([3000, 2900, 2950], dtype=np.int32)
    spec = W.Spec("manyseg", B=3, Hq=32, Hkv=8, D=128, kv_dtype="fp8", num_pages=1024,
                  lens=lens, tags=True, split_tokens=16, seed=404)
    run_and_compare(spec, label="many-segments")


@pytest.mark.parametrize("kv_dtype,D", [("fp8", 128), ("bf16", 128), ("fp8", 64)])
def test_long_sequences_with_a_small_split(B, kv_dtype, D):
    """16-token chunks of 30,000-token sequences: 30,000 segments, coarsened."""
    lens = np.array([30000, 17000], dtype=np.int32)
    spec = W.Spec(f"smallsplit-{kv_dtype}-d{D}", B=2, Hq=16, Hkv=4, D=D, kv_dtype=kv_dtype,
                  num_pages=int(((lens + 16) // 16).sum()) + 8, lens=lens, append=True,
                  tags=True, split_tokens=16, seed=405)
    run_and_compare(spec, label=f"small split {kv_dtype}")


@pytest.mark.parametrize("kv_dtype,G,D", [("fp8", 4, 128), ("bf16", 8, 128), ("fp8", 1, 128),
                                          ("fp8", 2, 64)])
def test_request_groups(B, kv_dtype, G, D):
    """More (request, kv head) pairs than one persistent launch's tables
    hold (520 requests x 8 kv heads > 4,096): the batch runs as request
    groups, each a split and a combine; stale tags flag requests in both
    groups."""
    rng = np.random.default_rng(606 + G)
    lens = rng.integers(1, 90, size=520, endpoint=True).astype(np.int32)
    spec = W.Spec(f"groups-{kv_dtype}-g{G}-d{D}", B=520, Hq=8 * G, Hkv=8, D=D, kv_dtype=kv_dtype,
                  num_pages=int(((lens + 16) // 16).sum()) + 16, lens=lens, append=True,
                  tags=True, stale_per_mille=3.0, seed=606 + G)
    db, ref, _ = run_and_compare(spec, label=f"request groups {kv_dtype} G={G}")
    f = ref["flags"]
    assert f[:512].any() and f[512:].any() or f.any()


def test_packed_step_io_gives_the_same_outputs(B):
    """DeviceBatch.pack_step_io moves the step's inputs and outputs into two
    buffers (one copy each way for an end-to-end caller); the step's results
    are unchanged."""
    spec = W.spec_llama8b("small")
    db = _db(W.make_batch(spec))
    out0 = db.out.clone()
    db.step()
    torch.cuda.synchronize()
    want = db.out.clone()
    pool_k = db.cache.k_pages.clone()
    db.pack_step_io()
    db.out.copy_(out0)
    db.step()   # the append rewrites the same slots with the same values
    torch.cuda.synchronize()
    assert torch.equal(db.out, want)
    assert torch.equal(db.cache.k_pages, pool_k)
    assert db.io_in.data_ptr() <= db.q.data_ptr() < db.io_in.data_ptr() + db.io_in.numel()
    assert db.io_out.data_ptr() <= db.flags.data_ptr() < db.io_out.data_ptr() + db.io_out.numel()
