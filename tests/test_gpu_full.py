"""GPU path vs the oracle at the workloads' full sizes, in the launch
configuration the benchmark times (automatic split unless the workload fixes
one), on sampled (request, kv head) pairs.

For each sampled pair the oracle rebuilds that head alone: it quantises the
head's bf16 rows (the same rows the GPU filled from) into a compact pool of its
own, appends the step's token, and attends with the G query heads of the
group.  The GPU's bytes and scales of the head's units must equal the
oracle's bit for bit, and its outputs must be within the contract tolerance.
Request flags are checked for the whole batch against the oracle's
tag/bounds check.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle_cases import assert_outputs_close, cache_dict, fill_pool, pages_dict
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


def _head_batch(spec, batch, b, h):
    """A one-request, one-kv-head batch holding head (b, h) on pages 0..k-1."""
    fill = int(batch.lens_bh("fill")[b, h])
    seq = int(batch.lens_bh("seq")[b, h])
    npages = max(1, -(-seq // 16))
    mini = W.Spec(f"{spec.name}-b{b}h{h}", B=1, Hq=spec.G, Hkv=1, D=spec.D,
                  kv_dtype=spec.kv_dtype, num_pages=npages, lens=np.array([fill], np.int32),
                  append=spec.append, tags=False, seed=spec.seed)
    mb = W.Batch(spec=mini, seq_lens=np.array([seq], np.int32),
                 fill_lens=np.array([fill], np.int32), positions=np.array([fill], np.int32),
                 len_strides=(1, 0), block_tables=np.arange(npages, dtype=np.int32)[None],
                 bt_strides=(npages, 0), max_pages=npages,
                 page_tags=np.zeros((npages, 1), np.uint32),
                 expected_tags=np.zeros((1, npages), np.uint32),
                 stale_units=np.zeros((0, 2), np.int64), live_units=npages)
    return mini, mb


def _check_head(db, b, h, flagged):
    spec, batch = db.spec, db.batch
    G, D = spec.G, spec.D
    gpu_out = db.out[b, h * G:(h + 1) * G].float().cpu().numpy().astype(np.float64)
    if flagged:
        assert not gpu_out.any()
        return
    mini, mb = _head_batch(spec, batch, b, h)
    fill = int(mb.fill_lens[0])
    kb = W.bf16_bits(db.k_rows[b:b + 1, h:h + 1, :fill].contiguous())
    vb = W.bf16_bits(db.v_rows[b:b + 1, h:h + 1, :fill].contiguous())
    k, v, ks, vs = fill_pool(mini, mb, kb, vb)
    cache = cache_dict(mini, mb, k, v, ks, vs, tags=False)
    pages = pages_dict(mini, mb, mb.seq_lens, tags=False)
    if spec.append:
        oracle.kv_append(cache, pages, mb.positions, W.bf16_bits(db.k_new[b:b + 1, h:h + 1]),
                         W.bf16_bits(db.v_new[b:b + 1, h:h + 1]))
    # the GPU's units of this head, in logical order
    npages = mb.max_pages
    phys = torch.from_numpy(batch.table_row(b, h)[:npages].astype(np.int64)).cuda()
    gk = db.cache.k_pages[phys, h]
    gv = db.cache.v_pages[phys, h]
    if spec.kv_dtype == "bf16":
        gk, gv = gk.view(torch.int16), gv.view(torch.int16)
    gk = gk.cpu().numpy().view(k.dtype)
    gv = gv.cpu().numpy().view(v.dtype)
    seq = int(mb.seq_lens[0])
    live = np.zeros((npages, 16), bool)
    live.reshape(-1)[:seq] = True
    assert np.array_equal(gk[live], k[:, 0][live]), (b, h)
    assert np.array_equal(gv[live], v[:, 0][live]), (b, h)
    if spec.kv_dtype == "fp8":
        assert np.array_equal(db.cache.k_scale[phys, h].cpu().numpy(), ks[:, 0]), (b, h)
        assert np.array_equal(db.cache.v_scale[phys, h].cpu().numpy(), vs[:, 0]), (b, h)
    q = W.bf16_bits(db.q[b:b + 1, h * G:(h + 1) * G].contiguous())
    ref, flags = oracle.paged_decode(cache, pages, q, G, spec.sm_scale, seq)
    assert not flags.any()
    assert_outputs_close(db.out[b:b + 1, h * G:(h + 1) * G], ref, (b, h))


def _flags_ref(db):
    spec, batch = db.spec, db.batch
    dummy8 = np.zeros(1, np.uint8)
    cache = dict(num_pages=spec.num_pages, num_kv_heads=spec.Hkv, head_dim=spec.D, dtype=1,
                 k_pages=dummy8, v_pages=dummy8, k_scale=np.zeros(1, np.float32),
                 v_scale=np.zeros(1, np.float32),
                 page_tags=batch.page_tags if db.cache.page_tags is not None else None)
    pages = pages_dict(spec, batch, batch.seq_lens, tags=db.cache.page_tags is not None)
    return oracle.validate(cache, pages, db.max_seq_len)


def _run(spec, samples, B, **kw):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    db = DeviceBatch(W.make_batch(spec), keep_rows=True, **kw)
    return _check_run(db, samples)


def _check_run(db, samples):
    spec = db.spec
    db.step()
    torch.cuda.synchronize()
    flags = db.flags.cpu().numpy()[:spec.B]
    want = _flags_ref(db)
    assert np.array_equal(flags, want), (flags, want)
    assert not db.append_flags.cpu().numpy()[:spec.B].any()
    for b, h in samples:
        _check_head(db, b, h, bool(want[b]))
    return db, want


def test_llama8b_full(B):
    spec = W.spec_llama8b("full")
    lens = spec.lens
    order = np.argsort(lens)
    samples = [(int(order[0]), 0), (int(order[-1]), 7), (int(order[len(order) // 2]), 3),
               (5, 5), (17, 2), (31, 6)]
    _run(spec, samples, B)


def test_long_context_full_split_4096(B):
    spec = W.spec_long("full")
    _run(spec, [(0, 0), (3, 7)], B)


def test_evict_full_stale_tags_and_per_head_lengths(B):
    spec = W.spec_evict("full")
    db, want = _run(spec, [], B)
    lens = db.batch.lens_bh()
    flagged = [b for b in range(spec.B) if want[b]]
    clean = [b for b in range(spec.B) if not want[b]]
    assert flagged, "the stale tags must flag some request"
    samples = [(flagged[0], 0)]
    for b in clean[:3]:
        samples.append((b, int(np.argmin(lens[b]))))    # the most-evicted head
        samples.append((b, int(np.argmax(lens[b]))))
    for b, h in samples:
        _check_head(db, b, h, bool(want[b]))


def test_evict_full_stale_tags_fused_check(B):
    """The tag check inside the attention kernel: same flags, sampled heads
    against the oracle."""
    spec = W.spec_evict("full")
    db, want = _run(spec, [], B, fused_tags=True)
    lens = db.batch.lens_bh()
    clean = [b for b in range(spec.B) if not want[b]]
    flagged = [b for b in range(spec.B) if want[b]]
    for b in clean[:2] + flagged[:1]:
        _check_head(db, b, int(np.argmin(lens[b])), bool(want[b]))
        _check_head(db, b, int(np.argmax(lens[b])), bool(want[b]))


def test_evict_full_without_tags(B):
    spec = W.spec_evict("full")
    db, want = _run(spec, [], B, tags=False)
    assert not want.any()
    lens = db.batch.lens_bh()
    for b in (0, 7, 15):
        _check_head(db, b, int(np.argmin(lens[b])), False)
        _check_head(db, b, int(np.argmax(lens[b])), False)


@pytest.mark.parametrize("batch,kv_dtype", [(64, "fp8"), (8, "bf16"), (32, "bf16"), (1, "fp8")])
def test_sweep_points_on_an_80_gb_pool(B, batch, kv_dtype):
    spec = W.spec_sweep(batch, kv_dtype)
    samples = [(0, 0), (batch - 1, 7)]
    db, _ = _run(spec, samples, B)
    del db
    torch.cuda.empty_cache()
