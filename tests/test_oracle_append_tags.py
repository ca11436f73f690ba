"""Pins of the oracle's kv_append (FP8 quantisation into page slots) and of its
integrity/bounds check (CPU only).

Quantisation pins: numpy's IEEE fp32 division for the scale, the format fact
that the absmax element lands on the largest code, exact codes for values that
are representable at a power-of-two scale, the half-spacing error bound, the
saturating reuse of a stored scale, and an exact bf16 copy.  Tag pins: brute
force over Python sets of the stale units.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle_cases import cache_dict, empty_pool, pages_dict
from paged_fp8_kv_decode_gb300 import workloads as W


def _one_unit_setup(kv_dtype="fp8", D=64, H=2, NP=8, tags=False):
    spec = W.Spec("u", B=1, Hq=H, Hkv=H, D=D, kv_dtype=kv_dtype, num_pages=NP,
                  lens=np.array([16], dtype=np.int32), tags=tags, seed=3)
    batch = W.make_batch(spec)
    k, v, ks, vs = empty_pool(spec)
    cache = cache_dict(spec, batch, k, v, ks, vs, tags=tags)
    pages = pages_dict(spec, batch, batch.seq_lens, tags=tags)
    return spec, batch, cache, pages


def _bits(x):
    return W.bf16_bits(torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16))


def test_full_unit_scale_is_absmax_over_448_and_absmax_hits_max_code(oracle):
    spec, batch, cache, pages = _one_unit_setup()
    kr = W.draw_bf16((1, 2, 16, 64), 7, 0.01)
    vr = W.draw_bf16((1, 2, 16, 64), 8, 0.01)
    oracle.kv_append(cache, pages, np.zeros(1, np.int32), W.bf16_bits(kr), W.bf16_bits(vr))
    for h in range(2):
        phys = int(batch.block_tables[0, 0])
        for rows, pool, sc in ((kr, cache["k_pages"], cache["k_scale"]),
                               (vr, cache["v_pages"], cache["v_scale"])):
            x = rows[0, h].float().numpy()
            amax = np.float32(np.abs(x).max())
            assert sc[phys, h] == np.float32(amax / np.float32(448.0))  # numpy IEEE fp32 div
            idx = np.unravel_index(np.abs(x).argmax(), x.shape)
            code = pool[phys, h][idx]
            assert code == (0xFE if x[idx] < 0 else 0x7E)


def test_power_of_two_scale_gives_exact_codes(oracle):
    """With absmax = 448 * 2^k the scale is 2^k and x = value(c) * 2^k must
    encode to c exactly."""
    spec, batch, cache, pages = _one_unit_setup(D=64)
    rng = np.random.Generator(np.random.PCG64(4))
    codes = rng.integers(0, 256, size=(1, 2, 16, 64)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x11
    # bf16 can hold values with at most 8 significant bits: e4m3 values qualify
    codes[..., 0] = 0x7E
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float32) * 0.25
    kb = W.bf16_bits(vals.to(torch.bfloat16))
    oracle.kv_append(cache, pages, np.zeros(1, np.int32), kb, kb)
    phys = int(batch.block_tables[0, 0])
    for h in range(2):
        assert cache["k_scale"][phys, h] == np.float32(0.25)
        got = cache["k_pages"][phys, h]
        want = codes[0, h].copy()
        want[want == 0x80] = 0x80  # -0 keeps its sign
        assert np.array_equal(got, want)


def test_dequant_error_within_half_spacing(oracle):
    spec, batch, cache, pages = _one_unit_setup(D=128)
    kr = W.draw_bf16((1, 2, 16, 128), 17, 0.01)
    oracle.kv_append(cache, pages, np.zeros(1, np.int32), W.bf16_bits(kr), W.bf16_bits(kr))
    phys = int(batch.block_tables[0, 0])
    for h in range(2):
        s = float(cache["k_scale"][phys, h])
        deq = torch.from_numpy(cache["k_pages"][phys, h].copy()).view(torch.float8_e4m3fn)
        deq = deq.to(torch.float64).numpy() * s
        x = kr[0, h].double().numpy()
        y = x / s
        e = np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -6)))
        half = np.where(np.abs(y) < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))
        # division rounding adds at most one fp32 ulp of y
        assert np.all(np.abs(deq / s - y) <= half + np.abs(y) * 2.0 ** -23 + 1e-30)


def test_append_reuses_stored_scale_and_saturates(oracle):
    spec, batch, cache, pages = _one_unit_setup(D=64)
    phys = int(batch.block_tables[0, 0])
    first = np.full((1, 2, 1, 64), 1.0, dtype=np.float32)
    oracle.kv_append(cache, pages, np.zeros(1, np.int32), _bits(first), _bits(first))
    assert cache["k_scale"][phys, 0] == np.float32(1.0 / 448.0)
    assert np.all(cache["k_pages"][phys, :, 0] == 0x7E)
    second = np.full((1, 2, 1, 64), 0.5, dtype=np.float32)
    second[..., 1] = 3.0    # beyond the stored scale's range -> saturates
    second[..., 2] = -3.0
    oracle.kv_append(cache, pages, np.ones(1, np.int32), _bits(second), _bits(second))
    assert cache["k_scale"][phys, 0] == np.float32(1.0 / 448.0)   # unchanged
    row = cache["k_pages"][phys, 0, 1]
    assert row[0] == 0x76       # 0.5 * 448 = 224 = 2^7 * 1.75 -> e=14, m=6
    assert row[1] == 0x7E and row[2] == 0xFE


def test_zero_unit_gets_scale_one(oracle):
    spec, batch, cache, pages = _one_unit_setup(D=64)
    z = np.zeros((1, 2, 1, 64), dtype=np.float32)
    oracle.kv_append(cache, pages, np.zeros(1, np.int32), _bits(z), _bits(z))
    phys = int(batch.block_tables[0, 0])
    assert np.all(cache["k_scale"][phys] == 1.0) and np.all(cache["v_scale"][phys] == 1.0)
    assert not cache["k_pages"][phys, :, 0].any()


def test_bf16_append_is_exact_copy(oracle):
    spec, batch, cache, pages = _one_unit_setup(kv_dtype="bf16", D=64)
    kr = W.draw_bf16((1, 2, 5, 64), 21, 0.01)
    oracle.kv_append(cache, pages, np.full(1, 9, np.int32), W.bf16_bits(kr), W.bf16_bits(kr))
    phys0, phys1 = int(batch.block_tables[0, 0]), -1
    assert np.array_equal(cache["k_pages"][phys0, :, 9:14], W.bf16_bits(kr)[0])


def test_append_checks_destination(oracle):
    """Tag mismatch, out-of-range page id and a position past the table each
    skip the write and set their flag bit."""
    spec = W.Spec("c", B=3, Hq=2, Hkv=2, D=64, kv_dtype="fp8", num_pages=8,
                  lens=np.array([16, 16, 16], dtype=np.int32), tags=True, seed=9)
    batch = W.make_batch(spec)
    k, v, ks, vs = empty_pool(spec)
    cache = cache_dict(spec, batch, k, v, ks, vs)
    cache["page_tags"] = batch.page_tags.copy()
    bt = batch.block_tables.copy()
    cache["page_tags"][bt[0, 0], 1] ^= np.uint32(5)       # request 0: stale tag on head 1
    bt[1, 0] = 8                                           # request 1: page id == pool size
    pages = pages_dict(spec, batch, batch.seq_lens)
    pages["block_tables"] = bt
    pos = np.array([3, 3, 16], dtype=np.int32)             # request 2: past its 1-page table
    kr = W.draw_bf16((3, 2, 1, 64), 1)
    before = cache["k_pages"].copy()
    flags = oracle.kv_append(cache, pages, pos, W.bf16_bits(kr), W.bf16_bits(kr))
    assert list(flags) == [oracle.FLAG_TAG, oracle.FLAG_PAGE, oracle.FLAG_LEN]
    changed = np.argwhere((cache["k_pages"] != before).any(axis=(2, 3)))
    # only request 0, head 0 was written
    assert [tuple(x) for x in changed] == [(bt[0, 0], 0)]


# --------------------------------------------------------------------------
# integrity tags: brute force over sets
# --------------------------------------------------------------------------
@pytest.mark.parametrize("per_mille", [1.0, 20.0])
def test_validate_flags_requests_touching_stale_units(oracle, per_mille):
    spec = W.spec_evict("small")
    spec.stale_per_mille = per_mille
    batch = W.make_batch(spec)
    k, v, ks, vs = empty_pool(spec)
    cache = cache_dict(spec, batch, k, v, ks, vs)
    pages = pages_dict(spec, batch, batch.seq_lens)
    flags = oracle.validate(cache, pages, 1 << 30)
    stale = {(int(p), int(h)) for p, h in batch.stale_units}
    assert len(stale) == round(batch.live_units * per_mille / 1000)
    lens = batch.lens_bh()
    want = []
    for b in range(spec.B):
        touched = set()
        for h in range(spec.Hkv):
            live = -(-int(lens[b, h]) // 16)
            touched |= {(int(batch.block_tables[b, h, p]), h) for p in range(live)}
        want.append(oracle.FLAG_TAG if touched & stale else 0)
    assert list(flags) == want
    assert any(want)
    if per_mille == 1.0:
        assert not all(want)      # both flagged and clean requests occur


def test_validate_bounds_and_padding(oracle):
    spec = W.spec_evict("small")
    spec.stale_per_mille = 0.0
    batch = W.make_batch(spec)
    k, v, ks, vs = empty_pool(spec)
    cache = cache_dict(spec, batch, k, v, ks, vs)
    lens = batch.seq_lens.copy()
    bt = batch.block_tables.copy()
    ex = batch.expected_tags.copy()
    # padding entries past each live length hold garbage: never read
    for b in range(spec.B):
        for h in range(spec.Hkv):
            live = -(-int(lens[b, h]) // 16)
            bt[b, h, live:] = -77
            ex[b, h, live:] = 0xDEAD
    lens[1, 2] = batch.max_pages * 16 + 1        # longer than the table -> LEN
    bt[2, 5, 0] = -1                             # negative page id -> PAGE
    bt[3, 0, 0] = spec.num_pages                 # page id == pool size -> PAGE
    pages = pages_dict(spec, batch, lens)
    pages.update(block_tables=bt, expected_tags=ex)
    flags = oracle.validate(cache, pages, 1 << 30)
    assert flags[0] == 0 and flags[4] == 0 and flags[5] == 0
    assert flags[1] == oracle.FLAG_LEN
    assert flags[2] == oracle.FLAG_PAGE and flags[3] == oracle.FLAG_PAGE
    # a length above the caller's max_seq_len bound is also LEN
    flags2 = oracle.validate(cache, pages_dict(spec, batch, batch.seq_lens), 10)
    assert all(f == oracle.FLAG_LEN for f in flags2)


def test_no_tags_means_no_tag_check(oracle):
    spec = W.spec_evict("small")
    spec.stale_per_mille = 50.0
    batch = W.make_batch(spec)
    k, v, ks, vs = empty_pool(spec)
    cache = cache_dict(spec, batch, k, v, ks, vs, tags=False)
    pages = pages_dict(spec, batch, batch.seq_lens, tags=False)
    assert not oracle.validate(cache, pages, 1 << 30).any()


def test_validate_checks_last_partial_page(oracle):
    """A stale tag on the last, partially filled page of a row is caught; one on
    the first padding entry after it is not."""
    spec = W.spec_evict("small")
    spec.stale_per_mille = 0.0
    batch = W.make_batch(spec)
    k, v, ks, vs = empty_pool(spec)
    cache = cache_dict(spec, batch, k, v, ks, vs)
    lens = batch.lens_bh()
    b, h = next((b, h) for b in range(spec.B) for h in range(spec.Hkv)
                if lens[b, h] % 16 != 0 and lens[b, h] > 16)
    last = -(-int(lens[b, h]) // 16) - 1
    ex = batch.expected_tags.copy()
    ex[b, h, last] ^= np.uint32(1)
    pages = pages_dict(spec, batch, batch.seq_lens)
    pages["expected_tags"] = ex
    flags = oracle.validate(cache, pages, 1 << 30)
    assert [int(f) for f in flags] == [oracle.FLAG_TAG if i == b else 0 for i in range(spec.B)]
    ex2 = batch.expected_tags.copy()
    bt2 = batch.block_tables.copy()
    if last + 1 < batch.max_pages:
        bt2[b, h, last + 1] = -5
        ex2[b, h, last + 1] = 7
    pages.update(expected_tags=ex2, block_tables=bt2)
    assert not oracle.validate(cache, pages, 1 << 30).any()
