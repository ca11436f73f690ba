"""Pins of the oracle's attention mass (CPU only).

The mass of token j of kv head h is the sum over the G query heads reading h
of token j's softmax weight ("Workers AI targets the inference bottleneck",
section "KV cache compression goes open source", 3rd paragraph: eviction keeps
the attention each entry received).  Pins from outside the oracle: the closed
forms (weights of a head sum to one, so a head's masses sum to G; uniform keys
give G/n each; one token gets G; a dominant key takes almost all of it),
brute force against torch's fp64 softmax on the dense gather, accumulation
across calls, and no contribution from flagged requests or empty heads."""
import numpy as np
import pytest
import torch

import oracle
from oracle_cases import cache_dict, fill_pool, pages_dict
from paged_fp8_kv_decode_gb300 import workloads as W
from test_oracle_attention import _dense_kv, _setup, _small_spec


def _mass(spec, batch, cache, pages, q, mass=None):
    return oracle.attention_mass(cache, pages, q, spec.Hq, spec.sm_scale,
                                 int(batch.seq_lens.max()), mass=mass)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_masses_of_a_head_sum_to_the_group_size(kv_dtype):
    spec = _small_spec(kv_dtype, [37, 100, 1, 16], Hq=8, Hkv=2)
    batch, cache, pages, q, *_ = _setup(spec)
    m = _mass(spec, batch, cache, pages, q)
    lens = batch.lens_bh("seq")
    for b in range(spec.B):
        for h in range(spec.Hkv):
            n = int(lens[b, h])
            assert abs(m[b, h, :n].sum() - spec.G) < 1e-12
            assert (m[b, h, :n] > 0).all() and not m[b, h, n:].any()


def test_brute_force_against_dense_softmax():
    spec = _small_spec("fp8", [53, 20, 77], Hq=4, Hkv=2)
    batch, cache, pages, q, _, _, qt = _setup(spec)
    m = _mass(spec, batch, cache, pages, q)
    K = _dense_kv(spec, batch, cache, "k")
    lens = batch.lens_bh("seq")
    for b in range(spec.B):
        for h in range(spec.Hkv):
            n = int(lens[b, h])
            qs = qt[b, h * spec.G:(h + 1) * spec.G].to(torch.float64)           # [G][D]
            w = torch.softmax(spec.sm_scale * qs @ K[b][h][:n].T, dim=-1)       # [G][n]
            np.testing.assert_allclose(m[b, h, :n], w.sum(0).numpy(), rtol=1e-12, atol=1e-15)


def test_uniform_keys_give_equal_mass():
    spec = _small_spec("bf16", [40, 9], Hq=4, Hkv=2)
    T = 40
    k = torch.ones((spec.B, spec.Hkv, T, spec.D), dtype=torch.float32).to(torch.bfloat16)
    batch, cache, pages, q, *_ = _setup(spec, k_rows=k)
    m = _mass(spec, batch, cache, pages, q)
    for b, n in enumerate([40, 9]):
        np.testing.assert_allclose(m[b, :, :n], spec.G / n, rtol=1e-12)


def test_one_token_and_a_dominant_key():
    spec = _small_spec("bf16", [1, 30], Hq=2, Hkv=1, D=64)
    T = 30
    k = torch.zeros((spec.B, 1, T, spec.D), dtype=torch.float32)
    qv = torch.zeros((spec.B, spec.Hq, spec.D), dtype=torch.float32)
    qv[1, :, 0] = 8.0
    k[1, 0, 17, 0] = 8.0        # score 8 * 8 / sqrt(64) = 8 for token 17, 0 for the rest
    batch, cache, pages, q, *_ = _setup(spec, k_rows=k.to(torch.bfloat16),
                                        q=qv.to(torch.bfloat16))
    m = _mass(spec, batch, cache, pages, q)
    assert m[0, 0, 0] == pytest.approx(2.0, abs=1e-15)
    w = np.exp(8.0) / (np.exp(8.0) + 29.0)
    assert m[1, 0, 17] == pytest.approx(2 * w, rel=1e-12)
    assert m[1, 0, 3] == pytest.approx(2 * (1 - w) / 29, rel=1e-12)


def test_calls_accumulate_and_skip_flagged_requests():
    spec = _small_spec("fp8", [33, 60, 12], Hq=4, Hkv=2)
    batch, cache, pages, q, *_ = _setup(spec)
    one = _mass(spec, batch, cache, pages, q)
    two = _mass(spec, batch, cache, pages, q, mass=one.copy())
    np.testing.assert_allclose(two, 2 * one, rtol=1e-15)
    # a stale tag on request 1: its heads receive nothing
    tags = cache["page_tags"].copy()
    tags[int(batch.table_row(1, 0)[0]), :] ^= 5
    cache2 = dict(cache, page_tags=tags)
    m = _mass(spec, batch, cache2, pages, q)
    assert not m[1].any()
    np.testing.assert_allclose(m[0], one[0], rtol=0)
    np.testing.assert_allclose(m[2], one[2], rtol=0)


def test_zero_length_heads_receive_nothing():
    lens = np.array([[0, 25], [19, 0]], dtype=np.int32)
    spec = _small_spec("bf16", lens, Hq=4, Hkv=2, per_head=True)
    batch, cache, pages, q, *_ = _setup(spec)
    m = _mass(spec, batch, cache, pages, q)
    assert not m[0, 0].any() and not m[1, 1].any()
    assert abs(m[0, 1, :25].sum() - 2) < 1e-12 and abs(m[1, 0, :19].sum() - 2) < 1e-12
