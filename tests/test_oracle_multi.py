"""Pins of the oracle's multi-query verify (CPU only).

The kq candidate tokens of a request are its last kq tokens; query token i
attends to the first n - kq + 1 + i tokens ("Workers AI targets the inference
bottleneck", section "Speculative decoding: predicting more than one token":
all candidates are verified in one pass).  Pins from outside the oracle:
fp64 brute force against torch's scaled_dot_product_attention with an explicit
causal mask over the dense gather, the closed form of uniform keys (mean of
the visible values), kq = 1 being plain decode, and the empty and flagged
cases."""
import numpy as np
import pytest
import torch

import oracle
from paged_fp8_kv_decode_gb300 import workloads as W
from test_oracle_attention import _dense_kv, _setup, _small_spec


def _q_multi(spec, kq, seed=3):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((spec.B, kq, spec.Hq, spec.D), generator=g).to(torch.bfloat16)
    return q, W.bf16_bits(q)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("kq", [1, 3, 5])
def test_brute_force_with_causal_mask(kv_dtype, kq):
    spec = _small_spec(kv_dtype, [40, 7, 66], Hq=4, Hkv=2)
    batch, cache, pages, *_ = _setup(spec)
    qt, qb = _q_multi(spec, kq)
    out, flags = oracle.paged_decode_multi(cache, pages, qb, spec.Hq, kq, spec.sm_scale,
                                           int(batch.seq_lens.max()))
    assert not flags.any()
    K = _dense_kv(spec, batch, cache, "k")
    V = _dense_kv(spec, batch, cache, "v")
    lens = batch.lens_bh("seq")
    for b in range(spec.B):
        for h in range(spec.Hkv):
            n = int(lens[b, h])
            qs = qt[b, :, h * spec.G:(h + 1) * spec.G].to(torch.float64).transpose(0, 1)  # [G][kq][D]
            # query i sees keys j <= n - kq + i
            keep = torch.arange(n)[None, :] <= (n - kq + torch.arange(kq))[:, None]      # [kq][n]
            if n >= kq:
                ref = torch.nn.functional.scaled_dot_product_attention(
                    qs, K[b][h][:n][None].expand(spec.G, -1, -1),
                    V[b][h][:n][None].expand(spec.G, -1, -1), attn_mask=keep,
                    scale=spec.sm_scale)                                              # [G][kq][D]
                got = torch.from_numpy(out[b, :, h * spec.G:(h + 1) * spec.G]).transpose(0, 1)
                np.testing.assert_allclose(got.numpy(), ref.numpy(), rtol=1e-9, atol=1e-12)
            else:
                for i in range(kq):
                    if n - kq + 1 + i <= 0:
                        assert not out[b, i, h * spec.G:(h + 1) * spec.G].any()


def test_one_query_token_is_plain_decode():
    spec = _small_spec("fp8", [53, 20], Hq=4, Hkv=2)
    batch, cache, pages, q, *_ = _setup(spec)
    multi, _ = oracle.paged_decode_multi(cache, pages, q[:, None].copy(), spec.Hq, 1,
                                         spec.sm_scale, int(batch.seq_lens.max()))
    plain, _ = oracle.paged_decode(cache, pages, q, spec.Hq, spec.sm_scale,
                                   int(batch.seq_lens.max()))
    np.testing.assert_array_equal(multi[:, 0], plain)


def test_uniform_keys_average_the_visible_prefix():
    spec = _small_spec("bf16", [30], Hq=2, Hkv=1)
    k = torch.ones((1, 1, 30, spec.D)).to(torch.bfloat16)
    batch, cache, pages, *_, v_rows, _ = _setup(spec, k_rows=k)
    kq = 4
    _, qb = _q_multi(spec, kq)
    out, _ = oracle.paged_decode_multi(cache, pages, qb, spec.Hq, kq, spec.sm_scale, 30)
    v = v_rows.to(torch.float64)[0, 0]
    for i in range(kq):
        want = v[:30 - kq + 1 + i].mean(0).numpy()
        for hq in range(spec.Hq):
            np.testing.assert_allclose(out[0, i, hq], want, rtol=1e-12, atol=1e-14)


def test_short_heads_and_flagged_requests_give_zero_rows():
    lens = np.array([[2, 30], [25, 1]], dtype=np.int32)
    spec = _small_spec("bf16", lens, Hq=4, Hkv=2, per_head=True)
    batch, cache, pages, *_ = _setup(spec)
    kq = 3
    _, qb = _q_multi(spec, kq)
    out, flags = oracle.paged_decode_multi(cache, pages, qb, spec.Hq, kq, spec.sm_scale, 30)
    assert not out[0, 0, 0:2].any()          # head 0 of request 0: n = 2, query 0 sees nothing
    assert out[0, 1, 0:2].any() and out[0, 2, 0:2].any()
    assert not out[1, 0, 2:4].any() and not out[1, 1, 2:4].any() and out[1, 2, 2:4].any()
    tags = cache["page_tags"].copy()
    tags[int(batch.table_row(1, 0)[0]), 0] ^= 1
    out2, flags2 = oracle.paged_decode_multi(dict(cache, page_tags=tags), pages, qb, spec.Hq, kq,
                                             spec.sm_scale, 30)
    assert flags2[1] == 1 and not out2[1].any()
    np.testing.assert_array_equal(out2[0], out[0])
