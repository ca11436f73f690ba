"""Pins of the oracle's paged decode attention (CPU only).

Each pin reaches the oracle from outside: a closed form (uniform keys give the
mean of V; one token gives that token's V; a dominant key gives its V), an
invariant (physical page placement, per-head tables that all agree), and brute
force against torch's fp64 scaled_dot_product_attention on the dense gather.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle_cases import cache_dict, empty_pool, fill_pool, pages_dict
from paged_fp8_kv_decode_gb300 import workloads as W


def _small_spec(kv_dtype, lens, Hq=4, Hkv=2, D=64, per_head=False, NP=64, seed=5):
    lens = np.asarray(lens, dtype=np.int32)
    return W.Spec("t", B=lens.shape[0], Hq=Hq, Hkv=Hkv, D=D, kv_dtype=kv_dtype, num_pages=NP,
                  lens=lens, per_head=per_head, tags=True, seed=seed)


def _setup(spec, k_rows=None, v_rows=None, q=None):
    batch = W.make_batch(spec)
    T = int(batch.fill_lens.max())
    if k_rows is None:
        k_rows = W.draw_kv_rows(spec, T, "k")
    if v_rows is None:
        v_rows = W.draw_kv_rows(spec, T, "v")
    if q is None:
        q = W.draw_q(spec)
    kb, vb = W.bf16_bits(k_rows), W.bf16_bits(v_rows)
    k, v, ks, vs = fill_pool(spec, batch, kb, vb)
    cache = cache_dict(spec, batch, k, v, ks, vs)
    pages = pages_dict(spec, batch, batch.seq_lens)
    return batch, cache, pages, W.bf16_bits(q), k_rows, v_rows, q


def _dense_kv(spec, batch, cache, which):
    """Dequantised K or V gathered to dense [B][Hkv][n][D] (fp64) through the
    block table, using torch's float8 decode (a library routine)."""
    pool = cache["k_pages"] if which == "k" else cache["v_pages"]
    scale = cache["k_scale"] if which == "k" else cache["v_scale"]
    lens = batch.lens_bh("seq")
    out = []
    for b in range(spec.B):
        row = []
        for h in range(spec.Hkv):
            n = int(lens[b, h])
            tbl = batch.table_row(b, h)
            toks = []
            for j in range(n):
                u = (int(tbl[j // 16]), h)
                raw = pool[u[0], u[1], j % 16]
                if spec.kv_dtype == "bf16":
                    val = torch.from_numpy(raw.view(np.int16).copy()).view(torch.bfloat16)
                    val = val.to(torch.float64)
                else:
                    val = torch.from_numpy(raw.copy()).view(torch.float8_e4m3fn)
                    val = val.to(torch.float64) * float(scale[u])
                toks.append(val)
            row.append(torch.stack(toks) if toks else torch.zeros(0, spec.D, dtype=torch.float64))
        out.append(row)
    return out


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_matches_dense_sdpa_bruteforce(oracle, kv_dtype):
    spec = _small_spec(kv_dtype, [37, 100, 1, 16, 17])
    batch, cache, pages, qb, _, _, q = _setup(spec)
    out, flags = oracle.paged_decode(cache, pages, qb, spec.Hq, spec.sm_scale, 200)
    assert not flags.any()
    K = _dense_kv(spec, batch, cache, "k")
    V = _dense_kv(spec, batch, cache, "v")
    qd = q.to(torch.float64)
    for b in range(spec.B):
        for hq in range(spec.Hq):
            h = hq // spec.G          # consecutive GQA grouping
            ref = torch.nn.functional.scaled_dot_product_attention(
                qd[b, hq][None, None, None, :], K[b][h][None, None], V[b][h][None, None],
                scale=spec.sm_scale)[0, 0, 0].numpy()
            np.testing.assert_allclose(out[b, hq], ref, rtol=1e-12, atol=1e-12)


def test_gqa_bruteforce_with_library_gqa(oracle):
    """torch's enable_gqa maps query head hq to kv head hq // G, like the oracle."""
    spec = _small_spec("fp8", [50, 33], Hq=8, Hkv=2)
    batch, cache, pages, qb, _, _, q = _setup(spec)
    out, _ = oracle.paged_decode(cache, pages, qb, spec.Hq, spec.sm_scale, 64)
    K = _dense_kv(spec, batch, cache, "k")
    V = _dense_kv(spec, batch, cache, "v")
    for b in range(spec.B):
        kk = torch.stack([K[b][h] for h in range(spec.Hkv)])[None]
        vv = torch.stack([V[b][h] for h in range(spec.Hkv)])[None]
        qq = q[b].to(torch.float64)[None, :, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, kk, vv, scale=spec.sm_scale, enable_gqa=True)[0, :, 0].numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_uniform_keys_give_mean_of_values(oracle, kv_dtype):
    spec = _small_spec(kv_dtype, [45, 80])
    T = 80
    krow = W.draw_bf16((1, 1, 1, spec.D), 99)
    k_rows = krow.expand(spec.B, spec.Hkv, T, spec.D).contiguous()
    batch, cache, pages, qb, _, v_rows, _ = _setup(spec, k_rows=k_rows)
    out, _ = oracle.paged_decode(cache, pages, qb, spec.Hq, spec.sm_scale, 128)
    V = _dense_kv(spec, batch, cache, "v")
    for b in range(spec.B):
        for hq in range(spec.Hq):
            mean = V[b][hq // spec.G].mean(dim=0).numpy()
            np.testing.assert_allclose(out[b, hq], mean, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_single_token_gives_its_value(oracle, kv_dtype):
    spec = _small_spec(kv_dtype, [1, 1, 1])
    batch, cache, pages, qb, _, _, _ = _setup(spec)
    out, _ = oracle.paged_decode(cache, pages, qb, spec.Hq, spec.sm_scale, 1)
    V = _dense_kv(spec, batch, cache, "v")
    for b in range(spec.B):
        for hq in range(spec.Hq):
            assert np.array_equal(out[b, hq], V[b][hq // spec.G][0].numpy())


def test_dominant_key_gives_its_value(oracle):
    """A key aligned with q and far larger than the rest takes all the weight."""
    spec = _small_spec("bf16", [70])
    T, star = 70, 53
    q = W.draw_q(spec)
    k_rows = W.draw_kv_rows(spec, T, "k") * 0.01
    for h in range(spec.Hkv):
        k_rows[0, h, star] = (q[0, h * spec.G].float() * 200).to(torch.bfloat16)
    batch, cache, pages, qb, _, _, _ = _setup(spec, k_rows=k_rows.contiguous(), q=q)
    out, _ = oracle.paged_decode(cache, pages, qb, spec.Hq, spec.sm_scale, 70)
    V = _dense_kv(spec, batch, cache, "v")
    for h in range(spec.Hkv):
        np.testing.assert_allclose(out[0, h * spec.G], V[0][h][star].numpy(), rtol=1e-9,
                                   atol=1e-12)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
def test_physical_placement_does_not_change_result(oracle, kv_dtype):
    """Contiguous pages vs a seeded permutation: bit-identical output."""
    spec = _small_spec(kv_dtype, [37, 100], NP=40)
    batch, cache, pages, qb, k_rows, v_rows, q = _setup(spec)
    out1, _ = oracle.paged_decode(cache, pages, qb, spec.Hq, spec.sm_scale, 100)
    # same logical content on pages 0..k-1 in order
    batch2 = W.make_batch(spec)
    need = (batch2.seq_lens + 15) // 16
    bt = np.full_like(batch2.block_tables, -1)
    off = 0
    for b in range(spec.B):
        bt[b, :need[b]] = np.arange(off, off + need[b])
        off += need[b]
    batch2.block_tables = bt
    batch2.expected_tags = np.zeros_like(bt, dtype=np.uint32)
    k, v, ks, vs = fill_pool(spec, batch2, W.bf16_bits(k_rows), W.bf16_bits(v_rows))
    c2 = cache_dict(spec, batch2, k, v, ks, vs, tags=False)
    p2 = pages_dict(spec, batch2, batch2.seq_lens, tags=False)
    out2, _ = oracle.paged_decode(c2, p2, qb, spec.Hq, spec.sm_scale, 100)
    assert not np.array_equal(batch.block_tables, bt)
    assert np.array_equal(out1, out2)


def test_per_head_tables_all_equal_match_shared_table(oracle):
    spec = _small_spec("fp8", [37, 100])
    batch, cache, pages, qb, k_rows, v_rows, _ = _setup(spec)
    out1, _ = oracle.paged_decode(cache, pages, qb, spec.Hq, spec.sm_scale, 100)
    # the same table repeated per head, lengths per head
    bt3 = np.repeat(batch.block_tables[:, None, :], spec.Hkv, axis=1).copy()
    ex3 = np.repeat(batch.expected_tags[:, None, :], spec.Hkv, axis=1).copy()
    lens2 = np.repeat(batch.seq_lens[:, None], spec.Hkv, axis=1).copy()
    p2 = dict(pages)
    p2.update(block_tables=bt3, bt_stride_b=spec.Hkv * batch.max_pages,
              bt_stride_h=batch.max_pages, expected_tags=ex3, seq_lens=lens2,
              len_stride_b=spec.Hkv, len_stride_h=1)
    out2, _ = oracle.paged_decode(cache, p2, qb, spec.Hq, spec.sm_scale, 100)
    assert np.array_equal(out1, out2)


def test_per_head_lengths_bruteforce(oracle):
    lens = np.array([[20, 3], [0, 47], [16, 33]], dtype=np.int32)
    spec = _small_spec("fp8", lens, per_head=True)
    batch, cache, pages, qb, _, _, q = _setup(spec)
    out, flags = oracle.paged_decode(cache, pages, qb, spec.Hq, spec.sm_scale, 64)
    assert not flags.any()
    K = _dense_kv(spec, batch, cache, "k")
    V = _dense_kv(spec, batch, cache, "v")
    for b in range(spec.B):
        for hq in range(spec.Hq):
            h = hq // spec.G
            if lens[b, h] == 0:
                assert not out[b, hq].any()      # zero-length head -> zeros
                continue
            ref = torch.nn.functional.scaled_dot_product_attention(
                q[b, hq].to(torch.float64)[None, None, None], K[b][h][None, None],
                V[b][h][None, None], scale=spec.sm_scale)[0, 0, 0].numpy()
            np.testing.assert_allclose(out[b, hq], ref, rtol=1e-12, atol=1e-12)


def test_flagged_request_outputs_zero(oracle):
    spec = _small_spec("fp8", [37, 100])
    batch, cache, pages, qb, _, _, _ = _setup(spec)
    tags = cache["page_tags"].copy()
    phys = int(batch.block_tables[1, 3])
    tags[phys, 1] ^= np.uint32(0x1234)
    cache2 = dict(cache, page_tags=tags)
    out, flags = oracle.paged_decode(cache2, pages, qb, spec.Hq, spec.sm_scale, 100)
    assert list(flags) == [0, oracle.FLAG_TAG]
    assert not out[1].any()
    assert out[0].any()
