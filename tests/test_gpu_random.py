"""Seeded random configurations against the oracle: kv dtype, head_dim, group
size, kv heads, batch, lengths (zero, one token, page edges, ragged tails),
shared or per-head tables, split size, tags with stale pages, separate or fused
tag check, plain / multi-query / attention-mass calls.  Each case is small
enough for the oracle to finish in well under a second; together they reach
combinations the hand-written cases do not."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle_cases import assert_outputs_close, cache_dict, fill_pool, pages_dict
from paged_fp8_kv_decode_gb300 import workloads as W
from test_gpu_parity import B  # noqa: F401  (fixture)

pytestmark = pytest.mark.gpu


def _random_spec(seed):
    rng = np.random.default_rng(seed)
    # weighted toward the persistent kernel's shapes (FP8, head_dim 128, G <= 4)
    kv_dtype = ["fp8", "fp8", "bf16"][rng.integers(3)]
    D = [64, 128, 128][rng.integers(3)]
    G = [1, 2, 4, 4, 8][rng.integers(5)]
    Hkv = int(rng.integers(1, 5))
    Bn = int(rng.integers(1, 7))
    per_head = bool(rng.integers(2))
    choices = np.array([0, 1, 15, 16, 17, 31, 33, 100, 255, 256, 257, 700, 1500])
    shape = (Bn, Hkv) if per_head else (Bn,)
    lens = rng.choice(choices, size=shape).astype(np.int32)
    lens.reshape(-1)[0] = max(lens.reshape(-1)[0], 40)          # at least one real head
    split = [0, 0, 16, 48, 256][rng.integers(5)]
    stale = [0.0, 0.0, 30.0][rng.integers(3)]
    need = (lens.astype(np.int64) + 15) // 16
    NP = int(need.sum() if not per_head else need.sum(axis=0).max()) + 8
    return W.Spec(f"rand{seed}", B=Bn, Hq=Hkv * G, Hkv=Hkv, D=D, kv_dtype=kv_dtype,
                  num_pages=NP, lens=lens, per_head=per_head, tags=True,
                  stale_per_mille=stale, split_tokens=split, seed=5000 + seed), rng


@pytest.mark.parametrize("seed", range(24))
def test_random_configuration(B, seed):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    spec, rng = _random_spec(seed)
    mode = ["plain", "multi", "mass"][seed % 3]
    fused = bool(rng.integers(2))
    batch = W.make_batch(spec)
    db = DeviceBatch(batch, keep_rows=True)
    L = max(1, int(batch.seq_lens.max()))
    k, v, ks, vs = fill_pool(spec, batch, W.bf16_bits(db.k_rows), W.bf16_bits(db.v_rows))
    cache = cache_dict(spec, batch, k, v, ks, vs)
    pages = pages_dict(spec, batch, batch.seq_lens)
    opt = B.PFKV_STAGE_FUSED_TAGS if fused else 0
    label = f"seed {seed} {mode} fused={fused} {spec}"
    if mode == "multi":
        kq = int(rng.integers(2, 5))
        g = torch.Generator(device="cuda").manual_seed(seed)
        q = torch.randn((spec.B, kq, spec.Hq, spec.D), generator=g, device="cuda").to(torch.bfloat16)
        out = torch.empty_like(q)
        ws = torch.empty(max(256, B.pfkv_decode_multi_workspace_size(db.cache, db.pages, spec.Hq, kq,
                                                                     spec.split_tokens, L)),
                         dtype=torch.uint8, device="cuda")
        B.pfkv_paged_decode_attn_multi(db.cache, db.pages, q, spec.sm_scale, spec.split_tokens, L,
                                       ws, out, db.flags, opt)
        torch.cuda.synchronize()
        ref, rflags = oracle.paged_decode_multi(cache, pages, W.bf16_bits(q), spec.Hq, kq,
                                                spec.sm_scale, L)
    else:
        q, out = db.q, db.out
        mass = None
        if mode == "mass":
            ws = torch.empty(max(256, B.pfkv_decode_mass_workspace_size(db.cache, db.pages, spec.Hq,
                                                                        spec.split_tokens, L)),
                             dtype=torch.uint8, device="cuda")
            mass = torch.zeros((spec.B, spec.Hkv, L), dtype=torch.float32, device="cuda")
            B.pfkv_paged_decode_attn_mass(db.cache, db.pages, q, spec.sm_scale, spec.split_tokens, L,
                                          ws, out, db.flags, mass, opt)
        else:
            ws = torch.empty(max(256, B.pfkv_decode_workspace_size(db.cache, db.pages, spec.Hq,
                                                                   spec.split_tokens, L)),
                             dtype=torch.uint8, device="cuda")
            fn = B.pfkv_paged_decode_attn_fused_tags if fused else B.pfkv_paged_decode_attn
            fn(db.cache, db.pages, q, spec.sm_scale, spec.split_tokens, L, ws, out, db.flags)
        torch.cuda.synchronize()
        ref, rflags = oracle.paged_decode(cache, pages, W.bf16_bits(q), spec.Hq, spec.sm_scale, L)
        if mass is not None:
            want = oracle.attention_mass(cache, pages, W.bf16_bits(q), spec.Hq, spec.sm_scale, L)
            got = mass.cpu().numpy().astype(np.float64)
            assert (np.abs(got - want) <= 1e-6 + 1e-3 * np.abs(want)).all(), label
    flags = db.flags.cpu().numpy()[:spec.B]
    assert np.array_equal(flags, rflags), (label, flags, rflags)
    assert_outputs_close(out, ref, label)
