"""Canary guards: no kernel writes outside the buffers a call is given.

The pages stress that a bookkeeping mistake in a paged cache shows up sooner
or later at scale ("Cloudflare quantizes Kimi and GLM caches for 41% faster
inference", 4th paragraph).  compute-sanitizer is closed on this machine, so
every buffer a call writes (out, flags, append flags, the workspace, the K/V
pools and their scales, the attention-mass totals) sits between two guard
regions of seeded random bytes, and each test checks, after the call, that
every guard byte is unchanged and that the guarded call's results equal an
unguarded call's.  The cases take every kernel path: the persistent split
kernel (8 and 12 workers, FP8 and BF16, head_dim 128 and 64, groups of 4
and 8, a coarsened split, request groups), the combine's query-head groups,
the per-chunk kernel (multi-query verify with more query tokens x kv heads
than a persistent launch holds), the fused tag check, the attention-mass pass
and multi-query verify.
"""
import dataclasses

import numpy as np
import pytest
import torch

from paged_fp8_kv_decode_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes each side: a multiple of 256, so every alignment the ABI asks for holds


@pytest.fixture(scope="module")
def B():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_fp8_kv_decode_gb300 import build as pbuild
    pbuild.build()
    from paged_fp8_kv_decode_gb300 import binding
    binding.lib()
    return binding


class Guarded:
    """A device buffer of `like`'s size and contents between two guards."""

    def __init__(self, like: torch.Tensor, seed: int):
        n = like.numel() * like.element_size()
        g = torch.Generator().manual_seed(seed)
        self.pattern = torch.randint(0, 256, (2 * GUARD + n,), generator=g, dtype=torch.uint8)
        self.buf = self.pattern.to(like.device)
        self.n = n
        self.t = self.buf[GUARD:GUARD + n].view(like.dtype).view(like.shape)
        self.t.copy_(like)

    def intact(self) -> bool:
        host = self.buf.cpu()
        return (torch.equal(host[:GUARD], self.pattern[:GUARD])
                and torch.equal(host[GUARD + self.n:], self.pattern[GUARD + self.n:]))


def _guard_all(tensors, seed):
    return {k: Guarded(v, seed + i) for i, (k, v) in enumerate(tensors.items()) if v is not None}


def _assert_intact(g, label):
    bad = [k for k, x in g.items() if not x.intact()]
    assert not bad, (label, bad)


def _cache(B, db, g):
    c = db.cache
    return B.Cache(g["k_pages"].t, g["v_pages"].t, g["k_scale"].t if "k_scale" in g else None,
                   g["v_scale"].t if "v_scale" in g else None, c.page_tags)


def _db(spec, max_seq_len=None):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    return DeviceBatch(W.make_batch(spec), max_seq_len=max_seq_len)


def _pool(db):
    return {"k_pages": db.cache.k_pages, "v_pages": db.cache.v_pages,
            "k_scale": db.cache.k_scale, "v_scale": db.cache.v_scale}


STEP_CASES = {
    "llama8b": (lambda: W.spec_llama8b("small"), None),
    "llama8b_split48": (lambda: dataclasses.replace(W.spec_llama8b("small"), split_tokens=48), None),
    "twelve_workers": (lambda: W.spec_llama8b("small"), 131072),
    "g8_bf16": (lambda: dataclasses.replace(W.spec_llama8b("small"), Hq=64, kv_dtype="bf16",
                                            name="g8"), None),
    "combine_groups": (lambda: W.Spec("comb", B=5, Hq=64, Hkv=8, D=128, kv_dtype="fp8",
                                      num_pages=400, lens=np.array([90, 600, 333, 61, 700], np.int32),
                                      append=True, split_tokens=64, seed=7005), None),
    "many_segments": (lambda: W.Spec("manyseg", B=3, Hq=32, Hkv=8, D=128, kv_dtype="fp8",
                                     num_pages=1024, lens=np.array([3000, 2900, 2950], np.int32),
                                     append=True, split_tokens=16, seed=404), None),
    "head_dim_64": (lambda: dataclasses.replace(W.spec_tiny(), append=True), None),
    "head_dim_64_fp8_long": (lambda: W.Spec("d64", B=3, Hq=16, Hkv=4, D=64, kv_dtype="fp8",
                                            num_pages=600, lens=np.array([4000, 1500, 33], np.int32),
                                            append=True, stale_per_mille=2.0, seed=919), 131072),
    "request_groups": (lambda: W.Spec("groups", B=520, Hq=32, Hkv=8, D=128, kv_dtype="fp8",
                                      num_pages=1200, lens=np.arange(520, dtype=np.int32) % 37 + 1,
                                      append=True, stale_per_mille=3.0, seed=515), None),
    "evict": (lambda: dataclasses.replace(W.spec_evict("small"), append=True), None),
}


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("case", sorted(STEP_CASES))
def test_decode_step_writes_only_its_buffers(B, case, fused):
    """pfkv_decode_step (append, validation, split, combine) into guarded
    buffers: guards intact, results equal to the same step unguarded."""
    make, bound = STEP_CASES[case]
    spec = make()
    ref = _db(spec, bound)
    g = _guard_all({**_pool(ref), "out": ref.out, "flags": ref.flags,
                    "append_flags": ref.append_flags, "workspace": ref.workspace}, seed=11)
    opt = B.PFKV_STAGE_FUSED_TAGS if fused else 0
    B.pfkv_decode_step(_cache(B, ref, g), ref.pages, ref.positions, ref.k_new, ref.v_new, ref.q,
                       spec.sm_scale, ref.split_tokens, ref.max_seq_len, g["workspace"].t,
                       g["out"].t, g["flags"].t, append_flags=g["append_flags"].t, options=opt)
    B.pfkv_decode_step(ref.cache, ref.pages, ref.positions, ref.k_new, ref.v_new, ref.q,
                       spec.sm_scale, ref.split_tokens, ref.max_seq_len, ref.workspace, ref.out,
                       ref.flags, append_flags=ref.append_flags, options=opt)
    torch.cuda.synchronize()
    _assert_intact(g, f"{case} fused={fused}")
    assert torch.equal(g["out"].t, ref.out), case
    assert torch.equal(g["flags"].t[:spec.B], ref.flags[:spec.B]), case
    assert torch.equal(g["append_flags"].t[:spec.B], ref.append_flags[:spec.B]), case
    assert torch.equal(g["k_pages"].t, ref.cache.k_pages) and torch.equal(g["v_pages"].t, ref.cache.v_pages)
    if ref.cache.k_scale is not None:
        assert torch.equal(g["k_scale"].t, ref.cache.k_scale)
        assert torch.equal(g["v_scale"].t, ref.cache.v_scale)


@pytest.mark.parametrize("case", ["llama8b", "evict", "head_dim_64", "many_segments"])
def test_attention_mass_writes_only_its_buffers(B, case):
    make, bound = STEP_CASES[case]
    spec = dataclasses.replace(make(), append=False)
    db = _db(spec, bound)
    L = db.max_seq_len
    need = B.pfkv_decode_mass_workspace_size(db.cache, db.pages, spec.Hq, spec.split_tokens, L)
    ws = torch.empty(max(256, need), dtype=torch.uint8, device="cuda")
    mass = torch.rand((spec.B, spec.Hkv, L), device="cuda")
    want_out, want_flags, want_mass = torch.empty_like(db.out), torch.zeros_like(db.flags), mass.clone()
    g = _guard_all({"out": db.out, "flags": db.flags, "workspace": ws, "mass": mass}, seed=23)
    B.pfkv_paged_decode_attn_mass(db.cache, db.pages, db.q, spec.sm_scale, spec.split_tokens, L,
                                  g["workspace"].t, g["out"].t, g["flags"].t, g["mass"].t)
    B.pfkv_paged_decode_attn_mass(db.cache, db.pages, db.q, spec.sm_scale, spec.split_tokens, L,
                                  ws, want_out, want_flags, want_mass)
    torch.cuda.synchronize()
    _assert_intact(g, case)
    assert torch.equal(g["out"].t, want_out) and torch.equal(g["mass"].t, want_mass), case
    assert torch.equal(g["flags"].t[:spec.B], want_flags[:spec.B]), case


@pytest.mark.parametrize("case,kq", [("llama8b", 3), ("evict", 3), ("head_dim_64", 3),
                                     ("many_segments", 3), ("g8_bf16", 3), ("llama8b", 520)])
def test_multi_query_writes_only_its_buffers(B, case, kq):
    """kq = 520 on 8 kv heads: the per-chunk kernel and its combine."""
    make, bound = STEP_CASES[case]
    spec = dataclasses.replace(make(), append=False)
    if kq > 3:
        spec = dataclasses.replace(spec, B=2, lens=spec.lens[:2])
    db = _db(spec, bound)
    L = db.max_seq_len
    gen = torch.Generator(device="cuda").manual_seed(99)
    q = torch.randn((spec.B, kq, spec.Hq, spec.D), generator=gen, device="cuda").to(torch.bfloat16)
    need = B.pfkv_decode_multi_workspace_size(db.cache, db.pages, spec.Hq, kq, spec.split_tokens, L)
    ws = torch.empty(max(256, need), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    want_out, want_flags = torch.empty_like(q), torch.zeros_like(db.flags)
    g = _guard_all({"out": out, "flags": db.flags, "workspace": ws}, seed=37)
    B.pfkv_paged_decode_attn_multi(db.cache, db.pages, q, spec.sm_scale, spec.split_tokens, L,
                                   g["workspace"].t, g["out"].t, g["flags"].t)
    B.pfkv_paged_decode_attn_multi(db.cache, db.pages, q, spec.sm_scale, spec.split_tokens, L, ws,
                                   want_out, want_flags)
    torch.cuda.synchronize()
    _assert_intact(g, case)
    assert torch.equal(g["out"].t, want_out), case
    assert torch.equal(g["flags"].t[:spec.B], want_flags[:spec.B]), case


def test_append_of_many_tokens_writes_only_its_buffers(B):
    """kv_append of several pages' worth of tokens per (request, kv head)."""
    spec = dataclasses.replace(W.spec_llama8b("small"), append=False)
    db = _db(spec)
    T = 40
    gen = torch.Generator(device="cuda").manual_seed(5)
    kn = torch.randn((spec.B, spec.Hkv, T, spec.D), generator=gen, device="cuda").to(torch.bfloat16)
    vn = torch.randn((spec.B, spec.Hkv, T, spec.D), generator=gen, device="cuda").to(torch.bfloat16)
    pos = (db.seq_lens - T - 3).clamp(min=0)
    want = {k: v.clone() for k, v in _pool(db).items()}
    want_flags = torch.zeros_like(db.append_flags)
    g = _guard_all({**_pool(db), "flags": db.append_flags}, seed=51)
    B.pfkv_kv_append(_cache(B, db, g), db.pages, pos, kn, vn, flags=g["flags"].t)
    B.pfkv_kv_append(B.Cache(want["k_pages"], want["v_pages"], want["k_scale"], want["v_scale"],
                             db.cache.page_tags), db.pages, pos, kn, vn, flags=want_flags)
    torch.cuda.synchronize()
    _assert_intact(g, "append")
    for k in want:
        assert torch.equal(g[k].t, want[k]), k
    assert torch.equal(g["flags"].t[:spec.B], want_flags[:spec.B])
