"""pfkv_paged_decode_attn_noalloc: the attention entry point for callers that
cannot allocate device memory at decode time (an engine whose GPU memory is all
given to weights and the KV pool, a plugin whose host framework owns every
allocation, a loop that must not risk a synchronising cudaMalloc).  It uses a
fixed workspace inside the library instead of one the caller passes.

Checked through the C ABI against pfkv_paged_decode_attn with a caller
workspace, on two calls in a row (the second reuses the array the first left
behind).  This file is named to be collected last and builds what it needs, so
it runs the same alone in a fresh process or after the other tests.
"""
import numpy as np
import pytest
import torch

from oracle_cases import ATOL, RTOL
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


def _close(a, b):
    a = a.float().cpu().numpy().astype(np.float64)
    b = b.float().cpu().numpy().astype(np.float64)
    return bool(np.all(np.abs(a - b) <= ATOL + RTOL * np.abs(b)))


@pytest.mark.parametrize("make_spec", [lambda: W.spec_llama8b("small"),
                                       lambda: W.spec_evict("small"),
                                       W.spec_tiny])
def test_noalloc_matches_caller_workspace_twice(B, make_spec):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    spec = make_spec()
    db = DeviceBatch(W.make_batch(spec))
    ref_out = torch.empty_like(db.out)
    ref_flags = torch.zeros_like(db.flags)
    B.pfkv_paged_decode_attn(db.cache, db.pages, db.q, spec.sm_scale, db.split_tokens,
                             db.max_seq_len, db.workspace, ref_out, ref_flags)
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(db.out, 7.0)
        flags = torch.full_like(db.flags, 0xEE)
        B.pfkv_paged_decode_attn_noalloc(db.cache, db.pages, db.q, spec.sm_scale,
                                         db.split_tokens, db.max_seq_len, out, flags)
        torch.cuda.synchronize()
        assert torch.equal(flags[:spec.B], ref_flags[:spec.B])
        assert _close(out, ref_out)


def test_noalloc_rejects_calls_beyond_its_workspace(B):
    """A call that would need more than the built-in workspace is refused
    with PFKV_ERR_WORKSPACE before anything runs; out is left untouched."""
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    spec = W.spec_llama8b("small")
    db = DeviceBatch(W.make_batch(spec))
    split, max_len = 16, 1 << 20    # many 16-token chunks: a large workspace
    need = B.pfkv_decode_workspace_size(db.cache, db.pages, spec.Hq, split, max_len)
    assert need > B.PFKV_NOALLOC_WORKSPACE_BYTES
    out = torch.full_like(db.out, 3.0)
    with pytest.raises(B.PfkvError) as e:
        B.pfkv_paged_decode_attn_noalloc(db.cache, db.pages, db.q, spec.sm_scale, split, max_len,
                                         out, db.flags)
    assert e.value.status == B.PFKV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out.float() == 3.0).all())
