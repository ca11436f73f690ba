"""pfkv_decode_step (kv_append + attention in one call; the append shares its
launch with the validation) against the two calls it replaces, on identical
inputs: the same pool bytes, scales, append flags, attention flags and
outputs, byte for byte.  The two-call path is checked against the oracle in
test_gpu_parity.py."""
import dataclasses

import numpy as np
import pytest
import torch

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


CASES = {
    "llama8b": lambda: W.spec_llama8b("small"),
    # two stale units among the live ones: some requests flagged, some not
    "llama8b-stale": lambda: dataclasses.replace(W.spec_llama8b("small"), stale_per_mille=1.0),
    "evict-append": lambda: dataclasses.replace(W.spec_evict("small"), append=True),
    "long-append": lambda: dataclasses.replace(W.spec_long("small"), append=True),
}


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_step_equals_append_then_attention(B, name, fused):
    from paged_fp8_kv_decode_gb300.device_batch import DeviceBatch
    spec = CASES[name]()
    batch = W.make_batch(spec)
    one = DeviceBatch(batch, fused_tags=fused)
    two = DeviceBatch(batch, fused_tags=fused)
    for _ in range(2):  # a second step appends over the same slots again
        one.step(one_call=True)
        two.step(one_call=False)
    torch.cuda.synchronize()
    for x, y in [(one.cache.k_pages, two.cache.k_pages), (one.cache.v_pages, two.cache.v_pages),
                 (one.cache.k_scale, two.cache.k_scale), (one.cache.v_scale, two.cache.v_scale),
                 (one.append_flags, two.append_flags), (one.flags, two.flags)]:
        if x is None:
            continue
        assert torch.equal(x, y), name
    assert torch.equal(one.out.view(torch.int16), two.out.view(torch.int16)), name
    if name == "llama8b-stale":
        f = one.flags.cpu().numpy()[:spec.B]
        assert f.any() and not f.all()
