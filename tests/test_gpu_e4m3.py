"""GPU e4m3 conversions against the oracle codec: every code (decode) and
every fp32 bit pattern (encode), bit for bit."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from paged_fp8_kv_decode_gb300 import build as pbuild
    pbuild.build()
    from paged_fp8_kv_decode_gb300 import binding
    return binding


def test_decode_all_codes(B):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8).cuda()
    out = torch.empty(256, dtype=torch.float32, device="cuda")
    B.pfkv_e4m3_decode(codes, out)
    got = out.cpu().numpy().astype(np.float64)
    ref = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_encode_every_fp32_bit_pattern(B):
    """All 2^32 fp32 inputs, in 16 slices of 2^28."""
    n = 1 << 28
    out = torch.empty(n, dtype=torch.uint8, device="cuda")
    for s in range(16):
        bits = np.arange(s * n, (s + 1) * n, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        xd = torch.from_numpy(x).cuda()
        B.pfkv_e4m3_encode(xd, out)
        ref = oracle.e4m3_encode(x)
        got = out.cpu().numpy()
        bad = np.nonzero(got != ref)[0]
        assert bad.size == 0, [(hex(int(bits[i])), hex(got[i]), hex(ref[i])) for i in bad[:8]]
        del xd
