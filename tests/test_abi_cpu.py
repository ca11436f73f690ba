"""The C ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching CUDA.
No call here launches a kernel."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pfkv.h")


@pytest.fixture(scope="module")
def B():
    from paged_fp8_kv_decode_gb300 import build as pbuild
    pbuild.build()
    from paged_fp8_kv_decode_gb300 import binding
    binding.lib()
    return binding


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(pfkv_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    assert names == sorted(["pfkv_abi_version", "pfkv_decode_workspace_size", "pfkv_e4m3_decode",
                            "pfkv_e4m3_encode", "pfkv_kv_append", "pfkv_decode_step", "pfkv_paged_decode_attn",
                            "pfkv_paged_decode_attn_fused_tags", "pfkv_paged_decode_attn_mass",
                            "pfkv_decode_mass_workspace_size", "pfkv_paged_decode_attn_multi",
                            "pfkv_decode_multi_workspace_size",
                            "pfkv_paged_decode_attn_noalloc", "pfkv_paged_decode_attn_stages",
                            "pfkv_status_string", "pfkv_selftest_bounded_wait", "pfkv_step_graph_create",
                            "pfkv_step_graph_destroy", "pfkv_step_graph_launch",
                            "pfkv_flags_status", "pfkv_stage_copy"])


def test_library_exports_every_declared_symbol(B):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared_functions():
        assert name in exported, name
        assert hasattr(B.lib(), name)
    # nothing but the C entry points is exported
    assert {n for n in exported if not n.startswith("pfkv_")} <= set()
    assert set(B.EXPORTED) == set(_declared_functions())


def test_status_strings_and_version(B):
    assert B.pfkv_abi_version() == 1
    for code in range(7):
        assert isinstance(B.pfkv_status_string(code), str)
    assert B.pfkv_status_string(0) == "ok"
    assert B.pfkv_status_string(99) == "unknown status"


def _structs(B, **over):
    c = dict(num_pages=8, num_kv_heads=2, page_size=16, head_dim=128, dtype=1,
             k_pages=0x10000, v_pages=0x20000, k_scale=0x30000, v_scale=0x40000, page_tags=None)
    p = dict(batch=2, max_pages=4, block_tables=0x50000, bt_stride_b=4, bt_stride_h=0,
             seq_lens=0x60000, len_stride_b=1, len_stride_h=0, expected_tags=None)
    for k, v in over.items():
        (c if k in c else p)[k] = v
    return B._CCache(**c), B._CPages(**p)


def _append(B, c, p, positions=0x70000, T=1, k=0x80000, v=0x90000, flags=None):
    return B.lib().pfkv_kv_append(ctypes.byref(c), ctypes.byref(p), positions, None, T, k, v,
                                  flags, None)


def _attn(B, c, p, Hq=4, q=0xA0000, ws=0xB0000, ws_bytes=1 << 30, out=0xC0000, split=0,
          max_len=64):
    return B.lib().pfkv_paged_decode_attn(ctypes.byref(c), ctypes.byref(p), q, Hq, 0.125, split,
                                          max_len, ws, ws_bytes, out, None, None)


@pytest.mark.parametrize("over,code", [
    (dict(page_size=32), 2), (dict(head_dim=96), 2), (dict(dtype=7), 1), (dict(num_pages=0), 1),
    (dict(k_pages=None), 1), (dict(k_scale=None), 1), (dict(k_pages=0x10008), 3),
    (dict(max_pages=0), 1), (dict(block_tables=None), 1), (dict(bt_stride_b=-1), 1),
    (dict(bt_stride_b=2), 1), (dict(page_tags=0x11000), 1), (dict(expected_tags=0x12000), 1),
    (dict(block_tables=0x50002), 3),
])
def test_host_rejects_bad_cache_or_pages(B, over, code):
    c, p = _structs(B, **over)
    assert _append(B, c, p) == code
    assert _attn(B, c, p) == code


def test_host_rejects_bad_call_arguments(B):
    c, p = _structs(B)
    assert _append(B, c, p, T=0) == 1
    assert _append(B, c, p, k=None) == 1
    assert _append(B, c, p, k=0x80008) == 3
    assert _append(B, c, p, positions=0x70002) == 3
    assert _append(B, c, p, flags=0xD0001) == 3
    assert _attn(B, c, p, Hq=3) == 1           # not a multiple of the kv heads
    assert _attn(B, c, p, Hq=6) == 2           # group size 3
    assert _attn(B, c, p, Hq=32) == 2          # group size 16
    assert _attn(B, c, p, split=24) == 1       # not a multiple of 16
    assert _attn(B, c, p, split=8192 + 16) == 2
    assert _attn(B, c, p, max_len=-1) == 1
    assert _attn(B, c, p, q=None) == 1
    assert _attn(B, c, p, out=0xC0004) == 3
    assert _attn(B, c, p, ws=None) == 4
    assert _attn(B, c, p, ws=0xB0010) == 3
    bad = ctypes.c_size_t(0)
    assert B.lib().pfkv_decode_workspace_size(ctypes.byref(c), ctypes.byref(p), 4, 0, 64,
                                              None) == 1


def test_stage_mask_is_checked(B):
    c, p = _structs(B)
    L = B.lib()
    # no stage bit (the option bits alone count as none), or an unknown bit
    for mask in (0, 8, 0x10, 0x18, 0x27, 0x20):
        assert L.pfkv_paged_decode_attn_stages(ctypes.byref(c), ctypes.byref(p), 0xA0000, 4, 0.125,
                                               0, 64, 0xB0000, 1 << 30, 0xC0000, None, mask,
                                               None) == 1


def test_fused_tag_entry_checks_arguments_like_the_plain_one(B):
    c, p = _structs(B)
    L = B.lib()
    def fused(Hq=4, split=0, max_len=64, ws=0xB0000):
        return L.pfkv_paged_decode_attn_fused_tags(ctypes.byref(c), ctypes.byref(p), 0xA0000, Hq,
                                                   0.125, split, max_len, ws, 1 << 30, 0xC0000,
                                                   None, None)
    assert fused(Hq=6) == 2
    assert fused(split=24) == 1
    assert fused(max_len=-1) == 1
    assert fused(ws=None) == 4
    assert fused(ws=0xB0010) == 3


def test_decode_step_checks_both_parts_before_any_launch(B):
    """pfkv_decode_step = kv_append + attention: the append's argument errors
    and the attention's come back with the same codes as from the two calls,
    and an unknown option bit is rejected (all before any device access)."""
    c, p = _structs(B)
    L = B.lib()
    def step(T=1, k=0x80000, positions=0x70000, Hq=4, split=0, ws=0xB0000, out=0xC0000, options=0):
        return L.pfkv_decode_step(ctypes.byref(c), ctypes.byref(p), positions, None, T, k, 0x90000,
                                  None, 0xA0000, Hq, 0.125, split, 64, ws, 1 << 30, out, None,
                                  options, None)
    assert step(options=0x1) == 1
    assert step(options=0x10) == 1
    assert step(T=0) == 1
    assert step(k=None) == 1
    assert step(k=0x80008) == 3
    assert step(positions=0x70002) == 3
    assert step(Hq=6) == 2
    assert step(split=24) == 1
    assert step(ws=None) == 4
    assert step(out=0xC0004) == 3
    for over, code in [(dict(page_size=32), 2), (dict(block_tables=None), 1)]:
        c2, p2 = _structs(B, **over)
        assert L.pfkv_decode_step(ctypes.byref(c2), ctypes.byref(p2), 0x70000, None, 1, 0x80000,
                                  0x90000, None, 0xA0000, 4, 0.125, 0, 64, 0xB0000, 1 << 30,
                                  0xC0000, None, 0, None) == code


def test_step_graph_argument_checks(B):
    """Checks that need no device: a missing handle pointer, no layers, an
    unknown option, a layer with only one of k_new / v_new."""
    c, p = _structs(B)
    L = B.lib()
    lay = (B._CLayer * 1)(B._CLayer(c, 0xA0000, 0, 0, 0xC0000, 0))
    h = ctypes.c_void_p(0)
    def create(layers=lay, n=1, opts=0, out=ctypes.byref(h)):
        return L.pfkv_step_graph_create(layers, n, ctypes.byref(p), 0xD0000, None, 1, None, 4,
                                        0.125, 0, 64, 0xB0000, 1 << 30, opts, out)
    assert create(out=None) == 1
    assert create(n=0) == 1
    assert create(layers=None) == 1
    assert create(opts=0x4) == 1
    half = (B._CLayer * 1)(B._CLayer(c, 0xA0000, 0xE0000, 0, 0xC0000, 0))
    assert create(layers=half) == 1
    assert h.value is None
    assert L.pfkv_step_graph_destroy(None) == 0
    assert L.pfkv_step_graph_launch(None, None) == 1


def test_mass_entry_checks_arguments(B):
    c, p = _structs(B)
    L = B.lib()
    def mass(buf=0xF0000, sb=8 * 64, sh=64, opts=0, Hq=4):
        return L.pfkv_paged_decode_attn_mass(ctypes.byref(c), ctypes.byref(p), 0xA0000, Hq, 0.125,
                                             0, 64, 0xB0000, 1 << 30, 0xC0000, None, buf, sb, sh,
                                             opts, None)
    assert mass(buf=None) == 1
    assert mass(buf=0xF0002) == 3
    assert mass(sb=-1) == 1
    assert mass(opts=0x2) == 1
    assert mass(Hq=6) == 2


def test_multi_entry_checks_arguments(B):
    c, p = _structs(B)
    L = B.lib()
    def multi(kq=3, opts=0, Hq=4, ws=0xB0000):
        return L.pfkv_paged_decode_attn_multi(ctypes.byref(c), ctypes.byref(p), 0xA0000, Hq, kq,
                                              0.125, 0, 64, ws, 1 << 30, 0xC0000, None, opts,
                                              None)
    assert multi(kq=0) == 1
    assert multi(kq=-2) == 1
    assert multi(opts=0x1) == 1
    assert multi(Hq=6) == 2
    assert multi(ws=None) == 4
    n = ctypes.c_size_t(0)
    assert L.pfkv_decode_multi_workspace_size(ctypes.byref(c), ctypes.byref(p), 4, 0, 0, 64,
                                              ctypes.byref(n)) == 1


def test_selftest_checks_its_pointer(B):
    assert B.lib().pfkv_selftest_bounded_wait(None, None) == 1
    assert B.lib().pfkv_selftest_bounded_wait(0x1002, None) == 3


def test_empty_batch_is_a_no_op(B):
    c, p = _structs(B, batch=0, block_tables=None, seq_lens=None)
    assert _append(B, c, p) == 0
    assert _attn(B, c, p) == 0


def test_e4m3_utilities_reject_bad_sizes(B):
    L = B.lib()
    assert L.pfkv_e4m3_encode(None, -1, None, None) == 1
    assert L.pfkv_e4m3_encode(None, 0, None, None) == 0
    assert L.pfkv_e4m3_encode(None, 5, None, None) == 1
    assert L.pfkv_e4m3_encode(0x1002, 5, 0x2000, None) == 3
    assert L.pfkv_e4m3_decode(0x1000, 5, 0x2002, None) == 3


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from paged_fp8_kv_decode_gb300 import binding
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "libpfkv.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()


def _header_enum(name):
    m = re.search(r"\b" + name + r"\s*=\s*(\d+)", open(HEADER).read())
    return int(m.group(1))


def _header_macro(name):
    m = re.search(r"#define\s+" + name + r"\s+\(?(\w+)u?\s*(<<\s*(\d+))?\)?", open(HEADER).read())
    v = int(m.group(1).rstrip("u"), 0)
    return v << int(m.group(3)) if m.group(3) else v


def test_binding_constants_match_the_header(B):
    """The binding's copies of the header's numbers, read from the header."""
    for name in ("PFKV_OK", "PFKV_ERR_INVALID_ARG", "PFKV_ERR_UNSUPPORTED", "PFKV_ERR_ALIGNMENT",
                 "PFKV_ERR_WORKSPACE", "PFKV_ERR_CUDA", "PFKV_ERR_DEVICE", "PFKV_KV_BF16",
                 "PFKV_KV_FP8_E4M3"):
        assert getattr(B, name) == _header_enum(name), name
    for name in ("PFKV_PAGE_SIZE", "PFKV_FLAG_TAG_MISMATCH", "PFKV_FLAG_BAD_PAGE",
                 "PFKV_FLAG_BAD_LENGTH", "PFKV_FLAG_DEVICE_TIMEOUT", "PFKV_STAGE_VALIDATE",
                 "PFKV_STAGE_SPLIT", "PFKV_STAGE_COMBINE", "PFKV_STAGE_ALL", "PFKV_STAGE_FUSED_TAGS",
                 "PFKV_STAGE_CUDA_CORES", "PFKV_NOALLOC_WORKSPACE_BYTES"):
        assert getattr(B, name) == _header_macro(name), name
    assert B.PFKV_NOALLOC_WORKSPACE_BYTES == 16 << 20


def test_flags_status_turns_device_timeouts_into_a_status(B):
    """Only PFKV_FLAG_DEVICE_TIMEOUT makes a status; data flags do not."""
    import numpy as np
    assert B.pfkv_flags_status(np.zeros(5, np.uint8)) == B.PFKV_OK
    data = np.array([B.PFKV_FLAG_TAG_MISMATCH, B.PFKV_FLAG_BAD_PAGE, B.PFKV_FLAG_BAD_LENGTH,
                     B.PFKV_FLAG_TAG_MISMATCH | B.PFKV_FLAG_BAD_LENGTH], np.uint8)
    assert B.pfkv_flags_status(data) == B.PFKV_OK
    for pos in range(4):
        f = data.copy()
        f[pos] |= B.PFKV_FLAG_DEVICE_TIMEOUT
        assert B.pfkv_flags_status(f) == B.PFKV_ERR_DEVICE
    assert B.pfkv_flags_status(np.zeros(0, np.uint8)) == B.PFKV_OK
    L = B.lib()
    assert L.pfkv_flags_status(None, 3) == B.PFKV_ERR_INVALID_ARG
    buf = np.zeros(4, np.uint8)
    assert L.pfkv_flags_status(buf.ctypes.data, -1) == B.PFKV_ERR_INVALID_ARG
    # only the first `batch` requests count
    buf[3] = B.PFKV_FLAG_DEVICE_TIMEOUT
    assert L.pfkv_flags_status(buf.ctypes.data, 3) == B.PFKV_OK
    assert L.pfkv_flags_status(buf.ctypes.data, 4) == B.PFKV_ERR_DEVICE


def test_stage_copy_checks_arguments_before_any_cuda_call(B):
    L = B.lib()
    assert L.pfkv_stage_copy(None, None, 0, None) == B.PFKV_OK          # nothing to copy
    assert L.pfkv_stage_copy(None, 0x10000, 64, None) == B.PFKV_ERR_INVALID_ARG
    assert L.pfkv_stage_copy(0x20000, None, 64, None) == B.PFKV_ERR_INVALID_ARG
    assert L.pfkv_stage_copy(0x20008, 0x10000, 64, None) == B.PFKV_ERR_ALIGNMENT
    assert L.pfkv_stage_copy(0x20000, 0x10000, 40, None) == B.PFKV_ERR_ALIGNMENT
    assert L.pfkv_stage_copy(0x10020, 0x10000, 64, None) == B.PFKV_ERR_INVALID_ARG  # overlap
    # valid arguments reach the device check: no GPU here
    assert L.pfkv_stage_copy(0x20000, 0x10000, 64, None) in (B.PFKV_ERR_CUDA, B.PFKV_ERR_UNSUPPORTED)
