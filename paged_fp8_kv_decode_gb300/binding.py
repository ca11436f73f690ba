"""ctypes binding of libpfkv.so (argument marshalling only).

Every function here has the name of the C entry point it calls (see
``include/pfkv.h`` for the full contract) and forwards torch CUDA tensors as
raw device pointers plus the caller's CUDA stream.  All computation runs in the
library's kernels; there is no fallback.  If the library has not been built,
the first call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpfkv.so")

PFKV_OK = 0
PFKV_ERR_INVALID_ARG = 1
PFKV_ERR_UNSUPPORTED = 2
PFKV_ERR_ALIGNMENT = 3
PFKV_ERR_WORKSPACE = 4
PFKV_ERR_CUDA = 5
PFKV_ERR_DEVICE = 6

PFKV_KV_BF16 = 0
PFKV_KV_FP8_E4M3 = 1
PFKV_PAGE_SIZE = 16

PFKV_FLAG_TAG_MISMATCH = 0x01
PFKV_FLAG_BAD_PAGE = 0x02
PFKV_FLAG_BAD_LENGTH = 0x04
PFKV_FLAG_DEVICE_TIMEOUT = 0x08

PFKV_STAGE_VALIDATE = 0x1
PFKV_STAGE_SPLIT = 0x2
PFKV_STAGE_COMBINE = 0x4
PFKV_STAGE_ALL = 0x7
PFKV_STAGE_FUSED_TAGS = 0x8
PFKV_STAGE_CUDA_CORES = 0x10

# every symbol include/pfkv.h declares
EXPORTED = ("pfkv_kv_append", "pfkv_decode_workspace_size", "pfkv_paged_decode_attn",
            "pfkv_decode_step",
            "pfkv_paged_decode_attn_stages", "pfkv_paged_decode_attn_fused_tags",
            "pfkv_paged_decode_attn_noalloc", "pfkv_paged_decode_attn_mass",
            "pfkv_decode_mass_workspace_size", "pfkv_paged_decode_attn_multi",
            "pfkv_decode_multi_workspace_size", "pfkv_step_graph_create", "pfkv_step_graph_launch",
            "pfkv_step_graph_destroy", "pfkv_selftest_bounded_wait", "pfkv_e4m3_encode", "pfkv_e4m3_decode", "pfkv_status_string",
            "pfkv_abi_version", "pfkv_flags_status", "pfkv_stage_copy")


class PfkvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {pfkv_status_string(status)} (status {status})")


class _CCache(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("k_pages", ctypes.c_void_p),
                ("v_pages", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("page_tags", ctypes.c_void_p)]


class _CPages(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("block_tables", ctypes.c_void_p), ("bt_stride_b", ctypes.c_int64),
                ("bt_stride_h", ctypes.c_int64), ("seq_lens", ctypes.c_void_p),
                ("len_stride_b", ctypes.c_int64), ("len_stride_h", ctypes.c_int64),
                ("expected_tags", ctypes.c_void_p)]


class _CLayer(ctypes.Structure):
    _fields_ = [("cache", _CCache), ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p),
                ("v_new", ctypes.c_void_p), ("out", ctypes.c_void_p), ("flags", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpfkv.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        L.pfkv_kv_append.argtypes = [ctypes.POINTER(_CCache), ctypes.POINTER(_CPages), P, P, I32,
                                     P, P, P, P]
        L.pfkv_kv_append.restype = ctypes.c_int
        L.pfkv_decode_workspace_size.argtypes = [ctypes.POINTER(_CCache),
                                                 ctypes.POINTER(_CPages), I32, I32, I32,
                                                 ctypes.POINTER(ctypes.c_size_t)]
        L.pfkv_decode_workspace_size.restype = ctypes.c_int
        L.pfkv_paged_decode_attn.argtypes = [ctypes.POINTER(_CCache), ctypes.POINTER(_CPages), P,
                                             I32, ctypes.c_float, I32, I32, P, ctypes.c_size_t,
                                             P, P, P]
        L.pfkv_paged_decode_attn.restype = ctypes.c_int
        L.pfkv_paged_decode_attn_stages.argtypes = [ctypes.POINTER(_CCache),
                                                    ctypes.POINTER(_CPages), P, I32,
                                                    ctypes.c_float, I32, I32, P, ctypes.c_size_t,
                                                    P, P, ctypes.c_uint32, P]
        L.pfkv_paged_decode_attn_stages.restype = ctypes.c_int
        L.pfkv_decode_step.argtypes = [ctypes.POINTER(_CCache), ctypes.POINTER(_CPages), P, P, I32,
                                       P, P, P, P, I32, ctypes.c_float, I32, I32, P,
                                       ctypes.c_size_t, P, P, ctypes.c_uint32, P]
        L.pfkv_decode_step.restype = ctypes.c_int
        L.pfkv_paged_decode_attn_fused_tags.argtypes = L.pfkv_paged_decode_attn.argtypes
        L.pfkv_paged_decode_attn_fused_tags.restype = ctypes.c_int
        L.pfkv_paged_decode_attn_noalloc.argtypes = [ctypes.POINTER(_CCache),
                                                     ctypes.POINTER(_CPages), P, I32,
                                                     ctypes.c_float, I32, I32, P, P, P]
        L.pfkv_paged_decode_attn_noalloc.restype = ctypes.c_int
        L.pfkv_decode_multi_workspace_size.argtypes = [ctypes.POINTER(_CCache),
                                                       ctypes.POINTER(_CPages), I32, I32, I32,
                                                       I32, ctypes.POINTER(ctypes.c_size_t)]
        L.pfkv_decode_multi_workspace_size.restype = ctypes.c_int
        L.pfkv_paged_decode_attn_multi.argtypes = [ctypes.POINTER(_CCache),
                                                   ctypes.POINTER(_CPages), P, I32, I32,
                                                   ctypes.c_float, I32, I32, P, ctypes.c_size_t,
                                                   P, P, ctypes.c_uint32, P]
        L.pfkv_paged_decode_attn_multi.restype = ctypes.c_int
        L.pfkv_decode_mass_workspace_size.argtypes = L.pfkv_decode_workspace_size.argtypes
        L.pfkv_decode_mass_workspace_size.restype = ctypes.c_int
        L.pfkv_paged_decode_attn_mass.argtypes = [ctypes.POINTER(_CCache), ctypes.POINTER(_CPages),
                                                  P, I32, ctypes.c_float, I32, I32, P,
                                                  ctypes.c_size_t, P, P, P, I64, I64,
                                                  ctypes.c_uint32, P]
        L.pfkv_paged_decode_attn_mass.restype = ctypes.c_int
        L.pfkv_step_graph_create.argtypes = [ctypes.POINTER(_CLayer), I32, ctypes.POINTER(_CPages),
                                             P, P, I32, P, I32, ctypes.c_float, I32, I32, P,
                                             ctypes.c_size_t, ctypes.c_uint32,
                                             ctypes.POINTER(ctypes.c_void_p)]
        L.pfkv_step_graph_create.restype = ctypes.c_int
        L.pfkv_step_graph_launch.argtypes = [P, P]
        L.pfkv_step_graph_launch.restype = ctypes.c_int
        L.pfkv_step_graph_destroy.argtypes = [P]
        L.pfkv_step_graph_destroy.restype = ctypes.c_int
        L.pfkv_selftest_bounded_wait.argtypes = [P, P]
        L.pfkv_selftest_bounded_wait.restype = ctypes.c_int
        L.pfkv_e4m3_encode.argtypes = [P, I64, P, P]
        L.pfkv_e4m3_encode.restype = ctypes.c_int
        L.pfkv_e4m3_decode.argtypes = [P, I64, P, P]
        L.pfkv_e4m3_decode.restype = ctypes.c_int
        L.pfkv_status_string.argtypes = [ctypes.c_int]
        L.pfkv_status_string.restype = ctypes.c_char_p
        L.pfkv_abi_version.argtypes = []
        L.pfkv_abi_version.restype = ctypes.c_int32
        L.pfkv_flags_status.argtypes = [P, I32]
        L.pfkv_flags_status.restype = ctypes.c_int
        L.pfkv_stage_copy.argtypes = [P, P, ctypes.c_size_t, P]
        L.pfkv_stage_copy.restype = ctypes.c_int
        _lib = L
    return _lib


def pfkv_status_string(status: int) -> str:
    return lib().pfkv_status_string(int(status)).decode()


def pfkv_abi_version() -> int:
    return int(lib().pfkv_abi_version())


def pfkv_stage_copy(dst, src, nbytes: Optional[int] = None, stream=None) -> None:
    """Copy ``nbytes`` (default: all of ``src``) from ``src`` to ``dst`` with a
    kernel; each a device tensor, a pinned host tensor or an address."""
    if nbytes is None:
        nbytes = src.numel() * src.element_size()
    _check(lib().pfkv_stage_copy(_ptr(dst), _ptr(src), int(nbytes), _stream(stream)),
           "pfkv_stage_copy")


def pfkv_flags_status(flags) -> int:
    """Status that a finished call's flags amount to (see include/pfkv.h):
    PFKV_ERR_DEVICE if a request carries PFKV_FLAG_DEVICE_TIMEOUT, else
    PFKV_OK.  ``flags``: host uint8 array or a tensor (copied to the host)."""
    import numpy as np
    if isinstance(flags, torch.Tensor):
        flags = flags.detach().to("cpu").numpy()
    a = np.ascontiguousarray(flags, dtype=np.uint8)
    return int(lib().pfkv_flags_status(a.ctypes.data if a.size else None, int(a.size)))


# --------------------------------------------------------------------------
# argument containers
# --------------------------------------------------------------------------
@dataclasses.dataclass
class Cache:
    """The page pool (caller-owned CUDA tensors).

    k_pages, v_pages: [num_pages][Hkv][16][head_dim], torch.bfloat16 or
    torch.uint8 (e4m3 codes); k_scale, v_scale: float32 [num_pages][Hkv] (FP8);
    page_tags: int32 (uint32 bit patterns) [num_pages][Hkv] or None."""
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    k_scale: Optional[torch.Tensor] = None
    v_scale: Optional[torch.Tensor] = None
    page_tags: Optional[torch.Tensor] = None

    @property
    def dtype(self) -> int:
        return PFKV_KV_BF16 if self.k_pages.dtype == torch.bfloat16 else PFKV_KV_FP8_E4M3

    def c_struct(self) -> _CCache:
        NP, H, PS, D = self.k_pages.shape
        return _CCache(NP, H, PS, D, self.dtype, _ptr(self.k_pages), _ptr(self.v_pages),
                       _ptr(self.k_scale), _ptr(self.v_scale), _ptr(self.page_tags))


@dataclasses.dataclass
class Pages:
    """The batch's block tables (int32), lengths (int32) and expected tags,
    with element strides (stride_h = 0: shared by every kv head)."""
    batch: int
    max_pages: int
    block_tables: torch.Tensor
    bt_stride_b: int
    bt_stride_h: int
    seq_lens: torch.Tensor
    len_stride_b: int
    len_stride_h: int
    expected_tags: Optional[torch.Tensor] = None

    def c_struct(self) -> _CPages:
        return _CPages(self.batch, self.max_pages, _ptr(self.block_tables), self.bt_stride_b,
                       self.bt_stride_h, _ptr(self.seq_lens), self.len_stride_b,
                       self.len_stride_h, _ptr(self.expected_tags))

    def with_lens(self, seq_lens: torch.Tensor) -> "Pages":
        return dataclasses.replace(self, seq_lens=seq_lens)


def _ptr(t) -> Optional[int]:
    """Address of a device tensor, or of a pinned host tensor (which the
    kernels read and write directly over the CPU-GPU link)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("device tensor or pinned host tensor expected")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != PFKV_OK:
        raise PfkvError(status, where)


# --------------------------------------------------------------------------
# entry points
# --------------------------------------------------------------------------
def pfkv_kv_append(cache: Cache, pages: Pages, positions: torch.Tensor, k_new: torch.Tensor,
                   v_new: torch.Tensor, new_lens: Optional[torch.Tensor] = None,
                   flags: Optional[torch.Tensor] = None, stream=None) -> None:
    """k_new, v_new: bf16 [B][Hkv][T][D]; positions/new_lens int32 with the
    length strides of ``pages``; flags uint8 [>= round_up(B, 4)] (OR-ed)."""
    c, p = cache.c_struct(), pages.c_struct()
    T = int(k_new.shape[2])
    _check(lib().pfkv_kv_append(ctypes.byref(c), ctypes.byref(p), _ptr(positions),
                                _ptr(new_lens), T, _ptr(k_new), _ptr(v_new), _ptr(flags),
                                _stream(stream)), "pfkv_kv_append")


def pfkv_decode_workspace_size(cache: Cache, pages: Pages, num_q_heads: int, split_tokens: int,
                               max_seq_len: int) -> int:
    c, p = cache.c_struct(), pages.c_struct()
    out = ctypes.c_size_t(0)
    _check(lib().pfkv_decode_workspace_size(ctypes.byref(c), ctypes.byref(p), int(num_q_heads),
                                            int(split_tokens), int(max_seq_len),
                                            ctypes.byref(out)), "pfkv_decode_workspace_size")
    return int(out.value)


def pfkv_paged_decode_attn(cache: Cache, pages: Pages, q: torch.Tensor, sm_scale: float,
                           split_tokens: int, max_seq_len: int, workspace: torch.Tensor,
                           out: torch.Tensor, flags: Optional[torch.Tensor] = None,
                           stream=None) -> None:
    """q, out: bf16 [B][Hq][D]; workspace: uint8 CUDA tensor of at least
    pfkv_decode_workspace_size(...) bytes; flags uint8 [>= round_up(B, 4)]."""
    c, p = cache.c_struct(), pages.c_struct()
    Hq = int(q.shape[1])
    _check(lib().pfkv_paged_decode_attn(ctypes.byref(c), ctypes.byref(p), _ptr(q), Hq,
                                        float(sm_scale), int(split_tokens), int(max_seq_len),
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _ptr(out), _ptr(flags), _stream(stream)),
           "pfkv_paged_decode_attn")


def pfkv_paged_decode_attn_stages(cache: Cache, pages: Pages, q: torch.Tensor, sm_scale: float,
                                  split_tokens: int, max_seq_len: int, workspace: torch.Tensor,
                                  out: torch.Tensor, flags: Optional[torch.Tensor], stages: int,
                                  stream=None) -> None:
    """pfkv_paged_decode_attn restricted to the PFKV_STAGE_* kernels in ``stages``."""
    c, p = cache.c_struct(), pages.c_struct()
    Hq = int(q.shape[1])
    _check(lib().pfkv_paged_decode_attn_stages(
        ctypes.byref(c), ctypes.byref(p), _ptr(q), Hq, float(sm_scale), int(split_tokens),
        int(max_seq_len), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(out), _ptr(flags), int(stages), _stream(stream)), "pfkv_paged_decode_attn_stages")


def pfkv_decode_step(cache: Cache, pages: Pages, positions: torch.Tensor, k_new: torch.Tensor,
                     v_new: torch.Tensor, q: torch.Tensor, sm_scale: float, split_tokens: int,
                     max_seq_len: int, workspace: torch.Tensor, out: torch.Tensor,
                     flags: Optional[torch.Tensor] = None,
                     append_flags: Optional[torch.Tensor] = None,
                     new_lens: Optional[torch.Tensor] = None, options: int = 0,
                     stream=None) -> None:
    """pfkv_kv_append then pfkv_paged_decode_attn in one call (the append and
    the validation share a launch); arguments as for the two calls."""
    c, p = cache.c_struct(), pages.c_struct()
    T = int(k_new.shape[2])
    Hq = int(q.shape[1])
    _check(lib().pfkv_decode_step(
        ctypes.byref(c), ctypes.byref(p), _ptr(positions), _ptr(new_lens), T, _ptr(k_new),
        _ptr(v_new), _ptr(append_flags), _ptr(q), Hq, float(sm_scale), int(split_tokens),
        int(max_seq_len), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(out), _ptr(flags), int(options), _stream(stream)), "pfkv_decode_step")


def pfkv_paged_decode_attn_fused_tags(cache: Cache, pages: Pages, q: torch.Tensor,
                                      sm_scale: float, split_tokens: int, max_seq_len: int,
                                      workspace: torch.Tensor, out: torch.Tensor,
                                      flags: Optional[torch.Tensor] = None, stream=None) -> None:
    """pfkv_paged_decode_attn with the tag check inside the attention kernel
    (same outputs and flags; see include/pfkv.h)."""
    c, p = cache.c_struct(), pages.c_struct()
    Hq = int(q.shape[1])
    _check(lib().pfkv_paged_decode_attn_fused_tags(
        ctypes.byref(c), ctypes.byref(p), _ptr(q), Hq, float(sm_scale), int(split_tokens),
        int(max_seq_len), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(out), _ptr(flags), _stream(stream)), "pfkv_paged_decode_attn_fused_tags")


def pfkv_decode_multi_workspace_size(cache: Cache, pages: Pages, num_q_heads: int,
                                     num_query_tokens: int, split_tokens: int,
                                     max_seq_len: int) -> int:
    c, p = cache.c_struct(), pages.c_struct()
    out = ctypes.c_size_t(0)
    _check(lib().pfkv_decode_multi_workspace_size(ctypes.byref(c), ctypes.byref(p),
                                                  int(num_q_heads), int(num_query_tokens),
                                                  int(split_tokens), int(max_seq_len),
                                                  ctypes.byref(out)),
           "pfkv_decode_multi_workspace_size")
    return int(out.value)


def pfkv_paged_decode_attn_multi(cache: Cache, pages: Pages, q: torch.Tensor, sm_scale: float,
                                 split_tokens: int, max_seq_len: int, workspace: torch.Tensor,
                                 out: torch.Tensor, flags: Optional[torch.Tensor] = None,
                                 options: int = 0, stream=None) -> None:
    """q, out: bf16 [B][kq][Hq][D]: the kq candidate tokens of each request,
    causal among themselves (see include/pfkv.h)."""
    c, p = cache.c_struct(), pages.c_struct()
    kq, Hq = int(q.shape[1]), int(q.shape[2])
    _check(lib().pfkv_paged_decode_attn_multi(
        ctypes.byref(c), ctypes.byref(p), _ptr(q), Hq, kq, float(sm_scale), int(split_tokens),
        int(max_seq_len), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(out), _ptr(flags), int(options), _stream(stream)), "pfkv_paged_decode_attn_multi")


def pfkv_decode_mass_workspace_size(cache: Cache, pages: Pages, num_q_heads: int,
                                    split_tokens: int, max_seq_len: int) -> int:
    c, p = cache.c_struct(), pages.c_struct()
    out = ctypes.c_size_t(0)
    _check(lib().pfkv_decode_mass_workspace_size(ctypes.byref(c), ctypes.byref(p),
                                                 int(num_q_heads), int(split_tokens),
                                                 int(max_seq_len), ctypes.byref(out)),
           "pfkv_decode_mass_workspace_size")
    return int(out.value)


def pfkv_paged_decode_attn_mass(cache: Cache, pages: Pages, q: torch.Tensor, sm_scale: float,
                                split_tokens: int, max_seq_len: int, workspace: torch.Tensor,
                                out: torch.Tensor, flags: Optional[torch.Tensor],
                                attn_mass: torch.Tensor, options: int = 0, stream=None) -> None:
    """pfkv_paged_decode_attn plus attn_mass[b][h][j] += the token's summed softmax
    weight over the group's query heads (attn_mass: float32 CUDA tensor, 3-D
    [B][Hkv][>= max_seq_len] with any strides)."""
    c, p = cache.c_struct(), pages.c_struct()
    Hq = int(q.shape[1])
    if attn_mass.dtype != torch.float32 or attn_mass.dim() != 3 or attn_mass.stride(2) != 1:
        raise ValueError("attn_mass: float32 [B][Hkv][L] with unit stride along tokens")
    _check(lib().pfkv_paged_decode_attn_mass(
        ctypes.byref(c), ctypes.byref(p), _ptr(q), Hq, float(sm_scale), int(split_tokens),
        int(max_seq_len), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(out), _ptr(flags), _ptr(attn_mass), int(attn_mass.stride(0)),
        int(attn_mass.stride(1)), int(options), _stream(stream)), "pfkv_paged_decode_attn_mass")


# bytes of the library's own workspace used by pfkv_paged_decode_attn_noalloc
PFKV_NOALLOC_WORKSPACE_BYTES = 16 << 20


def pfkv_paged_decode_attn_noalloc(cache: Cache, pages: Pages, q: torch.Tensor, sm_scale: float,
                                   split_tokens: int, max_seq_len: int, out: torch.Tensor,
                                   flags: Optional[torch.Tensor] = None, stream=None) -> None:
    """pfkv_paged_decode_attn with the library's built-in workspace, for
    callers that cannot allocate device memory (see include/pfkv.h)."""
    c, p = cache.c_struct(), pages.c_struct()
    Hq = int(q.shape[1])
    _check(lib().pfkv_paged_decode_attn_noalloc(
        ctypes.byref(c), ctypes.byref(p), _ptr(q), Hq, float(sm_scale), int(split_tokens),
        int(max_seq_len), _ptr(out), _ptr(flags), _stream(stream)),
        "pfkv_paged_decode_attn_noalloc")


@dataclasses.dataclass
class Layer:
    """One attention layer of a step graph: its pool and its q/new rows/out/flags
    (k_new and v_new both None: no append in this layer)."""
    cache: Cache
    q: torch.Tensor
    out: torch.Tensor
    k_new: Optional[torch.Tensor] = None
    v_new: Optional[torch.Tensor] = None
    flags: Optional[torch.Tensor] = None

    def c_struct(self) -> _CLayer:
        return _CLayer(self.cache.c_struct(), _ptr(self.q), _ptr(self.k_new), _ptr(self.v_new),
                       _ptr(self.out), _ptr(self.flags))


class StepGraph:
    """Owner of a pfkv_step_graph handle (destroyed with the object or close())."""

    def __init__(self, handle: int, keep):
        self.handle, self._keep = handle, keep

    def launch(self, stream=None) -> None:
        pfkv_step_graph_launch(self, stream)

    def close(self) -> None:
        if self.handle:
            h, self.handle = self.handle, 0
            _check(lib().pfkv_step_graph_destroy(h), "pfkv_step_graph_destroy")

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pfkv_step_graph_create(layers, pages: Pages, positions: Optional[torch.Tensor],
                           new_lens: Optional[torch.Tensor], num_new_tokens: int,
                           append_flags: Optional[torch.Tensor], num_q_heads: int,
                           sm_scale: float, split_tokens: int, max_seq_len: int,
                           workspace: torch.Tensor, options: int = 0) -> StepGraph:
    """Capture one decode step of ``layers`` (a list of Layer) as a CUDA graph."""
    arr = (_CLayer * len(layers))(*[l.c_struct() for l in layers])
    p = pages.c_struct()
    h = ctypes.c_void_p(0)
    _check(lib().pfkv_step_graph_create(arr, len(layers), ctypes.byref(p), _ptr(positions),
                                        _ptr(new_lens), int(num_new_tokens), _ptr(append_flags),
                                        int(num_q_heads), float(sm_scale), int(split_tokens),
                                        int(max_seq_len), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(),
                                        int(options), ctypes.byref(h)), "pfkv_step_graph_create")
    # the captured pointers stay valid only while these tensors live
    return StepGraph(int(h.value), (layers, pages, positions, new_lens, append_flags, workspace))


def pfkv_step_graph_launch(graph: StepGraph, stream=None) -> None:
    _check(lib().pfkv_step_graph_launch(graph.handle or None, _stream(stream)),
           "pfkv_step_graph_launch")


def pfkv_step_graph_destroy(graph: StepGraph) -> None:
    graph.close()


def pfkv_selftest_bounded_wait(result: torch.Tensor, stream=None) -> None:
    """result: int32 CUDA tensor of >= 1 element (see include/pfkv.h)."""
    _check(lib().pfkv_selftest_bounded_wait(_ptr(result), _stream(stream)),
           "pfkv_selftest_bounded_wait")


def pfkv_e4m3_encode(x: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    _check(lib().pfkv_e4m3_encode(_ptr(x), x.numel(), _ptr(out), _stream(stream)),
           "pfkv_e4m3_encode")


def pfkv_e4m3_decode(codes: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    _check(lib().pfkv_e4m3_decode(_ptr(codes), codes.numel(), _ptr(out), _stream(stream)),
           "pfkv_e4m3_decode")
