"""CPU oracle for paged FP8/BF16 KV-cache decode attention (test infrastructure).

Only tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  It shares no code with the CUDA library: the C source
``oracle.c`` is written from the method's definition (see its header for the
cited passages and the readings taken where the pages are silent).

All arrays are host numpy arrays.  bf16 tensors travel as their uint16 bit
patterns, e4m3 tensors as uint8 codes.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

FLAG_TAG = 1
FLAG_PAGE = 2
FLAG_LEN = 4
PAGE_SIZE = 16


class _Cache(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("k_pages", ctypes.c_void_p), ("v_pages", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("page_tags", ctypes.c_void_p)]


class _Pages(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("block_tables", ctypes.c_void_p),
                ("bt_stride_b", ctypes.c_int64), ("bt_stride_h", ctypes.c_int64),
                ("seq_lens", ctypes.c_void_p),
                ("len_stride_b", ctypes.c_int64), ("len_stride_h", ctypes.c_int64),
                ("expected_tags", ctypes.c_void_p)]


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_e4m3_to_double.restype = ctypes.c_double
        L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_from_float.restype = ctypes.c_uint8
        L.oracle_e4m3_from_float.argtypes = [ctypes.c_float]
        L.oracle_e4m3_encode_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        L.oracle_e4m3_decode_array.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
        L.oracle_unit_scale.restype = ctypes.c_float
        L.oracle_unit_scale.argtypes = [ctypes.c_float]
        L.oracle_quantize.restype = ctypes.c_uint8
        L.oracle_quantize.argtypes = [ctypes.c_float, ctypes.c_float]
        L.oracle_kv_append.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Pages),
                                       ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_validate.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Pages),
                                      ctypes.c_int32, ctypes.c_void_p]
        L.oracle_paged_decode.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Pages),
                                          ctypes.c_void_p, ctypes.c_int32, ctypes.c_double,
                                          ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
        L.oracle_attention_mass.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Pages),
                                            ctypes.c_void_p, ctypes.c_int32, ctypes.c_double,
                                            ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                                            ctypes.c_int64]
        L.oracle_paged_decode_multi.argtypes = [ctypes.POINTER(_Cache), ctypes.POINTER(_Pages),
                                                ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                                ctypes.c_double, ctypes.c_int32, ctypes.c_void_p,
                                                ctypes.c_void_p]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _need(a, dtype, name):
    if a is None:
        return None
    if not isinstance(a, np.ndarray) or a.dtype != dtype or not a.flags.c_contiguous:
        raise TypeError(f"{name}: expected a C-contiguous numpy array of {np.dtype(dtype)}")
    return a


# --------------------------------------------------------------------------
# e4m3 codec
# --------------------------------------------------------------------------
def e4m3_to_double(code: int) -> float:
    return lib().oracle_e4m3_to_double(int(code) & 0xFF)


def e4m3_from_float(x: float) -> int:
    return int(lib().oracle_e4m3_from_float(float(x)))


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape, dtype=np.float64)
    lib().oracle_e4m3_decode_array(_ptr(codes), codes.size, _ptr(out))
    return out


def unit_scale(absmax: float) -> float:
    return lib().oracle_unit_scale(float(absmax))


def quantize(x: float, scale: float) -> int:
    return int(lib().oracle_quantize(float(x), float(scale)))


# --------------------------------------------------------------------------
# paged cache
# --------------------------------------------------------------------------
def _cache(num_pages, num_kv_heads, head_dim, dtype, k_pages, v_pages, k_scale, v_scale,
           page_tags):
    pool_t = np.uint16 if dtype == 0 else np.uint8
    _need(k_pages, pool_t, "k_pages")
    _need(v_pages, pool_t, "v_pages")
    if dtype == 1:
        _need(k_scale, np.float32, "k_scale")
        _need(v_scale, np.float32, "v_scale")
    _need(page_tags, np.uint32, "page_tags")
    return _Cache(int(num_pages), int(num_kv_heads), int(head_dim), int(dtype),
                  _ptr(k_pages), _ptr(v_pages), _ptr(k_scale) if dtype == 1 else None,
                  _ptr(v_scale) if dtype == 1 else None, _ptr(page_tags))


def _pages(batch, max_pages, block_tables, bt_stride_b, bt_stride_h, seq_lens, len_stride_b,
           len_stride_h, expected_tags):
    _need(block_tables, np.int32, "block_tables")
    _need(seq_lens, np.int32, "seq_lens")
    _need(expected_tags, np.uint32, "expected_tags")
    return _Pages(int(batch), int(max_pages), _ptr(block_tables), int(bt_stride_b),
                  int(bt_stride_h), _ptr(seq_lens), int(len_stride_b), int(len_stride_h),
                  _ptr(expected_tags))


def kv_append(cache: dict, pages: dict, positions, k_new, v_new, new_lens=None, flags=None):
    """Write new tokens into the pool arrays of ``cache`` in place (see oracle.c).

    cache: num_pages, num_kv_heads, head_dim, dtype (0 bf16, 1 e4m3), k_pages,
           v_pages, k_scale, v_scale, page_tags (None: untracked)
    pages: batch, max_pages, block_tables, bt_stride_b, bt_stride_h, seq_lens,
           len_stride_b, len_stride_h, expected_tags (None: untracked)
    positions/new_lens: int32, indexed with the length strides.
    k_new/v_new: uint16 bf16 bits [B][Hkv][T][D].  flags: uint8 [B], OR-ed.
    Returns flags.
    """
    c = _cache(**cache)
    p = _pages(**pages)
    _need(positions, np.int32, "positions")
    _need(new_lens, np.int32, "new_lens")
    _need(k_new, np.uint16, "k_new")
    _need(v_new, np.uint16, "v_new")
    T = int(k_new.shape[2])
    if flags is None:
        flags = np.zeros(int(pages["batch"]), dtype=np.uint8)
    _need(flags, np.uint8, "flags")
    lib().oracle_kv_append(ctypes.byref(c), ctypes.byref(p), _ptr(positions), T, _ptr(new_lens),
                           _ptr(k_new), _ptr(v_new), _ptr(flags))
    return flags


def validate(cache: dict, pages: dict, max_seq_len: int) -> np.ndarray:
    c = _cache(**cache)
    p = _pages(**pages)
    flags = np.zeros(max(int(pages["batch"]), 1), dtype=np.uint8)
    lib().oracle_validate(ctypes.byref(c), ctypes.byref(p), int(max_seq_len), _ptr(flags))
    return flags[: int(pages["batch"])]


def paged_decode(cache: dict, pages: dict, q, num_q_heads: int, sm_scale: float,
                 max_seq_len: int):
    """fp64 decode attention.  q: uint16 bf16 bits [B][Hq][D].  Returns (out fp64, flags)."""
    c = _cache(**cache)
    p = _pages(**pages)
    _need(q, np.uint16, "q")
    B = int(pages["batch"])
    D = int(cache["head_dim"])
    out = np.zeros((B, int(num_q_heads), D), dtype=np.float64)
    flags = np.zeros(max(B, 1), dtype=np.uint8)
    lib().oracle_paged_decode(ctypes.byref(c), ctypes.byref(p), _ptr(q), int(num_q_heads),
                              float(sm_scale), int(max_seq_len), _ptr(out), _ptr(flags))
    return out, flags[:B]


def attention_mass(cache: dict, pages: dict, q, num_q_heads: int, sm_scale: float,
                   max_seq_len: int, mass=None, mass_strides=None):
    """fp64 attention mass (see oracle.c): adds, for each (b, h, j), the sum
    over the group's query heads of token j's softmax weight to ``mass``
    (float64, C-contiguous; default zeros [B][Hkv][max_seq_len]).  Returns mass."""
    c = _cache(**cache)
    p = _pages(**pages)
    _need(q, np.uint16, "q")
    B, H = int(pages["batch"]), int(cache["num_kv_heads"])
    if mass is None:
        mass = np.zeros((B, H, max(int(max_seq_len), 1)), dtype=np.float64)
    _need(mass, np.float64, "mass")
    sb, sh = mass_strides if mass_strides is not None else (mass.strides[0] // 8, mass.strides[1] // 8)
    lib().oracle_attention_mass(ctypes.byref(c), ctypes.byref(p), _ptr(q), int(num_q_heads),
                                float(sm_scale), int(max_seq_len), _ptr(mass), int(sb), int(sh))
    return mass


def paged_decode_multi(cache: dict, pages: dict, q, num_q_heads: int, kq: int,
                       sm_scale: float, max_seq_len: int):
    """fp64 multi-query verify (see oracle.c).  q: uint16 bf16 bits
    [B][kq][Hq][D].  Returns (out fp64 [B][kq][Hq][D], flags)."""
    c = _cache(**cache)
    p = _pages(**pages)
    _need(q, np.uint16, "q")
    B = int(pages["batch"])
    D = int(cache["head_dim"])
    out = np.zeros((B, int(kq), int(num_q_heads), D), dtype=np.float64)
    flags = np.zeros(max(B, 1), dtype=np.uint8)
    lib().oracle_paged_decode_multi(ctypes.byref(c), ctypes.byref(p), _ptr(q), int(num_q_heads),
                                    int(kq), float(sm_scale), int(max_seq_len), _ptr(out),
                                    _ptr(flags))
    return out, flags[:B]


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))
