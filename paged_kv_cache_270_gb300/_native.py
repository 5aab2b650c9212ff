"""ctypes binding of ``libpagedkv.so`` -- argument marshalling only.

Every function here has the name of the C entry point it calls and does
nothing but convert Python arguments, call it, and raise ``PAError`` on a
non-zero status.  All device work happens inside the library's CUDA kernels.
There is no fallback: if the library has not been built, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

PA_OK = 0
PA_ERR_INVALID = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_OUT_OF_BLOCKS = 3
PA_ERR_NO_MEMORY = 4
PA_ERR_CUDA = 5
PA_ERR_BOUNDS = 6
PA_ERR_TIMEOUT = 7

PA_FP16 = 0
PA_BF16 = 1
PA_FP8_E4M3 = 2
PA_FP32 = 3
PA_FP8_E4M3_BLOCK = 4

PA_SPLITS_BALANCED = -1  # num_splits: the balanced decode schedule

ERROR_NAMES = {PA_OK: "PA_OK", PA_ERR_INVALID: "PA_ERR_INVALID",
               PA_ERR_UNSUPPORTED: "PA_ERR_UNSUPPORTED",
               PA_ERR_OUT_OF_BLOCKS: "PA_ERR_OUT_OF_BLOCKS", PA_ERR_NO_MEMORY: "PA_ERR_NO_MEMORY",
               PA_ERR_CUDA: "PA_ERR_CUDA", PA_ERR_BOUNDS: "PA_ERR_BOUNDS",
               PA_ERR_TIMEOUT: "PA_ERR_TIMEOUT"}


class PAError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{ERROR_NAMES.get(code, code)}: {msg}")
        self.code = code


class pa_pool_desc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("num_blocks", ctypes.c_int),
                ("block_size", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("kv_dtype", ctypes.c_int),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


_lock = threading.Lock()
_lib = None

# (name, argtypes) of every exported entry point, in header order.
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_SIGS = [
    ("pa_last_error", [ctypes.c_char_p, _SZ]),
    ("pa_kv_bytes_per_token", [_I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    ("pa_pool_bytes", [ctypes.POINTER(pa_pool_desc), ctypes.POINTER(_SZ), ctypes.POINTER(_SZ)]),
    ("pa_pool_blocks_for_budget", [ctypes.POINTER(pa_pool_desc), _SZ, ctypes.POINTER(_I)]),
    ("pa_pool_create", [ctypes.POINTER(pa_pool_desc), _P, _P, ctypes.POINTER(_P)]),
    ("pa_pool_destroy", [_P]),
    ("pa_pool_get_desc", [_P, ctypes.POINTER(pa_pool_desc)]),
    ("pa_block_alloc", [_P, _I, _P]),
    ("pa_block_free", [_P, _I, _P]),
    ("pa_block_incref", [_P, _I, _P]),
    ("pa_block_refcount", [_P, ctypes.c_int32, ctypes.POINTER(_I)]),
    ("pa_pool_stats", [_P, ctypes.POINTER(_I), ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    ("pa_cow_prepare", [_P, _P, _I, ctypes.POINTER(ctypes.c_int32),
                        ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(_I)]),
    ("pa_prefix_hash", [_P, _I, ctypes.c_uint64, _P, ctypes.POINTER(_I)]),
    ("pa_prefix_lookup", [_P, _I, _P, _P, ctypes.POINTER(_I)]),
    ("pa_prefix_register", [_P, _I, _P, _P]),
    ("pa_prefix_evict", [_P, _I, ctypes.POINTER(_I)]),
    ("pa_prefix_stats", [_P, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_longlong),
                         ctypes.POINTER(ctypes.c_longlong)]),
    ("pa_copy_blocks", [_P, _I, _P, _I, _P]),
    ("pa_swap_block_bytes", [_P, ctypes.POINTER(_SZ)]),
    ("pa_swap_out", [_P, _I, _P, _P, _P]),
    ("pa_swap_in", [_P, _I, _P, _P, _P]),
    ("pa_reshape_and_cache", [_P, _I, _P, _P, _P, _I, _P]),
    ("pa_decode_num_splits", [_P, _I, _I, _I, ctypes.POINTER(_I)]),
    ("pa_decode_workspace_bytes", [_P, _I, _I, _I, _I, ctypes.POINTER(_SZ)]),
    ("pa_decode", [_P, _I, _P, _I, _P, _P, _I, _P, _I, _I, ctypes.c_float, _I, _P, _SZ, _P]),
    ("pa_prefill", [_P, _I, _P, _I, _P, _P, _P, _I, _P, _I, _I, _I, ctypes.c_float, _P]),
    ("pa_decode_no_alloc", [_P, _I, _P, _I, _P, _P, _I, _P, _I, _I, ctypes.c_float, _I, _P]),
    ("pa_set_pipeline_wait_limit_ns", [ctypes.c_uint64]),
    ("pa_get_device_error", [_P, ctypes.POINTER(_I), _P]),
]

PA_NOALLOC_SCRATCH_BYTES = 8 << 20


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded library.  Raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with "
                               "`python -m paged_kv_cache_270_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(path)
        for name, args in _SIGS:
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        _lib = L
        return L


def last_error() -> str:
    buf = ctypes.create_string_buffer(512)
    lib().pa_last_error(buf, 512)
    return buf.value.decode(errors="replace")


def _check(status: int) -> None:
    if status != PA_OK:
        raise PAError(status, last_error())


def _arr_ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def make_desc(n_layers, num_blocks, n_kv_heads, head_dim, kv_dtype, k_scale=1.0, v_scale=1.0,
              block_size=16) -> pa_pool_desc:
    return pa_pool_desc(n_layers, num_blocks, block_size, n_kv_heads, head_dim, kv_dtype,
                        k_scale, v_scale)


# ------------------------------------------------------------------ host calls
def pa_kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, kv_dtype: int) -> int:
    out = _SZ()
    _check(lib().pa_kv_bytes_per_token(n_layers, n_kv_heads, head_dim, kv_dtype, ctypes.byref(out)))
    return out.value


def pa_pool_bytes(desc: pa_pool_desc):
    k, v = _SZ(), _SZ()
    _check(lib().pa_pool_bytes(ctypes.byref(desc), ctypes.byref(k), ctypes.byref(v)))
    return k.value, v.value


def pa_pool_blocks_for_budget(desc: pa_pool_desc, budget_bytes: int) -> int:
    n = _I()
    _check(lib().pa_pool_blocks_for_budget(ctypes.byref(desc), budget_bytes, ctypes.byref(n)))
    return n.value


def pa_pool_create(desc: pa_pool_desc, k_cache_ptr: int, v_cache_ptr: int) -> int:
    h = _P()
    _check(lib().pa_pool_create(ctypes.byref(desc), k_cache_ptr, v_cache_ptr, ctypes.byref(h)))
    return h.value


def pa_pool_destroy(pool: int) -> None:
    _check(lib().pa_pool_destroy(pool))


def pa_pool_get_desc(pool: int) -> pa_pool_desc:
    d = pa_pool_desc()
    _check(lib().pa_pool_get_desc(pool, ctypes.byref(d)))
    return d


def pa_block_alloc(pool: int, n: int) -> np.ndarray:
    ids = np.zeros(max(n, 0), np.int32)
    _check(lib().pa_block_alloc(pool, n, _arr_ptr(ids)))
    return ids


def pa_block_free(pool: int, ids) -> None:
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    _check(lib().pa_block_free(pool, ids.size, _arr_ptr(ids)))


def pa_block_incref(pool: int, ids) -> None:
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    _check(lib().pa_block_incref(pool, ids.size, _arr_ptr(ids)))


def pa_block_refcount(pool: int, block: int) -> int:
    rc = _I()
    _check(lib().pa_block_refcount(pool, block, ctypes.byref(rc)))
    return rc.value


def pa_pool_stats(pool: int):
    u, f, s = _I(), _I(), _I()
    _check(lib().pa_pool_stats(pool, ctypes.byref(u), ctypes.byref(f), ctypes.byref(s)))
    return u.value, f.value, s.value


def pa_cow_prepare(pool: int, table_row: np.ndarray, ctx_len: int):
    """Returns (src, dst) and rewrites table_row (int32, in place), or None."""
    assert table_row.dtype == np.int32 and table_row.flags["C_CONTIGUOUS"]
    src, dst, n = ctypes.c_int32(), ctypes.c_int32(), _I()
    _check(lib().pa_cow_prepare(pool, _arr_ptr(table_row), ctx_len, ctypes.byref(src),
                                ctypes.byref(dst), ctypes.byref(n)))
    return (src.value, dst.value) if n.value else None


def pa_prefix_hash(tokens, parent: int = 0) -> np.ndarray:
    """Chain hashes (uint64) of the full 16-token blocks of `tokens`."""
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    out = np.zeros(max(tokens.size // 16, 1), np.uint64)
    n = _I()
    _check(lib().pa_prefix_hash(_arr_ptr(tokens) if tokens.size else None, tokens.size,
                                ctypes.c_uint64(parent), _arr_ptr(out), ctypes.byref(n)))
    return out[:n.value]


def pa_prefix_lookup(pool: int, hashes) -> np.ndarray:
    """Block ids of the leading cached blocks (each gains a reference)."""
    hashes = np.ascontiguousarray(hashes, dtype=np.uint64)
    ids = np.zeros(max(hashes.size, 1), np.int32)
    n = _I()
    _check(lib().pa_prefix_lookup(pool, hashes.size, _arr_ptr(hashes), _arr_ptr(ids),
                                  ctypes.byref(n)))
    return ids[:n.value]


def pa_prefix_register(pool: int, hashes, ids) -> None:
    hashes = np.ascontiguousarray(hashes, dtype=np.uint64)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    assert hashes.size == ids.size
    _check(lib().pa_prefix_register(pool, hashes.size, _arr_ptr(hashes) if hashes.size else None,
                                    _arr_ptr(ids) if ids.size else None))


def pa_prefix_evict(pool: int, max_blocks: int) -> int:
    n = _I()
    _check(lib().pa_prefix_evict(pool, max_blocks, ctypes.byref(n)))
    return n.value


def pa_prefix_stats(pool: int):
    e, lk, h = _I(), ctypes.c_longlong(), ctypes.c_longlong()
    _check(lib().pa_prefix_stats(pool, ctypes.byref(e), ctypes.byref(lk), ctypes.byref(h)))
    return e.value, lk.value, h.value


# ---------------------------------------------------------------- device calls
def pa_copy_blocks(pool: int, layer: int, pairs_ptr: int, n_pairs: int, stream: int) -> None:
    _check(lib().pa_copy_blocks(pool, layer, pairs_ptr, n_pairs, stream))


def pa_swap_block_bytes(pool: int) -> int:
    n = _SZ()
    _check(lib().pa_swap_block_bytes(pool, ctypes.byref(n)))
    return n.value


def pa_swap_out(pool: int, n: int, ids_ptr: int, host_ptr: int, stream: int) -> None:
    _check(lib().pa_swap_out(pool, n, ids_ptr, host_ptr, stream))


def pa_swap_in(pool: int, n: int, ids_ptr: int, host_ptr: int, stream: int) -> None:
    _check(lib().pa_swap_in(pool, n, ids_ptr, host_ptr, stream))


def pa_reshape_and_cache(pool: int, layer: int, k_ptr: int, v_ptr: int, slot_mapping_ptr: int,
                         T: int, stream: int) -> None:
    _check(lib().pa_reshape_and_cache(pool, layer, k_ptr, v_ptr, slot_mapping_ptr, T, stream))


def pa_decode_num_splits(pool: int, S: int, n_q_heads: int, max_blocks_per_seq: int) -> int:
    n = _I()
    _check(lib().pa_decode_num_splits(pool, S, n_q_heads, max_blocks_per_seq, ctypes.byref(n)))
    return n.value


def pa_decode_workspace_bytes(pool: int, S: int, n_q_heads: int, max_blocks_per_seq: int,
                              num_splits: int = 0) -> int:
    n = _SZ()
    _check(lib().pa_decode_workspace_bytes(pool, S, n_q_heads, max_blocks_per_seq, num_splits,
                                           ctypes.byref(n)))
    return n.value


def pa_decode(pool: int, layer: int, out_ptr: int, out_dtype: int, q_ptr: int, tables_ptr: int,
              max_blocks_per_seq: int, ctx_lens_ptr: int, S: int, n_q_heads: int,
              softmax_scale: float, num_splits: int, workspace_ptr: int, workspace_bytes: int,
              stream: int) -> None:
    _check(lib().pa_decode(pool, layer, out_ptr, out_dtype, q_ptr, tables_ptr, max_blocks_per_seq,
                           ctx_lens_ptr, S, n_q_heads, softmax_scale, num_splits, workspace_ptr,
                           workspace_bytes, stream))


def pa_prefill(pool: int, layer: int, out_ptr: int, out_dtype: int, q_ptr: int, q_start_ptr: int,
               tables_ptr: int, max_blocks_per_seq: int, ctx_lens_ptr: int, S: int,
               n_q_heads: int, max_chunk: int, softmax_scale: float, stream: int) -> None:
    _check(lib().pa_prefill(pool, layer, out_ptr, out_dtype, q_ptr, q_start_ptr, tables_ptr,
                            max_blocks_per_seq, ctx_lens_ptr, S, n_q_heads, max_chunk,
                            softmax_scale, stream))


def pa_decode_no_alloc(pool: int, layer: int, out_ptr: int, out_dtype: int, q_ptr: int,
                       tables_ptr: int, max_blocks_per_seq: int, ctx_lens_ptr: int, S: int,
                       n_q_heads: int, softmax_scale: float, num_splits: int, stream: int) -> None:
    _check(lib().pa_decode_no_alloc(pool, layer, out_ptr, out_dtype, q_ptr, tables_ptr,
                                    max_blocks_per_seq, ctx_lens_ptr, S, n_q_heads, softmax_scale,
                                    num_splits, stream))


def pa_set_pipeline_wait_limit_ns(ns: int) -> None:
    """Test-only: the limit of the kernels' pipeline waits in ns (0 = the default 2 s)."""
    _check(lib().pa_set_pipeline_wait_limit_ns(int(ns)))


def pa_get_device_error(pool: int, stream: int) -> int:
    code = _I()
    _check(lib().pa_get_device_error(pool, ctypes.byref(code), stream))
    return code.value
