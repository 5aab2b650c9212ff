"""fp64 CPU oracle for paged KV-cache decode -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package.  The product (the CUDA library and its
Python binding) never imports, links or calls it, and the two share no code:
the oracle is ``pa_oracle.c`` (plain C, fp64, compiled here with gcc, no
fast-math) plus the pure-Python allocator model in ``allocator_model.py``.

This module only compiles ``pa_oracle.c`` and marshals numpy arrays into it.
What each routine computes, and the page passage it follows, is documented in
``pa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libpa_oracle.so")

# The oracle's own dtype codes (see pa_oracle.c).
F16, BF16, E4M3, E4M3_BLK = 0, 1, 2, 3
_DTYPE_CODES = {"fp16": F16, "bf16": BF16, "fp8_e4m3": E4M3, "fp8_e4m3_block": E4M3_BLK}
FP8_DTYPES = ("fp8_e4m3", "fp8_e4m3_block")

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into a shared library (gcc -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, f32, f64 = ctypes.c_int, ctypes.c_float, ctypes.c_double
        lib.or_f16_value.argtypes = [ctypes.c_uint16]
        lib.or_f16_value.restype = f64
        lib.or_bf16_value.argtypes = [ctypes.c_uint16]
        lib.or_bf16_value.restype = f64
        lib.or_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_value.restype = f64
        lib.or_e4m3_encode.argtypes = [f32]
        lib.or_e4m3_encode.restype = ctypes.c_uint8
        lib.or_quantize_e4m3.argtypes = [f64, f32]
        lib.or_quantize_e4m3.restype = ctypes.c_uint8
        lib.or_kv_bytes_per_token.argtypes = [i32, i32, i32, i32]
        lib.or_kv_bytes_per_token.restype = ctypes.c_longlong
        lib.or_reshape_and_cache.argtypes = [i32, i32, i32, i32, i32, P, P, P, i32, f32, f32, P, P]
        lib.or_reshape_and_cache.restype = i32
        lib.or_copy_blocks.argtypes = [i32, i32, i32, i32, i32, P, i32, P, P]
        lib.or_copy_blocks.restype = i32
        lib.or_paged_attention.argtypes = [i32, i32, i32, i32, i32, i32, P, P, f32, f32, P, i32,
                                           P, i32, P, i32, f64, P, P]
        lib.or_paged_attention.restype = i32
        lib.or_paged_prefill.argtypes = [i32, i32, i32, i32, i32, i32, P, P, f32, f32, P, i32, P,
                                          P, i32, P, i32, f64, P]
        lib.or_paged_prefill.restype = i32
        lib.or_swap_gather.argtypes = [i32, i32, i32, i32, i32, P, i32, P, P, P]
        lib.or_swap_gather.restype = i32
        lib.or_swap_record_bytes.argtypes = [i32, i32, i32, i32]
        lib.or_swap_record_bytes.restype = ctypes.c_longlong
        lib.or_slab_attention.argtypes = [P, P, i32, i32, i32, P, i32, P, i32, f64, P]
        lib.or_slab_attention.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def dtype_code(name: str) -> int:
    return _DTYPE_CODES[name]


# --------------------------------------------------------------------- scalars
def f16_value(bits: int) -> float:
    return _load().or_f16_value(bits)


def bf16_value(bits: int) -> float:
    return _load().or_bf16_value(bits)


def e4m3_value(code: int) -> float:
    return _load().or_e4m3_value(code)


def e4m3_encode(y: float) -> int:
    return _load().or_e4m3_encode(y)


def quantize_e4m3(x: float, scale: float) -> int:
    return _load().or_quantize_e4m3(x, scale)


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, d_head: int, precision_bytes: int) -> int:
    return _load().or_kv_bytes_per_token(n_layers, n_kv_heads, d_head, precision_bytes)


def value16(dtype: str, bits: np.ndarray) -> np.ndarray:
    """Decode an array of 16-bit patterns to fp64 through the oracle's decoders."""
    lib = _load()
    fn = lib.or_bf16_value if dtype == "bf16" else lib.or_f16_value
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    out = np.fromiter((fn(int(b)) for b in flat), dtype=np.float64, count=flat.size)
    return out.reshape(np.shape(bits))


def e4m3_table() -> np.ndarray:
    """fp64 value of each of the 256 E4M3 codes."""
    lib = _load()
    return np.array([lib.or_e4m3_value(c) for c in range(256)], dtype=np.float64)


# ---------------------------------------------------------------------- pools
def tiles_bytes(kv_dtype: str, num_blocks: int, block_size: int, n_kv_heads: int,
                head_dim: int) -> int:
    """Bytes of the code tiles of one K or V region."""
    b = 1 if kv_dtype in FP8_DTYPES else 2
    return num_blocks * n_kv_heads * block_size * head_dim * b


def pool_bytes(kv_dtype: str, num_blocks: int, block_size: int, n_kv_heads: int,
               head_dim: int) -> int:
    """Bytes of one K or V region: the tiles, then (block-scaled FP8) the fp32
    scale table [num_blocks][n_kv_heads]."""
    n = tiles_bytes(kv_dtype, num_blocks, block_size, n_kv_heads, head_dim)
    if kv_dtype == "fp8_e4m3_block":
        n += 4 * num_blocks * n_kv_heads
    return n


def tile_scales(kv_dtype: str, num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int,
                region: np.ndarray) -> np.ndarray:
    """The scale table of a block-scaled region, as float32 [num_blocks][n_kv_heads]."""
    assert kv_dtype == "fp8_e4m3_block"
    off = tiles_bytes(kv_dtype, num_blocks, block_size, n_kv_heads, head_dim)
    return region[off:off + 4 * num_blocks * n_kv_heads].view(np.float32).reshape(
        num_blocks, n_kv_heads)


def reshape_and_cache(kv_dtype: str, num_blocks: int, block_size: int, n_kv_heads: int,
                      head_dim: int, k_bits: np.ndarray, v_bits: np.ndarray,
                      slot_mapping: np.ndarray, k_scale: float, v_scale: float,
                      k_pool: np.ndarray, v_pool: np.ndarray) -> int:
    """Write tokens [T][Hkv][d] (16-bit patterns) into the byte pools in place."""
    k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert k_pool.dtype == np.uint8 and v_pool.dtype == np.uint8
    T = slots.shape[0]
    assert k_bits.size == T * n_kv_heads * head_dim
    return _load().or_reshape_and_cache(
        dtype_code(kv_dtype), num_blocks, block_size, n_kv_heads, head_dim, _ptr(k_bits),
        _ptr(v_bits), _ptr(slots), T, k_scale, v_scale, _ptr(k_pool), _ptr(v_pool))


def copy_blocks(kv_dtype: str, num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int,
                pairs: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray) -> int:
    pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    return _load().or_copy_blocks(dtype_code(kv_dtype), num_blocks, block_size, n_kv_heads,
                                  head_dim, _ptr(pairs), pairs.shape[0], _ptr(k_pool),
                                  _ptr(v_pool))


def paged_attention(kv_dtype: str, q_dtype: str, num_blocks: int, block_size: int,
                    n_kv_heads: int, head_dim: int, k_pool: np.ndarray, v_pool: np.ndarray,
                    k_scale: float, v_scale: float, q_bits: np.ndarray,
                    block_tables: np.ndarray, ctx_lens: np.ndarray, softmax_scale: float,
                    want_probs: bool = False):
    """fp64 paged decode attention; returns out [S][Hq][d] (and probs if asked)."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    S, Hq, d = q_bits.shape
    assert d == head_dim
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    out = np.zeros((S, Hq, d), dtype=np.float64)
    probs = None
    if want_probs:
        probs = np.zeros((S, Hq, max(int(ctx.max(initial=0)), 1)), dtype=np.float64)
    st = _load().or_paged_attention(
        dtype_code(kv_dtype), dtype_code(q_dtype), num_blocks, block_size, n_kv_heads, head_dim,
        _ptr(k_pool), _ptr(v_pool), k_scale, v_scale, _ptr(q_bits), Hq, _ptr(tables),
        tables.shape[1], _ptr(ctx), S, softmax_scale, _ptr(out), _ptr(probs))
    if st != 0:
        raise ValueError(f"oracle paged_attention status {st}")
    return (out, probs) if want_probs else out


def slab_attention(K: np.ndarray, V: np.ndarray, q: np.ndarray, ctx_lens: np.ndarray,
                   softmax_scale: float) -> np.ndarray:
    """Attention over contiguous K/V slabs [S][max_ctx][Hkv][d] (fp64)."""
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    q = np.ascontiguousarray(q, dtype=np.float64)
    ctx = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    S, max_ctx, Hkv, d = K.shape
    Hq = q.shape[1]
    out = np.zeros((S, Hq, d), dtype=np.float64)
    st = _load().or_slab_attention(_ptr(K), _ptr(V), max_ctx, Hkv, d, _ptr(q), Hq, _ptr(ctx), S,
                                   softmax_scale, _ptr(out))
    if st != 0:
        raise ValueError(f"oracle slab_attention status {st}")
    return out


def paged_prefill(kv_dtype: str, q_dtype: str, num_blocks: int, block_size: int, n_kv_heads: int,
                  head_dim: int, k_pool: np.ndarray, v_pool: np.ndarray, k_scale: float,
                  v_scale: float, q_bits: np.ndarray, q_start: np.ndarray,
                  block_tables: np.ndarray, ctx_lens: np.ndarray,
                  softmax_scale: float) -> np.ndarray:
    """fp64 causal attention of each chunk over its paged history; out [T][Hq][d]."""
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    T, Hq, d = q_bits.shape
    assert d == head_dim
    qs = np.ascontiguousarray(q_start, dtype=np.int32)
    tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    S = ctx.shape[0]
    assert qs.shape[0] == S + 1 and qs[-1] == T
    out = np.zeros((T, Hq, d), dtype=np.float64)
    st = _load().or_paged_prefill(
        dtype_code(kv_dtype), dtype_code(q_dtype), num_blocks, block_size, n_kv_heads, head_dim,
        _ptr(k_pool), _ptr(v_pool), k_scale, v_scale, _ptr(q_bits), Hq, _ptr(qs), _ptr(tables),
        tables.shape[1], _ptr(ctx), S, softmax_scale, _ptr(out))
    if st != 0:
        raise ValueError(f"oracle paged_prefill status {st}")
    return out


def swap_gather(kv_dtype: str, num_blocks: int, block_size: int, n_kv_heads: int, head_dim: int,
                ids: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray) -> np.ndarray:
    """One layer's swap buffer of blocks `ids`: per block its K tiles, its V tiles
    and, for block-scaled pools, its K and V scales padded to 16 bytes."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    rec = _load().or_swap_record_bytes(dtype_code(kv_dtype), block_size, n_kv_heads, head_dim)
    buf = np.zeros(rec * ids.size, np.uint8)
    st = _load().or_swap_gather(dtype_code(kv_dtype), num_blocks, block_size, n_kv_heads, head_dim,
                                _ptr(ids), ids.size, _ptr(k_pool), _ptr(v_pool), _ptr(buf))
    if st != 0:
        raise ValueError("oracle swap_gather: id out of range")
    return buf
