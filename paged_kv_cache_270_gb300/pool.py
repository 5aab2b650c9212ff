"""PyTorch-facing wrapper of the C ABI: device memory and streams come from
PyTorch, every computation from the library's CUDA kernels.

``KVPool`` owns the two device regions of a pool (as uint8 tensors) and the
library's pool handle, and forwards each call to the C entry point of the same
name with the tensors' device pointers and the current CUDA stream.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from . import _native as N

KV_DTYPES = {"fp16": N.PA_FP16, "bf16": N.PA_BF16, "fp8_e4m3": N.PA_FP8_E4M3,
             "fp8_e4m3_block": N.PA_FP8_E4M3_BLOCK}
_TORCH_OUT = {N.PA_FP16: torch.float16, N.PA_BF16: torch.bfloat16, N.PA_FP32: torch.float32}


def _stream_handle(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")


class KVPool:
    def __init__(self, n_layers: int, num_blocks: int, n_kv_heads: int, head_dim: int,
                 kv_dtype: str, k_scale: float = 1.0, v_scale: float = 1.0, device="cuda"):
        self.kv_dtype = kv_dtype
        self.code = KV_DTYPES[kv_dtype]
        self.desc = N.make_desc(n_layers, num_blocks, n_kv_heads, head_dim, self.code, k_scale,
                                v_scale)
        kb, vb = N.pa_pool_bytes(self.desc)
        self.device = torch.device(device)
        if self.device.type == "cuda" and self.device.index is None:
            self.device = torch.device("cuda", torch.cuda.current_device())
        self.k_cache = torch.empty(kb, dtype=torch.uint8, device=self.device)
        self.v_cache = torch.empty(vb, dtype=torch.uint8, device=self.device)
        self.handle = N.pa_pool_create(self.desc, self.k_cache.data_ptr(), self.v_cache.data_ptr())
        self.n_layers, self.num_blocks = n_layers, num_blocks
        self.n_kv_heads, self.head_dim = n_kv_heads, head_dim
        self.elem_bytes = 1 if kv_dtype in ("fp8_e4m3", "fp8_e4m3_block") else 2
        self.block_scaled = kv_dtype == "fp8_e4m3_block"
        # bytes of one layer's tiles in each region (a block-scaled region ends
        # with the scale table [n_layers][num_blocks][n_kv_heads] of fp32)
        self.layer_bytes = num_blocks * n_kv_heads * 16 * head_dim * self.elem_bytes
        self.in_dtype = torch.float16 if kv_dtype == "fp16" else torch.bfloat16
        self.in_code = N.PA_FP16 if kv_dtype == "fp16" else N.PA_BF16

    # ----------------------------------------------------------------- life
    def close(self):
        if getattr(self, "handle", None):
            N.pa_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ----------------------------------------------------------- allocator
    def alloc(self, n: int) -> np.ndarray:
        return N.pa_block_alloc(self.handle, n)

    def free(self, ids) -> None:
        N.pa_block_free(self.handle, ids)

    def incref(self, ids) -> None:
        N.pa_block_incref(self.handle, ids)

    def refcount(self, block: int) -> int:
        return N.pa_block_refcount(self.handle, block)

    def stats(self):
        return N.pa_pool_stats(self.handle)

    def cow_prepare(self, table_row: np.ndarray, ctx_len: int):
        return N.pa_cow_prepare(self.handle, table_row, ctx_len)

    # -------------------------------------------------------- prefix cache
    def prefix_lookup(self, hashes) -> np.ndarray:
        return N.pa_prefix_lookup(self.handle, hashes)

    def prefix_register(self, hashes, ids) -> None:
        N.pa_prefix_register(self.handle, hashes, ids)

    def prefix_evict(self, max_blocks: int) -> int:
        return N.pa_prefix_evict(self.handle, max_blocks)

    def prefix_stats(self):
        return N.pa_prefix_stats(self.handle)

    # --------------------------------------------------------------- views
    def layer_view(self, which: str, layer: int = 0) -> torch.Tensor:
        """uint8 view [num_blocks, n_kv_heads, 16, head_dim * elem_bytes] of one layer."""
        buf = self.k_cache if which == "k" else self.v_cache
        per = self.layer_bytes
        return buf[layer * per:(layer + 1) * per].view(self.num_blocks, self.n_kv_heads, 16,
                                                         self.head_dim * self.elem_bytes)

    def scale_view(self, which: str, layer: int = 0) -> torch.Tensor:
        """float32 view [num_blocks, n_kv_heads] of one layer's K or V tile scales
        (block-scaled FP8 pools)."""
        if not self.block_scaled:
            raise ValueError("only block-scaled FP8 pools keep per-tile scales")
        buf = self.k_cache if which == "k" else self.v_cache
        n = self.num_blocks * self.n_kv_heads * 4
        off = self.n_layers * self.layer_bytes + layer * n
        return buf[off:off + n].view(torch.float32).view(self.num_blocks, self.n_kv_heads)

    # --------------------------------------------------------- device calls
    def reshape_and_cache(self, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                          layer: int = 0, stream=None) -> None:
        _need(k, "k", self.in_dtype, self.device)
        _need(v, "v", self.in_dtype, self.device)
        _need(slot_mapping, "slot_mapping", torch.int64, self.device)
        T = slot_mapping.numel()
        if k.numel() != T * self.n_kv_heads * self.head_dim or v.numel() != k.numel():
            raise ValueError("k and v must be [T, n_kv_heads, head_dim]")
        N.pa_reshape_and_cache(self.handle, layer, k.data_ptr(), v.data_ptr(),
                               slot_mapping.data_ptr(), T, _stream_handle(stream))

    def copy_blocks(self, pairs: torch.Tensor, layer: int = 0, stream=None) -> None:
        _need(pairs, "pairs", torch.int32, self.device)
        N.pa_copy_blocks(self.handle, layer, pairs.data_ptr(), pairs.numel() // 2,
                         _stream_handle(stream))

    def swap_block_bytes(self) -> int:
        return N.pa_swap_block_bytes(self.handle)

    def swap_out(self, ids: torch.Tensor, host_buf: torch.Tensor, stream=None) -> None:
        """Copy blocks `ids` (device int32) into pinned host memory `host_buf`."""
        _need(ids, "ids", torch.int32, self.device)
        if not host_buf.is_pinned():
            raise ValueError("host_buf must be pinned host memory")
        if host_buf.numel() * host_buf.element_size() < ids.numel() * self.swap_block_bytes():
            raise ValueError("host_buf too small")
        N.pa_swap_out(self.handle, ids.numel(), ids.data_ptr(), host_buf.data_ptr(),
                      _stream_handle(stream))

    def swap_in(self, ids: torch.Tensor, host_buf: torch.Tensor, stream=None) -> None:
        """Copy a swap buffer back into blocks `ids` (device int32)."""
        _need(ids, "ids", torch.int32, self.device)
        if not host_buf.is_pinned():
            raise ValueError("host_buf must be pinned host memory")
        if host_buf.numel() * host_buf.element_size() < ids.numel() * self.swap_block_bytes():
            raise ValueError("host_buf too small")
        N.pa_swap_in(self.handle, ids.numel(), ids.data_ptr(), host_buf.data_ptr(),
                     _stream_handle(stream))

    def num_splits(self, S: int, n_q_heads: int, max_blocks_per_seq: int) -> int:
        return N.pa_decode_num_splits(self.handle, S, n_q_heads, max_blocks_per_seq)

    def workspace_bytes(self, S: int, n_q_heads: int, max_blocks_per_seq: int,
                        num_splits: int = 0) -> int:
        return N.pa_decode_workspace_bytes(self.handle, S, n_q_heads, max_blocks_per_seq,
                                           num_splits)

    def decode(self, q: torch.Tensor, block_tables: torch.Tensor, ctx_lens: torch.Tensor,
               out: torch.Tensor | None = None, out_dtype: torch.dtype | None = None,
               softmax_scale: float | None = None, num_splits: int = 0, layer: int = 0,
               workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        _need(q, "q", self.in_dtype, self.device)
        _need(block_tables, "block_tables", torch.int32, self.device)
        _need(ctx_lens, "ctx_lens", torch.int32, self.device)
        S, Hq, D = q.shape
        if D != self.head_dim:
            raise ValueError("q head_dim mismatch")
        max_blocks = block_tables.shape[1]
        if out is None:
            out = torch.empty((S, Hq, D), dtype=out_dtype or q.dtype, device=self.device)
        _need(out, "out", None, self.device)
        code = {v: k for k, v in _TORCH_OUT.items()}[out.dtype]
        if softmax_scale is None:
            softmax_scale = 1.0 / math.sqrt(D)
        ws_bytes = N.pa_decode_workspace_bytes(self.handle, S, Hq, max_blocks, num_splits)
        ws_ptr = 0
        if ws_bytes:
            if workspace is None or workspace.numel() * workspace.element_size() < ws_bytes:
                workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device)
            ws_ptr = workspace.data_ptr()
        N.pa_decode(self.handle, layer, out.data_ptr(), code, q.data_ptr(),
                    block_tables.data_ptr(), max_blocks, ctx_lens.data_ptr(), S, Hq,
                    float(softmax_scale), num_splits, ws_ptr, ws_bytes, _stream_handle(stream))
        return out

    def prefill(self, q: torch.Tensor, q_start: torch.Tensor, block_tables: torch.Tensor,
                ctx_lens: torch.Tensor, max_chunk: int, out: torch.Tensor | None = None,
                out_dtype: torch.dtype | None = None, softmax_scale: float | None = None,
                layer: int = 0, stream=None) -> torch.Tensor:
        """Causal attention of packed chunks q [T, Hq, D] (rows q_start[s] ..
        q_start[s+1]-1 for sequence s) over their paged history."""
        _need(q, "q", self.in_dtype, self.device)
        _need(q_start, "q_start", torch.int32, self.device)
        _need(block_tables, "block_tables", torch.int32, self.device)
        _need(ctx_lens, "ctx_lens", torch.int32, self.device)
        T, Hq, D = q.shape
        if out is None:
            out = torch.empty((T, Hq, D), dtype=out_dtype or q.dtype, device=self.device)
        _need(out, "out", None, self.device)
        code = {v: k for k, v in _TORCH_OUT.items()}[out.dtype]
        if softmax_scale is None:
            softmax_scale = 1.0 / math.sqrt(D)
        N.pa_prefill(self.handle, layer, out.data_ptr(), code, q.data_ptr(), q_start.data_ptr(),
                     block_tables.data_ptr(), block_tables.shape[1], ctx_lens.data_ptr(),
                     ctx_lens.numel(), Hq, int(max_chunk), float(softmax_scale),
                     _stream_handle(stream))
        return out

    def device_error(self, stream=None) -> int:
        return N.pa_get_device_error(self.handle, _stream_handle(stream))
