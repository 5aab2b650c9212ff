"""Shared helpers for the GPU parity tests: fill a device pool through the
library and an oracle pool through the oracle from the same seeded inputs,
run both decodes, and compare with the stated tolerances.

Tolerances (from the decode specification):
  * cache bytes written by pa_reshape_and_cache / pa_copy_blocks: bit-exact;
  * bf16 / fp16 output: max |gpu - oracle| <= 1e-2 * max|V|, max|V| over the
    (dequantised) values the oracle reads;
  * fp32 output (check mode): per (sequence, query head) row,
    max_i |gpu - oracle| / max_i |oracle| <= 1e-4.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_270_gb300 import _native as N
from paged_kv_cache_270_gb300 import workloads as W
from paged_kv_cache_270_gb300.pool import KVPool

BF16_TOL = 1e-2
FP32_ROW_TOL = 1e-4


def bits_to_torch(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.float16 if dtype == "fp16" else torch.bfloat16)
    return t.to(device)


def new_pool(w: W.Workload, fill_byte: int | None = 0, num_blocks=None) -> KVPool:
    p = KVPool(1, num_blocks or w.num_blocks, w.n_kv_heads, w.head_dim, w.kv_dtype, w.k_scale,
               w.v_scale)
    if fill_byte is not None:
        p.k_cache.fill_(fill_byte)
        p.v_cache.fill_(fill_byte)
    return p


def oracle_pools(w: W.Workload, fill_byte: int = 0, num_blocks=None):
    nb = num_blocks or w.num_blocks
    n = oracle.pool_bytes(w.kv_dtype, nb, 16, w.n_kv_heads, w.head_dim)
    return np.full(n, fill_byte, np.uint8), np.full(n, fill_byte, np.uint8)


def fill_both(w: W.Workload, pool: KVPool | None, opools, seqs=None, ctx=None, tables=None,
              chunk_tokens=65536, num_blocks=None):
    """Write tokens [0, ctx[s]) of each sequence in `seqs` into the GPU pool
    (pa_reshape_and_cache) and the oracle pools (oracle.reshape_and_cache)."""
    seqs = range(w.S) if seqs is None else seqs
    ctx = w.ctx_lens if ctx is None else ctx
    tables = w.block_tables if tables is None else tables
    nb = num_blocks or w.num_blocks
    for s in seqs:
        n = int(ctx[s])
        for lo in range(0, n, chunk_tokens):
            hi = min(n, lo + chunk_tokens)
            k, v = w.kv_bits(s, lo, hi)
            pos = np.arange(lo, hi, dtype=np.int64)
            slots = tables[s, pos // 16].astype(np.int64) * 16 + pos % 16
            if pool is not None:
                pool.reshape_and_cache(bits_to_torch(k, w.in_dtype), bits_to_torch(v, w.in_dtype),
                                       torch.from_numpy(slots).cuda())
            if opools is not None:
                st = oracle.reshape_and_cache(w.kv_dtype, nb, 16, w.n_kv_heads, w.head_dim, k, v,
                                              slots, w.k_scale, w.v_scale, *opools)
                assert st == 0


def oracle_decode(w: W.Workload, opools, q_bits, ctx=None, tables=None, num_blocks=None):
    return oracle.paged_attention(w.kv_dtype, w.in_dtype, num_blocks or w.num_blocks, 16,
                                  w.n_kv_heads, w.head_dim, opools[0], opools[1], w.k_scale,
                                  w.v_scale, q_bits,
                                  w.block_tables if tables is None else tables,
                                  w.ctx_lens if ctx is None else ctx, w.softmax_scale)


def gpu_decode(w: W.Workload, pool: KVPool, q_bits, ctx=None, tables=None, out_dtype=None,
               num_splits=0):
    q = bits_to_torch(q_bits, w.in_dtype)
    t = torch.from_numpy(np.ascontiguousarray(w.block_tables if tables is None else tables,
                                              dtype=np.int32)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(w.ctx_lens if ctx is None else ctx,
                                              dtype=np.int32)).cuda()
    out = pool.decode(q, t, c, out_dtype=out_dtype, num_splits=num_splits,
                      softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    return out


def vmax_of(w: W.Workload, opools, num_blocks=None) -> float:
    """max |V| over the values the oracle reads (dequantised for FP8)."""
    vp = opools[1]
    if w.kv_dtype == "fp8_e4m3_block":
        nb = num_blocks or w.num_blocks
        n = oracle.tiles_bytes(w.kv_dtype, nb, 16, w.n_kv_heads, w.head_dim)
        table = np.abs(oracle.e4m3_table())
        table[np.isnan(table)] = 0
        sc = oracle.tile_scales(w.kv_dtype, nb, 16, w.n_kv_heads, w.head_dim, vp).astype(np.float64)
        sc[~np.isfinite(sc)] = 0
        tile_max = table[vp[:n].reshape(nb, w.n_kv_heads, -1)].max(axis=2)
        return float((tile_max * sc).max())
    if w.kv_dtype == "fp8_e4m3":
        table = np.abs(oracle.e4m3_table()) * w.v_scale
        table[np.isnan(table)] = 0
        return float(table[np.unique(vp)].max())
    bits = vp.view(np.uint16)
    vals = W.bits_to_f32(bits, w.in_dtype)
    vals = vals[np.isfinite(vals)]
    return float(np.abs(vals).max())


def check_half(out: torch.Tensor, ref: np.ndarray, vmax: float):
    got = out.float().cpu().double().numpy()
    err = np.abs(got - ref).max()
    assert np.all(np.isfinite(got)), "non-finite output"
    assert err <= BF16_TOL * vmax, f"max|err| {err:.3e} > 1e-2 * max|V| = {BF16_TOL * vmax:.3e}"
    return err


def check_fp32(out: torch.Tensor, ref: np.ndarray):
    got = out.cpu().double().numpy()
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - ref).max(axis=-1)
    scale = np.abs(ref).max(axis=-1)
    zero = scale == 0
    assert np.all(err[zero] == 0), "nonzero output where the oracle row is zero"
    rel = np.where(zero, 0.0, err / np.where(zero, 1.0, scale))
    worst = float(rel.max(initial=0.0))
    assert worst <= FP32_ROW_TOL, f"row relative error {worst:.3e} > 1e-4"
    return worst


def pool_bytes_equal(pool: KVPool, opools, blocks=None):
    """Bit-exact comparison of the device pool with the oracle pool (all blocks
    or the listed physical ids)."""
    for which, op in (("k", opools[0]), ("v", opools[1])):
        dev = pool.layer_view(which).cpu().numpy()
        ref = op[:dev.size].reshape(dev.shape)
        if blocks is not None:
            dev, ref = dev[blocks], ref[blocks]
        if not np.array_equal(dev, ref):
            bad = np.argwhere(dev != ref)
            raise AssertionError(f"{which} pool differs at {len(bad)} bytes, first {bad[:4]}")
        if pool.block_scaled:  # the tiles' scales, bit for bit
            ds = pool.scale_view(which).cpu().numpy().view(np.uint32)
            rs = oracle.tile_scales(pool.kv_dtype, pool.num_blocks, 16, pool.n_kv_heads,
                                    pool.head_dim, op).view(np.uint32)
            if blocks is not None:
                ds, rs = ds[blocks], rs[blocks]
            if not np.array_equal(ds, rs):
                bad = np.argwhere(ds != rs)
                raise AssertionError(f"{which} scales differ at {len(bad)} tiles, first {bad[:4]}")


def full_size_sampled_check(name, sample):
    """A full-size 70B-shaped decode in the launches the benchmark times (the
    automatic split count) and with the balanced schedule; the oracle
    checks the sampled sequences one by one: their blocks bit for bit (block
    scales too), their bf16 and fp32 outputs within tolerance."""
    w = W.make(name)
    w.compute_fp8_scales()
    pool = new_pool(w, None)
    fill_both(w, pool, None, chunk_tokens=1 << 17)
    q = w.q_bits()
    outs = [(gpu_decode(w, pool, q, num_splits=ns),
             gpu_decode(w, pool, q, out_dtype=torch.float32, num_splits=ns))
            for ns in (0, N.PA_SPLITS_BALANCED)]
    assert pool.device_error() == N.PA_OK
    for s in sample:
        n = int(w.ctx_lens[s])
        ids = w.block_tables[s, :-(-n // 16)]
        ow = W.Workload(**{**w.__dict__, "ctx_lens": w.ctx_lens[s:s + 1],
                           "block_tables": np.arange(len(ids), dtype=np.int32)[None, :],
                           "num_blocks": len(ids)})
        op = oracle_pools(ow, 0)
        for lo in range(0, n, 1 << 16):
            hi = min(n, lo + (1 << 16))
            k, v = w.kv_bits(s, lo, hi)
            oracle.reshape_and_cache(w.kv_dtype, len(ids), 16, w.n_kv_heads, w.head_dim, k, v,
                                     np.arange(lo, hi, dtype=np.int64), w.k_scale, w.v_scale, *op)
        ref = oracle_decode(ow, op, q[s:s + 1])
        for out, out32 in outs:
            check_half(out[s:s + 1], ref, vmax_of(ow, op))
            check_fp32(out32[s:s + 1], ref)
        tile = w.n_kv_heads * 16 * w.head_dim
        for which, o in (("k", op[0]), ("v", op[1])):
            dev = pool.layer_view(which)[torch.from_numpy(ids.astype(np.int64)).cuda()]
            assert np.array_equal(dev.cpu().numpy().ravel(), o[:len(ids) * tile]), \
                f"{which} cache bytes differ (sequence {s})"
            if w.block_scaled:
                dsc = pool.scale_view(which)[torch.from_numpy(ids.astype(np.int64)).cuda()]
                assert np.array_equal(dsc.cpu().numpy(),
                                      oracle.tile_scales(w.kv_dtype, len(ids), 16, w.n_kv_heads,
                                                         w.head_dim, o))
