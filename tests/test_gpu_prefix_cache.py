"""Prefix caching end to end on the GPU: a request whose prompt starts with a
cached prefix reuses the cached blocks, writes and prefills only its own
tokens, and gets the same attention results as a request that prefilled
everything into private blocks."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import bits_to_torch, check_fp32, check_half
from paged_kv_cache_270_gb300 import _native as N
from paged_kv_cache_270_gb300 import workloads as W
from paged_kv_cache_270_gb300.pool import KVPool

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_270_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()


def _write(pool, k, v, table, lo, hi):
    pos = np.arange(lo, hi, dtype=np.int64)
    slots = np.asarray(table)[pos // 16].astype(np.int64) * 16 + pos % 16
    pool.reshape_and_cache(bits_to_torch(k, "bf16"), bits_to_torch(v, "bf16"),
                           torch.from_numpy(slots).cuda())


def test_cached_prefix_gives_identical_attention():
    ps = W.PrefixShare()
    P, X = 2048, 300
    rng = np.random.default_rng(12)
    prompt = rng.integers(0, 128000, P).astype(np.int32)
    suffix = rng.integers(0, 128000, X).astype(np.int32)
    kp, vp = ps.prefix_kv(P)
    ks, vs = ps.suffix_kv(0, X)
    k_all, v_all = np.concatenate([kp, ks]), np.concatenate([vp, vs])

    pool = KVPool(1, 512, 8, 128, "bf16")
    pool.k_cache.fill_(0xFF)
    pool.v_cache.fill_(0xFF)
    # request A: prefill the prompt, register its full blocks
    ha = N.pa_prefix_hash(prompt)
    assert len(pool.prefix_lookup(ha)) == 0
    ta = pool.alloc(len(ha))
    _write(pool, kp, vp, ta, 0, P)
    pool.prefix_register(ha, ta)
    torch.cuda.synchronize()
    cached_bytes = pool.layer_view("k")[torch.from_numpy(ta.astype(np.int64)).cuda()].clone()

    # request B: prompt + own tokens; leading blocks come from the cache
    hb = N.pa_prefix_hash(np.concatenate([prompt, suffix]))
    hit = pool.prefix_lookup(hb)
    assert np.array_equal(hit, ta)                       # 128 hits, same blocks
    nb = -(-(P + X) // 16)
    tb = np.concatenate([hit, pool.alloc(nb - len(hit))]).astype(np.int32)
    _write(pool, ks, vs, tb, P, P + X)                   # only B's own tokens
    assert pool.refcount(int(ta[0])) == 3                # A, B and the cache

    # reference pool: B's whole prompt in private blocks, no sharing
    ref = KVPool(1, 512, 8, 128, "bf16")
    ref.k_cache.fill_(0xFF)
    ref.v_cache.fill_(0xFF)
    tr = ref.alloc(nb)
    _write(ref, k_all, v_all, tr, 0, P + X)

    q = bits_to_torch(ps.q_bits(X)[:X], "bf16")          # B's chunk queries (X rows)
    qs = torch.tensor([0, X], dtype=torch.int32, device="cuda")
    ctx = torch.tensor([P + X], dtype=torch.int32, device="cuda")
    outs = {}
    for name, pl, tab in (("cached", pool, tb), ("private", ref, tr)):
        t = torch.from_numpy(np.asarray(tab, np.int32)[None, :]).cuda()
        pre = pl.prefill(q, qs, t, ctx, max_chunk=X, out_dtype=torch.float32)
        dec = pl.decode(q[-1:].contiguous(), t, ctx, out_dtype=torch.float32)
        outs[name] = (pre, dec)
    torch.cuda.synchronize()
    assert torch.equal(outs["cached"][0], outs["private"][0])
    assert torch.equal(outs["cached"][1], outs["private"][1])
    # the cached prefix blocks were not written by request B
    after = pool.layer_view("k")[torch.from_numpy(ta.astype(np.int64)).cuda()]
    assert torch.equal(after, cached_bytes)
    assert pool.device_error() == N.PA_OK and ref.device_error() == N.PA_OK

    # sampled rows against the oracle (a row of the chunk = a decode at its position)
    nbytes = oracle.pool_bytes("bf16", nb, 16, 8, 128)
    okp, ovp = np.zeros(nbytes, np.uint8), np.zeros(nbytes, np.uint8)
    oracle.reshape_and_cache("bf16", nb, 16, 8, 128, k_all, v_all,
                             np.arange(P + X, dtype=np.int64), 1.0, 1.0, okp, ovp)
    qb = ps.q_bits(X)[:X]
    vmax = float(np.abs(W.bits_to_f32(v_all, "bf16")).max())
    for j in (0, 1, 150, X - 1):
        r = oracle.paged_attention("bf16", "bf16", nb, 16, 8, 128, okp, ovp, 1.0, 1.0,
                                   qb[j:j + 1], np.arange(nb, dtype=np.int32)[None, :],
                                   np.array([P + j + 1], np.int32), 1.0 / np.sqrt(128))
        check_fp32(outs["cached"][0][j:j + 1], r)
        check_half(outs["cached"][0][j:j + 1].to(torch.bfloat16), r, vmax)

    # both requests finish: the prompt blocks stay cached until evicted
    pool.free(tb)
    pool.free(ta)
    assert pool.stats()[0] == len(ta)
    assert pool.prefix_evict(1 << 20) == len(ta)
    assert pool.stats() == (0, 512, 0)
