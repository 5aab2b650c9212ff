"""GPU parity of the guided split layout: the automatic split count s of a
launch that takes more than one wave of CTAs becomes min(2 s, 8) splits whose
sizes fall geometrically (ratio 0.55), with the split index as the slowest grid
dimension, so the last CTAs handed out are the short last splits.  Checked
against the fp64 oracle on the 8B-shaped ragged FP8 batch (where the automatic
count is 8 guided splits) and on ragged batches of every pool type with empty
contexts, beside an explicit uniform split count on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (check_fp32, check_half, fill_both, gpu_decode, new_pool, oracle_decode,
                         oracle_pools, vmax_of)
from paged_kv_cache_270_gb300 import _native as N
from paged_kv_cache_270_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_270_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()


def test_guided_layout_on_the_8b_ragged_batch():
    w = W.make("llama3_8b_fp8")
    w.compute_fp8_scales()
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    # 64 x 8 units over 258 table columns: four uniform splits (2048 CTAs, more
    # than one wave), so the automatic layout is eight guided splits
    assert pool.num_splits(w.S, w.n_q_heads, w.max_blocks) == 8
    assert pool.workspace_bytes(w.S, w.n_q_heads, w.max_blocks, 0) == \
        w.S * w.n_q_heads * 8 * (w.head_dim + 2) * 4
    q = w.q_bits()
    ref = oracle_decode(w, op, q)
    vmax = vmax_of(w, op)
    outs = []
    for _ in range(3):
        outs.append(gpu_decode(w, pool, q))
    check_half(outs[0], ref, vmax)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    check_fp32(gpu_decode(w, pool, q, out_dtype=torch.float32), ref)
    check_half(gpu_decode(w, pool, q, num_splits=8), ref, vmax)  # the same count, uniform
    assert pool.device_error() == N.PA_OK


def _ragged(kv_dtype, S, Hkv, G, d, seed):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1, 3000, S).astype(np.int32)
    ctx[::37] = 0
    ctx[1] = 3000
    need = -(-ctx // 16)
    nb = int(need.sum()) + 5
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.zeros((S, int(need.max())), np.int32)
    used = 0
    for s, k in enumerate(need):
        tables[s, :k] = perm[used:used + k]
        used += int(k)
    return W.Workload(name="guided", index=9, kv_dtype=kv_dtype, n_q_heads=Hkv * G, n_kv_heads=Hkv,
                      head_dim=d, ctx_lens=ctx, num_blocks=nb, block_tables=tables, kv_seed=seed)


@pytest.mark.parametrize("kv_dtype,d,G", [("fp16", 64, 2), ("bf16", 128, 4), ("fp8_e4m3", 128, 8),
                                          ("fp8_e4m3_block", 128, 8)])
def test_guided_layout_ragged_with_empty_contexts(kv_dtype, d, G):
    w = _ragged(kv_dtype, 96, 8, G, d, seed=41)  # several waves at the automatic count: guided
    w.compute_fp8_scales()
    pool = new_pool(w, 0xFF)
    op = oracle_pools(w, 0xFF)
    fill_both(w, pool, op)
    q = w.q_bits()
    ref = oracle_decode(w, op, q)
    vmax = vmax_of(w, op)
    n = pool.num_splits(w.S, w.n_q_heads, w.max_blocks)
    assert 2 <= n <= 8
    out = gpu_decode(w, pool, q)
    check_half(out, ref, vmax)
    for s in np.flatnonzero(w.ctx_lens == 0):
        assert torch.all(out[s] == 0)
    check_fp32(gpu_decode(w, pool, q, out_dtype=torch.float32), ref)
    check_half(gpu_decode(w, pool, q, num_splits=3), ref, vmax)
    assert pool.device_error() == N.PA_OK
