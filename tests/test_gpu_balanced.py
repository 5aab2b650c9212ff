"""GPU parity of the balanced decode schedule (num_splits = PA_SPLITS_BALANCED,
batches of up to 4096 sequences) against the fp64 oracle.

The schedule cuts the pages of every (sequence, kv head) unit, in order, into
equal contiguous ranges, one per CTA, so one unit may be spread over hundreds
of CTAs (merged by the job kernel) and one CTA may finish dozens of short
units.  These cases drive both extremes and contexts of zero anywhere in the batch,
against fixed splits on the same inputs."""
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


def _workload(ctx, kv_dtype="fp8_e4m3", Hkv=8, G=8, d=128, seed=0, extra_cols=1):
    ctx = np.asarray(ctx, np.int32)
    rng = np.random.default_rng([seed, 77])
    need = -(-np.maximum(ctx, 0) // 16)
    nb = int(need.sum()) + 3
    perm = rng.permutation(nb).astype(np.int32)
    max_blocks = int(need.max(initial=1)) + extra_cols
    tables = np.zeros((len(ctx), max_blocks), np.int32)
    used = 0
    for s, k in enumerate(need):
        tables[s, :k] = perm[used:used + k]
        tables[s, k:] = rng.integers(-7, 10**6, max_blocks - k)  # never read
        used += int(k)
    return W.Workload(name="balanced", index=9, kv_dtype=kv_dtype, n_q_heads=Hkv * G, n_kv_heads=Hkv,
                      head_dim=d, ctx_lens=ctx, num_blocks=nb, block_tables=tables, kv_seed=seed)


BAL = N.PA_SPLITS_BALANCED


def _check(w, splits=(BAL,), fill=0xFF):
    w.compute_fp8_scales()
    pool = new_pool(w, fill)  # fill None: the device pool keeps whatever it held
    op = oracle_pools(w, 0 if fill is None else fill)
    fill_both(w, pool, op)
    q = w.q_bits()
    ref = oracle_decode(w, op, q)
    vmax = vmax_of(w, op)
    outs = {}
    for ns in splits:
        out = gpu_decode(w, pool, q, num_splits=ns)
        check_half(out, ref, vmax)
        check_fp32(gpu_decode(w, pool, q, out_dtype=torch.float32, num_splits=ns), ref)
        outs[ns] = out
    assert pool.device_error() == N.PA_OK
    return pool, outs


def test_balanced_schedule_sizes():
    w = _workload([100] * 4)
    pool = new_pool(w, 0)
    assert pool.num_splits(4, w.n_q_heads, w.max_blocks) >= 1  # the automatic choice: fixed splits
    # the balanced workspace: two partial slots and one job per CTA, four CTAs per SM at most
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    ws = pool.workspace_bytes(4, w.n_q_heads, w.max_blocks, BAL)
    per_cta = 2 * w.G * (w.head_dim + 2) * 4 + 16
    assert ws % per_cta == 0 and sms <= ws // per_cta <= 4 * sms
    with pytest.raises(N.PAError) as e:
        pool.workspace_bytes(4097, w.n_q_heads, w.max_blocks, BAL)
    assert e.value.code == N.PA_ERR_UNSUPPORTED


@pytest.mark.parametrize("kv_dtype", ["fp16", "bf16", "fp8_e4m3", "fp8_e4m3_block"])
def test_ragged_with_empty_contexts(kv_dtype):
    """Lengths from 0 to 3000 with empty contexts first, in the middle and
    last; every output against the oracle, balanced and fixed splits."""
    rng = np.random.default_rng(5)
    ctx = rng.integers(1, 3000, 40)
    ctx[[0, 7, 8, 39]] = 0
    ctx[[3, 4]] = [1, 16]
    G = 4 if kv_dtype in ("fp16", "bf16") else 8
    w = _workload(ctx, kv_dtype=kv_dtype, Hkv=4, G=G, d=128 if kv_dtype != "fp16" else 64, seed=11)
    pool, outs = _check(w, splits=(BAL, 3))
    for s in (0, 7, 8, 39):
        assert torch.all(outs[BAL][s] == 0)


def test_one_unit_spread_over_hundreds_of_ctas():
    """One kv head of one 131072-token sequence: 8192 pages, so every CTA of
    the launch holds a piece of the one unit and the merge job combines
    hundreds of partials (several rounds of 128)."""
    w = _workload([131072], kv_dtype="fp8_e4m3", Hkv=1, G=8, d=128, seed=3)
    _check(w, fill=None)


def test_long_and_short_sequences_mixed():
    """A few long sequences among many short ones (the case a split count
    chosen for the longest sequence serves badly)."""
    ctx = [40000, 17, 33, 2, 65536, 500, 1, 0, 3000, 16] * 3
    w = _workload(ctx, kv_dtype="bf16", Hkv=2, G=4, d=128, seed=4)
    _check(w, splits=(BAL, 7), fill=None)


def test_many_short_units_per_cta():
    """3000 sequences of 1 to 48 tokens: each CTA finishes dozens of units
    (one merge of its warps and one output row per unit)."""
    rng = np.random.default_rng(8)
    ctx = rng.integers(1, 49, 3000)
    ctx[::97] = 0
    w = _workload(ctx, kv_dtype="fp8_e4m3", Hkv=8, G=2, d=64, seed=8)
    _check(w)


def test_balanced_equals_itself_under_block_relabelling():
    """The schedule depends on the context lengths only, so relabelling the
    physical blocks leaves the output bit-identical."""
    rng = np.random.default_rng(12)
    ctx = rng.integers(0, 2000, 50)
    w = _workload(ctx, kv_dtype="fp8_e4m3", Hkv=8, G=8, d=128, seed=12, extra_cols=0)
    w.compute_fp8_scales()
    pool = new_pool(w, 0)
    fill_both(w, pool, None)
    q = w.q_bits()
    out = gpu_decode(w, pool, q, num_splits=BAL).cpu()
    perm = np.random.default_rng(13).permutation(w.num_blocks)
    pool2 = new_pool(w, 0)
    for which in ("k", "v"):
        pool2.layer_view(which)[torch.from_numpy(perm).cuda()] = pool.layer_view(which)
    tables2 = w.block_tables.copy()
    for s, n in enumerate(w.ctx_lens):
        k = -(-int(n) // 16)
        tables2[s, :k] = perm[w.block_tables[s, :k]]
    out2 = gpu_decode(w, pool2, q, tables=tables2, num_splits=BAL).cpu()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_bad_ids_and_lengths_are_reported():
    w = _workload([40, 300, 5], kv_dtype="fp8_e4m3", Hkv=2, G=4, d=128, seed=2)
    w.compute_fp8_scales()
    pool = new_pool(w, 0)
    fill_both(w, pool, None)
    q = w.q_bits()
    tables = w.block_tables.copy()
    tables[1, 3] = w.num_blocks + 5
    gpu_decode(w, pool, q, tables=tables, num_splits=BAL)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    gpu_decode(w, pool, q, ctx=np.array([40, 16 * w.max_blocks + 1, 5], np.int32), num_splits=BAL)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    gpu_decode(w, pool, q, ctx=np.array([40, -3, 5], np.int32), num_splits=BAL)
    assert pool.device_error() == N.PA_ERR_BOUNDS
    gpu_decode(w, pool, q, num_splits=BAL)
    assert pool.device_error() == N.PA_OK


def test_one_long_sequence_among_short_ones():
    """The 8B-shaped FP8 batch of one 131072-token sequence among 127 short ones,
    scaled down 16 times (one of 8192 tokens among 7 short): balanced and the
    automatic split count against the oracle, every row."""
    w = W.make("llama3_8b_fp8_long_short", scale_down=16)
    _check(w, splits=(BAL, 0))
