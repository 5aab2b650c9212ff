"""The kernels' bounded waits on a GPU: with the pipeline-wait limit lowered
to 1 ns (pa_set_pipeline_wait_limit_ns, a test-only entry point) a wait that
is not satisfied at once gives up, so decode (balanced schedule and fixed
splits) and both prefill kernels (tcgen05 and mma.sync) unwind: they record
PA_ERR_TIMEOUT in the device error word, drain the copies they issued (those
waits keep their 2 s limit), free their tensor memory and return.  Nothing
hangs and nothing faults; with the default limit restored the same calls
succeed and match the fp64 oracle, so the context stays usable."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (bits_to_torch, check_fp32, check_half, fill_both, gpu_decode, new_pool,
                         oracle_decode, oracle_pools, vmax_of)
from paged_kv_cache_270_gb300 import _native as N
from paged_kv_cache_270_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_270_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()


class short_waits:
    """Pipeline waits give up after 1 ns inside the block; the default after."""

    def __enter__(self):
        torch.cuda.synchronize()
        N.pa_set_pipeline_wait_limit_ns(1)

    def __exit__(self, *exc):
        torch.cuda.synchronize()
        N.pa_set_pipeline_wait_limit_ns(0)


def test_decode_timeout_then_recovery():
    w = W.make("llama3_70b_fp8_b", scale_down=4)  # 64 x 1024 tokens, FP8
    w.compute_fp8_scales()
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    q = w.q_bits()
    assert pool.device_error() == N.PA_OK
    with short_waits():
        for ns in (N.PA_SPLITS_BALANCED, 4):  # the balanced schedule, then fixed splits
            gpu_decode(w, pool, q, num_splits=ns)
            assert pool.device_error() == N.PA_ERR_TIMEOUT, f"num_splits={ns}"
    ref = oracle_decode(w, op, q)
    for ns in (N.PA_SPLITS_BALANCED, 4):
        out = gpu_decode(w, pool, q, num_splits=ns)
        assert pool.device_error() == N.PA_OK
        check_half(out, ref, vmax_of(w, op))
    check_fp32(gpu_decode(w, pool, q, out_dtype=torch.float32), ref)


def _prefill_case(kv_dtype, d, G, pairs, seed, Hkv=2):
    ctx = np.array([h + c for h, c in pairs], np.int32)
    chunks = np.array([c for _, c in pairs], np.int32)
    rng = np.random.default_rng(seed)
    nb = int(np.sum(-(-ctx // 16))) + 2
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.zeros((len(ctx), int(-(-ctx.max() // 16))), np.int32)
    used = 0
    for s, n in enumerate(ctx):
        k = -(-int(n) // 16)
        tables[s, :k] = perm[used:used + k]
        used += k
    w = W.Workload(name="timeout", index=13, kv_dtype=kv_dtype, n_q_heads=Hkv * G, n_kv_heads=Hkv,
                   head_dim=d, ctx_lens=ctx, num_blocks=nb, block_tables=tables, kv_seed=seed)
    w.compute_fp8_scales()
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    x = rng.standard_normal((int(chunks.sum()), w.n_q_heads, d)).astype(np.float32)
    qb = W.f32_to_f16_bits(x) if w.in_dtype == "fp16" else W.f32_to_bf16_bits(x)
    q_start = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    args = (bits_to_torch(qb, w.in_dtype), torch.from_numpy(q_start).cuda(),
            torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda())
    ref = oracle.paged_prefill(kv_dtype, w.in_dtype, nb, 16, Hkv, d, op[0], op[1], w.k_scale,
                               w.v_scale, qb, q_start, tables, ctx, w.softmax_scale)
    return w, pool, op, args, int(chunks.max()), ref


@pytest.mark.parametrize("kv_dtype,d,G", [("fp8_e4m3", 128, 8),   # the tcgen05 kernel
                                          ("bf16", 128, 4),       # the tcgen05 kernel, 16-bit
                                          ("fp16", 64, 2)])       # the mma.sync kernel
def test_prefill_timeout_then_recovery(kv_dtype, d, G):
    w, pool, op, args, max_chunk, ref = _prefill_case(kv_dtype, d, G, [(2000, 300), (500, 128)],
                                                      seed=17)
    assert pool.device_error() == N.PA_OK
    with short_waits():
        pool.prefill(*args, max_chunk=max_chunk, softmax_scale=w.softmax_scale)
        torch.cuda.synchronize()
        assert pool.device_error() == N.PA_ERR_TIMEOUT
    out = pool.prefill(*args, max_chunk=max_chunk, softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert pool.device_error() == N.PA_OK
    check_half(out, ref, vmax_of(w, op))


def test_default_limit_restored_by_zero():
    """0 sets the default back: a normal decode right after reports no error."""
    N.pa_set_pipeline_wait_limit_ns(0)
    w = W.make("tiny_fp16")
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    out = gpu_decode(w, pool, w.q_bits())
    assert pool.device_error() == N.PA_OK
    check_half(out, oracle_decode(w, op, w.q_bits()), vmax_of(w, op))
