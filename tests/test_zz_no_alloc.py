"""pa_decode_no_alloc: the decode entry point for callers that cannot allocate
device memory (a plugin whose host framework owns every allocation, a serving
loop that must not allocate once running).  It keeps its split partials in a
fixed array inside the library instead of a caller workspace.

Checked here through the C ABI: two calls in a row, on different shapes, each
bit for bit against pa_decode with a caller workspace and the same schedule,
and against the fp64 oracle within the tolerances the other decode tests use;
an automatic split count that must be lowered to fit the fixed array; and the
clear error for an explicit split count whose partials exceed it.  This file is
collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import (check_fp32, check_half, fill_both, new_pool, oracle_decode, oracle_pools,
                         vmax_of)
from paged_kv_cache_270_gb300 import _native as N
from paged_kv_cache_270_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_kv_cache_270_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    oracle.build()


def _inputs(w):
    q = torch.from_numpy(w.q_bits().view(np.int16)).view(torch.bfloat16).cuda()
    if w.in_dtype == "fp16":
        q = q.view(torch.float16)
    t = torch.from_numpy(np.ascontiguousarray(w.block_tables, np.int32)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(w.ctx_lens, np.int32)).cuda()
    return q, t, c


def _both(w, pool, q, t, c, out_dtype, num_splits):
    """(pa_decode with a workspace, pa_decode_no_alloc) for the same call."""
    S, Hq, D = q.shape
    code = {torch.float32: N.PA_FP32, torch.bfloat16: N.PA_BF16, torch.float16: N.PA_FP16}
    stream = torch.cuda.current_stream().cuda_stream
    ws_bytes = N.pa_decode_workspace_bytes(pool.handle, S, Hq, t.shape[1], num_splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    ref = torch.empty((S, Hq, D), dtype=out_dtype, device="cuda")
    got = torch.full((S, Hq, D), float("nan"), dtype=out_dtype, device="cuda")
    N.pa_decode(pool.handle, 0, ref.data_ptr(), code[out_dtype], q.data_ptr(), t.data_ptr(),
                t.shape[1], c.data_ptr(), S, Hq, w.softmax_scale, num_splits, ws.data_ptr(),
                ws_bytes, stream)
    N.pa_decode_no_alloc(pool.handle, 0, got.data_ptr(), code[out_dtype], q.data_ptr(),
                         t.data_ptr(), t.shape[1], c.data_ptr(), S, Hq, w.softmax_scale,
                         num_splits, stream)
    torch.cuda.synchronize()
    return ref, got


def _same_bits(a, b):
    """Bit-for-bit equality of two outputs of the same dtype."""
    view = torch.int32 if a.dtype == torch.float32 else torch.int16
    return torch.equal(a.view(view), b.view(view))


def test_no_alloc_matches_decode_on_two_calls_in_a_row():
    # call 1: long FP8 contexts split 24 ways (partials in the fixed array)
    w1 = W.make("llama3_70b_fp8_a", scale_down=16)
    w1.compute_fp8_scales()
    p1 = new_pool(w1, 0)
    op1 = oracle_pools(w1, 0)
    fill_both(w1, p1, op1)
    q1, t1, c1 = _inputs(w1)
    want1 = oracle_decode(w1, op1, w1.q_bits())
    ref, got = _both(w1, p1, q1, t1, c1, torch.bfloat16, 24)
    assert _same_bits(got, ref)
    check_half(got, want1, vmax_of(w1, op1))
    ref32, got32 = _both(w1, p1, q1, t1, c1, torch.float32, 24)
    assert _same_bits(got32, ref32)
    check_fp32(got32, want1)

    # call 2: another shape and dtype right after, the balanced schedule, the
    # automatic split count and fixed splits; stale partials of call 1 are still
    # in the array and must not leak in
    w2 = W.make("llama3_8b_bf16", scale_down=4)
    p2 = new_pool(w2, 0)
    op2 = oracle_pools(w2, 0)
    fill_both(w2, p2, op2)
    q2, t2, c2 = _inputs(w2)
    want2 = oracle_decode(w2, op2, w2.q_bits())
    for ns in (N.PA_SPLITS_BALANCED, 0, 3):
        ref, got = _both(w2, p2, q2, t2, c2, torch.bfloat16, ns)
        assert _same_bits(got, ref)
        check_half(got, want2, vmax_of(w2, op2))
        ref32, got32 = _both(w2, p2, q2, t2, c2, torch.float32, ns)
        assert _same_bits(got32, ref32)
        check_fp32(got32, want2)
    assert p1.device_error() == N.PA_OK


def test_no_alloc_lowers_an_automatic_split_count_to_fit():
    """The automatic split count here is two uniform splits (4100 single-head
    sequences against 760 resident CTAs, every one taken as 2048 pages long),
    which pa_decode runs as four guided splits; neither's partials (2 x 4100 x
    8 heads x (128 + 2) floats, 34 MB, for two) fit the 8 MiB array, so the
    entry point takes the largest uniform count that fits (one split, no
    partials), and matches pa_decode at that count."""
    rng = np.random.default_rng(31)
    S, Hkv, G, d, max_blocks = 4100, 1, 8, 128, 2048
    ctx = rng.integers(1, 60, S).astype(np.int32)
    need = -(-ctx // 16)
    nb = int(need.sum())
    perm = rng.permutation(nb).astype(np.int32)
    tables = np.zeros((S, max_blocks), np.int32)
    used = 0
    for s, k in enumerate(need):
        tables[s, :k] = perm[used:used + k]
        used += int(k)
    w = W.Workload(name="lowered", index=9, kv_dtype="fp8_e4m3", n_q_heads=Hkv * G,
                   n_kv_heads=Hkv, head_dim=d, ctx_lens=ctx, num_blocks=nb, block_tables=tables,
                   kv_seed=31)
    w.compute_fp8_scales()
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    q, t, c = _inputs(w)
    auto = N.pa_decode_num_splits(pool.handle, S, w.n_q_heads, max_blocks)
    per_split = S * w.n_q_heads * (d + 2) * 4
    assert auto >= 2 and auto * per_split > N.PA_NOALLOC_SCRATCH_BYTES, \
        f"the automatic count ({auto}) should need more than the array here"
    fit = max(s for s in range(1, auto + 1)
              if N.pa_decode_workspace_bytes(pool.handle, S, w.n_q_heads, max_blocks, s)
              <= N.PA_NOALLOC_SCRATCH_BYTES)
    stream = torch.cuda.current_stream().cuda_stream
    got = torch.full((S, w.n_q_heads, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    N.pa_decode_no_alloc(pool.handle, 0, got.data_ptr(), N.PA_BF16, q.data_ptr(), t.data_ptr(),
                         max_blocks, c.data_ptr(), S, w.n_q_heads, w.softmax_scale, 0, stream)
    ref = pool.decode(q, t, c, num_splits=fit, softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert _same_bits(got, ref)
    rows = np.sort(rng.choice(S, 64, replace=False))
    sub = W.Workload(**{**w.__dict__, "ctx_lens": ctx[rows], "block_tables": tables[rows]})
    want = oracle_decode(sub, op, w.q_bits()[rows])
    check_half(got[torch.from_numpy(rows).cuda()], want, vmax_of(w, op))
    assert pool.device_error() == N.PA_OK


def test_no_alloc_rejects_scratch_beyond_its_maximum():
    w = W.make("tiny_fp16")
    pool = new_pool(w, 0)
    S, Hq, D, max_blocks = 4096, 4, 64, 4096
    per_split = S * Hq * (D + 2) * 4
    too_many = N.PA_NOALLOC_SCRATCH_BYTES // per_split + 1
    with pytest.raises(N.PAError) as e:
        # rejected on the host before anything is launched (pointers unused)
        N.pa_decode_no_alloc(pool.handle, 0, 16, N.PA_FP16, 16, 16, max_blocks, 16, S, Hq, 0.125,
                             too_many, 0)
    assert e.value.code == N.PA_ERR_INVALID
    assert "static maximum" in str(e.value)
