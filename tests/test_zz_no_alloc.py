"""pa_decode_no_alloc: the decode entry point for callers that cannot allocate
device memory (a plugin whose host framework owns every allocation, a serving
loop that must not allocate once running).  It keeps its split partials in a
fixed array inside the library instead of a caller workspace.

Checked here through the C ABI: two calls in a row, on different shapes, each
against pa_decode with a caller workspace and the same split count, within the
tolerances the other decode tests use; and the clear error for a split count
whose partials exceed the fixed array.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import check_fp32, check_half, fill_both, new_pool, oracle_pools, vmax_of
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


def _as_ref(t):
    return t.double().cpu().numpy()


def test_no_alloc_matches_decode_on_two_calls_in_a_row():
    # call 1: long FP8 contexts split 24 ways (partials in the fixed array)
    w1 = W.make("llama3_70b_fp8_a", scale_down=16)
    w1.compute_fp8_scales()
    p1 = new_pool(w1, 0)
    op1 = oracle_pools(w1, 0)
    fill_both(w1, p1, op1)
    q1, t1, c1 = _inputs(w1)
    ref, got = _both(w1, p1, q1, t1, c1, torch.bfloat16, 24)
    check_half(got, _as_ref(ref), vmax_of(w1, op1))
    ref32, got32 = _both(w1, p1, q1, t1, c1, torch.float32, 24)
    check_fp32(got32, _as_ref(ref32))

    # call 2: another shape and dtype right after, automatic splits; stale
    # partials of call 1 are still in the array and must not leak in
    w2 = W.make("llama3_8b_bf16", scale_down=4)
    p2 = new_pool(w2, 0)
    op2 = oracle_pools(w2, 0)
    fill_both(w2, p2, op2)
    q2, t2, c2 = _inputs(w2)
    for ns in (0, 3):
        ref, got = _both(w2, p2, q2, t2, c2, torch.bfloat16, ns)
        check_half(got, _as_ref(ref), vmax_of(w2, op2))
    ref32, got32 = _both(w2, p2, q2, t2, c2, torch.float32, 3)
    check_fp32(got32, _as_ref(ref32))
    assert p1.device_error() == N.PA_OK


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
