"""GPU parity of block swap-out / swap-in to pinned host memory."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import fill_both, gpu_decode, new_pool
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


@pytest.mark.parametrize("kv_dtype,d", [("bf16", 128), ("fp8_e4m3", 128), ("fp16", 64)])
def test_swap_out_and_in_bit_exact(kv_dtype, d):
    L, nb, hkv = 3, 64, 4
    pool = KVPool(L, nb, hkv, d, kv_dtype, 0.5, 0.5)
    rng = np.random.default_rng(5)
    k_host = rng.integers(0, 256, pool.k_cache.numel(), dtype=np.uint8)
    v_host = rng.integers(0, 256, pool.v_cache.numel(), dtype=np.uint8)
    pool.k_cache.copy_(torch.from_numpy(k_host))
    pool.v_cache.copy_(torch.from_numpy(v_host))
    ids = np.array([7, 0, 63, 12, 12, 40], np.int32)
    per = pool.swap_block_bytes()
    buf = torch.zeros(len(ids) * per, dtype=torch.uint8).pin_memory()
    pool.swap_out(torch.from_numpy(ids).cuda(), buf)
    torch.cuda.synchronize()
    layer = k_host.size // L
    got = buf.numpy().reshape(len(ids), L, -1)
    for l in range(L):
        want = oracle.swap_gather(kv_dtype, nb, 16, hkv, d, ids, k_host[l * layer:(l + 1) * layer],
                                  v_host[l * layer:(l + 1) * layer]).reshape(len(ids), -1)
        assert np.array_equal(got[:, l, :], want)
    # swap back into other blocks, after wiping the pool
    pool.k_cache.fill_(0xEE)
    pool.v_cache.fill_(0xEE)
    dst = np.array([1, 2, 3, 4, 5, 6], np.int32)
    pool.swap_in(torch.from_numpy(dst).cuda(), buf)
    torch.cuda.synchronize()
    for l in range(L):
        kk = pool.layer_view("k", l).cpu().numpy().reshape(nb, -1)
        vv = pool.layer_view("v", l).cpu().numpy().reshape(nb, -1)
        src_k = k_host[l * layer:(l + 1) * layer].reshape(nb, -1)
        src_v = v_host[l * layer:(l + 1) * layer].reshape(nb, -1)
        for s, t in zip(ids, dst):
            assert np.array_equal(kk[t], src_k[s]) and np.array_equal(vv[t], src_v[s])
        assert np.all(kk[0] == 0xEE) and np.all(kk[7:] == 0xEE)
    assert pool.device_error() == N.PA_OK


def test_decode_after_swap_round_trip_is_bit_identical():
    """A sequence's pages go to host memory, the blocks are reused by someone
    else, and the pages come back into different blocks: same output."""
    w = W.make("llama3_8b_bf16", scale_down=8)
    pool = new_pool(w, 0)
    fill_both(w, pool, None)
    q = w.q_bits()
    before = gpu_decode(w, pool, q).cpu()
    s = 3
    nbk = -(-int(w.ctx_lens[s]) // 16)
    old = w.block_tables[s, :nbk].copy()
    buf = torch.empty(nbk * pool.swap_block_bytes(), dtype=torch.uint8).pin_memory()
    pool.swap_out(torch.from_numpy(old).cuda(), buf)
    # someone else overwrites those blocks
    pool.layer_view("k")[torch.from_numpy(old.astype(np.int64)).cuda()] = 0x7F
    pool.layer_view("v")[torch.from_numpy(old.astype(np.int64)).cuda()] = 0x7F
    new = np.array(w.spare_blocks[:nbk], np.int32)
    assert len(new) == nbk
    pool.swap_in(torch.from_numpy(new).cuda(), buf)
    tables = w.block_tables.copy()
    tables[s, :nbk] = new
    after = gpu_decode(w, pool, q, tables=tables).cpu()
    assert torch.equal(before.view(torch.int16), after.view(torch.int16))
    assert pool.device_error() == N.PA_OK


def test_swap_rejects_unpinned_and_flags_bad_ids():
    pool = KVPool(1, 8, 2, 64, "fp16")
    ids = torch.tensor([1, 2], dtype=torch.int32, device="cuda")
    pageable = np.zeros(2 * pool.swap_block_bytes(), np.uint8)  # kept alive for the call
    with pytest.raises(N.PAError):
        N.pa_swap_out(pool.handle, 2, ids.data_ptr(), pageable.ctypes.data, 0)
    assert np.all(pageable == 0)
    buf = torch.zeros(2 * pool.swap_block_bytes(), dtype=torch.uint8).pin_memory()
    pool.swap_out(torch.tensor([1, 8], dtype=torch.int32, device="cuda"), buf)
    assert pool.device_error() == N.PA_ERR_BOUNDS
