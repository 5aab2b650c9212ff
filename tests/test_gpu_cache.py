"""GPU parity of the cache-writing kernels: pa_reshape_and_cache (16-bit copy
and FP8 E4M3 quantisation) and pa_copy_blocks, bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_harness import bits_to_torch, fill_both, new_pool, oracle_pools, pool_bytes_equal
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


@pytest.mark.parametrize("name,sd", [("tiny_fp16", 1), ("llama3_8b_bf16", 8),
                                     ("llama3_8b_fp8", 8), ("llama3_70b_fp8_b", 64)])
def test_reshape_bit_exact(name, sd):
    w = W.make(name, scale_down=sd, steps=1) if name == "llama3_8b_fp8" else W.make(name, sd)
    w.compute_fp8_scales()
    pool = new_pool(w, 0)
    op = oracle_pools(w, 0)
    fill_both(w, pool, op)
    torch.cuda.synchronize()
    pool_bytes_equal(pool, op)
    assert pool.device_error() == N.PA_OK


@pytest.mark.parametrize("scale", [1.0, 0.125, float(np.float32(4.75) / np.float32(448.0)),
                                   float(np.float32(1e-3))])
def test_fp8_quantiser_all_bf16_patterns(scale):
    """Every bf16 bit pattern (NaN excluded: parity unpinned) through the cache
    quantiser: codes must equal the oracle's E4M3 RNE-satfinite codes."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = W.bits_to_f32(bits, "bf16")
    bits = bits[~np.isnan(f)]
    T, Hkv, d = 0, 1, 128
    pad = (-bits.size) % d
    bits = np.concatenate([bits, np.zeros(pad, np.uint16)])
    T = bits.size // d
    k = bits.reshape(T, Hkv, d)
    v = k[::-1].copy()
    nb = (T + 15) // 16
    pool = KVPool(1, nb, Hkv, d, "fp8_e4m3", scale, scale)
    pool.k_cache.zero_()
    pool.v_cache.zero_()
    slots = np.arange(T, dtype=np.int64)
    pool.reshape_and_cache(bits_to_torch(k, "bf16"), bits_to_torch(v, "bf16"),
                           torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    kp = np.zeros(nb * 16 * d, np.uint8)
    vp = np.zeros_like(kp)
    oracle.reshape_and_cache("fp8_e4m3", nb, 16, Hkv, d, k, v, slots, scale, scale, kp, vp)
    assert np.array_equal(pool.k_cache.cpu().numpy(), kp)
    assert np.array_equal(pool.v_cache.cpu().numpy(), vp)


def test_reshape_skips_negative_and_flags_out_of_range():
    w = W.make("tiny_fp16")
    pool = new_pool(w, 0x5A)
    op = oracle_pools(w, 0x5A)
    k, v = w.kv_bits(0, 0, 4)
    slots = np.array([3, -1, 17, w.num_blocks * 16 + 5], np.int64)
    pool.reshape_and_cache(bits_to_torch(k, "fp16"), bits_to_torch(v, "fp16"),
                           torch.from_numpy(slots).cuda())
    assert pool.device_error() == N.PA_ERR_BOUNDS
    assert pool.device_error() == N.PA_OK  # reading clears it
    st = oracle.reshape_and_cache("fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim, k, v, slots,
                                  1.0, 1.0, *op)
    assert st == -1
    pool_bytes_equal(pool, op)


def test_reshape_multi_layer_offsets():
    w = W.make("tiny_fp16")
    pool = KVPool(3, w.num_blocks, w.n_kv_heads, w.head_dim, "fp16")
    pool.k_cache.zero_()
    pool.v_cache.zero_()
    k, v = w.kv_bits(1, 0, 20)
    slots = w.slots(1, 0, 20)
    pool.reshape_and_cache(bits_to_torch(k, "fp16"), bits_to_torch(v, "fp16"),
                           torch.from_numpy(slots).cuda(), layer=1)
    torch.cuda.synchronize()
    op = oracle_pools(w, 0)
    oracle.reshape_and_cache("fp16", w.num_blocks, 16, w.n_kv_heads, w.head_dim, k, v, slots, 1, 1,
                             *op)
    assert np.array_equal(pool.layer_view("k", 1).cpu().numpy().ravel(), op[0])
    assert not pool.layer_view("k", 0).any() and not pool.layer_view("k", 2).any()


@pytest.mark.parametrize("kv_dtype,d", [("fp16", 64), ("bf16", 128), ("fp8_e4m3", 128)])
def test_copy_blocks_bit_exact(kv_dtype, d):
    nb, hkv = 40, 4
    pool = KVPool(2, nb, hkv, d, kv_dtype, 0.5, 0.25)
    g = torch.Generator(device="cpu").manual_seed(9)
    init_k = torch.randint(0, 256, (pool.k_cache.numel(),), generator=g, dtype=torch.uint8)
    init_v = torch.randint(0, 256, (pool.v_cache.numel(),), generator=g, dtype=torch.uint8)
    pool.k_cache.copy_(init_k)
    pool.v_cache.copy_(init_v)
    pairs = np.array([[3, 9], [5, 0], [39, 12]], np.int32)
    pool.copy_blocks(torch.from_numpy(pairs).cuda(), layer=1)
    torch.cuda.synchronize()
    per = init_k.numel() // 2
    kp = init_k.numpy()[per:].copy()
    vp = init_v.numpy()[per:].copy()
    oracle.copy_blocks(kv_dtype, nb, 16, hkv, d, pairs, kp, vp)
    assert np.array_equal(pool.layer_view("k", 1).cpu().numpy().ravel(), kp)
    assert np.array_equal(pool.layer_view("v", 1).cpu().numpy().ravel(), vp)
    # layer 0 untouched
    assert np.array_equal(pool.layer_view("k", 0).cpu().numpy().ravel(), init_k.numpy()[:per])
    bad = torch.tensor([[1, nb]], dtype=torch.int32, device="cuda")
    pool.copy_blocks(bad)
    assert pool.device_error() == N.PA_ERR_BOUNDS
