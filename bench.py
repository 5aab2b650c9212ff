#!/usr/bin/env python
"""Paged decode benchmark on GB300: KV-read HBM GB/s and decode tokens/s.

Workload (default): Llama-3.1-70B-shaped single-layer decode over an FP8 E4M3
paged KV cache -- 64 query heads, 8 KV heads, head dim 128, 16-token blocks,
block tables random permutations of the pool -- in two batches:
  A: 4 sequences x 131,072 tokens  (long context; split along the pages)
  B: 256 sequences x 4,096 tokens
One step = for each batch: pa_reshape_and_cache of the step's new token of
every sequence (quantised into its slot) then pa_decode of one query token per
sequence against its whole context.  The pool (3 GiB) is larger than L2, so
no flush is needed between steps.

Output: one JSON line (rank 0).  `value` = K+V bytes the decode reads per
step / step time.  `e2e` = the same metric measured through the C ABI with the
step's inputs copied from pinned host memory and the output read back, every
step.  `--impl reference` times the fp64 CPU oracle on a bounded sample of the
same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import multiprocessing as mp
import os
import re
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = ("paged decode: KV-read HBM GB/s (% of GB300 peak) and decode tokens/s, 1 GPU")
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

WORKLOADS = {
    "llama3_70b_fp8": ["llama3_70b_fp8_a", "llama3_70b_fp8_b"],
    "llama3_70b_fp8_a": ["llama3_70b_fp8_a"],
    "llama3_70b_fp8_b": ["llama3_70b_fp8_b"],
    "llama3_70b_fp8_block": ["llama3_70b_fp8_block_a", "llama3_70b_fp8_block_b"],
    "llama3_70b_fp8_block_a": ["llama3_70b_fp8_block_a"],
    "llama3_70b_fp8_block_b": ["llama3_70b_fp8_block_b"],
    "llama3_8b_bf16": ["llama3_8b_bf16"],
    "llama3_8b_fp8": ["llama3_8b_fp8"],
    "llama3_8b_fp8_long_short": ["llama3_8b_fp8_long_short"],
    "llama3_70b_fp8_prefill": ["llama3_70b_fp8_prefill"],
    "prefix_cache_bf16": ["prefix_cache_bf16"],
    "kv_swap_fp8": ["kv_swap_fp8"],
}
SWAP_METRIC = "KV page swap to host memory: GB/s out + in (gather / scatter of blocks), 1 GPU"
PREFIX_METRIC = ("prefill with block-hash prefix caching: prompt tokens served per second "
                 "(shared 2048-token system prompt), 1 GPU")
PREFILL_METRIC = "chunked prefill attention over a paged FP8 KV cache: TFLOP/s, 1 GPU"
DESCRIPTION = {
    "llama3_70b_fp8": "Llama-3.1-70B-shaped single-layer decode, FP8 E4M3 paged KV (per-tensor "
                      "scales amax/448), Hq 64 / Hkv 8 / d 128, 16-token blocks, random block "
                      "tables; batch A 4 x 131072 tokens + batch B 256 x 4096 tokens",
    "llama3_70b_fp8_a": "Llama-3.1-70B-shaped FP8 decode, 4 x 131072 tokens",
    "llama3_70b_fp8_b": "Llama-3.1-70B-shaped FP8 decode, 256 x 4096 tokens",
    "llama3_70b_fp8_block": "Llama-3.1-70B-shaped single-layer decode, FP8 E4M3 paged KV with a "
                            "dynamic scale per (block, kv head) tile (MaxAbs/448 taken as tokens "
                            "are written), Hq 64 / Hkv 8 / d 128, 16-token blocks, random block "
                            "tables; batch A 4 x 131072 tokens + batch B 256 x 4096 tokens",
    "llama3_70b_fp8_block_a": "Llama-3.1-70B-shaped block-scaled FP8 decode, 4 x 131072 tokens",
    "llama3_70b_fp8_block_b": "Llama-3.1-70B-shaped block-scaled FP8 decode, 256 x 4096 tokens",
    "llama3_8b_bf16": "Llama-3.1-8B-shaped bf16 decode, 64 seqs, ctx U[512,4096]",
    "llama3_8b_fp8": "Llama-3.1-8B-shaped FP8 decode, 64 seqs, ctx U[512,4096], 1% K outliers",
    "llama3_8b_fp8_long_short": "Llama-3.1-8B-shaped FP8 decode, one 131072-token sequence among "
                                "127 of U[128,1024] tokens",
    "kv_swap_fp8": "Llama-3.1-70B-shaped FP8 pool (Hkv 8, d 128, 16384 blocks of 32 KiB): each "
                   "step swaps 8192 scattered blocks (256 MiB) out to pinned host memory and back "
                   "into 8192 other blocks",
    "prefix_cache_bf16": "Llama-3.1-8B-shaped bf16 (Hq 32 / Hkv 8 / d 128): 64 requests whose "
                         "prompts share a 2048-token system prompt, each with its own U[128,1024] "
                         "suffix; a step hashes and looks up every prompt, writes and prefills "
                         "only the uncached tokens, then releases the requests",
    "llama3_70b_fp8_prefill": "Llama-3.1-70B-shaped chunked prefill, FP8 E4M3 paged KV, Hq 64 / "
                              "Hkv 8 / d 128: 4 sequences each prefilling a 2048-token chunk after "
                              "6144 cached tokens (one 8192-token packet), causal",
}

# DRAM traffic per decode launch from one ncu capture, valid only while the
# decode source (its code: comments and blank lines do not count) is the one
# measured.
NCU_TRAFFIC = {
    # hash of the decode source with comments and blank lines removed (see _source_sha)
    "source_sha256": "1fffa0627ca9a67c2af353fbfdac22678835d4f261f9384f609d9a64fae42a63",
    # dram__bytes_read.sum + dram__bytes_write.sum of one decode launch
    "bytes_per_launch": {"llama3_70b_fp8_a": 1073987328 + 3501568,
                         "llama3_70b_fp8_b": 2151997952 + 4874240,
                         "llama3_70b_fp8_block_a": 1076081664 + 2970112,
                         "llama3_70b_fp8_block_b": 2156272128 + 4859136},
}

# --------------------------------------------------------------------- workers
def _gen_amax(args):
    name, s, lo, hi = args
    from paged_kv_cache_270_gb300 import workloads as W
    w = W.make(name)
    k, v = w.kv_bits(s, lo, hi)
    return (float(np.abs(W.bits_to_f32(k, w.in_dtype)).max(initial=0)),
            float(np.abs(W.bits_to_f32(v, w.in_dtype)).max(initial=0)))


def _gen_bits(args):
    name, s, lo, hi = args
    from paged_kv_cache_270_gb300 import workloads as W
    w = W.make(name)
    k, v = w.kv_bits(s, lo, hi)
    return s, lo, hi, k, v


def _oracle_prefill_worker(args):
    """Times the fp64 oracle's chunked prefill on the last `rows` queries of one
    sequence; returns (flops, t_start, t_end)."""
    name, s, rows, k_scale, v_scale = args
    import oracle
    from paged_kv_cache_270_gb300 import workloads as W
    w = W.make(name)
    n = int(w.ctx_lens[s])
    nb = -(-n // 16)
    nbytes = oracle.pool_bytes(w.kv_dtype, nb, 16, w.n_kv_heads, w.head_dim)
    kp, vp = np.zeros(nbytes, np.uint8), np.zeros(nbytes, np.uint8)
    k, v = w.kv_bits(s, 0, n)
    oracle.reshape_and_cache(w.kv_dtype, nb, 16, w.n_kv_heads, w.head_dim, k, v,
                             np.arange(n, dtype=np.int64), k_scale, v_scale, kp, vp)
    q = w.prefill_q_bits()[s * w.chunk + w.chunk - rows: (s + 1) * w.chunk]
    t0 = time.time()
    oracle.paged_prefill(w.kv_dtype, w.in_dtype, nb, 16, w.n_kv_heads, w.head_dim, kp, vp,
                         k_scale, v_scale, q, np.array([0, rows], np.int32),
                         np.arange(nb, dtype=np.int32)[None, :], np.array([n], np.int32),
                         w.softmax_scale)
    t1 = time.time()
    keys = rows * n - rows * (rows - 1) // 2
    return 4 * w.head_dim * w.n_q_heads * keys, t0, t1


def _oracle_worker(args):
    """Times the fp64 oracle (gather + textbook attention) on some sequences of
    a workload; returns (kv bytes, t_start, t_end)."""
    name, seqs, k_scale, v_scale = args
    import oracle
    from paged_kv_cache_270_gb300 import workloads as W
    w = W.make(name)
    w.k_scale, w.v_scale = k_scale, v_scale
    ids = []
    for s in seqs:
        ids += list(w.block_tables[s, : -(-int(w.ctx_lens[s]) // 16)])
    remap = {b: i for i, b in enumerate(ids)}
    tables = np.zeros((len(seqs), w.max_blocks), np.int32)
    nbytes = oracle.pool_bytes(w.kv_dtype, len(ids), 16, w.n_kv_heads, w.head_dim)
    kp, vp = np.zeros(nbytes, np.uint8), np.zeros(nbytes, np.uint8)
    for r, s in enumerate(seqs):
        n = int(w.ctx_lens[s])
        nb = -(-n // 16)
        tables[r, :nb] = [remap[b] for b in w.block_tables[s, :nb]]
        k, v = w.kv_bits(s, 0, n)
        pos = np.arange(n, dtype=np.int64)
        slots = tables[r, pos // 16].astype(np.int64) * 16 + pos % 16
        oracle.reshape_and_cache(w.kv_dtype, len(ids), 16, w.n_kv_heads, w.head_dim, k, v, slots,
                                 w.k_scale, w.v_scale, kp, vp)
    q = w.q_bits()[list(seqs)]
    ctx = w.ctx_lens[list(seqs)]
    t0 = time.time()
    oracle.paged_attention(w.kv_dtype, w.in_dtype, len(ids), 16, w.n_kv_heads, w.head_dim, kp, vp,
                           w.k_scale, w.v_scale, q, tables, ctx, w.softmax_scale)
    t1 = time.time()
    return w.kv_bytes(ctx), t0, t1


# ------------------------------------------------------------------- helpers
def _env_rank():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def _measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _p10_p90(xs):
    """10th and 90th percentiles (nearest rank) of per-launch times, ms."""
    v = sorted(xs)
    if not v:
        return None
    return [round(v[int(0.1 * (len(v) - 1))], 4), round(v[int(0.9 * (len(v) - 1))], 4)]


def _source_sha():
    """sha256 of the decode kernel's code: pa_decode.cu and pa_device.cuh with
    // comments, trailing blanks and empty lines removed, so that editing a
    comment keeps the recorded traffic valid and any code change voids it."""
    h = hashlib.sha256()
    for f in ("pa_decode.cu", "pa_device.cuh"):
        with open(os.path.join(ROOT, "paged_kv_cache_270_gb300", "csrc", f)) as fh:
            lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in fh.read().splitlines())
            h.update(("\n".join(ln for ln in lines if ln.strip()) + "\n").encode())
    return h.hexdigest()


class ClockSampler:
    """Samples SM clock, power and clock-event reasons through NVML while the
    timed region runs (read-only queries)."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x1: "gpu_idle"}

    def __init__(self, device_index: int):
        self.samples = []
        self.ok = False
        self.max_mhz = None
        try:
            import torch
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            props = torch.cuda.get_device_properties(device_index)
            bus = f"{props.pci_domain_id:08x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
            self.h = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reasons = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except Exception:
            self.ok = False

    def _sample(self):
        c, p, r = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c))
        self.nvml.nvmlDeviceGetPowerUsage(self.h, ctypes.byref(p))
        self._reasons(self.h, ctypes.byref(r))
        self.samples.append((c.value, p.value / 1000.0, r.value))

    def __enter__(self):
        self._stop = threading.Event()
        if self.ok:
            self._sample()

            def loop():
                while not self._stop.is_set():
                    self._sample()
                    time.sleep(0.002)
            self._t = threading.Thread(target=loop, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self.ok:
            self._t.join()
            self._sample()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["nvml unavailable"]}
        reasons = set()
        for _, _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(s[0] for s in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "power_w_max": max(s[1] for s in self.samples), "samples": len(self.samples)}


# --------------------------------------------------------------- GPU batches
class Batch:
    """One workload batch resident on the GPU: filled pool plus the step's inputs."""

    def __init__(self, name, pool_procs, num_splits=0):
        import torch

        from paged_kv_cache_270_gb300 import _native as N
        from paged_kv_cache_270_gb300 import workloads as W
        from paged_kv_cache_270_gb300.pool import KVPool
        self.N = N
        w = W.make(name)
        self.w = w
        S, Hq, D = w.S, w.n_q_heads, w.head_dim
        chunks = []
        for s in range(S):
            n = int(w.final_ctx()[s])
            for lo in range(0, n, 16384):
                chunks.append((name, s, lo, min(n, lo + 16384)))
        if w.kv_dtype == "fp8_e4m3":
            ka = va = 0.0
            for a, b in pool_procs.imap_unordered(_gen_amax, chunks, chunksize=4):
                ka, va = max(ka, a), max(va, b)
            w.k_scale = float(np.float32(ka) / np.float32(448.0))
            w.v_scale = float(np.float32(va) / np.float32(448.0))
        self.pool = KVPool(1, w.num_blocks, w.n_kv_heads, D, w.kv_dtype, w.k_scale, w.v_scale)
        in_t = torch.float16 if w.in_dtype == "fp16" else torch.bfloat16
        self.in_t = in_t
        ctx = w.ctx_lens
        last_k = np.zeros((S, w.n_kv_heads, D), np.uint16)
        last_v = np.zeros_like(last_k)
        for s, lo, hi, k, v in pool_procs.imap(_gen_bits, chunks, chunksize=2):
            pos = np.arange(lo, hi, dtype=np.int64)
            slots = w.block_tables[s, pos // 16].astype(np.int64) * 16 + pos % 16
            self.pool.reshape_and_cache(
                torch.from_numpy(k.view(np.int16)).view(in_t).cuda(non_blocking=False),
                torch.from_numpy(v.view(np.int16)).view(in_t).cuda(non_blocking=False),
                torch.from_numpy(slots).cuda())
            if lo <= ctx[s] - 1 < hi:
                last_k[s] = k[ctx[s] - 1 - lo]
                last_v[s] = v[ctx[s] - 1 - lo]
        torch.cuda.synchronize()
        self.S, self.Hq, self.D = S, Hq, D
        self.max_blocks = w.max_blocks
        # host copies (pinned) of every per-step input, for the end-to-end run
        q_bits = w.q_bits()
        new_slots = (w.block_tables[np.arange(S), (ctx - 1) // 16].astype(np.int64) * 16 +
                     (ctx - 1) % 16)
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()  # noqa: E731
        self.h_q = pin(q_bits.view(np.int16)).view(in_t)
        self.h_k = pin(last_k.view(np.int16)).view(in_t)
        self.h_v = pin(last_v.view(np.int16)).view(in_t)
        self.h_slots = pin(new_slots)
        self.h_tables = pin(w.block_tables.astype(np.int32))
        self.h_ctx = pin(ctx.astype(np.int32))
        self.d_q = self.h_q.cuda()
        self.d_k = self.h_k.cuda()
        self.d_v = self.h_v.cuda()
        self.d_slots = self.h_slots.cuda()
        self.d_tables = self.h_tables.cuda()
        self.d_ctx = self.h_ctx.cuda()
        self.d_out = torch.empty((S, Hq, D), dtype=in_t, device="cuda")
        # 0: the library's automatic schedule; else a fixed split count
        self.num_splits = num_splits
        self.splits = num_splits or self.pool.num_splits(S, Hq, self.max_blocks)
        self.ws_bytes = self.pool.workspace_bytes(S, Hq, self.max_blocks, num_splits)
        self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device="cuda")
        self.kv_bytes = w.kv_bytes()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in
                             (self.h_q, self.h_k, self.h_v, self.h_slots, self.h_tables,
                              self.h_ctx))
        self.d2h_bytes = self.d_out.numel() * self.d_out.element_size()
        # cache write + decode, + the merge: always with the balanced schedule
        # (splits -1), with fixed splits when there are several
        self.launches = 2 + (1 if self.splits != 1 else 0)
        self.softmax_scale = w.softmax_scale
        self.out_code = N.PA_FP16 if w.in_dtype == "fp16" else N.PA_BF16

    def reshape(self, stream):
        self.N.pa_reshape_and_cache(self.pool.handle, 0, self.d_k.data_ptr(), self.d_v.data_ptr(),
                                    self.d_slots.data_ptr(), self.S, stream)

    def decode(self, stream):
        self.N.pa_decode(self.pool.handle, 0, self.d_out.data_ptr(), self.out_code,
                         self.d_q.data_ptr(), self.d_tables.data_ptr(), self.max_blocks,
                         self.d_ctx.data_ptr(), self.S, self.Hq, self.softmax_scale, self.num_splits,
                         self.ws.data_ptr(), self.ws_bytes, stream)


class Staging:
    """The step's host<->device traffic for the end-to-end run, packed: every
    batch's per-step inputs sit in one pinned host buffer whose device twin the
    kernels read (the batches' device tensors become views into it), and the
    outputs of all batches in one device buffer with a pinned host twin.  A step
    then moves its inputs with one host-to-device copy and its results with one
    device-to-host copy.  (Overlapping the second batch's copies with the first
    batch's decode on a copy stream measured slower: the step moves ~10 MB, and
    the cross-stream waits cost more than they hide.)"""
    FIELDS = ("q", "k", "v", "slots", "tables", "ctx")

    def __init__(self, batches):
        import torch
        align = lambda n: (n + 255) // 256 * 256  # noqa: E731
        nbytes = lambda t: t.numel() * t.element_size()  # noqa: E731
        self.in_rng, self.out_rng = [], []
        off_in = off_out = 0
        for b in batches:
            n = sum(align(nbytes(getattr(b, "h_" + f))) for f in self.FIELDS)
            self.in_rng.append((off_in, off_in + n))
            off_in += n
            n = align(nbytes(b.d_out))
            self.out_rng.append((off_out, off_out + n))
            off_out += n
        self.h_in = torch.empty(off_in, dtype=torch.uint8).pin_memory()
        self.d_in = torch.empty(off_in, dtype=torch.uint8, device="cuda")
        self.h_out = torch.empty(off_out, dtype=torch.uint8).pin_memory()
        self.d_out = torch.empty(off_out, dtype=torch.uint8, device="cuda")
        for b, (off, _) in zip(batches, self.in_rng):
            for f in self.FIELDS:
                h = getattr(b, "h_" + f)
                n = nbytes(h)
                self.h_in[off:off + n].copy_(h.contiguous().view(-1).view(torch.uint8))
                setattr(b, "d_" + f, self.d_in[off:off + n].view(h.dtype).view(h.shape))
                off += align(n)
        self.d_in.copy_(self.h_in)
        for b, (off, _) in zip(batches, self.out_rng):
            n = nbytes(b.d_out)
            b.d_out = self.d_out[off:off + n].view(b.d_out.dtype).view(b.d_out.shape)
        self.h2d_bytes = sum(b.h2d_bytes for b in batches)
        self.d2h_bytes = sum(b.d2h_bytes for b in batches)

    def step(self, batches, sh):
        """One end-to-end step: inputs in, reshape + decode per batch, results out."""
        self.d_in.copy_(self.h_in, non_blocking=True)
        for b in batches:
            b.reshape(sh)
            b.decode(sh)
        self.h_out.copy_(self.d_out, non_blocking=True)


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(names, scales, seconds, procs, pool, single_core=True):
    """Time the oracle on a bounded sample of the workload's sequences, one
    process per core (and, with single_core, in one process on a smaller sample)."""
    # calibrate: one short sequence set first, then size the sample
    from paged_kv_cache_270_gb300 import workloads as W
    jobs = []
    for name in names[-1:]:  # the batch with the most sequences: short ones sample evenly
        w = W.make(name)
        order = np.random.default_rng(17).permutation(w.S)
        jobs.append((name, w, order))
    name, w, order = jobs[-1]
    probe = pool.map(_oracle_worker, [(name, [int(order[0])], *scales[name])])
    b, t0, t1 = probe[0]
    per_byte = (t1 - t0) / b
    results, sample_desc = [], []
    budget = seconds * procs
    for name, w, order in jobs:
        per_seq = w.kv_bytes(w.ctx_lens[:1]) * per_byte
        n = max(1, min(w.S, int(budget / len(jobs) / max(per_seq, 1e-9))))
        seqs = [int(s) for s in order[:n]]
        groups = [seqs[i::procs] for i in range(procs) if seqs[i::procs]]
        results += pool.map(_oracle_worker, [(name, g, *scales[name]) for g in groups])
        sample_desc.append(f"{name}: {n} of {w.S} sequences")
    total = sum(r[0] for r in results)
    wall = max(r[2] for r in results) - min(r[1] for r in results)
    rec = {"value": total / wall / 1e9, "unit": "GB/s", "cores": procs, "kind": "oracle",
           "cpu_model": _cpu_model(), "host_cores": os.cpu_count(),
           "sample": "; ".join(sample_desc) + f" ({total / 1e6:.0f} MB of K+V, "
                     f"{wall:.1f} s wall, fp64 gather + softmax attention, one process per core)"}
    if single_core:
        # the same oracle in one process (one core), on a sample of about seconds / 2
        name, w, order = jobs[-1]
        n1 = max(1, min(w.S, int(seconds / 2 / max(w.kv_bytes(w.ctx_lens[:1]) * per_byte, 1e-9))))
        one = pool.map(_oracle_worker, [(name, [int(s) for s in order[:n1]], *scales[name])])[0]
        rec["single_core"] = {"value": one[0] / (one[2] - one[1]) / 1e9, "unit": "GB/s", "cores": 1,
                              "sample": f"{name}: {n1} of {w.S} sequences ({one[0] / 1e6:.0f} MB "
                                        f"of K+V, {one[2] - one[1]:.1f} s)"}
    return rec


_ARM_PARTS = {"0xd0c": "Neoverse-N1", "0xd40": "Neoverse-V1", "0xd49": "Neoverse-N2",
              "0xd4f": "Neoverse-V2", "0xd8e": "Neoverse-N3", "0xd84": "Neoverse-V3"}


def _cpu_model():
    """The host CPU's model from /proc/cpuinfo (x86: "model name"; Arm: the
    implementer and part numbers, named for the Neoverse cores)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return None
    m = re.search(r"^model name\s*:\s*(.+)$", info, re.M)
    if m:
        return m.group(1).strip()
    impl = re.search(r"^CPU implementer\s*:\s*(\S+)", info, re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)", info, re.M)
    if part:
        name = _ARM_PARTS.get(part.group(1).lower(), "Arm core")
        return f"{name} (implementer {impl.group(1) if impl else '?'}, part {part.group(1)})"
    return None


# ----------------------------------------------------------- config records
# The default run also measures the other decode configurations (one record
# each, in the line's "configs"): the headline value stays on the 70B batches.
def _bt(a, dtype):
    """uint16 bit patterns -> a CUDA tensor of the 16-bit dtype."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.view(torch.float16 if dtype == "fp16" else torch.bfloat16).cuda()


def _decode_call(pool, q, tables, ctx, out, ws, ws_bytes, stream, scale, num_splits=0):
    from paged_kv_cache_270_gb300 import _native as N
    S, Hq, _ = q.shape
    N.pa_decode(pool.handle, 0, out.data_ptr(), pool.in_code, q.data_ptr(), tables.data_ptr(),
                tables.shape[-1], ctx.data_ptr(), S, Hq, scale, num_splits,
                ws.data_ptr() if ws_bytes else 0, ws_bytes, stream)


def _median_ms(fn, iters, warmup, stream):
    """Median time of fn() in ms, each call between CUDA events on `stream`."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    for e0, e1 in ev:
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)


def record_8b_bf16(pool_procs, peak):
    """Config 1: Llama-3.1-8B-shaped bf16 decode, 64 sequences of U[512, 4096]."""
    import torch
    from paged_kv_cache_270_gb300 import _native as N
    b = Batch("llama3_8b_bf16", pool_procs)
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)
    rec = {"workload": DESCRIPTION["llama3_8b_bf16"], "kv_bytes": b.kv_bytes,
           "timing": "median of 50 decode calls, CUDA events"}
    for key, ns in (("automatic", 0), ("balanced", N.PA_SPLITS_BALANCED)):
        ws_bytes = b.pool.workspace_bytes(b.S, b.Hq, b.max_blocks, ns)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        ms = _median_ms(lambda: _decode_call(b.pool, b.d_q, b.d_tables, b.d_ctx, b.d_out, ws, ws_bytes,
                                             sh, b.softmax_scale, ns), 50, 10, stream)
        rec[key] = {"schedule": f"{b.splits} splits" if ns == 0 else "balanced",
                    "decode_ms_median": round(ms, 5), "decode_kv_gbs": round(b.kv_bytes / ms / 1e6, 1),
                    "frac_of_measured_peak": round(b.kv_bytes / ms / 1e6 / peak, 4),
                    "tokens_per_s": round(b.S / ms * 1e3, 1)}
    rec["device_error"] = b.pool.device_error()
    b.pool.close()
    return rec


def record_long_short(pool_procs, peak):
    """A batch whose lengths differ by orders of magnitude (8B shapes, FP8): one
    131072-token sequence among 127 short ones.  The automatic split count
    takes every sequence as the table's width (the lengths live on the
    device), so the long sequence's few CTAs set the time; the balanced
    schedule cuts all pages into equal ranges.  Decode calls back to back."""
    import torch
    from paged_kv_cache_270_gb300 import _native as N
    b = Batch("llama3_8b_fp8_long_short", pool_procs)
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)
    rec = {"workload": DESCRIPTION["llama3_8b_fp8_long_short"], "kv_bytes": b.kv_bytes,
           "timing": "20 decode calls back to back between two events, median of 5 runs"}
    for key, ns in (("automatic", 0), ("balanced", N.PA_SPLITS_BALANCED)):
        ws_bytes = b.pool.workspace_bytes(b.S, b.Hq, b.max_blocks, ns)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")

        def calls():
            for _ in range(20):
                _decode_call(b.pool, b.d_q, b.d_tables, b.d_ctx, b.d_out, ws, ws_bytes, sh, b.softmax_scale, ns)

        ms = _median_ms(calls, 5, 1, stream) / 20
        rec[key] = {"schedule": (f"{b.pool.num_splits(b.S, b.Hq, b.max_blocks)} splits" if ns == 0
                                 else "balanced"),
                    "decode_ms": round(ms, 5), "decode_kv_gbs": round(b.kv_bytes / ms / 1e6, 1),
                    "frac_of_measured_peak": round(b.kv_bytes / ms / 1e6 / peak, 4)}
    rec["device_error"] = b.pool.device_error()
    b.pool.close()
    return rec


def record_8b_fp8_steps(pool_procs, peak):
    """Config 2: the 8B shapes over an FP8 cache (per-tensor scales amax/448, 1%
    of K x8), 32 decode steps of (write one token per sequence, decode), new
    blocks taken from the pool's spare blocks when a sequence crosses a block
    boundary.  Every step's inputs are resident before the timed region."""
    import torch
    from paged_kv_cache_270_gb300 import workloads as W
    from paged_kv_cache_270_gb300.pool import KVPool
    w = W.make("llama3_8b_fp8")
    S, steps, D, Hkv = w.S, w.steps, w.head_dim, w.n_kv_heads
    fin = w.final_ctx()
    amax_chunks = [(w.name, s, lo, min(int(n), lo + 16384)) for s, n in enumerate(fin)
                   for lo in range(0, int(n), 16384)]
    ka = va = 0.0
    for a_, b_ in pool_procs.imap_unordered(_gen_amax, amax_chunks, chunksize=4):
        ka, va = max(ka, a_), max(va, b_)
    k_scale = float(np.float32(ka) / np.float32(448.0))
    v_scale = float(np.float32(va) / np.float32(448.0))
    pool = KVPool(1, w.num_blocks, Hkv, D, "fp8_e4m3", k_scale, v_scale)
    ctx0 = w.ctx_lens
    fill = [(w.name, s, lo, min(int(n), lo + 16384)) for s, n in enumerate(ctx0)
            for lo in range(0, int(n), 16384)]
    for s, lo, hi, k, v in pool_procs.imap(_gen_bits, fill, chunksize=2):
        pos = np.arange(lo, hi, dtype=np.int64)
        slots = w.block_tables[s, pos // 16].astype(np.int64) * 16 + pos % 16
        pool.reshape_and_cache(_bt(k, "bf16"), _bt(v, "bf16"), torch.from_numpy(slots).cuda())
    tables = w.block_tables.copy()
    spare = list(w.spare_blocks)
    t_all, s_all, c_all, q_all = [], [], [], []
    new_blocks = 0
    for j in range(steps):
        pos = ctx0 + j
        for s in np.nonzero(pos % 16 == 0)[0]:
            tables[s, pos[s] // 16] = spare.pop(0)
            new_blocks += 1
        s_all.append(tables[np.arange(S), pos // 16].astype(np.int64) * 16 + pos % 16)
        t_all.append(tables.copy())
        c_all.append(pos + 1)
        q_all.append(w.q_bits(j))
    # the new tokens of every step: [steps][S][Hkv][D]
    kv = [w.kv_bits(s, int(ctx0[s]), int(ctx0[s]) + steps) for s in range(S)]
    k_all = np.stack([k for k, _ in kv], axis=1)
    v_all = np.stack([v for _, v in kv], axis=1)
    d_t = torch.from_numpy(np.stack(t_all).astype(np.int32)).cuda()
    d_s = torch.from_numpy(np.stack(s_all)).cuda()
    d_c = torch.from_numpy(np.stack(c_all).astype(np.int32)).cuda()
    d_k, d_v, d_q = _bt(k_all, "bf16"), _bt(v_all, "bf16"), _bt(np.stack(q_all), "bf16")
    out = torch.empty((S, w.n_q_heads, D), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)
    from paged_kv_cache_270_gb300 import _native as N
    kv_bytes = int(sum(int(c.sum()) for c in c_all)) * 2 * Hkv * D
    rec = {"workload": DESCRIPTION["llama3_8b_fp8"] + ", 32 steps of (write one token per "
                                                       "sequence, decode)",
           "steps": steps, "new_blocks": new_blocks, "kv_bytes_all_steps": kv_bytes,
           "timing": "median of 5 runs of the 32-step loop (CUDA events); decode calls timed "
                     "one by one in one more run (an event between each cache write and its "
                     "decode, so no launch overlap); back to back: the last step's decode "
                     "called 50 times in a row between two events, median of 5 such runs"}
    for key, ns in (("automatic", 0), ("balanced", N.PA_SPLITS_BALANCED)):
        ws_bytes = pool.workspace_bytes(S, w.n_q_heads, w.max_blocks, ns)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        dec_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)]

        def run(evs=None):
            for j in range(steps):
                N.pa_reshape_and_cache(pool.handle, 0, d_k[j].data_ptr(), d_v[j].data_ptr(),
                                       d_s[j].data_ptr(), S, sh)
                if evs:
                    evs[j][0].record(stream)
                _decode_call(pool, d_q[j], d_t[j], d_c[j], out, ws, ws_bytes, sh, w.softmax_scale, ns)
                if evs:
                    evs[j][1].record(stream)

        loop_ms = _median_ms(run, 5, 2, stream)
        run(dec_ev)
        torch.cuda.synchronize()
        dec_ms = [e0.elapsed_time(e1) for e0, e1 in dec_ev]
        last = steps - 1

        def back_to_back():
            for _ in range(50):
                _decode_call(pool, d_q[last], d_t[last], d_c[last], out, ws, ws_bytes, sh, w.softmax_scale, ns)

        b2b_ms = _median_ms(back_to_back, 5, 1, stream) / 50
        b2b_bytes = int(c_all[last].sum()) * 2 * Hkv * D
        rec[key] = {"schedule": (f"{pool.num_splits(S, w.n_q_heads, w.max_blocks)} splits" if ns == 0
                                 else "balanced"),
                    "step_ms": round(loop_ms / steps, 5),
                    "step_kv_gbs": round(kv_bytes / loop_ms / 1e6, 1),
                    "decode_ms_median": round(statistics.median(dec_ms), 5),
                    "decode_kv_gbs": round(kv_bytes / sum(dec_ms) / 1e6, 1),
                    "decode_frac_of_measured_peak": round(kv_bytes / sum(dec_ms) / 1e6 / peak, 4),
                    "decode_back_to_back_ms": round(b2b_ms, 5),
                    "decode_back_to_back_kv_gbs": round(b2b_bytes / b2b_ms / 1e6, 1),
                    "decode_back_to_back_frac_of_measured_peak": round(b2b_bytes / b2b_ms / 1e6 / peak, 4),
                    "tokens_per_s": round(S * steps / loop_ms * 1e3, 1)}
    rec["device_error"] = pool.device_error()
    pool.close()
    return rec


def record_prefix_share(peak):
    """Config 4: 64 requests sharing a 2048-token prefix (128 refcounted blocks)
    plus a U[128, 1024] suffix each, one decode; and best-of-8 over a 2008-token
    prompt: copy-on-write of the shared tail block, then 64 steps of (write one
    token per branch, decode).  Logical bytes count every sequence's pages,
    unique bytes each physical page once (the 8 MiB prefix can stay in L2)."""
    import torch
    from paged_kv_cache_270_gb300 import _native as N
    from paged_kv_cache_270_gb300 import workloads as W
    from paged_kv_cache_270_gb300.pool import KVPool
    ps = W.PrefixShare()
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)
    R, P, Hkv, D = ps.n_requests, ps.prefix_tokens, ps.n_kv_heads, ps.head_dim
    tok_bytes = 2 * Hkv * D * 2
    pool = KVPool(1, 4096, Hkv, D, "bf16")
    prefix = pool.alloc(P // 16)
    kp, vp = ps.prefix_kv()
    pos = np.arange(P, dtype=np.int64)
    pool.reshape_and_cache(_bt(kp, "bf16"), _bt(vp, "bf16"),
                           torch.from_numpy(prefix[pos // 16].astype(np.int64) * 16 + pos % 16).cuda())
    suf = ps.suffix_lens()
    ctx = (P + suf).astype(np.int32)
    tables = np.zeros((R, -(-int(ctx.max()) // 16)), np.int32)
    for r in range(R):
        if r:
            pool.incref(prefix)
        own = pool.alloc(-(-int(suf[r]) // 16))
        tables[r, :len(prefix)] = prefix
        tables[r, len(prefix):len(prefix) + len(own)] = own
        k, v = ps.suffix_kv(r, int(suf[r]))
        p_ = np.arange(int(suf[r]), dtype=np.int64)
        pool.reshape_and_cache(_bt(k, "bf16"), _bt(v, "bf16"),
                               torch.from_numpy(own[p_ // 16].astype(np.int64) * 16 + p_ % 16).cuda())
    used, _, shared = pool.stats()
    q = _bt(ps.q_bits(R), "bf16")
    d_t, d_c = torch.from_numpy(tables).cuda(), torch.from_numpy(ctx).cuda()
    out = torch.empty((R, ps.n_q_heads, D), dtype=torch.bfloat16, device="cuda")
    ws_bytes = pool.workspace_bytes(R, ps.n_q_heads, tables.shape[1], 0)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    scale = 1.0 / math.sqrt(D)
    ms = _median_ms(lambda: _decode_call(pool, q, d_t, d_c, out, ws, ws_bytes, sh, scale), 50, 10,
                    stream)
    logical = int(ctx.sum()) * tok_bytes
    unique = (P + int(suf.sum())) * tok_bytes
    err = pool.device_error()
    pool.close()
    shared_rec = {"requests": R, "blocks_used": used, "blocks_shared": shared,
                  "blocks_unshared_layout": int(np.sum(-(-ctx // 16))),
                  "logical_kv_bytes": logical, "unique_kv_bytes": unique,
                  "decode_ms_median": round(ms, 5),
                  "logical_gbs": round(logical / ms / 1e6, 1),
                  "unique_gbs": round(unique / ms / 1e6, 1),
                  "unique_frac_of_measured_peak": round(unique / ms / 1e6 / peak, 4),
                  "device_error": err}

    # best of 8 over a 2008-token prompt (its tail block holds 8 tokens)
    prompt, branches, new_tok = 2008, 8, 64
    pool = KVPool(1, 512, Hkv, D, "bf16")
    nb = -(-prompt // 16)
    pblocks = pool.alloc(nb)
    kp, vp = ps.prefix_kv(prompt)
    pos = np.arange(prompt, dtype=np.int64)
    pool.reshape_and_cache(_bt(kp, "bf16"), _bt(vp, "bf16"),
                           torch.from_numpy(pblocks[pos // 16].astype(np.int64) * 16 + pos % 16).cuda())
    width = -(-(prompt + new_tok) // 16)
    tables = np.zeros((branches, width), np.int32)
    for b in range(branches):
        if b:
            pool.incref(pblocks)
        tables[b, :nb] = pblocks
    pairs = []
    for b in range(branches):
        row = np.ascontiguousarray(tables[b])
        got = pool.cow_prepare(row, prompt)
        tables[b] = row
        if got:
            pairs.append(got)
    d_pairs = torch.from_numpy(np.array(pairs, np.int32)).cuda()
    copy_ms = _median_ms(lambda: pool.copy_blocks(d_pairs), 20, 3, stream)
    t_all, s_all, c_all = [], [], []
    c = np.full(branches, prompt, np.int32)
    for j in range(new_tok):
        for b in range(branches):
            if c[b] % 16 == 0:
                tables[b, c[b] // 16] = pool.alloc(1)[0]
        s_all.append(tables[np.arange(branches), c // 16].astype(np.int64) * 16 + c % 16)
        t_all.append(tables.copy())
        c = c + 1
        c_all.append(c.copy())
    used, _, shared = pool.stats()
    d_t = torch.from_numpy(np.stack(t_all)).cuda()
    d_s = torch.from_numpy(np.stack(s_all)).cuda()
    d_c = torch.from_numpy(np.stack(c_all)).cuda()
    kq = [ps.suffix_kv(1000 + j, branches) for j in range(new_tok)]
    d_k = _bt(np.stack([k for k, _ in kq]), "bf16")
    d_v = _bt(np.stack([v for _, v in kq]), "bf16")
    d_q = _bt(np.stack([ps.q_bits(branches, j) for j in range(new_tok)]), "bf16")
    out = torch.empty((branches, ps.n_q_heads, D), dtype=torch.bfloat16, device="cuda")
    ws_bytes = pool.workspace_bytes(branches, ps.n_q_heads, width, 0)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")

    def steps():
        for j in range(new_tok):
            N.pa_reshape_and_cache(pool.handle, 0, d_k[j].data_ptr(), d_v[j].data_ptr(),
                                   d_s[j].data_ptr(), branches, sh)
            _decode_call(pool, d_q[j], d_t[j], d_c[j], out, ws, ws_bytes, sh, scale)

    loop_ms = _median_ms(steps, 5, 2, stream)
    err = pool.device_error()
    pool.close()
    logical = int(sum(int(x.sum()) for x in c_all)) * tok_bytes
    return {"workload": "Llama-3.1-8B-shaped bf16 (Hq 32 / Hkv 8 / d 128): 64 requests sharing "
                        "a 2048-token prefix, each with a U[128,1024] suffix; best-of-8 over a "
                        "2008-token prompt with copy-on-write of the shared tail block",
            "shared_prefix_decode": shared_rec,
            "best_of_8": {"prompt_tokens": prompt, "branches": branches, "cow_copies": len(pairs),
                          "blocks_used": used, "blocks_unshared_layout": branches * width,
                          "copy_blocks_ms": round(copy_ms, 5),
                          "step_ms": round(loop_ms / new_tok, 5),
                          "tokens_per_s": round(branches * new_tok / loop_ms * 1e3, 1),
                          "logical_gbs": round(logical / loop_ms / 1e6, 1),
                          "device_error": err},
            "timing": "CUDA events; decode: median of 50 calls; best-of-8: median of 5 runs of "
                      "the 64-step loop; the copy: median of 20 calls"}


def config_records(pool_procs, peak):
    recs = {}
    for name, fn in (("llama3_8b_bf16", lambda: record_8b_bf16(pool_procs, peak)),
                     ("llama3_8b_fp8_steps", lambda: record_8b_fp8_steps(pool_procs, peak)),
                     ("prefix_share_bf16", lambda: record_prefix_share(peak)),
                     ("llama3_8b_fp8_long_short", lambda: record_long_short(pool_procs, peak))):
        recs[name] = fn()
        if recs[name].get("device_error") or \
                any(v.get("device_error") for v in recs[name].values() if isinstance(v, dict)):
            raise RuntimeError(f"device error in the {name} record")
    return recs


# ------------------------------------------------------------------- arms
def run_gb300(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    names = WORKLOADS[args.workload]
    ctx_mp = mp.get_context("spawn")
    procs = max(1, os.cpu_count() or 1)
    with ctx_mp.Pool(procs) as pool_procs:
        batches = [Batch(n, pool_procs, args.decode_splits) for n in names]
        staging = Staging(batches)
        scales = {b.w.name: (b.w.k_scale, b.w.v_scale) for b in batches}
        stream = torch.cuda.current_stream()
        sh = int(stream.cuda_stream)

        def step(evs=None):
            for i, b in enumerate(batches):
                b.reshape(sh)
                if evs is not None:
                    evs[i][0].record(stream)
                b.decode(sh)
                if evs is not None:
                    evs[i][1].record(stream)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        for b in batches:
            err = b.pool.device_error()
            if err:
                raise RuntimeError(f"device error {err} in {b.w.name}")
        K = args.steps
        evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in batches]
               for _ in range(K)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sampler = ClockSampler(local_rank)
        _barrier(world)
        torch.cuda.synchronize()
        with sampler:
            start.record(stream)
            for k in range(K):
                step(evs[k])
            end.record(stream)
            torch.cuda.synchronize()
        _barrier(world)
        t = start.elapsed_time(end) / 1e3
        t_max = _max_over_ranks(t, world)
        dec_ms = [[evs[k][i][0].elapsed_time(evs[k][i][1]) for k in range(K)]
                  for i in range(len(batches))]

        # end to end through the C ABI: pinned host inputs in, result out, every step
        e2e = None
        if not args.no_e2e:
            for _ in range(max(1, args.warmup // 2)):
                staging.step(batches, sh)
                torch.cuda.synchronize()
            _barrier(world)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(K):
                staging.step(batches, sh)
                stream.synchronize()  # the step's results are in host memory
            e1.record(stream)
            torch.cuda.synchronize()
            te = _max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
            kv = sum(b.kv_bytes for b in batches)
            e2e = {"value": world * kv * K / te / 1e9, "unit": "GB/s",
                   "h2d_bytes_per_step": staging.h2d_bytes,
                   "d2h_bytes_per_step": staging.d2h_bytes,
                   "ms_per_step": te / K * 1e3}
        for b in batches:
            err = b.pool.device_error()
            if err:
                raise RuntimeError(f"device error {err} in {b.w.name}")

        configs = None
        if args.workload == "llama3_70b_fp8" and world == 1 and not args.no_configs:
            configs = config_records(pool_procs, _measured_peak()[0])

        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu:
            cpu = cpu_baseline(names, scales, args.cpu_seconds, procs, pool_procs)

    if rank != 0:
        return
    kv = sum(b.kv_bytes for b in batches)
    value = world * kv * K / t_max / 1e9
    peak, peak_kind = _measured_peak()
    dec_avg = [statistics.fmean(d) / 1e3 for d in dec_ms]  # s per launch, per batch
    achieved = kv / sum(dec_avg) / 1e9
    sha = _source_sha()
    traffic = None
    if NCU_TRAFFIC["source_sha256"] == sha and all(
            b.w.name in NCU_TRAFFIC["bytes_per_launch"] for b in batches):
        traffic = sum(NCU_TRAFFIC["bytes_per_launch"][b.w.name] for b in batches)
    per_batch = {}
    for b, d in zip(batches, dec_ms):
        per_batch[b.w.name] = {
            "sequences": b.S, "tokens_per_seq": int(b.w.ctx_lens.max()), "kv_bytes": b.kv_bytes,
            "splits": b.splits, "schedule": "balanced" if b.splits < 0 else "fixed splits",
            "decode_ms_median": statistics.median(d),
            "decode_ms_p10_p90": _p10_p90(d),
            "decode_kv_gbs": b.kv_bytes / (statistics.median(d) / 1e3) / 1e9}
    launches = K * sum(b.launches for b in batches)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(t_max / K * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e4m3 KV / f16 tensor-core MMA / f32 accumulate" if batches[0].w.kv_dtype == "fp8_e4m3"
                  else "e4m3 KV with f32 scale per tile / f16 tensor-core MMA / f32 accumulate"
                  if batches[0].w.block_scaled else f"{batches[0].w.kv_dtype} KV / f32 accumulate"),
        "data": "synthetic (seeded N(0,1) q/k/v, random block tables)",
        "config": {"workload": DESCRIPTION[args.workload],
                   "l2": "inputs larger than L2 (KV pool "
                         f"{sum(b.pool.k_cache.numel() * 2 for b in batches) / 2**30:.2f} GiB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "tokens_per_s": round(world * sum(b.S for b in batches) * K / t_max, 1),
        "frac_of_spec_8tbs": round(value / SPEC_HBM_GBS, 4),
        "frac_of_measured_peak": round(value / peak, 4),
        "batches": per_batch,
        "roofline": {"kernel": "pa_decode (decode kernel + its merge kernel)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (hbm_gbs)", "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_step": kv},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "configs": configs,
        "clocks": sampler.summary(),
    }
    print(json.dumps(line), flush=True)


def _peak_tflops():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (bf16_tflops, burst)"
    except Exception:
        return 1900.0, "fallback"


def _prefill_mma_work(w):
    """The MMA work the tcgen05 prefill kernel issues for this packet, by kind.
    A CTA holds 128 rows (128 / G query tokens x the G heads of one kv head)
    and walks the 128-key blocks up to its last query's position; per block it
    issues S = Q K^T as two E4M3 passes (the query's two E4M3 terms) and
    O += P V as one binary16 pass, each M = N = K = 128 (masked keys of the
    diagonal blocks included).  Returns (e4m3 flops, f16 flops, blocks)."""
    G = w.n_q_heads // w.n_kv_heads
    tok = 128 // G
    blocks = 0
    for n in (int(x) for x in w.ctx_lens):
        for lo in range(0, w.chunk, tok):
            pos_last = n - w.chunk + min(w.chunk, lo + tok) - 1
            blocks += (pos_last // 16 + 1 + 7) // 8
    blocks *= w.n_kv_heads
    per_pass = 2 * 128 * 128 * 128
    return 2 * per_pass * blocks, per_pass * blocks, blocks


def run_prefill(args, rank, world, local_rank):
    """Chunked prefill: per step, write the chunk's K/V into its slots, then the
    causal attention of the chunk's queries over each sequence's pages."""
    import torch

    from paged_kv_cache_270_gb300 import _native as N
    from paged_kv_cache_270_gb300 import workloads as W
    from paged_kv_cache_270_gb300.pool import KVPool
    torch.cuda.set_device(local_rank)
    name = args.workload
    w = W.make(name)
    procs = max(1, os.cpu_count() or 1)
    with mp.get_context("spawn").Pool(procs) as pp:
        chunks = [(name, s, lo, min(int(w.ctx_lens[s]), lo + 16384))
                  for s in range(w.S) for lo in range(0, int(w.ctx_lens[s]), 16384)]
        ka = va = 0.0
        for a_, b_ in pp.imap_unordered(_gen_amax, chunks, chunksize=2):
            ka, va = max(ka, a_), max(va, b_)
        w.k_scale = float(np.float32(ka) / np.float32(448.0))
        w.v_scale = float(np.float32(va) / np.float32(448.0))
        pool = KVPool(1, w.num_blocks, w.n_kv_heads, w.head_dim, w.kv_dtype, w.k_scale, w.v_scale)
        in_t = torch.bfloat16
        new_k, new_v, new_slots = [], [], []
        for s, lo, hi, k, v in pp.imap(_gen_bits, chunks, chunksize=1):
            pos = np.arange(lo, hi, dtype=np.int64)
            slots = w.block_tables[s, pos // 16].astype(np.int64) * 16 + pos % 16
            pool.reshape_and_cache(torch.from_numpy(k.view(np.int16)).view(in_t).cuda(),
                                   torch.from_numpy(v.view(np.int16)).view(in_t).cuda(),
                                   torch.from_numpy(slots).cuda())
            first = int(w.ctx_lens[s]) - w.chunk  # the chunk's K/V are rewritten every step
            sel = pos >= first
            new_k.append(k[sel]); new_v.append(v[sel]); new_slots.append(slots[sel])
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu:
            rows = 16
            res = pp.map(_oracle_prefill_worker,
                         [(name, s % w.S, rows, w.k_scale, w.v_scale) for s in range(procs)])
            fl = sum(r[0] for r in res)
            wall = max(r[2] for r in res) - min(r[1] for r in res)
            cpu = {"value": fl / wall / 1e12, "unit": "TFLOP/s", "cores": procs, "kind": "oracle",
                   "sample": f"{procs} x the last {rows} queries of a 2048-token chunk "
                             f"({fl / 1e9:.1f} GFLOP, {wall:.1f} s wall, fp64)"}
    pin = lambda a_: torch.from_numpy(np.ascontiguousarray(a_)).pin_memory()  # noqa: E731
    h_q = pin(w.prefill_q_bits().view(np.int16)).view(in_t)
    h_k = pin(np.concatenate(new_k).view(np.int16)).view(in_t)
    h_v = pin(np.concatenate(new_v).view(np.int16)).view(in_t)
    h_slots = pin(np.concatenate(new_slots))
    h_qs = pin((np.arange(w.S + 1) * w.chunk).astype(np.int32))
    h_tab = pin(w.block_tables.astype(np.int32))
    h_ctx = pin(w.ctx_lens.astype(np.int32))
    hs = [h_q, h_k, h_v, h_slots, h_qs, h_tab, h_ctx]
    ds = [t.cuda() for t in hs]
    d_q, d_k, d_v, d_slots, d_qs, d_tab, d_ctx = ds
    d_out = torch.empty_like(d_q)
    h_out = torch.empty(d_out.shape, dtype=in_t).pin_memory()
    stream = torch.cuda.current_stream()
    sh = int(stream.cuda_stream)
    T = w.S * w.chunk

    def step(ev=None):
        N.pa_reshape_and_cache(pool.handle, 0, d_k.data_ptr(), d_v.data_ptr(), d_slots.data_ptr(),
                               T, sh)
        if ev is not None:
            ev[0].record(stream)
        N.pa_prefill(pool.handle, 0, d_out.data_ptr(), N.PA_BF16, d_q.data_ptr(), d_qs.data_ptr(),
                     d_tab.data_ptr(), w.max_blocks, d_ctx.data_ptr(), w.S, w.n_q_heads, w.chunk,
                     w.softmax_scale, sh)
        if ev is not None:
            ev[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if pool.device_error():
        raise RuntimeError("device error in prefill warm-up")
    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local_rank)
    _barrier(world)
    torch.cuda.synchronize()
    with sampler:
        e0.record(stream)
        for k in range(K):
            step(evs[k])
        e1.record(stream)
        torch.cuda.synchronize()
    _barrier(world)
    t_max = _max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    pre_ms = [ev[0].elapsed_time(ev[1]) for ev in evs]
    e2e = None
    if not args.no_e2e:
        # End to end, per sequence on the public API: a sequence's q, K/V and slots
        # go up on a copy stream while the previous sequence computes, and its
        # output comes back while the next one computes.
        cs = torch.cuda.Stream()
        C, Hq = w.chunk, w.n_q_heads
        h_qs1 = pin(np.array([0, C], np.int32))
        d_qs1 = h_qs1.cuda()
        small = [(d_tab, h_tab), (d_ctx, h_ctx), (d_qs1, h_qs1)]
        per_seq = [[(d_[s * C:(s + 1) * C], h_[s * C:(s + 1) * C]) for d_, h_ in
                    ((d_q, h_q), (d_k, h_k), (d_v, h_v), (d_slots, h_slots))] for s in range(w.S)]
        e2e_h2d = sum(h_.numel() * h_.element_size() for _, h_ in small) + sum(
            h_.numel() * h_.element_size() for seq in per_seq for _, h_ in seq)

        def e2e_step():
            cs.wait_stream(stream)
            ready = []
            with torch.cuda.stream(cs):
                for d_, h_ in small:
                    d_.copy_(h_, non_blocking=True)
                for seq in per_seq:
                    for d_, h_ in seq:
                        d_.copy_(h_, non_blocking=True)
                    ev_ = torch.cuda.Event()
                    ev_.record(cs)
                    ready.append(ev_)
            done = []
            for s_, ev_ in enumerate(ready):
                stream.wait_event(ev_)
                N.pa_reshape_and_cache(pool.handle, 0, d_k[s_ * C].data_ptr(), d_v[s_ * C].data_ptr(),
                                       d_slots[s_ * C:].data_ptr(), C, sh)
                N.pa_prefill(pool.handle, 0, d_out[s_ * C].data_ptr(), N.PA_BF16, d_q[s_ * C].data_ptr(),
                             d_qs1.data_ptr(), d_tab[s_].data_ptr(), w.max_blocks, d_ctx[s_:].data_ptr(), 1,
                             Hq, C, w.softmax_scale, sh)
                ev_ = torch.cuda.Event()
                ev_.record(stream)
                done.append(ev_)
            with torch.cuda.stream(cs):
                for s_, ev_ in enumerate(done):
                    cs.wait_event(ev_)
                    h_out[s_ * C:(s_ + 1) * C].copy_(d_out[s_ * C:(s_ + 1) * C], non_blocking=True)
            stream.wait_stream(cs)
            stream.synchronize()  # the step's results are in host memory
        for _ in range(2):
            e2e_step()
        _barrier(world)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(K):
            e2e_step()
        f1.record(stream)
        torch.cuda.synchronize()
        te = _max_over_ranks(f0.elapsed_time(f1) / 1e3, world)
        e2e = {"value": round(world * w.prefill_flops() * K / te / 1e12, 2), "unit": "TFLOP/s",
               "h2d_bytes_per_step": e2e_h2d,
               "d2h_bytes_per_step": h_out.numel() * h_out.element_size(),
               "ms_per_step": round(te / K * 1e3, 4)}
        # the per-sequence calls give the same result as the packet call
        ref_out = d_out.clone()
        step()
        torch.cuda.synchronize()
        if not torch.equal(ref_out, d_out) or not torch.equal(h_out, d_out.cpu()):
            raise RuntimeError("per-sequence prefill differs from the packet call")
    if pool.device_error():
        raise RuntimeError("device error in prefill")
    if rank != 0:
        return
    flops = w.prefill_flops()
    peak, peak_kind = _peak_tflops()
    achieved = flops / (statistics.fmean(pre_ms) / 1e3) / 1e12
    # against the peaks of the MMA kinds issued: e4m3 at twice the measured
    # bf16 rate (the nominal dense ratio, 4.5 / 2.25 PFLOP/s), binary16 at it
    f8_fl, f16_fl, blocks = _prefill_mma_work(w)
    t_peak = f8_fl / (2 * peak * 1e12) + f16_fl / (peak * 1e12)
    t_kernel = statistics.fmean(pre_ms) / 1e3
    mix = {"e4m3_flops_issued": f8_fl, "f16_flops_issued": f16_fl, "blocks": blocks,
           "e4m3_peak_tflops": round(2 * peak, 1), "f16_peak_tflops": peak,
           "ms_at_peak": round(t_peak * 1e3, 4), "frac": round(t_peak / t_kernel, 4)}
    line = {
        "metric": PREFILL_METRIC, "value": round(world * flops * K / t_max / 1e12, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(t_max / K * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 KV; tcgen05 MMA: e4m3 x e4m3 (Q K^T, q as two e4m3 terms) and f16 x f16 (P V); "
                 "f32 accumulate in tensor memory",
        "data": "synthetic (seeded N(0,1) q/k/v, random block tables)",
        "config": {"workload": DESCRIPTION[name], "tokens_per_step": T,
                   "flops_per_step": flops, "parallelism": "1 GPU" if world == 1 else
                   f"replicas x{world}"},
        "prefill_ms_median": round(statistics.median(pre_ms), 4),
        "prefill_ms_p10_p90": _p10_p90(pre_ms),
        "tokens_per_s": round(world * T * K / t_max, 1),
        "roofline": {"kernel": "prefill_tc_kernel (tcgen05)", "bound": "tensor", "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "algorithmic_flops_per_step": flops,
                     "mma_mix": mix},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": 2 * K, "clocks": sampler.summary(),
    }
    print(json.dumps(line), flush=True)


def run_prefix_cache(args, rank, world, local_rank):
    """Prompts sharing a system prompt, served with and without the prefix cache."""
    import torch

    from paged_kv_cache_270_gb300 import _native as N
    from paged_kv_cache_270_gb300 import workloads as W
    from paged_kv_cache_270_gb300.pool import KVPool
    torch.cuda.set_device(local_rank)
    ps = W.PrefixShare()
    R, P = ps.n_requests, ps.prefix_tokens
    suf = ps.suffix_lens()
    rng = np.random.default_rng(ps.seed + 7)
    system = rng.integers(0, 128000, P).astype(np.int32)
    prompts = [np.concatenate([system, rng.integers(0, 128000, int(n)).astype(np.int32)])
               for n in suf]
    kp, vp = ps.prefix_kv(P)
    sk = [ps.suffix_kv(r, int(n)) for r, n in enumerate(suf)]
    bt = lambda a_: torch.from_numpy(np.ascontiguousarray(a_).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    d_kp, d_vp = bt(kp), bt(vp)
    d_ks, d_vs = bt(np.concatenate([k for k, _ in sk])), bt(np.concatenate([v for _, v in sk]))
    d_kf = bt(np.concatenate([np.concatenate([kp, k]) for k, _ in sk]))
    d_vf = bt(np.concatenate([np.concatenate([vp, v]) for _, v in sk]))
    ctx = (P + suf).astype(np.int32)
    width = int(-(-ctx.max() // 16))
    q_suf = bt(ps.q_bits(int(suf.sum())))
    q_full = bt(ps.q_bits(int(ctx.sum()), step=1))
    d_ctx = torch.from_numpy(ctx).cuda()
    qs_suf = torch.from_numpy(np.concatenate([[0], np.cumsum(suf)]).astype(np.int32)).cuda()
    qs_full = torch.from_numpy(np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)).cuda()
    out_suf, out_full = torch.empty_like(q_suf), torch.empty_like(q_full)
    blocks_needed = int(sum(-(-int(c) // 16) for c in ctx))
    cached = KVPool(1, 128 + blocks_needed, 8, 128, "bf16")
    plain = KVPool(1, blocks_needed, 8, 128, "bf16")
    sh = int(torch.cuda.current_stream().cuda_stream)
    # the system prompt is prefilled once and registered
    sys_hashes = N.pa_prefix_hash(system)
    sys_ids = cached.alloc(len(sys_hashes))
    pos = np.arange(P, dtype=np.int64)
    cached.reshape_and_cache(d_kp, d_vp, torch.from_numpy(sys_ids[pos // 16].astype(np.int64) * 16
                                                           + pos % 16).cuda())
    cached.prefix_register(sys_hashes, sys_ids)
    N.pa_block_free(cached.handle, sys_ids)  # only the cache holds the system prompt now

    def serve(pool, use_cache):
        tables = np.zeros((R, width), np.int32)
        slots, held = [], []
        lookups = hits = 0
        for r in range(R):
            n = int(ctx[r])
            hit = np.zeros(0, np.int32)
            if use_cache:
                hs = N.pa_prefix_hash(prompts[r])
                hit = N.pa_prefix_lookup(pool.handle, hs)
                lookups += len(hs)
                hits += len(hit)
            own = N.pa_block_alloc(pool.handle, -(-n // 16) - len(hit))
            row = np.concatenate([hit, own]).astype(np.int32)
            tables[r, :len(row)] = row
            held.append(row)
            first = P if use_cache else 0
            p_ = np.arange(first, n, dtype=np.int64)
            slots.append(row[p_ // 16].astype(np.int64) * 16 + p_ % 16)
        d_slots = torch.from_numpy(np.concatenate(slots)).cuda()
        d_tab = torch.from_numpy(tables).cuda()
        if use_cache:
            N.pa_reshape_and_cache(pool.handle, 0, d_ks.data_ptr(), d_vs.data_ptr(),
                                   d_slots.data_ptr(), d_slots.numel(), sh)
            N.pa_prefill(pool.handle, 0, out_suf.data_ptr(), N.PA_BF16, q_suf.data_ptr(),
                         qs_suf.data_ptr(), d_tab.data_ptr(), width, d_ctx.data_ptr(), R, 32,
                         int(suf.max()), 1.0 / math.sqrt(128), sh)
        else:
            N.pa_reshape_and_cache(pool.handle, 0, d_kf.data_ptr(), d_vf.data_ptr(),
                                   d_slots.data_ptr(), d_slots.numel(), sh)
            N.pa_prefill(pool.handle, 0, out_full.data_ptr(), N.PA_BF16, q_full.data_ptr(),
                         qs_full.data_ptr(), d_tab.data_ptr(), width, d_ctx.data_ptr(), R, 32,
                         int(ctx.max()), 1.0 / math.sqrt(128), sh)
        torch.cuda.synchronize()
        for row in held:
            N.pa_block_free(pool.handle, row)
        return lookups, hits

    res = {}
    for mode, pool in (("cached", cached), ("uncached", plain)):
        for _ in range(args.warmup):
            serve(pool, mode == "cached")
        if pool.device_error():
            raise RuntimeError("device error in prefix-cache warm-up")
        _barrier(world)
        t0 = time.perf_counter()
        lk = ht = 0
        for _ in range(args.steps):
            a_, b_ = serve(pool, mode == "cached")
            lk += a_
            ht += b_
        t = _max_over_ranks(time.perf_counter() - t0, world)
        res[mode] = (t / args.steps, lk, ht)
    if rank != 0:
        return
    tokens = int(ctx.sum())
    t_c, lk, ht = res["cached"]
    t_u = res["uncached"][0]
    line = {"metric": PREFIX_METRIC, "value": round(world * tokens / t_c, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_c * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 KV / bf16 tensor-core MMA / f32 accumulate",
            "data": "synthetic (seeded token ids and N(0,1) q/k/v)",
            "config": {"workload": DESCRIPTION["prefix_cache_bf16"], "prompt_tokens": tokens,
                       "requests": R, "timing": "host wall clock around whole steps "
                       "(hashing, lookups, allocation, uploads, kernels, releases)"},
            "uncached_tokens_per_s": round(world * tokens / t_u, 1),
            "uncached_ms_per_step": round(t_u * 1e3, 3),
            "speedup_vs_uncached": round(t_u / t_c, 3),
            "block_hit_rate": round(ht / max(lk, 1), 4),
            "gpu_launches": 2 * args.steps, "e2e": None, "cpu_baseline": None}
    print(json.dumps(line), flush=True)


def run_swap(args, rank, world, local_rank):
    """Block swap-out / swap-in bandwidth next to contiguous host copies."""
    import torch

    from paged_kv_cache_270_gb300.pool import KVPool
    torch.cuda.set_device(local_rank)
    nb, n = 16384, 8192
    pool = KVPool(1, nb, 8, 128, "fp8_e4m3", 0.01, 0.01)
    g = torch.Generator(device="cuda").manual_seed(3)
    pool.k_cache.copy_(torch.randint(0, 256, (pool.k_cache.numel(),), dtype=torch.uint8,
                                     device="cuda", generator=g))
    pool.v_cache.copy_(torch.randint(0, 256, (pool.v_cache.numel(),), dtype=torch.uint8,
                                     device="cuda", generator=g))
    perm = np.random.default_rng(9).permutation(nb).astype(np.int32)
    src = torch.from_numpy(perm[:n]).cuda()
    dst = torch.from_numpy(perm[n:]).cuda()
    per = pool.swap_block_bytes()
    buf = torch.empty(n * per, dtype=torch.uint8).pin_memory()
    dev = torch.empty(n * per, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        _barrier(world)
        a_, b_ = ev(), ev()
        a_.record(stream)
        for _ in range(args.steps):
            fn()
        b_.record(stream)
        torch.cuda.synchronize()
        return _max_over_ranks(a_.elapsed_time(b_) / 1e3 / args.steps, world)

    t_out = timed(lambda: pool.swap_out(src, buf))
    t_in = timed(lambda: pool.swap_in(dst, buf))
    t_d2h = timed(lambda: buf.copy_(dev, non_blocking=True))
    t_h2d = timed(lambda: dev.copy_(buf, non_blocking=True))
    if pool.device_error():
        raise RuntimeError("device error in swap")
    if rank != 0:
        return
    nbytes = n * per
    gb = lambda t: round(nbytes / t / 1e9, 1)  # noqa: E731
    line = {"metric": SWAP_METRIC, "value": round(world * 2 * nbytes / (t_out + t_in) / 1e9, 1),
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round((t_out + t_in) * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u8",
            "data": "synthetic (random bytes, random block ids)",
            "config": {"workload": DESCRIPTION["kv_swap_fp8"], "bytes_each_way": nbytes},
            "swap_out_gbs": gb(t_out), "swap_in_gbs": gb(t_in),
            "contiguous_d2h_gbs": gb(t_d2h), "contiguous_h2d_gbs": gb(t_h2d),
            "frac_of_contiguous": {"out": round(t_d2h / t_out, 3), "in": round(t_h2d / t_in, 3)},
            "gpu_launches": 2 * args.steps, "e2e": None, "cpu_baseline": None}
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The fp64 oracle on the host cores, a bounded sample of the workload per step."""
    if rank != 0:
        return
    names = WORKLOADS[args.workload]
    from paged_kv_cache_270_gb300 import workloads as W
    procs = max(1, os.cpu_count() or 1)
    ctx_mp = mp.get_context("spawn")
    scales = {}
    with ctx_mp.Pool(procs) as pool:
        for name in names:
            w = W.make(name)
            if w.kv_dtype == "fp8_e4m3":
                chunks = [(name, s, lo, min(int(w.ctx_lens[s]), lo + 16384))
                          for s in range(w.S) for lo in range(0, int(w.ctx_lens[s]), 16384)]
                ka = va = 0.0
                for a, b in pool.imap_unordered(_gen_amax, chunks, chunksize=4):
                    ka, va = max(ka, a), max(va, b)
                scales[name] = (float(np.float32(ka) / np.float32(448.0)),
                                float(np.float32(va) / np.float32(448.0)))
            else:
                scales[name] = (1.0, 1.0)
        per_step = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
        for _ in range(args.warmup):
            cpu_baseline(names, scales, per_step / 4, procs, pool, single_core=False)
        vals, t_total = [], 0.0
        last = None
        for _ in range(args.steps):
            t0 = time.time()
            last = cpu_baseline(names, scales, per_step, procs, pool, single_core=False)
            t_total += time.time() - t0
            vals.append(last["value"])
    value = statistics.fmean(vals)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(t_total / args.steps * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) q/k/v, random block tables)",
            "config": {"workload": DESCRIPTION[args.workload],
                       "sample_per_step": last["sample"] if last else None},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": procs,
                             "kind": "oracle", "sample": last["sample"] if last else None,
                             "cpu_model": _cpu_model()},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama3_70b_fp8")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--decode-splits", type=int, default=0,
                    help="decode with this fixed split count (or -1: the balanced schedule) "
                         "instead of the automatic split count")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the records of the other decode configurations (default workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = _env_rank()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "gb300" else "gloo")
    try:
        if args.workload == "kv_swap_fp8":
            if args.impl == "reference":
                if rank == 0:
                    print(json.dumps({"impl": "reference", "unavailable":
                                      "the oracle leg covers the decode workloads only"}))
            else:
                run_swap(args, rank, world, local_rank)
        elif args.workload == "prefix_cache_bf16":
            if args.impl == "reference":
                if rank == 0:
                    print(json.dumps({"impl": "reference", "unavailable":
                                      "the oracle leg covers the decode workloads only"}))
            else:
                run_prefix_cache(args, rank, world, local_rank)
        elif args.workload.endswith("_prefill"):
            if args.impl == "reference":
                if rank == 0:
                    print(json.dumps({"impl": "reference", "unavailable":
                                      "the oracle leg covers the decode workloads only"}))
            else:
                run_prefill(args, rank, world, local_rank)
        elif args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gb300(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
