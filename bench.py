#!/usr/bin/env python3
"""Benchmark of the SAW-INT4 hot path on one GB300 (per rank).

Headline workload (the largest single-GPU configuration, Qwen3-32B-shaped
high concurrency): 64 layers, 64 q-heads, 8 kv-heads, head_dim 128, h = 128,
page 16, 256 sequences with contexts uniform in [4096, 8192], shuffled page
tables, K and V rotated.  One step = for every layer, append each sequence's
new token into that layer's paged INT4 cache and decode-attend over its
whole context (saw_decode_step: one fused launch per layer), replayed as one
CUDA graph.  value = algorithmic bytes of the step / step time (GB/s).

Also printed (rank 0, one JSON line): the decode kernel's HBM roofline
fraction, the quantize-append throughput of a 131072-token prefill chunk
(top-level tokens/s and fraction), the Qwen3-4B-shaped latency step (batch 1,
context 32768), decode alone on the other workloads, the end-to-end rate
through the public API with host buffers, and the CPU oracle timed on
bounded samples (all host cores and one core) together with its parity check
of the GPU's outputs on those samples.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl saw|reference]

--impl reference times the CPU oracle (test infrastructure) on the host
cores on a bounded sample of the headline workload: this method has no
installable reference implementation.  Under torchrun each rank runs an
independent replica (the path has no exchange step): value = bytes of all
ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "decode-attn KV GB/s & % HBM roofline; quantize-append tokens/s (1×GB300)"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ------------------------------------------------------------------ ncu traffic record

# The decode kernel's device code: these files whole, and the kernel's
# parameter block from saw_internal.h (the host-side declarations there do
# not change the kernel).
DECODE_SOURCES = ["paged_decode.cu", "saw_device.cuh", "saw_quant_row.cuh"]
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def decode_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_paged_kv_gb300", "csrc")
    for f in DECODE_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(csrc, "saw_internal.h"), "rb") as fh:
        text = fh.read()
    start = text.index(b"struct DecodeParams {")
    h.update(text[start:text.index(b"};", start) + 2])
    return h.hexdigest()


def decode_traffic(workload: str):
    """(DRAM bytes per launch, where the figure comes from) of the fused
    decode-step kernel on `workload`, from the committed ncu record
    (dram__bytes_read.sum + dram__bytes_write.sum of one capture).  The
    figure holds only for the sources it was captured from: when the
    kernel's sources have changed since, (None, the reason) is returned."""
    digest = decode_sources_sha256()
    recorded = []
    try:
        with open(TRAFFIC_RECORD) as fh:
            for line in fh:
                parts = line.split()
                if line.startswith("#") or len(parts) != 5 or parts[1] != workload:
                    continue
                recorded.append(parts[3])
                if parts[3] == digest:
                    return int(parts[4]), (f"ncu capture of one launch of {parts[0]} on "
                                           f"{workload} ({parts[2]})")
    except OSError:
        return None, "no ncu traffic record"
    if recorded:
        return None, (f"the decode kernel's sources (sha256 {digest[:12]}) changed since the "
                      f"ncu capture of {workload} (sha256 {recorded[-1][:12]}): not re-measured")
    return None, f"no ncu capture of the decode kernel on {workload}"


# ------------------------------------------------------------------ ranks

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_group(world: int):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("gloo")


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def reduce_over_ranks(seconds: float, units: float, world: int):
    """(max time over ranks, sum of units over ranks).  Replicas only: no data
    moves between ranks; this host-side reduction only aggregates timings."""
    if world <= 1:
        return seconds, units
    t = torch.tensor([seconds], dtype=torch.float64)
    u = torch.tensor([units], dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(u.item())


# ------------------------------------------------------------------ peaks, clocks

def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, earlier GB300 measurement)"


def read_tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s), burst figure: the prefill kernel is
    timed on its own.  Its MMAs are binary16, which runs at the bf16 rate."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"
    except Exception:
        return 1900.0, "fallback (1.9 PFLOP/s bf16 burst, earlier GB300 measurement)"


CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons (read-only)."""

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for r in csv.reader(io.StringIO(f.read())):
                if len(r) >= 9:
                    rows.append([x.strip() for x in r])
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        busy = [s for s in sm if s > 0]
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ workload

def time_events(fn, iters: int, stream) -> list[float]:
    """Per-iteration device time (ms) of fn() with CUDA events on `stream`."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(iters)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


class StepCase:
    """A decode step over every layer of a workload: per layer, the fused
    saw_decode_step appends each sequence's new token (position seq_len - 1)
    and attends over its whole context (one launch per layer).  Each layer's
    cache is prefilled with every token but the last of each sequence."""

    def __init__(self, wl, device):
        import bit_paged_kv_gb300 as saw
        from bit_paged_kv_gb300 import workloads as W
        self.saw, self.W, self.wl, self.dev = saw, W, wl, device
        self.lens = W.seq_lens(wl)
        self.L = int(self.lens.max())
        self.bt_cpu, self.npages = W.page_tables(wl, self.lens)
        self.bt = self.bt_cpu.to(device)
        self.lens_d = self.lens.to(device)
        B, Hq, Hkv, D, P = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size
        nb = saw.saw_cache_bytes(self.npages, P, Hkv, D)
        self.pre = [int(x) - 1 for x in self.lens.tolist()]
        self.n_pre = sum(self.pre)
        self.pre_slots = W.prefill_slots(self.bt, self.pre, P)
        self.kc, self.vc = [], []
        status = torch.zeros(1, dtype=torch.int32, device=device)
        # per-step inputs: each layer's new token of every sequence (the next
        # rows of the layer's stream after the prefill) and q
        self.knew = torch.empty(wl.num_layers, B, Hkv, D, dtype=torch.bfloat16, device=device)
        self.vnew = torch.empty(wl.num_layers, B, Hkv, D, dtype=torch.bfloat16, device=device)
        for layer in range(wl.num_layers):
            kc = torch.empty(nb, dtype=torch.uint8, device=device)
            vc = torch.empty(nb, dtype=torch.uint8, device=device)
            k = W.kv_rows(wl, layer, W.K, self.n_pre + B, device)
            v = W.kv_rows(wl, layer, W.V, self.n_pre + B, device)
            saw.saw_quantize_append(k[:self.n_pre], v[:self.n_pre], self.pre_slots, kc, vc,
                                    self.npages, P, wl.rotate_k, wl.rotate_v, wl.block_h,
                                    dev_status=status)
            self.knew[layer] = k[self.n_pre:]
            self.vnew[layer] = v[self.n_pre:]
            del k, v
            self.kc.append(kc)
            self.vc.append(vc)
        self.slot = torch.cat([W.slots_for(self.bt, P, b, int(Lb) - 1, int(Lb))
                               for b, Lb in enumerate(self.lens.tolist())])
        self.q = torch.stack([W.q_rows(wl, l, device) for l in range(wl.num_layers)])
        self.out = torch.empty(wl.num_layers, B, Hq, D, dtype=torch.float32, device=device)
        self.splits, self.pps = saw.saw_decode_plan(B, Hkv, P, self.L, 0)
        wsb = saw.saw_decode_workspace_bytes(B, Hq, Hkv, D, P, self.L, 0)
        self.ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=device) if wsb else None
        self.status = status
        torch.cuda.synchronize()
        assert int(status.item()) == 0

    def pre_rows(self, layer):
        """The bfloat16 K and V rows the prefill appended to `layer`."""
        W, wl = self.W, self.wl
        return (W.kv_rows(wl, layer, W.K, self.n_pre, self.dev),
                W.kv_rows(wl, layer, W.V, self.n_pre, self.dev))

    def decode_step(self, layer):
        """The fused step of one layer: append the new tokens, then attend."""
        wl = self.wl
        self.saw.saw_decode_step(self.q[layer], self.knew[layer], self.vnew[layer],
                                 self.kc[layer], self.vc[layer], self.bt, self.lens_d, self.L,
                                 wl.num_kv_heads, self.npages, wl.page_size, wl.rotate_k,
                                 wl.rotate_v, wl.block_h, self.out[layer], self.ws,
                                 flags=self.saw.SAW_STEP_EARLY_PAGES, dev_status=self.status)

    def step(self):
        for layer in range(self.wl.num_layers):
            self.decode_step(layer)

    def launches_per_step(self) -> int:
        return self.wl.num_layers

    def decode_bytes(self) -> int:
        return self.W.decode_bytes(self.wl, self.lens.tolist())

    def layer_bytes(self) -> int:
        """Algorithmic bytes of one fused decode step of one layer."""
        return self.decode_bytes() + self.W.append_bytes(self.wl, self.wl.num_seqs)

    def step_bytes(self) -> int:
        return self.wl.num_layers * self.layer_bytes()

    def release(self):
        del self.kc, self.vc, self.q, self.knew, self.vnew, self.out, self.ws
        torch.cuda.empty_cache()


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm (sets kernel attributes outside capture)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def append_chunk_measure(device, stream, iters: int = 20, keep: bool = False):
    """Quantize-append of one 131072-token prefill chunk (8 kv-heads, K and V,
    page 64), rotated (h = 128 and 64) and unrotated.  Inputs are 512 MB,
    larger than L2.  keep: also return host copies of the rows, slots and
    the h = 128 cache bytes (for the oracle's leg)."""
    import bit_paged_kv_gb300 as saw
    from bit_paged_kv_gb300 import workloads as W
    wl = W.LONG_PREFILL.variant(num_seqs=1)
    T = wl.len_hi
    lens = torch.tensor([T], dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens)
    k = W.kv_rows(wl, 0, W.K, T, device)
    v = W.kv_rows(wl, 0, W.V, T, device)
    slots = W.prefill_slots(bt.to(device), [T], wl.page_size)
    nb = saw.saw_cache_bytes(npages, wl.page_size, wl.num_kv_heads, wl.head_dim)
    kc = torch.empty(nb, dtype=torch.uint8, device=device)
    vc = torch.empty(nb, dtype=torch.uint8, device=device)
    res = {}
    nbytes = W.append_bytes(wl, T)
    for name, rk, rv, h in (("rotated_h128", True, True, 128), ("rotated_h64", True, True, 64),
                            ("unrotated", False, False, 128)):
        def fn():
            saw.saw_quantize_append(k, v, slots, kc, vc, npages, wl.page_size, rk, rv, h)
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            t = statistics.median(time_events(fn, iters, stream))
        res[name] = {"tokens_per_s": T / (t * 1e-3), "ms": t, "gbs": nbytes / (t * 1e-3) / 1e9}
    kept = None
    if keep:
        # the h = 128 result, for the oracle's leg (rows, slots, cache bytes)
        saw.saw_quantize_append(k, v, slots, kc, vc, npages, wl.page_size, True, True, 128)
        torch.cuda.synchronize()
        kept = {"wl": wl, "k": np_bits(k).reshape(T, -1), "v": np_bits(v).reshape(T, -1),
                "slots": slots.cpu().numpy(), "npages": npages,
                "kc_gpu": kc.cpu().numpy(), "vc_gpu": vc.cpu().numpy()}
    del k, v, kc, vc
    torch.cuda.empty_cache()
    return res, nbytes, T, kept


def fill_caches(wl, layer, lens, bt, npages, device, chunk_tokens=1 << 18,
                dtype=torch.bfloat16, meta_bf16=False):
    """One layer's K and V caches holding every token of every sequence,
    written by the library's quantize-append (seeded synthetic rows of
    `dtype`, metadata as bfloat16 if meta_bf16)."""
    import bit_paged_kv_gb300 as saw
    from bit_paged_kv_gb300 import workloads as W
    P = wl.page_size
    lens_l = [int(x) for x in lens.tolist()]
    total = sum(lens_l)
    nb = saw.saw_cache_bytes(npages, P, wl.num_kv_heads, wl.head_dim)
    kc = torch.empty(nb, dtype=torch.uint8, device=device)
    vc = torch.empty(nb, dtype=torch.uint8, device=device)
    slots = W.prefill_slots(bt.to(device), lens_l, P)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    for a in range(0, total, chunk_tokens):
        b = min(total, a + chunk_tokens)
        k = W.kv_rows(wl, layer, W.K, b - a, device, token_offset=a, dtype=dtype)
        v = W.kv_rows(wl, layer, W.V, b - a, device, token_offset=a, dtype=dtype)
        saw.saw_quantize_append(k, v, slots[a:b], kc, vc, npages, P, wl.rotate_k, wl.rotate_v,
                                wl.block_h, dev_status=status, meta_bf16=meta_bf16)
        del k, v
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return kc, vc


def decode_config_measure(device, stream, layers: int = 2, reps: int = 10, only=None, keep=None):
    """Decode-only throughput of the bandwidth-bound workloads (Qwen3-8B
    concurrent, Qwen3-32B high concurrency in its three rotation variants,
    long context at h 128 and 64): `layers` distinct layer caches (each
    larger than L2) decoded in turn, CUDA events around reps passes.  keep:
    names whose first layer (cache, q, output) is copied to the host for the
    oracle's leg; returned as a third item."""
    import bit_paged_kv_gb300 as saw
    from bit_paged_kv_gb300 import workloads as W
    kept = {}
    c32 = W.QWEN3_32B_HIGH_CONCURRENCY
    cases = [("qwen3-8b-concurrent", W.QWEN3_8B_CONCURRENT),
             ("qwen3-32b-high-concurrency k+v", c32),
             ("qwen3-32b-high-concurrency k-only", c32.variant(rotate_k=True, rotate_v=False)),
             ("qwen3-32b-high-concurrency unrotated", c32.variant(rotate_k=False, rotate_v=False)),
             ("long-131072 h128", W.LONG_PREFILL),
             ("long-131072 h64", W.LONG_PREFILL.variant(block_h=64))]
    if only is not None:
        cases = [(n, w) for n, w in cases if n in only]
    res = {}
    for name, wl in cases:
        lens = W.seq_lens(wl)
        bt, npages = W.page_tables(wl, lens)
        btd, lensd = bt.to(device), lens.to(device)
        B, Hq, D = wl.num_seqs, wl.num_q_heads, wl.head_dim
        Lmax = int(lens.max())
        caches = [fill_caches(wl, l, lens, bt, npages, device) for l in range(layers)]
        qs = [W.q_rows(wl, l, device) for l in range(layers)]
        wsb = saw.saw_decode_workspace_bytes(B, Hq, wl.num_kv_heads, D, wl.page_size, Lmax, 0)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=device) if wsb else None
        out = torch.empty(B, Hq, D, dtype=torch.float32, device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize()  # the zero fills ran on the default stream

        def one_pass():
            for l in range(layers):
                saw.saw_paged_decode_int4(qs[l], caches[l][0], caches[l][1], btd, lensd, Lmax,
                                          wl.num_kv_heads, npages, wl.page_size, wl.rotate_k,
                                          wl.rotate_v, wl.block_h, out, ws, dev_status=status)
        with torch.cuda.stream(stream):
            for _ in range(2):
                one_pass()
            t = statistics.median(time_events(one_pass, reps, stream)) / layers
        assert int(status.item()) == 0
        if keep and name in keep:
            saw.saw_paged_decode_int4(qs[0], caches[0][0], caches[0][1], btd, lensd, Lmax,
                                      wl.num_kv_heads, npages, wl.page_size, wl.rotate_k,
                                      wl.rotate_v, wl.block_h, out, ws, dev_status=status)
            torch.cuda.synchronize()
            assert int(status.item()) == 0
            kept[name] = {"wl": wl, "kc": caches[0][0].cpu().numpy(),
                          "vc": caches[0][1].cpu().numpy(), "q": np_bits(qs[0]),
                          "out": out.cpu().numpy(), "bt": bt.numpy(), "lens": lens.numpy(),
                          "npages": npages}
        nbytes = W.decode_bytes(wl, lens.tolist())
        splits, pps = saw.saw_decode_plan(B, wl.num_kv_heads, wl.page_size, Lmax, 0)
        res[name] = {"ms_per_layer": t, "gbs": nbytes / (t * 1e-3) / 1e9,
                     "bytes_per_layer": nbytes, "splits": splits, "pages_per_split": pps,
                     "seqs": B, "tokens": int(lens.sum())}
        del caches, qs, ws, out
        torch.cuda.empty_cache()
    if only is not None:
        return res, None, kept
    a = res["qwen3-32b-high-concurrency k+v"]["ms_per_layer"]
    k1 = res["qwen3-32b-high-concurrency k-only"]["ms_per_layer"]
    u = res["qwen3-32b-high-concurrency unrotated"]["ms_per_layer"]
    overhead = {"k+v_vs_unrotated": a / u - 1.0, "k-only_vs_unrotated": k1 / u - 1.0}
    return res, overhead, kept


def fill_caches_bf16(wl, layer, lens, bt, npages, device, chunk_tokens=1 << 18):
    """One layer's BF16 K and V caches holding every token of every sequence
    (the same seeded rows as fill_caches), written by saw_bf16_append."""
    import bit_paged_kv_gb300 as saw
    from bit_paged_kv_gb300 import workloads as W
    P = wl.page_size
    lens_l = [int(x) for x in lens.tolist()]
    total = sum(lens_l)
    n = saw.saw_bf16_cache_bytes(npages, P, wl.num_kv_heads, wl.head_dim) // 2
    kc = torch.empty(n, dtype=torch.int16, device=device)
    vc = torch.empty(n, dtype=torch.int16, device=device)
    slots = W.prefill_slots(bt.to(device), lens_l, P)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    for a in range(0, total, chunk_tokens):
        b = min(total, a + chunk_tokens)
        k = W.kv_rows(wl, layer, W.K, b - a, device, token_offset=a)
        v = W.kv_rows(wl, layer, W.V, b - a, device, token_offset=a)
        saw.saw_bf16_append(k, v, slots[a:b], kc, vc, npages, P, dev_status=status)
        del k, v
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return kc, vc


def concurrency_sweep(device, stream, batches=(1, 4, 16, 64, 128, 256), reps=10,
                      min_pool=600_000_000):
    """INT4 (rotated, saw_paged_decode_int4) against BF16 (saw_paged_decode_bf16)
    decode attention on the qwen3-8b-concurrent shape (Hq 32, Hkv 8, page 16,
    lengths uniform in [2048, 16384]) at 1..256 concurrent sequences.  Each
    side decodes enough copies of its layer cache in turn (at least 600 MB,
    2..64 copies) that every pass reads from HBM, not L2."""
    import bit_paged_kv_gb300 as saw
    from bit_paged_kv_gb300 import workloads as W
    base = W.QWEN3_8B_CONCURRENT
    rows = []
    for B in batches:
        wl = base.variant(num_seqs=B)
        lens = W.seq_lens(wl)
        bt, npages = W.page_tables(wl, lens)
        btd, lensd = bt.to(device), lens.to(device)
        Hq, Hkv, D, P = wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size
        Lmax = int(lens.max())
        q = W.q_rows(wl, 0, device)
        out = torch.empty(B, Hq, D, dtype=torch.float32, device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        row = {"seqs": B, "tokens": int(lens.sum())}
        for kind in ("int4", "bf16"):
            if kind == "int4":
                kc, vc = fill_caches(wl, 0, lens, bt, npages, device, chunk_tokens=1 << 20)
                wsb = saw.saw_decode_workspace_bytes(B, Hq, Hkv, D, P, Lmax, 0)
                nbytes = W.decode_bytes(wl, lens.tolist())
            else:
                kc, vc = fill_caches_bf16(wl, 0, lens, bt, npages, device, chunk_tokens=1 << 20)
                wsb = saw.saw_decode_bf16_workspace_bytes(B, Hq, Hkv, D, P, Lmax)
                nbytes = W.decode_bytes_bf16(wl, lens.tolist())
            cache_bytes = 2 * kc.numel() * kc.element_size()
            copies = max(2, min(64, -(-min_pool // cache_bytes)))
            pool = [(kc, vc)] + [(kc.clone(), vc.clone()) for _ in range(copies - 1)]
            ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=device) if wsb else None
            torch.cuda.synchronize()  # the zero fill and the clones ran on the default stream

            def one_pass():
                for k_, v_ in pool:
                    if kind == "int4":
                        saw.saw_paged_decode_int4(q, k_, v_, btd, lensd, Lmax, Hkv, npages, P,
                                                  wl.rotate_k, wl.rotate_v, wl.block_h, out, ws,
                                                  dev_status=status)
                    else:
                        saw.saw_paged_decode_bf16(q, k_, v_, btd, lensd, Lmax, Hkv, npages, P,
                                                  out, ws, dev_status=status)
            with torch.cuda.stream(stream):
                for _ in range(2):
                    one_pass()
                t = statistics.median(time_events(one_pass, reps, stream)) / copies
            assert int(status.item()) == 0
            row[kind] = {"ms_per_layer": t, "gbs": nbytes / (t * 1e-3) / 1e9,
                         "bytes_per_layer": nbytes, "copies": copies,
                         "decode_tokens_per_s_36_layers": B / (36 * t * 1e-3)}
            del pool, kc, vc, ws
            torch.cuda.empty_cache()
        row["int4_speedup"] = row["bf16"]["ms_per_layer"] / row["int4"]["ms_per_layer"]
        rows.append(row)
    return rows


def prefill_flops(num_q_heads: int, head_dim: int, seq_len: int, q_len: int) -> int:
    """Useful FLOPs of causal attention for one chunk: each query at position
    p does 2 D FLOPs per key for Q K^T and 2 D for P V over p + 1 keys."""
    first = seq_len - q_len + 1        # keys seen by the first query
    keys = (first + seq_len) * q_len // 2
    return 4 * head_dim * num_q_heads * keys


def prefill_measure(device, stream, reps: int = 5):
    """saw_prefill_attn_int4 on the long-context workload (Hq 32, Hkv 8, page
    64, h 128, K and V rotated; the cache holds 131072 tokens): the last
    8192-token chunk at context 131072, and a whole 16384-token prompt.  L2
    is flushed (a 256 MB write) before every timed launch."""
    import bit_paged_kv_gb300 as saw
    from bit_paged_kv_gb300 import workloads as W
    wl = W.LONG_PREFILL.variant(num_seqs=1)
    Lfull = wl.len_hi
    lens_full = torch.tensor([Lfull], dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens_full)
    kc, vc = fill_caches(wl, 0, lens_full, bt, npages, device)
    btd = bt.to(device)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    peak, peak_src = read_tensor_peak()
    g = torch.Generator(device=device).manual_seed(11)
    res = {}
    for name, L, n in (("chunk 8192 at context 131072", Lfull, 8192),
                       ("prompt 16384", 16384, 16384)):
        q = torch.randn(n, wl.num_q_heads, wl.head_dim, generator=g, device=device).to(torch.bfloat16)
        out = torch.empty(n, wl.num_q_heads, wl.head_dim, dtype=torch.float32, device=device)
        cu = torch.tensor([0, n], dtype=torch.int32, device=device)
        sl = torch.tensor([L], dtype=torch.int32, device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

        def run():
            saw.saw_prefill_attn_int4(q, cu, kc, vc, btd, sl, n, L, wl.num_kv_heads, npages,
                                      wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h, out,
                                      dev_status=status)
        times = []
        with torch.cuda.stream(stream):
            run()
            for _ in range(reps):
                flush.fill_(1)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                run()
                b.record(stream)
                b.synchronize()
                times.append(a.elapsed_time(b))
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        t = statistics.median(times)
        fl = prefill_flops(wl.num_q_heads, wl.head_dim, L, n)
        tf = fl / (t * 1e-3) / 1e12
        res[name] = {"ms": t, "flops": fl, "tflops": tf, "frac": tf / peak,
                     "tokens_per_s": n / (t * 1e-3)}
        del q, out
    del kc, vc, flush
    torch.cuda.empty_cache()
    return res, peak, peak_src


def variants_measure(device, stream, reps: int = 10):
    """head_dim 64 and 256: decode alone (the tensor-core decode built for
    those sizes) on the
    qwen3-8b-concurrent shape (64 sequences, lengths in [2048, 16384], K and V
    rotated with h = head_dim, two layer caches decoded in turn), and the
    quantize-append of a 131072-token chunk (Hkv 8, K and V, page 64)."""
    import bit_paged_kv_gb300 as saw
    from bit_paged_kv_gb300 import workloads as W
    res = {}
    for D in (64, 256):
        wl = W.QWEN3_8B_CONCURRENT.variant(head_dim=D, block_h=D)
        lens = W.seq_lens(wl)
        bt, npages = W.page_tables(wl, lens)
        btd, lensd = bt.to(device), lens.to(device)
        B, Hq = wl.num_seqs, wl.num_q_heads
        Lmax = int(lens.max())
        caches = [fill_caches(wl, l, lens, bt, npages, device, chunk_tokens=1 << 20) for l in range(2)]
        qs = [W.q_rows(wl, l, device) for l in range(2)]
        wsb = saw.saw_decode_workspace_bytes(B, Hq, wl.num_kv_heads, D, wl.page_size, Lmax, 0)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=device) if wsb else None
        out = torch.empty(B, Hq, D, dtype=torch.float32, device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

        def one_pass():
            for l in range(2):
                saw.saw_paged_decode_int4(qs[l], caches[l][0], caches[l][1], btd, lensd, Lmax,
                                          wl.num_kv_heads, npages, wl.page_size, True, True, D,
                                          out, ws, dev_status=status)
        with torch.cuda.stream(stream):
            for _ in range(2):
                one_pass()
            t = statistics.median(time_events(one_pass, reps, stream)) / 2
        assert int(status.item()) == 0
        nbytes = W.decode_bytes(wl, lens.tolist())
        res[f"decode head_dim {D}"] = {"ms_per_layer": t, "gbs": nbytes / (t * 1e-3) / 1e9,
                                       "bytes_per_layer": nbytes}
        del caches, qs, ws, out
        torch.cuda.empty_cache()
        # bulk append
        wa = W.LONG_PREFILL.variant(num_seqs=1, head_dim=D, block_h=D)
        T = wa.len_hi
        lens1 = torch.tensor([T], dtype=torch.int32)
        bt1, np1 = W.page_tables(wa, lens1)
        k = W.kv_rows(wa, 0, W.K, T, device)
        v = W.kv_rows(wa, 0, W.V, T, device)
        slots = W.prefill_slots(bt1.to(device), [T], wa.page_size)
        nb = saw.saw_cache_bytes(np1, wa.page_size, wa.num_kv_heads, D)
        kc = torch.empty(nb, dtype=torch.uint8, device=device)
        vc = torch.empty(nb, dtype=torch.uint8, device=device)
        torch.cuda.synchronize()

        def app():
            saw.saw_quantize_append(k, v, slots, kc, vc, np1, wa.page_size, True, True, D)
        with torch.cuda.stream(stream):
            for _ in range(3):
                app()
            t = statistics.median(time_events(app, reps, stream))
        ab = W.append_bytes(wa, T)
        res[f"append head_dim {D}"] = {"ms": t, "gbs": ab / (t * 1e-3) / 1e9,
                                       "tokens_per_s": T / (t * 1e-3), "bytes": ab}
        del k, v, kc, vc
        torch.cuda.empty_cache()
    return res


def formats_measure(device, stream, reps: int = 10):
    """The format variants (binary16 input, bfloat16 metadata, both) beside
    the plain formats, on two shapes: decode alone on qwen3-8b-concurrent
    (64 sequences, lengths in [2048, 16384], head_dim 128, K and V rotated,
    two layer caches decoded in turn), and the quantize-append of a
    131072-token chunk (Hkv 8, K and V, page 64, h 128).  The algorithmic
    bytes are the same for every format."""
    import bit_paged_kv_gb300 as saw
    from bit_paged_kv_gb300 import workloads as W
    res = {}
    fmts = [("bf16 input, fp16 meta", torch.bfloat16, False),
            ("fp16 input, fp16 meta", torch.float16, False),
            ("bf16 input, bf16 meta", torch.bfloat16, True),
            ("fp16 input, bf16 meta", torch.float16, True)]
    wl = W.QWEN3_8B_CONCURRENT
    lens = W.seq_lens(wl)
    bt, npages = W.page_tables(wl, lens)
    btd, lensd = bt.to(device), lens.to(device)
    B, Hq, D = wl.num_seqs, wl.num_q_heads, wl.head_dim
    Lmax = int(lens.max())
    nbytes = W.decode_bytes(wl, lens.tolist())
    wa = W.LONG_PREFILL.variant(num_seqs=1)
    T = wa.len_hi
    lens1 = torch.tensor([T], dtype=torch.int32)
    bt1, np1 = W.page_tables(wa, lens1)
    slots = W.prefill_slots(bt1.to(device), [T], wa.page_size)
    ab = W.append_bytes(wa, T)
    for name, dt, bfm in fmts:
        caches = [fill_caches(wl, l, lens, bt, npages, device, chunk_tokens=1 << 20, dtype=dt,
                              meta_bf16=bfm) for l in range(2)]
        qs = [W.q_rows(wl, l, device, dtype=dt) for l in range(2)]
        wsb = saw.saw_decode_workspace_bytes(B, Hq, wl.num_kv_heads, D, wl.page_size, Lmax, 0)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=device) if wsb else None
        out = torch.empty(B, Hq, D, dtype=torch.float32, device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

        def one_pass():
            for l in range(2):
                saw.saw_paged_decode_int4(qs[l], caches[l][0], caches[l][1], btd, lensd, Lmax,
                                          wl.num_kv_heads, npages, wl.page_size, wl.rotate_k,
                                          wl.rotate_v, wl.block_h, out, ws, dev_status=status,
                                          meta_bf16=bfm)
        with torch.cuda.stream(stream):
            for _ in range(2):
                one_pass()
            t = statistics.median(time_events(one_pass, reps, stream)) / 2
        assert int(status.item()) == 0
        entry = {"decode_ms_per_layer": t, "decode_gbs": nbytes / (t * 1e-3) / 1e9}
        del caches, qs, ws, out
        torch.cuda.empty_cache()
        k = W.kv_rows(wa, 0, W.K, T, device, dtype=dt)
        v = W.kv_rows(wa, 0, W.V, T, device, dtype=dt)
        nb = saw.saw_cache_bytes(np1, wa.page_size, wa.num_kv_heads, wa.head_dim)
        kc = torch.empty(nb, dtype=torch.uint8, device=device)
        vc = torch.empty(nb, dtype=torch.uint8, device=device)
        torch.cuda.synchronize()

        def app():
            saw.saw_quantize_append(k, v, slots, kc, vc, np1, wa.page_size, True, True,
                                    wa.block_h, meta_bf16=bfm)
        with torch.cuda.stream(stream):
            for _ in range(3):
                app()
            ta = statistics.median(time_events(app, reps, stream))
        entry.update({"append_ms": ta, "append_gbs": ab / (ta * 1e-3) / 1e9})
        res[name] = entry
        del k, v, kc, vc
        torch.cuda.empty_cache()
    return res


def np_bits(t):
    """bfloat16 / float16 tensor -> numpy uint16 bit patterns on the host."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def sample_decode_bytes(wl, lens, seqs, kv_heads_per_seq: int, pairs: int, appended: bool) -> int:
    """Algorithmic bytes of an oracle decode sample: K and V codes and
    (scale, zero) of every attended (token, kv-head), the sequences' block
    tables, q in and out for each (sequence, q-head) pair, and the appended
    token's rows when the sample includes the step's append."""
    from bit_paged_kv_gb300 import workloads as W
    P, D = wl.page_size, wl.head_dim
    per_row = D // 2 + 4
    n = 0
    for b in seqs:
        L = int(lens[b])
        n += 2 * per_row * L * kv_heads_per_seq + 4 * ((L + P - 1) // P)
    n += pairs * D * (2 + 4)
    if appended:
        n += len(seqs) * W.append_bytes(wl.variant(num_kv_heads=kv_heads_per_seq), 1)
    return n


def timed_passes(fn, min_seconds: float, max_passes: int):
    """Call fn() until min_seconds have gone (at least once); (seconds, passes)."""
    passes, t0 = 0, time.perf_counter()
    while True:
        fn()
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= max_passes:
            return dt, passes


def rel_max_err(got, ref) -> float:
    import numpy as np
    scale = float(np.max(np.abs(ref)))
    d = float(np.max(np.abs(got - ref)))
    return d / scale if scale > 0 else d


def cpu_oracle_legs(samples, threads: int, min_seconds: float = 1.5):
    """The oracle (as it stands), timed on the host cores on bounded samples
    of the GPU workloads, at all cores and at one core; while it runs, its
    results are compared with the GPU's outputs of the same inputs.

    samples: host copies of what the GPU computed (see run_saw).  Returns
    (legs, parity): legs[name] = {value, unit, cores, sample}; parity[name]
    = the comparison of that sample with the GPU (cache bytes equal, attention
    max |o_gpu - o_ref| / max |o_ref| against 2e-3)."""
    import numpy as np

    import oracle
    oracle.load()
    legs, parity = {}, {}

    # quantize-append: the long-context prefill chunk, R-canon butterfly
    a = samples["append"]
    wl = a["wl"]
    T = a["k"].shape[0]
    for cores, n in ((threads, T), (1, min(T, 8192))):
        kc = np.zeros_like(a["kc_gpu"])
        vc = np.zeros_like(a["vc_gpu"])

        def run(n=n, kc=kc, vc=vc, cores=cores):
            oracle.quantize_append(a["k"][:n], a["v"][:n], a["slots"][:n], wl.num_kv_heads,
                                   wl.head_dim, kc, vc, a["npages"], wl.page_size, wl.rotate_k,
                                   wl.rotate_v, wl.block_h, threads=cores)
        dt, passes = timed_passes(run, min_seconds, 20)
        legs[f"append cores={cores}"] = {
            "value": n * passes / dt, "unit": "tokens/s", "cores": cores,
            "sample": f"{n} tokens of the {T}-token chunk (Hkv {wl.num_kv_heads}, K and V, "
                      f"h {wl.block_h}), {passes} pass(es), {dt:.1f} s"}
        if n == T:
            parity["append long-131072 chunk"] = {
                "bytes_equal": bool(np.array_equal(kc, a["kc_gpu"]) and
                                    np.array_equal(vc, a["vc_gpu"])),
                "what": f"every cache byte of the {T}-token chunk"}

    # decode legs: the fused step's layer (configs 2 and 4), decode alone (config 5)
    for name, d in samples["decode"].items():
        wl = d["wl"]
        G = wl.num_q_heads // wl.num_kv_heads
        kc, vc = d["kc"], d["vc"]
        if d.get("new") is not None:
            # the step appended each sequence's new token: the oracle appends
            # the same rows into a copy of the GPU's cache; identical bytes
            # mean the GPU wrote exactly the oracle's codes and (scale, zero)
            kn, vn, sl = d["new"]
            kr, vr = kc.copy(), vc.copy()
            oracle.quantize_append(kn, vn, sl, wl.num_kv_heads, wl.head_dim, kr, vr, d["npages"],
                                   wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                                   threads=threads)
            if d.get("pre") is not None:
                # and the whole layer from scratch: prefill rows, then the new tokens
                kp, vp, sp = d["pre"]
                kr, vr = np.zeros_like(kc), np.zeros_like(vc)
                oracle.quantize_append(kp, vp, sp, wl.num_kv_heads, wl.head_dim, kr, vr,
                                       d["npages"], wl.page_size, wl.rotate_k, wl.rotate_v,
                                       wl.block_h, threads=threads)
                oracle.quantize_append(kn, vn, sl, wl.num_kv_heads, wl.head_dim, kr, vr,
                                       d["npages"], wl.page_size, wl.rotate_k, wl.rotate_v,
                                       wl.block_h, threads=threads)
            eq = bool(np.array_equal(kr, kc) and np.array_equal(vr, vc))
            del kr, vr
        else:
            eq = None
        for cores, seqs, heads in ((threads, d["seqs_all"], range(wl.num_q_heads)),
                                   (1, d["seqs_one"], range(d.get("heads_one", wl.num_q_heads)))):
            pairs = [(b, h) for b in seqs for h in heads]
            ref = {}

            def run(pairs=pairs, cores=cores, ref=ref):
                ref["o"] = oracle.decode(d["q"], kc, vc, d["bt"], d["lens"], wl.num_q_heads,
                                         wl.num_kv_heads, wl.head_dim, d["npages"], wl.page_size,
                                         wl.rotate_k, wl.rotate_v, wl.block_h, pairs=pairs,
                                         threads=cores)
            dt, passes = timed_passes(run, min_seconds, 50)
            kvh = len({h // G for h in heads})
            nbytes = sample_decode_bytes(wl, d["lens"], seqs, kvh, len(pairs),
                                         appended=d.get("new") is not None)
            legs[f"{name} cores={cores}"] = {
                "value": nbytes * passes / dt / 1e9, "unit": "GB/s", "cores": cores,
                "sample": f"one layer, {len(seqs)} sequence(s) x {len(list(heads))} q-head(s) "
                          f"({len(pairs)} rows, fp64), {passes} pass(es), {dt:.1f} s"}
            if cores == threads:
                got = d["out"][[b for b, _ in pairs], [h for _, h in pairs]]
                err = rel_max_err(got, ref["o"])
                parity[name] = {"cache_bytes_equal": eq, "attn_rel_err": err, "tol": 2e-3,
                                "finite": bool(np.all(np.isfinite(got))),
                                "ok": bool(err <= 2e-3 and eq is not False and
                                           np.all(np.isfinite(got))),
                                "what": f"{len(pairs)} rows of one layer's output" +
                                        (", and the cache bytes after the step's append"
                                         if eq is not None else "")}
    return legs, parity


# ------------------------------------------------------------------ arms

HEADLINE_WORKLOAD = ("qwen3-32b-high-concurrency: 64 layers, Hq 64, Hkv 8 (GQA 8), head_dim 128, "
                     "h 128, page 16, 256 sequences, context uniform in [4096, 8192], shuffled "
                     "page tables, K and V rotated; step = per layer, append each sequence's new "
                     "token and attend over its whole context (saw_decode_step, one launch per "
                     "layer)")


def headline_config(world: int) -> dict:
    """The `config` object of both arms (the same workload and metric)."""
    step_bytes = StepBytes.headline()
    return {"workload": HEADLINE_WORKLOAD,
            "l2": f"inputs larger than L2: 64 distinct layer caches of 1.71 GB, "
                  f"{step_bytes / 1e9:.1f} GB read per step",
            "parallelism": f"replicas x{world}"}


def graph_step_timing(case, stream, steps: int, warmup: int, sampler=None):
    """CUDA-graph the step, warm it up, and time `steps` replays with CUDA
    events on the launching stream (synchronised on both sides)."""
    graph = capture(case.step, stream)
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler is not None:
        sampler.mark(True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(steps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.mark(False)
    return graph, start.elapsed_time(end) * 1e-3


def e2e_measure(case, graph, stream, iters: int, world: int):
    """The same step end to end through the public API: every step's inputs
    (q, new K and V rows of every layer) come in from pinned host memory and
    its attention output goes back, pipelined as a server would: two sets of
    device inputs and outputs, each with its own captured step, so that
    while step s runs on `stream`, a copy stream brings step s-1's output
    out and step s+1's inputs in.  The timed region runs from the first
    step's input copy to the last step's output copy."""
    q_h = case.q.cpu().pin_memory()
    k_h = case.knew.cpu().pin_memory()
    v_h = case.vnew.cpu().pin_memory()
    o_h = torch.empty(case.out.shape, dtype=case.out.dtype).pin_memory()
    first = (case.q, case.knew, case.vnew, case.out)
    second = tuple(torch.empty_like(t) for t in first)
    case.q, case.knew, case.vnew, case.out = second
    graphs = [graph, capture(case.step, stream)]
    case.q, case.knew, case.vnew, case.out = first
    sets = [first, second]
    copy = torch.cuda.Stream(device=case.q.device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    inputs_in = [ev(), ev()]   # set b holds its step's inputs
    step_done = [ev(), ev()]   # set b's step has run (its output is ready)

    def upload(b):
        q, kn, vn, _ = sets[b]
        q.copy_(q_h, non_blocking=True)
        kn.copy_(k_h, non_blocking=True)
        vn.copy_(v_h, non_blocking=True)
        inputs_in[b].record(copy)

    def run(n):
        with torch.cuda.stream(copy):
            upload(0)
        for s in range(n):
            b = s & 1
            stream.wait_event(inputs_in[b])
            with torch.cuda.stream(stream):
                graphs[b].replay()
            step_done[b].record(stream)
            with torch.cuda.stream(copy):
                if s >= 1:  # step s-1's output, then step s+1's inputs into its set
                    copy.wait_event(step_done[b ^ 1])
                    o_h.copy_(sets[b ^ 1][3], non_blocking=True)
                if s + 1 < n:  # set b^1 is free: its step has run (waited above)
                    upload(b ^ 1)
        with torch.cuda.stream(copy):
            copy.wait_event(step_done[(n - 1) & 1])
            o_h.copy_(sets[(n - 1) & 1][3], non_blocking=True)

    run(3)
    torch.cuda.synchronize()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(copy)
    run(iters)
    e2.record(copy)
    torch.cuda.synchronize()
    del graphs[1], second
    t, nbytes = reduce_over_ranks(s2.elapsed_time(e2) * 1e-3, case.step_bytes() * iters, world)
    h2d = (q_h.numel() + k_h.numel() + v_h.numel()) * 2
    d2h = o_h.numel() * 4
    return {"value": nbytes / t / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": t / iters * 1e3,
            "how": "every step: pinned host q and new K/V rows of every layer copied in, "
                   "graph step, attention output of every layer copied out; double-buffered "
                   "device inputs/outputs, the copies of steps s-1 and s+1 on a second "
                   "stream overlapping step s"}


def step_sample_for_oracle(case, layer: int, seqs_all, seqs_one, heads_one=None,
                           with_prefill=False) -> dict:
    """Host copies of one layer of a fused step (after the step ran): cache
    bytes, q, the appended rows and slots, the output; optionally the
    prefill rows, so that the oracle can rebuild the whole layer."""
    wl = case.wl
    B = wl.num_seqs
    d = {"wl": wl, "kc": case.kc[layer].cpu().numpy(), "vc": case.vc[layer].cpu().numpy(),
         "q": np_bits(case.q[layer]), "out": case.out[layer].cpu().numpy(),
         "bt": case.bt_cpu.numpy(), "lens": case.lens.numpy(), "npages": case.npages,
         "new": (np_bits(case.knew[layer]).reshape(B, -1), np_bits(case.vnew[layer]).reshape(B, -1),
                 case.slot.cpu().numpy()),
         "seqs_all": list(seqs_all), "seqs_one": list(seqs_one)}
    if heads_one is not None:
        d["heads_one"] = heads_one
    if with_prefill:
        k, v = case.pre_rows(layer)
        d["pre"] = (np_bits(k).reshape(case.n_pre, -1), np_bits(v).reshape(case.n_pre, -1),
                    case.pre_slots.cpu().numpy())
        del k, v
    return d


def run_saw(args):
    rank, world, local = dist_env()
    init_group(world)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    from bit_paged_kv_gb300 import workloads as W

    peak, peak_src = read_peaks()
    stream = torch.cuda.Stream(device)
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    samples = {"decode": {}}

    # ---- headline: the config-4 decode step over all 64 layers
    wl = W.QWEN3_32B_HIGH_CONCURRENCY
    t_fill = time.perf_counter()
    case = StepCase(wl, device)
    fill_s = time.perf_counter() - t_fill
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    graph, elapsed = graph_step_timing(case, stream, args.steps, args.warmup, sampler)
    clocks = sampler.stop()
    barrier(world)
    step_bytes = case.step_bytes()
    t_max, bytes_all = reduce_over_ranks(elapsed, step_bytes * args.steps, world)
    value = bytes_all / t_max / 1e9
    status = int(case.status.item())
    launches = case.launches_per_step() * args.steps
    dec_ms = elapsed * 1e3 / launches
    achieved = case.layer_bytes() / (dec_ms * 1e-3) / 1e9
    traffic, traffic_src = decode_traffic(wl.name)
    e2e = e2e_measure(case, graph, stream, max(3, args.steps // 4), world)
    head_plan = {"splits": case.splits, "pages_per_split": case.pps}
    if want_cpu:
        last = wl.num_layers - 1
        samples["decode"]["qwen3-32b-high-concurrency step"] = step_sample_for_oracle(
            case, last, seqs_all=range(0, wl.num_seqs, 2), seqs_one=[0, 1])
    del graph
    case.release()
    del case

    # ---- the Qwen3-4B-shaped latency step (batch 1, context 32768, 36 layers)
    lw = W.QWEN3_4B_LATENCY
    lat = StepCase(lw, device)
    lat_steps = max(50, 10 * args.steps)
    lgraph, lt = graph_step_timing(lat, stream, lat_steps, max(args.warmup, 5))
    lat_ms = lt * 1e3 / (lat_steps * lat.launches_per_step())
    lat_traffic, lat_traffic_src = decode_traffic(lw.name)
    latency = {
        "workload": "qwen3-4b-latency: 36 layers, Hq 32, Hkv 8, head_dim 128, h 128, page 16, "
                    "batch 1, context 32768, K-only rotation; step = per layer 1-token "
                    "quantize-append + paged decode (saw_decode_step), one CUDA graph per step",
        "value": lat.step_bytes() * lat_steps / lt / 1e9, "unit": "GB/s",
        "ms_per_step": lt * 1e3 / lat_steps, "steps": lat_steps,
        "decode_plan": {"splits": lat.splits, "pages_per_split": lat.pps},
        "roofline": {"bound": "hbm", "achieved": lat.layer_bytes() / (lat_ms * 1e-3) / 1e9,
                     "peak": peak, "unit": "GB/s",
                     "frac": lat.layer_bytes() / (lat_ms * 1e-3) / 1e9 / peak,
                     "traffic": lat_traffic, "traffic_source": lat_traffic_src,
                     "bytes_per_launch": lat.layer_bytes(), "ms_per_launch": lat_ms},
        "e2e": e2e_measure(lat, lgraph, stream, max(10, lat_steps // 4), world),
        "device_status": int(lat.status.item()),
    }
    if want_cpu:
        samples["decode"]["qwen3-4b-latency step"] = step_sample_for_oracle(
            lat, lw.num_layers - 1, seqs_all=[0], seqs_one=[0], heads_one=lw.group,
            with_prefill=True)
    del lgraph
    lat.release()
    del lat

    # ---- quantize-append of a 131072-token prefill chunk
    app, app_bytes, app_T, app_keep = append_chunk_measure(device, stream, keep=want_cpu)
    samples["append"] = app_keep
    # ---- decode alone on the bandwidth-bound workloads, and the other rows
    dec_cfg = dec_rot = None
    if not args.no_decode_configs:
        dec_cfg, dec_rot, kept = decode_config_measure(device, stream,
                                                       keep={"long-131072 h128"} if want_cpu else None)
        if want_cpu:
            k5 = kept["long-131072 h128"]
            k5.update(seqs_all=list(range(k5["wl"].num_seqs)), seqs_one=[0],
                      heads_one=k5["wl"].group)
            samples["decode"]["long-131072 h128"] = k5
    sweep = None if args.no_decode_configs else concurrency_sweep(device, stream)
    pre = None if args.no_decode_configs else prefill_measure(device, stream)
    var = None if args.no_decode_configs else variants_measure(device, stream)
    fmtv = None if args.no_decode_configs else formats_measure(device, stream)

    cpu = parity = None
    if want_cpu:
        import oracle
        threads = oracle.host_threads()
        legs, parity = cpu_oracle_legs(samples, threads)
        head = legs["qwen3-32b-high-concurrency step cores=%d" % threads]
        cpu = {"value": head["value"], "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": "fp64 decode of " + head["sample"] + " of the config-4 step (its "
                         "appended tokens included); the other legs below",
               "legs": legs}
    del samples

    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_max / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int4 KV (bf16 in, f32 rotation/softmax, f16 MMA f32 accumulate)",
        "data": "synthetic",
        "config": headline_config(world),
        "execution": "one CUDA graph per step (64 launches)",
        "decode_plan": head_plan,
        "fill_s": fill_s,
        "roofline": {
            "bound": "hbm",
            "kernel": "saw_decode_step: paged_decode_kernel<head_dim 128, page 16, wide (GQA 8), "
                      "append>, 4-warp CTAs (four per SM), one per (sequence, kv-head) "
                      "(256 new tokens appended, 1.57e6 cached tokens attended per layer)",
            "achieved": achieved,
            "peak": peak,
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "traffic_source": traffic_src,
            "bytes_per_launch": case_layer_bytes(wl),
            "ms_per_launch": dec_ms,
            "timing": "CUDA events around the timed region on the launching stream / "
                      f"{launches} launches",
            "peak_source": peak_src,
        },
        "quantize_append_tokens_per_s": app["rotated_h128"]["tokens_per_s"],
        "quantize_append_frac": app["rotated_h128"]["gbs"] / peak,
        "quantize_append": {
            "workload": "131072-token prefill chunk, Hkv 8, head_dim 128, K and V, page 64",
            "tokens_per_s": app["rotated_h128"]["tokens_per_s"],
            "roofline": {"bound": "hbm", "achieved": app["rotated_h128"]["gbs"], "peak": peak,
                         "unit": "GB/s", "frac": app["rotated_h128"]["gbs"] / peak,
                         "bytes_per_launch": app_bytes},
            "variants": app,
            "rotation_overhead": app["rotated_h128"]["ms"] / app["unrotated"]["ms"] - 1.0,
        },
        "latency_step": latency,
        "decode_configs": None if dec_cfg is None else {
            "what": "saw_paged_decode_int4 alone, automatic split plan, distinct layer caches "
                    "decoded in turn (each larger than L2); GB/s = algorithmic bytes / time",
            "peak": peak,
            "results": {k: dict(v, frac=v["gbs"] / peak) for k, v in dec_cfg.items()},
            "rotation_overhead": dec_rot,
        },
        "int4_vs_bf16": None if sweep is None else {
            "what": "decode attention of one layer, INT4 (K and V rotated, h 128) vs the BF16 "
                    "cache baseline, qwen3-8b-concurrent shape (Hq 32, Hkv 8, page 16, lengths "
                    "uniform in [2048, 16384]) at 1..256 concurrent sequences; tokens/s = "
                    "sequences / (36 layers x time per layer), attention only",
            "results": sweep,
        },
        "prefill_attn": None if pre is None else {
            "what": "saw_prefill_attn_int4 (causal, INT4 cache, q and V-output rotation), "
                    "long-context shape: Hq 32, Hkv 8, page 64, h 128, K and V rotated",
            "roofline": {"bound": "tensor", "peak": pre[1], "unit": "TFLOP/s",
                         "peak_source": pre[2],
                         "flops": "useful causal FLOPs: 4 * head_dim * Hq per (query, visible key)"},
            "results": pre[0],
        },
        "head_dim_variants": None if var is None else {
            "what": "head_dim 64 and 256, h = head_dim; decode on the qwen3-8b-concurrent "
                    "shape, append on a 131072-token chunk; GB/s = algorithmic bytes / time",
            "peak": peak,
            "results": {k: dict(v, frac=v["gbs"] / peak) for k, v in var.items()},
        },
        "format_variants": None if fmtv is None else {
            "what": "binary16 input and bfloat16 metadata beside the plain formats (head_dim "
                    "128, h 128); decode on the qwen3-8b-concurrent shape, append on a "
                    "131072-token chunk; GB/s = algorithmic bytes / time (the same bytes "
                    "for every format)",
            "peak": peak,
            "results": {k: dict(v, decode_frac=v["decode_gbs"] / peak,
                                append_frac=v["append_gbs"] / peak) for k, v in fmtv.items()},
        },
        "e2e": e2e,
        "cpu_baseline": cpu,
        "parity": parity,
        "gpu_launches": launches,
        "clocks": clocks,
        "device_status": status,
    }
    print(json.dumps(line))


def case_layer_bytes(wl) -> int:
    from bit_paged_kv_gb300 import workloads as W
    lens = W.seq_lens(wl)
    return W.decode_bytes(wl, lens.tolist()) + W.append_bytes(wl, wl.num_seqs)


def run_reference(args):
    """The CPU oracle (test infrastructure, as it stands) on a bounded sample
    of the headline workload per step, on the same host cores the GPU arm's
    cpu_baseline uses.  Step k: the fused step of layer 0 for sequence k mod 4
    of the Qwen3-32B-shaped workload -- append its new token (8 kv-heads, K and
    V), then fp64 decode of its 64 q-heads over its whole context."""
    rank, world, local = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from bit_paged_kv_gb300 import workloads as W
    oracle.load()
    wl = W.QWEN3_32B_HIGH_CONCURRENCY
    P, Hkv, D, Hq = wl.page_size, wl.num_kv_heads, wl.head_dim, wl.num_q_heads
    nseq = 4
    lens = W.seq_lens(wl)[:nseq]
    bt, npages = W.page_tables(wl, lens)
    threads = oracle.host_threads()

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    # prefill every token but each sequence's last, the rows drawn on the host
    pre = [int(x) - 1 for x in lens.tolist()]
    n_pre = sum(pre)
    k = bits(W.kv_rows(wl, 0, W.K, n_pre + nseq, "cpu")).reshape(n_pre + nseq, -1)
    v = bits(W.kv_rows(wl, 0, W.V, n_pre + nseq, "cpu")).reshape(n_pre + nseq, -1)
    slots = W.prefill_slots(bt, pre, P).numpy()
    new_slots = np.array([int(bt[b, (int(L) - 1) // P]) * P + (int(L) - 1) % P
                          for b, L in enumerate(lens.tolist())], dtype=np.int32)
    nb = oracle.cache_bytes(npages, P, Hkv, D)
    kc, vc = np.zeros(nb, np.uint8), np.zeros(nb, np.uint8)
    oracle.quantize_append(k[:n_pre], v[:n_pre], slots, Hkv, D, kc, vc, npages, P, wl.rotate_k,
                           wl.rotate_v, wl.block_h, threads=threads)
    q = bits(W.q_rows(wl, 0, "cpu", num_seqs=nseq))
    btn, lensn = bt.numpy(), lens.numpy()

    def step(i):
        b = i % nseq
        oracle.quantize_append(k[n_pre + b:n_pre + b + 1], v[n_pre + b:n_pre + b + 1],
                               new_slots[b:b + 1], Hkv, D, kc, vc, npages, P, wl.rotate_k,
                               wl.rotate_v, wl.block_h)
        oracle.decode(q, kc, vc, btn, lensn, Hq, Hkv, D, npages, P, wl.rotate_k, wl.rotate_v,
                      wl.block_h, pairs=[(b, h) for h in range(Hq)], threads=threads)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    nbytes = sum(sample_decode_bytes(wl, lensn, [i % nseq], Hkv, Hq, appended=True)
                 for i in range(args.steps))
    value = nbytes / dt / 1e9
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 attention, f32 quantizer",
        "data": "synthetic",
        "config": headline_config(world),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step: layer 0, one of the first {nseq} sequences "
                                   f"(cycled): append its new token (Hkv {Hkv}, K and V) and "
                                   f"fp64 decode of its {Hq} q-heads over its context"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


class StepBytes:
    @staticmethod
    def headline() -> int:
        from bit_paged_kv_gb300 import workloads as W
        wl = W.QWEN3_32B_HIGH_CONCURRENCY
        return wl.num_layers * case_layer_bytes(wl)


def run_profile(args):
    """Small, fixed loops for ncu captures (no timing, no JSON):
    decode: the latency case's fused step over --profile-layers layer caches
    (35.7 MB each, more than L2 in total), three passes;
    step4: the same on the Qwen3-32B-shaped workload (1.71 GB per layer;
    use --profile-layers 2), three passes;
    append: three quantize-appends of the 131072-token chunk;
    bf16: three BF16-cache decodes of 16 qwen3-8b-concurrent sequences
    (about 600 MB of cache, more than L2);
    prefill: three 2048-token chunks at context 16384 (long-context shape);
    variant: three head_dim 256 (--profile-head-dim 64: 64) decodes of 16
    qwen3-8b-concurrent sequences."""
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    import __graft_entry__
    __graft_entry__.build()
    from bit_paged_kv_gb300 import workloads as W
    if args.profile in ("decode", "step4"):
        if args.profile == "decode":
            wl = W.QWEN3_4B_LATENCY.variant(num_layers=args.profile_layers)
        else:
            wl = W.QWEN3_32B_HIGH_CONCURRENCY.variant(num_layers=args.profile_layers)
        case = StepCase(wl, device)
        for _ in range(3):
            for layer in range(wl.num_layers):
                case.decode_step(layer)
        torch.cuda.synchronize()
        assert int(case.status.item()) == 0
    elif args.profile == "prefill":
        import bit_paged_kv_gb300 as saw
        wl = W.LONG_PREFILL.variant(num_seqs=1)
        L, n = 16384, 2048
        lens = torch.tensor([L], dtype=torch.int32)
        bt, npages = W.page_tables(wl, lens)
        kc, vc = fill_caches(wl, 0, lens, bt, npages, device)
        q = torch.randn(n, wl.num_q_heads, wl.head_dim, device=device).to(torch.bfloat16)
        out = torch.empty(n, wl.num_q_heads, wl.head_dim, dtype=torch.float32, device=device)
        cu = torch.tensor([0, n], dtype=torch.int32, device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        for _ in range(3):
            saw.saw_prefill_attn_int4(q, cu, kc, vc, bt.to(device), lens.to(device), n, L,
                                      wl.num_kv_heads, npages, wl.page_size, wl.rotate_k,
                                      wl.rotate_v, wl.block_h, out, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
    elif args.profile == "bf16":
        import bit_paged_kv_gb300 as saw
        wl = W.QWEN3_8B_CONCURRENT.variant(num_seqs=16)
        lens = W.seq_lens(wl)
        bt, npages = W.page_tables(wl, lens)
        kc, vc = fill_caches_bf16(wl, 0, lens, bt, npages, device)
        B, Hq, D = wl.num_seqs, wl.num_q_heads, wl.head_dim
        Lmax = int(lens.max())
        q = W.q_rows(wl, 0, device)
        out = torch.empty(B, Hq, D, dtype=torch.float32, device=device)
        wsb = saw.saw_decode_bf16_workspace_bytes(B, Hq, wl.num_kv_heads, D, wl.page_size, Lmax)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        for _ in range(3):
            saw.saw_paged_decode_bf16(q, kc, vc, bt.to(device), lens.to(device), Lmax,
                                      wl.num_kv_heads, npages, wl.page_size, out, ws,
                                      dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
    elif args.profile == "variant":
        # head_dim 256 (or --profile-head-dim) decode on 16 sequences of the
        # qwen3-8b-concurrent shape
        import bit_paged_kv_gb300 as saw
        hd = args.profile_head_dim
        wl = W.QWEN3_8B_CONCURRENT.variant(num_seqs=16, head_dim=hd, block_h=hd)
        lens = W.seq_lens(wl)
        bt, npages = W.page_tables(wl, lens)
        kc, vc = fill_caches(wl, 0, lens, bt, npages, device)
        B, Hq, D = wl.num_seqs, wl.num_q_heads, wl.head_dim
        Lmax = int(lens.max())
        q = W.q_rows(wl, 0, device)
        out = torch.empty(B, Hq, D, dtype=torch.float32, device=device)
        wsb = saw.saw_decode_workspace_bytes(B, Hq, wl.num_kv_heads, D, wl.page_size, Lmax, 0)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        torch.cuda.synchronize()
        for _ in range(3):
            saw.saw_paged_decode_int4(q, kc, vc, bt.to(device), lens.to(device), Lmax,
                                      wl.num_kv_heads, npages, wl.page_size, True, True, D, out,
                                      ws, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
    else:
        append_chunk_measure(device, torch.cuda.current_stream(device), iters=1)
    torch.cuda.synchronize()
    print(f"profile {args.profile} done")


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["saw", "reference"], default="saw")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode-configs", action="store_true",
                    help="skip the decode-only measurements of the other workloads")
    ap.add_argument("--profile", choices=["decode", "step4", "append", "bf16", "prefill",
                                          "variant"],
                    default=None,
                    help="run a small fixed loop for an ncu capture instead of the benchmark")
    ap.add_argument("--profile-layers", type=int, default=8)
    ap.add_argument("--profile-head-dim", type=int, default=256, choices=[64, 256],
                    help="head dimension of --profile variant")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.profile:
        run_profile(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_saw(args)


if __name__ == "__main__":
    main()
