#!/usr/bin/env python3
"""Benchmark of the SAW-INT4 hot path on one GB300 (per rank).

Default workload (the Qwen3-4B-shaped latency case): 36 layers, 32 q-heads,
8 kv-heads, head_dim 128, h = 128, page 16, batch 1, context 32768, K-only
rotation.  One step = for every layer, quantize-append the new token's K/V
into that layer's paged INT4 cache, then decode-attend over the 32768
cached tokens (saw_decode_step: one fused launch per layer).  The step is
replayed as one CUDA graph.

Printed (rank 0, one JSON line): KV GB/s of the whole step (algorithmic
bytes / step time), the decode kernel's HBM roofline fraction, the
quantize-append throughput of a 131072-token prefill chunk, the end-to-end
rate through the public API with host buffers, and the CPU oracle's rate.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl saw|reference]

--impl reference times the CPU oracle (test infrastructure) on the host
cores on a bounded sample of the same workload: this method has no
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

DECODE_SOURCES = ["paged_decode.cu", "saw_device.cuh", "saw_internal.h", "saw_quant_row.cuh"]


def decode_traffic():
    """DRAM bytes per launch of the decode kernel from the committed ncu
    record (profiles/dram_traffic.txt), or None when the kernel's sources
    have changed since that capture."""
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, "bit_paged_kv_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.txt")) as fh:
            for line in fh:
                parts = line.split()
                if len(parts) == 4 and not line.startswith("#") and parts[2] == h.hexdigest():
                    return int(parts[3]), "ncu capture in profiles/paged_decode_qwen3-4b-latency.md"
    except OSError:
        pass
    return None, "no ncu capture of the current kernel sources"


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


class LatencyCase:
    """Qwen3-4B-shaped decode step: per layer a 1-token append + decode."""

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
        self.kc = [torch.empty(nb, dtype=torch.uint8, device=device) for _ in range(wl.num_layers)]
        self.vc = [torch.empty(nb, dtype=torch.uint8, device=device) for _ in range(wl.num_layers)]
        status = torch.zeros(1, dtype=torch.int32, device=device)
        # prefill every layer's cache with all but the last token of each sequence
        for layer in range(wl.num_layers):
            pre = [int(x) - 1 for x in self.lens.tolist()]
            k = W.kv_rows(wl, layer, W.K, sum(pre), device)
            v = W.kv_rows(wl, layer, W.V, sum(pre), device)
            slots = W.prefill_slots(self.bt, pre, P)
            saw.saw_quantize_append(k, v, slots, self.kc[layer], self.vc[layer], self.npages, P,
                                    wl.rotate_k, wl.rotate_v, wl.block_h, dev_status=status)
            del k, v
        # per-step inputs: each layer's new token (the last one of each sequence) and q
        self.slot = torch.cat([W.slots_for(self.bt, P, b, int(Lb) - 1, int(Lb))
                               for b, Lb in enumerate(self.lens.tolist())])
        self.knew = torch.stack([W.kv_rows(wl, l, W.K, 1, device, token_offset=self.L - 1)
                                 for l in range(wl.num_layers)]).expand(-1, B, -1, -1).contiguous()
        self.vnew = torch.stack([W.kv_rows(wl, l, W.V, 1, device, token_offset=self.L - 1)
                                 for l in range(wl.num_layers)]).expand(-1, B, -1, -1).contiguous()
        self.q = torch.stack([W.q_rows(wl, l, device) for l in range(wl.num_layers)])
        self.out = torch.empty(wl.num_layers, B, Hq, D, dtype=torch.float32, device=device)
        self.splits, self.pps = saw.saw_decode_plan(B, Hkv, P, self.L, 0)
        wsb = saw.saw_decode_workspace_bytes(B, Hq, Hkv, D, P, self.L, 0)
        self.ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device=device) if wsb else None
        self.status = status
        torch.cuda.synchronize()
        assert int(status.item()) == 0

    def append(self, layer):
        wl = self.wl
        self.saw.saw_quantize_append(self.knew[layer], self.vnew[layer], self.slot,
                                     self.kc[layer], self.vc[layer], self.npages, wl.page_size,
                                     wl.rotate_k, wl.rotate_v, wl.block_h,
                                     dev_status=self.status)

    def decode(self, layer):
        wl = self.wl
        self.saw.saw_paged_decode_int4(self.q[layer], self.kc[layer], self.vc[layer], self.bt,
                                       self.lens_d, self.L, wl.num_kv_heads, self.npages,
                                       wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                                       self.out[layer], self.ws, dev_status=self.status)

    def decode_step(self, layer):
        """The fused step of one layer: append the new token, then attend."""
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

    def step_bytes(self) -> int:
        W, wl = self.W, self.wl
        return wl.num_layers * (W.decode_bytes(wl, self.lens.tolist()) +
                                W.append_bytes(wl, wl.num_seqs))

    def decode_bytes(self) -> int:
        return self.W.decode_bytes(self.wl, self.lens.tolist())

    def layer_bytes(self) -> int:
        """Algorithmic bytes of one fused decode step of one layer."""
        return self.decode_bytes() + self.W.append_bytes(self.wl, self.wl.num_seqs)


def capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # warm (sets kernel attributes outside capture)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def decode_kernel_times(case, stream, reps: int):
    """Average device time of one layer's fused decode step (one kernel),
    from external event records captured around every layer's call inside a
    graph of the step; falls back to graph time / layers."""
    nl = case.wl.num_layers
    try:
        evs = [(torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True)) for _ in range(nl)]
    except TypeError:
        evs = None
    if evs is not None:
        def fn():
            s = torch.cuda.current_stream()
            for layer in range(nl):
                evs[layer][0].record(s)
                case.decode_step(layer)
                evs[layer][1].record(s)
        try:
            g = capture(fn, stream)
            acc = []
            for _ in range(reps):
                g.replay()
                torch.cuda.synchronize()
                acc.extend(a.elapsed_time(b) for a, b in evs)
            return statistics.mean(acc), "external events around each layer's call in the step graph"
        except Exception:
            pass
    g = capture(case.step, stream)
    t = time_events(g.replay, reps, stream)
    return statistics.mean(t) / nl, "step graph time / layers (includes launch gaps)"


def append_chunk_measure(device, stream, iters: int = 20):
    """Quantize-append of one 131072-token prefill chunk (8 kv-heads, K and V,
    page 64), rotated (h = 128 and 64) and unrotated.  Inputs are 512 MB,
    larger than L2."""
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
    return res, nbytes, T


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


def decode_config_measure(device, stream, layers: int = 2, reps: int = 10, only=None):
    """Decode-only throughput of the bandwidth-bound workloads (Qwen3-8B
    concurrent, Qwen3-32B high concurrency in its three rotation variants,
    long context at h 128 and 64): `layers` distinct layer caches (each
    larger than L2) decoded in turn, CUDA events around reps passes."""
    import bit_paged_kv_gb300 as saw
    from bit_paged_kv_gb300 import workloads as W
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
        nbytes = W.decode_bytes(wl, lens.tolist())
        splits, pps = saw.saw_decode_plan(B, wl.num_kv_heads, wl.page_size, Lmax, 0)
        res[name] = {"ms_per_layer": t, "gbs": nbytes / (t * 1e-3) / 1e9,
                     "bytes_per_layer": nbytes, "splits": splits, "pages_per_split": pps,
                     "seqs": B, "tokens": int(lens.sum())}
        del caches, qs, ws, out
        torch.cuda.empty_cache()
    if only is not None:
        return res, None
    a = res["qwen3-32b-high-concurrency k+v"]["ms_per_layer"]
    k1 = res["qwen3-32b-high-concurrency k-only"]["ms_per_layer"]
    u = res["qwen3-32b-high-concurrency unrotated"]["ms_per_layer"]
    overhead = {"k+v_vs_unrotated": a / u - 1.0, "k-only_vs_unrotated": k1 / u - 1.0}
    return res, overhead


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
    """head_dim 64 and 256 (variant kernels): decode alone on the
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


def cpu_oracle_decode_sample(case, layers, threads, min_seconds=10.0, max_passes=40):
    """Time the oracle (as it stands) on the step's work for `layers`:
    append the new token, then decode every q-head over the layer's pages;
    whole passes over the layers are repeated until min_seconds have gone."""
    import numpy as np

    import oracle
    wl = case.wl

    def bits(t):
        return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

    hosts = []
    for layer in layers:
        hosts.append((case.kc[layer].cpu().numpy(), case.vc[layer].cpu().numpy(),
                      bits(case.knew[layer]).reshape(wl.num_seqs, -1),
                      bits(case.vnew[layer]).reshape(wl.num_seqs, -1), bits(case.q[layer])))
    slots = case.slot.cpu().numpy()
    bt = case.bt_cpu.numpy()
    lens = case.lens.numpy()
    passes = 0
    t0 = time.perf_counter()
    while True:  # whole passes over the layers until min_seconds (re-appending is idempotent)
        for kc, vc, kn, vn, q in hosts:
            oracle.quantize_append(kn, vn, slots, wl.num_kv_heads, wl.head_dim, kc, vc,
                                   case.npages, wl.page_size, wl.rotate_k, wl.rotate_v,
                                   wl.block_h)
            oracle.decode(q, kc, vc, bt, lens, wl.num_q_heads, wl.num_kv_heads, wl.head_dim,
                          case.npages, wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                          threads=threads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= max_passes:
            break
    nbytes = passes * len(layers) * (case.W.decode_bytes(wl, case.lens.tolist()) +
                                     case.W.append_bytes(wl, wl.num_seqs))
    return nbytes / dt / 1e9, dt, passes


# ------------------------------------------------------------------ arms

def run_saw(args):
    rank, world, local = dist_env()
    init_group(world)
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import __graft_entry__
    __graft_entry__.build()
    from bit_paged_kv_gb300 import workloads as W

    wl = W.QWEN3_4B_LATENCY
    case = LatencyCase(wl, device)
    stream = torch.cuda.Stream(device)
    graph = capture(case.step, stream)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark(True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(args.steps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    sampler.mark(False)
    clocks = sampler.stop()
    barrier(world)
    elapsed = start.elapsed_time(end) * 1e-3
    step_bytes = case.step_bytes()
    t_max, bytes_all = reduce_over_ranks(elapsed, step_bytes * args.steps, world)
    value = bytes_all / t_max / 1e9
    status = int(case.status.item())

    # dominant (and only) kernel: one fused decode step per layer.  Its
    # average launch duration is the timed region's device time over the
    # launches in it; launches overlap slightly (programmatic dependent
    # launch), so this is what a launch costs in the step.
    dec_ms = elapsed * 1e3 / (args.steps * case.launches_per_step())
    dec_how = ("CUDA events around the timed region on the launching stream / "
               f"{case.launches_per_step()} launches per step")
    iso_ms, iso_how = decode_kernel_times(case, stream, reps=max(20, min(200, args.steps // 10)))
    peak, peak_src = read_peaks()
    achieved = case.layer_bytes() / (dec_ms * 1e-3) / 1e9
    traffic, traffic_src = decode_traffic()

    # end to end through the public API with host buffers
    q_h = case.q.cpu().pin_memory()
    k_h = case.knew.cpu().pin_memory()
    v_h = case.vnew.cpu().pin_memory()
    o_h = torch.empty(case.out.shape, dtype=case.out.dtype).pin_memory()

    def e2e_step():
        case.q.copy_(q_h, non_blocking=True)
        case.knew.copy_(k_h, non_blocking=True)
        case.vnew.copy_(v_h, non_blocking=True)
        graph.replay()
        o_h.copy_(case.out, non_blocking=True)

    e2e_iters = max(10, args.steps // 4)
    with torch.cuda.stream(stream):
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for _ in range(e2e_iters):
            e2e_step()
        e2.record(stream)
    torch.cuda.synchronize()
    t_e2e, bytes_e2e = reduce_over_ranks(s2.elapsed_time(e2) * 1e-3, step_bytes * e2e_iters, world)
    h2d = q_h.numel() * 2 + k_h.numel() * 2 + v_h.numel() * 2
    d2h = o_h.numel() * 4

    # quantize-append of a 131072-token prefill chunk
    app, app_bytes, app_T = append_chunk_measure(device, stream)
    # decode alone on the bandwidth-bound workloads
    dec_cfg, dec_rot = (None, None) if args.no_decode_configs else decode_config_measure(device, stream)
    sweep = None if args.no_decode_configs else concurrency_sweep(device, stream)
    pre = None if args.no_decode_configs else prefill_measure(device, stream)
    var = None if args.no_decode_configs else variants_measure(device, stream)
    fmtv = None if args.no_decode_configs else formats_measure(device, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        threads = oracle.host_threads()
        layers = list(range(min(args.cpu_layers, wl.num_layers)))
        gbs, dt, passes = cpu_oracle_decode_sample(case, layers, threads)
        cpu = {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": f"{passes} pass(es) over {len(layers)} of the 36 layers of the step "
                         f"(1-token append + fp64 decode of all 32 q-heads over 32768 tokens), "
                         f"{dt:.1f} s wall"}

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
        "config": {
            "workload": "qwen3-4b-latency: 36 layers, Hq 32, Hkv 8, head_dim 128, h 128, page 16, "
                        "batch 1, context 32768, K-only rotation; step = per layer 1-token "
                        "quantize-append + paged decode (saw_decode_step, one launch per layer)",
            "l2": f"inputs larger than L2: 36 distinct layer caches, "
                  f"{step_bytes / 1e9:.2f} GB read per step",
            "execution": "one CUDA graph per step",
            "decode_plan": {"splits": case.splits, "pages_per_split": case.pps},
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "saw_decode_step: paged_decode_kernel<16, packed, append> (1 token "
                      "appended, 32768 attended, merge in the last split)",
            "achieved": achieved,
            "peak": peak,
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "traffic_source": traffic_src,
            "bytes_per_launch": case.layer_bytes(),
            "ms_per_launch": dec_ms,
            "timing": dec_how,
            "ms_per_launch_bracketed": iso_ms,
            "bracketed_timing": iso_how + " (events between launches stop their overlap)",
            "peak_source": peak_src,
        },
        "quantize_append": {
            "workload": "131072-token prefill chunk, Hkv 8, head_dim 128, K and V, page 64",
            "tokens_per_s": app["rotated_h128"]["tokens_per_s"],
            "roofline": {"bound": "hbm", "achieved": app["rotated_h128"]["gbs"], "peak": peak,
                         "unit": "GB/s", "frac": app["rotated_h128"]["gbs"] / peak,
                         "bytes_per_launch": app_bytes},
            "variants": app,
            "rotation_overhead": app["rotated_h128"]["ms"] / app["unrotated"]["ms"] - 1.0,
        },
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
            "what": "head_dim 64 and 256 (CUDA-core decode kernel, warp-per-row append), "
                    "h = head_dim; decode on the qwen3-8b-concurrent shape, append on a "
                    "131072-token chunk; GB/s = algorithmic bytes / time",
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
        "e2e": {"value": bytes_e2e / t_e2e / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "how": "pinned host q/k/v copied in, graph step, output copied out, every step"},
        "cpu_baseline": cpu,
        "gpu_launches": case.launches_per_step() * args.steps,
        "clocks": clocks,
        "device_status": status,
    }
    print(json.dumps(line))


def run_reference(args):
    """The CPU oracle on a bounded sample of the same workload per step."""
    rank, world, local = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    from bit_paged_kv_gb300 import workloads as W
    oracle.load()
    wl = W.QWEN3_4B_LATENCY
    lens = W.seq_lens(wl)
    L = int(lens[0])
    bt, npages = W.page_tables(wl, lens)
    P, Hkv, D, G = wl.page_size, wl.num_kv_heads, wl.head_dim, wl.group

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    # sample: layer 0, kv-head 0 and its G q-heads, full 32768-token context
    k = W.kv_rows(wl, 0, W.K, L, "cpu")
    v = W.kv_rows(wl, 0, W.V, L, "cpu")
    slots = W.prefill_slots(bt, [L], P).numpy()
    nb = oracle.cache_bytes(npages, P, Hkv, D)
    kc, vc = np.zeros(nb, np.uint8), np.zeros(nb, np.uint8)
    kb, vb = bits(k).reshape(L, -1), bits(v).reshape(L, -1)
    threads = oracle.host_threads()
    oracle.quantize_append(kb[:-1], vb[:-1], slots[:-1], Hkv, D, kc, vc, npages, P, wl.rotate_k,
                           wl.rotate_v, wl.block_h, threads=threads)
    q = bits(W.q_rows(wl, 0, "cpu"))
    pairs = [(0, h) for h in range(G)]

    def step():
        oracle.quantize_append(kb[-1:], vb[-1:], slots[-1:], Hkv, D, kc, vc, npages, P,
                               wl.rotate_k, wl.rotate_v, wl.block_h)
        oracle.decode(q, kc, vc, bt.numpy(), lens.numpy(), wl.num_q_heads, Hkv, D, npages, P,
                      wl.rotate_k, wl.rotate_v, wl.block_h, pairs=pairs, threads=min(threads, G))

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    per_row = D // 2 + 4
    # algorithmic bytes of the sample: one kv-head's K and V rows over the
    # context, its block-table entries, G q rows in and out, one appended token
    sample_bytes = (2 * per_row * L + 4 * -(-L // P) + G * D * (2 + 4)
                    + W.append_bytes(wl, 1))
    value = sample_bytes * args.steps / dt / 1e9
    cores = min(threads, G)
    print(json.dumps({
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 attention, f32 quantizer",
        "data": "synthetic",
        "config": {"workload": "qwen3-4b-latency (same as the GPU arm)",
                   "parallelism": "host threads"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"per step: layer 0, kv-head 0 with its {G} q-heads over "
                                   f"{L} tokens (1-token append + fp64 decode)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def run_profile(args):
    """Small, fixed loops for ncu captures (no timing, no JSON):
    decode: the latency case's decode over --profile-layers layer caches
    (35.7 MB each, more than L2 in total), three passes;
    append: three quantize-appends of the 131072-token chunk;
    bf16: three BF16-cache decodes of 16 qwen3-8b-concurrent sequences
    (about 600 MB of cache, more than L2);
    prefill: three 2048-token chunks at context 16384 (long-context shape)."""
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    import __graft_entry__
    __graft_entry__.build()
    from bit_paged_kv_gb300 import workloads as W
    if args.profile == "decode":
        wl = W.QWEN3_4B_LATENCY.variant(num_layers=args.profile_layers)
        case = LatencyCase(wl, device)
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
        # head_dim 256 decode on 16 sequences of the qwen3-8b-concurrent shape
        import bit_paged_kv_gb300 as saw
        wl = W.QWEN3_8B_CONCURRENT.variant(num_seqs=16, head_dim=256, block_h=256)
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
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["saw", "reference"], default="saw")
    ap.add_argument("--cpu-layers", type=int, default=36)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode-configs", action="store_true",
                    help="skip the decode-only measurements of the other workloads")
    ap.add_argument("--profile", choices=["decode", "append", "bf16", "prefill", "variant"],
                    default=None,
                    help="run a small fixed loop for an ncu capture instead of the benchmark")
    ap.add_argument("--profile-layers", type=int, default=8)
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
