"""Host-side benchmark logic, on CPU: the max-over-ranks / sum-of-units
reduction with two gloo ranks, and the reference arm (the CPU oracle)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    bench.init_group(world)
    t, u = bench.reduce_over_ranks(seconds=1.0 + rank, units=10.0 * (rank + 1), world=world)
    bench.barrier(world)
    q.put((rank, t, u))


def test_reduce_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for _, t, u in res:
        assert t == 2.0 and u == 30.0


def test_single_rank_is_identity():
    assert bench.reduce_over_ranks(1.5, 7.0, 1) == (1.5, 7.0)


def _run(args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=e, timeout=600)


def test_reference_arm_prints_one_line():
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _run(["--impl", "reference", "--steps", "3", "--warmup", "3"],
             env={"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_floor():
    r = _run(["--impl", "reference", "--warmup", "2"])
    assert r.returncode != 0


def _oracle_samples():
    """Stand-ins for the host copies run_saw hands to the oracle's legs: the
    caches and outputs are the oracle's own, so every check must pass."""
    import numpy as np
    import torch

    import oracle
    from bit_paged_kv_gb300 import workloads as W
    wl = W.TINY.variant(num_seqs=3, len_lo=40, len_hi=90, rotate_v=False)
    lens = W.seq_lens(wl)
    bt, npages = W.page_tables(wl, lens)
    T = int(lens.sum())
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    k = bits(W.kv_rows(wl, 0, W.K, T, "cpu")).reshape(T, -1)
    v = bits(W.kv_rows(wl, 0, W.V, T, "cpu")).reshape(T, -1)
    slots = W.prefill_slots(bt, lens.tolist(), wl.page_size).numpy()
    nb = oracle.cache_bytes(npages, wl.page_size, wl.num_kv_heads, wl.head_dim)
    kc, vc = np.zeros(nb, np.uint8), np.zeros(nb, np.uint8)
    oracle.quantize_append(k, v, slots, wl.num_kv_heads, wl.head_dim, kc, vc, npages,
                           wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h)
    q = bits(W.q_rows(wl, 0, "cpu"))
    out = oracle.decode(q, kc, vc, bt.numpy(), lens.numpy(), wl.num_q_heads, wl.num_kv_heads,
                        wl.head_dim, npages, wl.page_size, wl.rotate_k, wl.rotate_v,
                        wl.block_h).reshape(wl.num_seqs, wl.num_q_heads, wl.head_dim)
    # the "new" token of each sequence is its last one
    last = np.cumsum(lens.numpy()) - 1
    dec = {"wl": wl, "kc": kc, "vc": vc, "q": q, "out": out, "bt": bt.numpy(),
           "lens": lens.numpy(), "npages": npages, "new": (k[last], v[last], slots[last]),
           "seqs_all": [0, 1, 2], "seqs_one": [0], "heads_one": wl.group}
    app = {"wl": wl, "k": k, "v": v, "slots": slots, "npages": npages,
           "kc_gpu": kc.copy(), "vc_gpu": vc.copy()}
    return {"append": app, "decode": {"tiny step": dec}}


def test_oracle_legs_time_and_check():
    s = _oracle_samples()
    legs, parity = bench.cpu_oracle_legs(s, threads=2, min_seconds=0.01)
    assert {"append cores=2", "append cores=1", "tiny step cores=2",
            "tiny step cores=1"} <= set(legs)
    for leg in legs.values():
        assert leg["value"] > 0 and leg["cores"] in (1, 2)
    assert parity["tiny step"]["ok"] and parity["tiny step"]["cache_bytes_equal"]
    assert parity["tiny step"]["attn_rel_err"] < 1e-12
    assert parity["append long-131072 chunk"]["bytes_equal"]


def test_oracle_legs_catch_a_wrong_byte_and_a_wrong_output():
    s = _oracle_samples()
    d = s["decode"]["tiny step"]
    P, Hkv = d["wl"].page_size, d["wl"].num_kv_heads
    slot = int(d["new"][2][1])  # the appended token of sequence 1
    chunk = (slot // P * Hkv + 1) * 1088  # its kv-head 1 chunk
    d["kc"][chunk + (slot % P) * 64 + 3] ^= 0x10
    _, parity = bench.cpu_oracle_legs(s, threads=2, min_seconds=0.01)
    assert parity["tiny step"]["cache_bytes_equal"] is False
    assert not parity["tiny step"]["ok"]
    s = _oracle_samples()
    d = s["decode"]["tiny step"]
    d["out"] = d["out"].copy()
    d["out"][2, 1, 5] += 0.01 * float(abs(d["out"]).max())
    _, parity = bench.cpu_oracle_legs(s, threads=2, min_seconds=0.01)
    p = parity["tiny step"]
    assert p["cache_bytes_equal"] and not p["ok"] and p["attn_rel_err"] > 2e-3


def test_both_arms_share_the_config():
    c = bench.headline_config(1)
    assert c == bench.headline_config(1)
    assert "qwen3-32b-high-concurrency" in c["workload"]
