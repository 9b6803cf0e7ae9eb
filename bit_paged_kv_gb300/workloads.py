"""Seeded synthetic inputs for the SAW-INT4 hot path.

Shapes follow the models the gist.science SAW-INT4 page lists (Qwen3-4B,
8B, 32B; s.3 point 4) and its block size h = 128 (s.4); value distributions
reproduce what the pages blame for naive INT4's failure -- a few channels
with unusually large values (youngju.dev "Why Naive INT4 Breaks"; gist.science
s.2, range heterogeneity across channels).  The pages' accuracy suites are not
used: these tensors stand in for the activations a real model would produce.

This module holds no step of the method: it only draws numbers and lays out
page tables.  Both the CUDA path and the oracle consume its outputs.
Every draw comes from its own torch.Generator seeded with
seed * 1_000_000 + layer * 16 + stream, so a tensor never depends on what
else was generated.  Values differ between a CPU and a CUDA generator; a
parity check always feeds the same generated tensor to both sides.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

# stream ids within a layer
K, V, Q, K_OUTLIERS, V_OUTLIERS, K_BIAS, LENS, PAGES = range(8)
GEN_CHUNK_TOKENS = 16384  # token rows drawn per generator call (fixes the stream layout)


@dataclass(frozen=True)
class Workload:
    name: str
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_h: int
    page_size: int
    rotate_k: bool
    rotate_v: bool
    num_seqs: int
    len_lo: int              # context length after the append, uniform in [len_lo, len_hi]
    len_hi: int
    dist: str = "normal"     # "normal" or "student_t"
    nu: int = 4              # Student-t degrees of freedom (integer)
    scale: float = 1.0
    outliers: str = "per_head"   # "per_head": n channels per kv-head; "pairs": a fraction of (head, ch)
    outlier_count: int = 4
    outlier_frac: float = 0.0
    outlier_mult: float = 20.0
    k_bias_std: float = 0.0  # per-layer per-channel bias added to every K row
    shuffle_pages: bool = False
    seed: int = 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def variant(self, **kw) -> "Workload":
        return replace(self, **kw)


TINY = Workload("tiny", 1, 4, 2, 128, 128, 16, True, True, 4, 256, 256)

QWEN3_4B_LATENCY = Workload(
    "qwen3-4b-latency", 36, 32, 8, 128, 128, 16, True, False, 1, 32768, 32768,
    outliers="pairs", outlier_frac=0.01, outlier_mult=15.0, k_bias_std=2.0)

QWEN3_8B_CONCURRENT = Workload(
    "qwen3-8b-concurrent", 36, 32, 8, 128, 128, 16, True, True, 64, 2048, 16384,
    dist="student_t", nu=4)

QWEN3_32B_HIGH_CONCURRENCY = Workload(
    "qwen3-32b-high-concurrency", 64, 64, 8, 128, 128, 16, True, True, 256, 4096, 8192,
    dist="student_t", nu=4, shuffle_pages=True)

LONG_PREFILL = Workload(
    "long-131072", 1, 32, 8, 128, 128, 64, True, True, 8, 131072, 131072,
    dist="student_t", nu=3)

ALL = {w.name: w for w in (TINY, QWEN3_4B_LATENCY, QWEN3_8B_CONCURRENT,
                           QWEN3_32B_HIGH_CONCURRENCY, LONG_PREFILL)}


def generator(wl: Workload, layer: int, stream: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed * 1_000_000 + layer * 16 + stream)
    return g


def seq_lens(wl: Workload) -> torch.Tensor:
    """Context lengths (after the decode step's append), int32 on the CPU."""
    if wl.len_lo == wl.len_hi:
        return torch.full((wl.num_seqs,), wl.len_lo, dtype=torch.int32)
    g = generator(wl, 0, LENS, "cpu")
    return torch.randint(wl.len_lo, wl.len_hi + 1, (wl.num_seqs,), generator=g,
                         dtype=torch.int64).to(torch.int32)


def page_tables(wl: Workload, lens: torch.Tensor, spare_pages: int = 0):
    """Block tables [B, max_blocks] int32 (unused entries -1) and the page count.

    Pages are handed out sequence after sequence; with shuffle_pages the ids
    are a seeded random permutation, so a sequence's pages are scattered."""
    P = wl.page_size
    per = [(int(L) + P - 1) // P for L in lens.tolist()]
    total = sum(per) + spare_pages
    ids = torch.arange(total, dtype=torch.int64)
    if wl.shuffle_pages:
        ids = ids[torch.randperm(total, generator=generator(wl, 0, PAGES, "cpu"))]
    max_blocks = max(per) if per else 0
    bt = torch.full((len(per), max(max_blocks, 1)), -1, dtype=torch.int32)
    nxt = 0
    for b, n in enumerate(per):
        bt[b, :n] = ids[nxt:nxt + n].to(torch.int32)
        nxt += n
    return bt, total


def slots_for(block_tables: torch.Tensor, page_size: int, seq: int, begin: int,
              end: int) -> torch.Tensor:
    """Slot ids of tokens [begin, end) of one sequence (int32, same device)."""
    j = torch.arange(begin, end, device=block_tables.device, dtype=torch.int64)
    return (block_tables[seq, j // page_size].to(torch.int64) * page_size + j % page_size).to(torch.int32)


def prefill_slots(block_tables: torch.Tensor, lens, page_size: int) -> torch.Tensor:
    """Slots of every token of every sequence, sequence-major (int32)."""
    parts = [slots_for(block_tables, page_size, b, 0, int(L)) for b, L in enumerate(list(lens))]
    if not parts:
        return torch.zeros(0, dtype=torch.int32, device=block_tables.device)
    return torch.cat(parts)


def _base(wl: Workload, g: torch.Generator, n: int, device) -> torch.Tensor:
    if wl.dist == "normal":
        x = torch.randn(n, generator=g, device=device)
    elif wl.dist == "student_t":
        # t = Z / sqrt(chi2_nu / nu), chi2_nu a sum of nu squared normals
        z = torch.randn(n, generator=g, device=device)
        chi = torch.zeros(n, device=device)
        for _ in range(wl.nu):
            chi += torch.randn(n, generator=g, device=device).square()
        x = z / torch.sqrt(chi / wl.nu)
    else:
        raise ValueError(wl.dist)
    return x * wl.scale


def outlier_gain(wl: Workload, layer: int, tensor: int, device) -> torch.Tensor:
    """Per-(kv-head, channel) multiplier [Hkv, D]: 1, or outlier_mult on the
    outlier channels.  Channel sets are fixed for all tokens of the layer."""
    Hkv, D = wl.num_kv_heads, wl.head_dim
    g = generator(wl, layer, K_OUTLIERS if tensor == K else V_OUTLIERS, "cpu")
    gain = torch.ones(Hkv, D)
    if wl.outliers == "per_head":
        for h in range(Hkv):
            idx = torch.randperm(D, generator=g)[:wl.outlier_count]
            gain[h, idx] = wl.outlier_mult
    elif wl.outliers == "pairs":
        n = max(1, int(round(wl.outlier_frac * Hkv * D)))
        idx = torch.randperm(Hkv * D, generator=g)[:n]
        gain.view(-1)[idx] = wl.outlier_mult
    return gain.to(device)


def k_bias(wl: Workload, layer: int, device) -> torch.Tensor | None:
    if wl.k_bias_std == 0.0:
        return None
    g = generator(wl, layer, K_BIAS, "cpu")
    return (torch.randn(wl.num_kv_heads, wl.head_dim, generator=g) * wl.k_bias_std).to(device)


def kv_rows(wl: Workload, layer: int, tensor: int, num_tokens: int, device,
            token_offset: int = 0, dtype=torch.bfloat16) -> torch.Tensor:
    """[num_tokens, Hkv, D] of K (tensor=K) or V (tensor=V) rows for tokens
    [token_offset, token_offset + num_tokens) of the layer's stream, rounded
    to `dtype` (bfloat16, or float16 for the binary16-input variant)."""
    Hkv, D = wl.num_kv_heads, wl.head_dim
    gain = outlier_gain(wl, layer, tensor, device)
    bias = k_bias(wl, layer, device) if tensor == K else None
    out = torch.empty(num_tokens, Hkv, D, dtype=dtype, device=device)
    g = generator(wl, layer, tensor, device)
    # walk the stream chunk by chunk so a slice does not depend on its neighbours
    first = token_offset // GEN_CHUNK_TOKENS
    last = (token_offset + num_tokens + GEN_CHUNK_TOKENS - 1) // GEN_CHUNK_TOKENS
    for ch in range(0, last):
        x = _base(wl, g, GEN_CHUNK_TOKENS * Hkv * D, device)
        if ch < first:
            continue
        lo = ch * GEN_CHUNK_TOKENS
        a, b = max(lo, token_offset), min(lo + GEN_CHUNK_TOKENS, token_offset + num_tokens)
        x = x.view(GEN_CHUNK_TOKENS, Hkv, D)[a - lo:b - lo] * gain
        if bias is not None:
            x = x + bias
        out[a - token_offset:b - token_offset] = x.to(dtype)
    return out


def q_rows(wl: Workload, layer: int, device, num_seqs: int | None = None,
           dtype=torch.bfloat16) -> torch.Tensor:
    B = wl.num_seqs if num_seqs is None else num_seqs
    g = generator(wl, layer, Q, device)
    return torch.randn(B, wl.num_q_heads, wl.head_dim, generator=g, device=device).to(dtype)


def decode_bytes(wl: Workload, lens) -> int:
    """Algorithmic HBM bytes of one decode pass over one layer: K and V codes
    plus (scale, zero) of every attended (token, kv-head), the block-table
    entries, q in and the output out."""
    P, D, Hkv, Hq = wl.page_size, wl.head_dim, wl.num_kv_heads, wl.num_q_heads
    per_row = D // 2 + 4
    toks = sum(int(L) for L in lens)
    pages = sum((int(L) + P - 1) // P for L in lens)
    B = len(list(lens))
    return 2 * per_row * toks * Hkv + 4 * pages + B * Hq * D * (2 + 4) + 4 * B


def decode_bytes_bf16(wl: Workload, lens) -> int:
    """The same for a BF16 cache: K and V bfloat16 rows of every attended
    (token, kv-head), block-table entries, q in and the output out."""
    P, D, Hkv, Hq = wl.page_size, wl.head_dim, wl.num_kv_heads, wl.num_q_heads
    toks = sum(int(L) for L in lens)
    pages = sum((int(L) + P - 1) // P for L in lens)
    B = len(list(lens))
    return 2 * 2 * D * toks * Hkv + 4 * pages + B * Hq * D * (2 + 4) + 4 * B


def append_bytes(wl: Workload, num_tokens: int, with_v: bool = True) -> int:
    """Algorithmic HBM bytes of one quantize-append of num_tokens tokens:
    bfloat16 rows in, codes and (scale, zero) out, one slot id per token."""
    D, Hkv = wl.head_dim, wl.num_kv_heads
    per_row = 2 * D + D // 2 + 4
    return num_tokens * (Hkv * per_row * (2 if with_v else 1) + 4)


def max_len(lens) -> int:
    return max((int(L) for L in lens), default=0)

