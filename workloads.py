"""Seeded synthetic inputs for MLA decode (shared by the tests, the oracle
checks and the benchmark).

This module holds no attention arithmetic: it only draws random numbers and
lays them out.  Every tensor is drawn on the CPU from torch generators seeded
from ``(seed, stream, chunk)`` with splitmix64, so the values do not depend on
the thread count.  Values are N(0, 1) drawn in float32 and rounded to bf16
(round-to-nearest-even); indices are drawn without replacement.

Workloads (latent d_c = 512, rope d_r = 64, one row = [c | k_rope] = 576 bf16,
scale = 1/sqrt(576)):

  dense_t256       dense, B=1, H=16, context T=256 (d_pos = 255)
  dense_t8192      dense, B=1, H=16, context T=8192 (d_pos = 8191)
  sparse_k2048     sparse, B=1, H=16, 65,536-row cache, top-k 2048 unique unsorted
  sparse_b64       sparse, B=64, H=16, per-request cache length ~ U[4096, 131072],
                   packed ragged cache, top-k 2048 unique unsorted per request
  graph_h128       dense, B=1, H=128, start context 32,768, 64 decode steps that each
                   append one new row at position d_pos and advance d_pos

Draw order per workload (stream ids): lengths (sparse_b64 only), q, kv, indices;
graph_h128 adds the 64 new rows and the 64 per-step queries.

FP8 caches (``to_e4m3``): the same bf16 draws, stored as OCP E4M3 bytes with
one scale per cache, amax / 448 (PyTorch's float8_e4m3fn rounding,
nearest-even); the oracle and the GPU both read those bytes.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
import os

import torch

D_LATENT = 512
D_ROPE = 64
D_ROW = D_LATENT + D_ROPE
SCALE = 1.0 / math.sqrt(D_ROW)

_MASK64 = (1 << 64) - 1
_CHUNK_ROWS = 8192


def _splitmix64(x: int) -> int:
    x = (x + 0x9E3779B97F4A7C15) & _MASK64
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
    return z ^ (z >> 31)


def _seed(seed: int, stream: int, chunk: int) -> int:
    s = _splitmix64(seed & _MASK64)
    s = _splitmix64(s ^ (stream & _MASK64))
    s = _splitmix64(s ^ (chunk & _MASK64))
    return s & ((1 << 63) - 1)


def _gen(seed: int, stream: int, chunk: int) -> torch.Generator:
    return torch.Generator().manual_seed(_seed(seed, stream, chunk))


def randn_bf16(rows: int, cols: int, *, seed: int, stream: int, out: torch.Tensor | None = None,
               threads: int | None = None) -> torch.Tensor:
    """[rows, cols] bf16 of N(0,1) values, drawn in chunks of 8192 rows."""
    if out is None:
        out = torch.empty(rows, cols, dtype=torch.bfloat16)
    n_chunks = (rows + _CHUNK_ROWS - 1) // _CHUNK_ROWS

    def fill(i: int) -> None:
        r0 = i * _CHUNK_ROWS
        r1 = min(rows, r0 + _CHUNK_ROWS)
        g = _gen(seed, stream, i)
        out[r0:r1] = torch.randn(r1 - r0, cols, generator=g, dtype=torch.float32).to(torch.bfloat16)

    if n_chunks <= 1:
        if n_chunks == 1:
            fill(0)
        return out
    threads = threads or min(n_chunks, os.cpu_count() or 1)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fill, range(n_chunks)))
    return out


def unique_indices(n: int, k: int, *, seed: int, stream: int, chunk: int = 0) -> torch.Tensor:
    """k distinct ids from range(n), in random (unsorted) order, int32."""
    if k > n:
        raise ValueError("k > n")
    g = _gen(seed, stream, chunk)
    return torch.randperm(n, generator=g)[:k].to(torch.int32)


@dataclass
class DenseInputs:
    q: torch.Tensor            # bf16 [B, H, 576]
    kv: torch.Tensor           # bf16 [rows, 576]
    d_pos: torch.Tensor        # int32 [B]; request b attends rows row_offset[b] + 0 .. d_pos[b]
    row_offset: torch.Tensor   # int64 [B]
    scale: float = SCALE


@dataclass
class SparseInputs:
    q: torch.Tensor            # bf16 [B, H, 576]
    kv: torch.Tensor           # bf16 [sum(cache_len), 576] packed segments
    indices: torch.Tensor      # int32 [B, topk], request-local row ids
    cache_len: torch.Tensor    # int32 [B]
    row_offset: torch.Tensor   # int64 [B], exclusive prefix sum of cache_len
    scale: float = SCALE


@dataclass
class GraphInputs:
    q_steps: torch.Tensor      # bf16 [steps, B, H, 576]; step k uses q_steps[k]
    kv: torch.Tensor           # bf16 [T0 + steps, 576]; rows >= T0 start as zeros
    new_rows: torch.Tensor     # bf16 [steps, B, 576]; step k writes new_rows[k] at row d_pos
    d_pos0: int                # d_pos before step 0 (= T0)
    steps: int
    scale: float = SCALE
    meta: dict = field(default_factory=dict)


def dense(B: int, H: int, T: int, *, seed: int = 0, capacity: int | None = None) -> DenseInputs:
    """Dense decode: every request attends rows 0..T-1 of its own segment."""
    cap = capacity if capacity is not None else T
    if cap < T:
        raise ValueError("capacity < T")
    q = randn_bf16(B * H, D_ROW, seed=seed, stream=1).view(B, H, D_ROW)
    kv = randn_bf16(B * cap, D_ROW, seed=seed, stream=2)
    d_pos = torch.full((B,), T - 1, dtype=torch.int32)
    row_offset = torch.arange(B, dtype=torch.int64) * cap
    return DenseInputs(q=q, kv=kv, d_pos=d_pos, row_offset=row_offset)


def sparse(B: int, H: int, cache_len, topk: int, *, seed: int = 0) -> SparseInputs:
    """Sparse decode over a packed ragged cache; ``cache_len`` is an int or a list."""
    if isinstance(cache_len, int):
        lens = torch.full((B,), cache_len, dtype=torch.int32)
    else:
        lens = torch.as_tensor(cache_len, dtype=torch.int32)
    if lens.numel() != B:
        raise ValueError("cache_len must have B entries")
    offs = torch.zeros(B, dtype=torch.int64)
    if B > 1:
        offs[1:] = torch.cumsum(lens.to(torch.int64), 0)[:-1]
    total = int(lens.to(torch.int64).sum())
    q = randn_bf16(B * H, D_ROW, seed=seed, stream=1).view(B, H, D_ROW)
    kv = randn_bf16(total, D_ROW, seed=seed, stream=2)
    idx = torch.stack([unique_indices(int(lens[b]), topk, seed=seed, stream=3, chunk=b) for b in range(B)])
    return SparseInputs(q=q, kv=kv, indices=idx.contiguous(), cache_len=lens, row_offset=offs)


def ragged_lengths(B: int, lo: int, hi: int, *, seed: int = 0) -> torch.Tensor:
    """Per-request cache lengths uniform on [lo, hi] (inclusive), int32."""
    g = _gen(seed, 0, 0)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def graph(H: int, T0: int, steps: int, *, B: int = 1, seed: int = 0) -> GraphInputs:
    """Multi-step decode: the cache holds T0 rows; step k appends new_rows[k]
    at row d_pos = T0 + k, attends rows 0..d_pos and then advances d_pos."""
    if B != 1:
        raise ValueError("the multi-step workload is batch 1")
    q_steps = randn_bf16(steps * B * H, D_ROW, seed=seed, stream=1).view(steps, B, H, D_ROW)
    kv = torch.zeros(T0 + steps, D_ROW, dtype=torch.bfloat16)
    randn_bf16(T0, D_ROW, seed=seed, stream=2, out=kv[:T0])
    new_rows = randn_bf16(steps * B, D_ROW, seed=seed, stream=4).view(steps, B, D_ROW)
    return GraphInputs(q_steps=q_steps, kv=kv, new_rows=new_rows, d_pos0=T0, steps=steps)


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------
WORKLOADS = {
    "dense_t256": dict(kind="dense", B=1, H=16, T=256),
    "dense_t8192": dict(kind="dense", B=1, H=16, T=8192),
    "sparse_k2048": dict(kind="sparse", B=1, H=16, cache=65536, topk=2048),
    "sparse_b64": dict(kind="sparse", B=64, H=16, len_lo=4096, len_hi=131072, topk=2048),
    "graph_h128": dict(kind="graph", B=1, H=128, T0=32768, steps=64),
}


def make(name: str, *, seed: int = 0):
    w = WORKLOADS[name]
    if w["kind"] == "dense":
        return dense(w["B"], w["H"], w["T"], seed=seed)
    if w["kind"] == "sparse":
        if "cache" in w:
            return sparse(w["B"], w["H"], w["cache"], w["topk"], seed=seed)
        lens = ragged_lengths(w["B"], w["len_lo"], w["len_hi"], seed=seed)
        return sparse(w["B"], w["H"], lens.tolist(), w["topk"], seed=seed)
    if w["kind"] == "graph":
        return graph(w["H"], w["T0"], w["steps"], B=w["B"], seed=seed)
    raise KeyError(name)


E4M3_MAX = 448.0


def to_e4m3(kv: torch.Tensor):
    """Quantise a bf16 cache to E4M3 bytes with one scale (amax / 448, so the
    largest magnitude maps to the largest finite E4M3 value).  Returns the
    uint8 bytes (same shape) and the float scale; the value of a byte b is
    e4m3(b) * scale."""
    amax = float(kv.float().abs().max()) if kv.numel() else 0.0
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    q8 = (kv.float() / scale).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q8.view(torch.uint8), scale
