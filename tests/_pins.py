"""Pins for the fp64 oracle: checks against facts fixed by the mathematics,
independent of the oracle's own code.

Each ``pin_*`` takes an optional ``lib`` (another build of the oracle source,
used by the tests that plant mistakes) and raises AssertionError on failure.

What pins what:
  pin_bruteforce_*       the definition evaluated at 50 significant digits with
                         exact rational scores (Fraction) and Decimal exp/ln, on
                         tiny shapes (d_c=8, d_r=4), batch 2, ragged, masked ids
  pin_numpy_reference    numpy/scipy float64 softmax at the real dims (512 + 64)
  pin_uniform_scores     q = 0: out = mean of the attended c rows, lse = ln n
  pin_single_row         one attended row: out = that row's c, lse = its score
  pin_identical_rows     all c rows equal v: out = v for any q
  pin_split_invariance   split emulation (S = 1..64) equals the two-pass result
  pin_sparse_is_dense    sparse with ids = a permutation of 0..T-1 equals dense
  pin_permutation        reordering the id list does not change the result
  pin_argmax_limit       q scaled up: out tends to the arg-max row
  pin_e4m3_decoding      FP8 (E4M3) bytes: PyTorch's float8_e4m3fn widening of all 256
  pin_e4m3_decode        FP8-cache decode: numpy float64 softmax over the cache
                         dequantised by PyTorch's widening times the scale
"""
from __future__ import annotations

from decimal import Decimal, getcontext
from fractions import Fraction
import math

import numpy as np
import torch

import oracle
import workloads


def _f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening bf16 -> float64 (bf16 -> fp32 is exact, fp32 -> fp64 is exact)."""
    return t.float().double().numpy()


def _attended(kind, B, d_pos=None, row_offset=None, indices=None, cache_len=None):
    """Attended absolute row ids per request, written from the definition."""
    rows = []
    for b in range(B):
        base = int(row_offset[b]) if row_offset is not None else 0
        if kind == "dense":
            rows.append([base + t for t in range(int(d_pos[b]) + 1)])
        else:
            rows.append([base + int(i) for i in indices[b] if 0 <= int(i) < int(cache_len[b])])
    return rows


def _decimal_reference(q, kv, rows, scale, dc):
    """out/lse from the definition at 50 digits (exact scores, Decimal exp/ln)."""
    getcontext().prec = 50
    qf = _f64(q)
    kvf = _f64(kv)
    B, H, D = qf.shape
    sc = Fraction(scale)
    out = np.zeros((B, H, dc))
    lse = np.zeros((B, H))
    for b in range(B):
        for h in range(H):
            weights = []
            for r in rows[b]:
                s = sum((Fraction(float(qf[b, h, i])) * Fraction(float(kvf[r, i])) for i in range(D)),
                        Fraction(0)) * sc
                weights.append((Decimal(s.numerator) / Decimal(s.denominator)).exp())
            if not weights:
                lse[b, h] = -math.inf
                continue
            Z = sum(weights, Decimal(0))
            lse[b, h] = float(Z.ln())
            for f in range(dc):
                num = sum((w * Decimal(float(kvf[r, f])) for w, r in zip(weights, rows[b])), Decimal(0))
                out[b, h, f] = float(num / Z)
    return out, lse


def _close(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    if fin.any():
        err = np.abs(a[fin] - b[fin]) / np.maximum(1.0, np.abs(b[fin]))
        assert err.max() <= tol, f"{what}: max scaled err {err.max():.3e} > {tol:.1e}"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: non-finite entries differ"


# --------------------------------------------------------------------------
def pin_bruteforce_dense(lib=None):
    dc, dr = 8, 4
    B, H, cap = 2, 3, 13
    q = workloads.randn_bf16(B * H, dc + dr, seed=11, stream=1).view(B, H, dc + dr)
    kv = workloads.randn_bf16(B * cap, dc + dr, seed=11, stream=2)
    d_pos = torch.tensor([12, 5], dtype=torch.int32)
    off = torch.tensor([0, cap], dtype=torch.int64)
    scale = 1.0 / math.sqrt(dc + dr)
    out, lse = oracle.decode(q, kv, scale=scale, d_latent=dc, d_rope=dr, d_pos=d_pos, row_offset=off, lib=lib)
    ref_o, ref_l = _decimal_reference(q, kv, _attended("dense", B, d_pos=d_pos, row_offset=off), scale, dc)
    _close(lse, ref_l, 1e-13, "dense lse vs 50-digit definition")
    _close(out, ref_o, 1e-13, "dense out vs 50-digit definition")


def pin_bruteforce_sparse(lib=None):
    dc, dr = 8, 4
    B, H = 2, 2
    lens = torch.tensor([20, 9], dtype=torch.int32)
    off = torch.tensor([0, 20], dtype=torch.int64)
    kv = workloads.randn_bf16(29, dc + dr, seed=12, stream=2)
    q = workloads.randn_bf16(B * H, dc + dr, seed=12, stream=1).view(B, H, dc + dr)
    # includes out-of-range ids (-1, len, len + 3) that must be masked
    idx = torch.tensor([[3, 19, -1, 7, 20, 0], [8, 9, 2, 12, 4, 0]], dtype=torch.int32)
    scale = 0.37
    out, lse = oracle.decode(q, kv, scale=scale, d_latent=dc, d_rope=dr, indices=idx, cache_len=lens,
                             row_offset=off, lib=lib)
    rows = _attended("sparse", B, row_offset=off, indices=idx, cache_len=lens)
    ref_o, ref_l = _decimal_reference(q, kv, rows, scale, dc)
    _close(lse, ref_l, 1e-13, "sparse lse vs 50-digit definition")
    _close(out, ref_o, 1e-13, "sparse out vs 50-digit definition")


def _numpy_reference(q, kv, rows, scale, dc):
    from scipy.special import logsumexp
    qf = _f64(q)
    kvf = _f64(kv)
    B, H, _ = qf.shape
    out = np.zeros((B, H, dc))
    lse = np.zeros((B, H))
    for b in range(B):
        K = kvf[rows[b]]                       # [n, D]
        s = (qf[b] @ K.T) * scale              # [H, n]
        lse[b] = logsumexp(s, axis=1)
        p = np.exp(s - lse[b][:, None])
        out[b] = p @ K[:, :dc]
    return out, lse


def pin_numpy_reference(lib=None):
    D = workloads.D_ROW
    B, H, cap = 2, 4, 700
    q = workloads.randn_bf16(B * H, D, seed=13, stream=1).view(B, H, D)
    kv = workloads.randn_bf16(B * cap, D, seed=13, stream=2)
    d_pos = torch.tensor([699, 321], dtype=torch.int32)
    off = torch.tensor([0, cap], dtype=torch.int64)
    s = workloads.SCALE
    out, lse = oracle.decode(q, kv, scale=s, d_pos=d_pos, row_offset=off, lib=lib)
    ro, rl = _numpy_reference(q, kv, _attended("dense", B, d_pos=d_pos, row_offset=off), s, 512)
    _close(lse, rl, 1e-12, "dense lse vs numpy")
    _close(out, ro, 1e-12, "dense out vs numpy")
    lens = torch.tensor([700, 650], dtype=torch.int32)
    off2 = torch.tensor([0, 700], dtype=torch.int64)
    kv2 = workloads.randn_bf16(1350, D, seed=13, stream=5)
    idx = torch.stack([workloads.unique_indices(700, 97, seed=13, stream=3, chunk=0),
                       workloads.unique_indices(650, 97, seed=13, stream=3, chunk=1)])
    out, lse = oracle.decode(q, kv2, scale=s, indices=idx, cache_len=lens, row_offset=off2, lib=lib)
    rows = _attended("sparse", B, row_offset=off2, indices=idx, cache_len=lens)
    ro, rl = _numpy_reference(q, kv2, rows, s, 512)
    _close(lse, rl, 1e-12, "sparse lse vs numpy")
    _close(out, ro, 1e-12, "sparse out vs numpy")


def pin_uniform_scores(lib=None):
    D = workloads.D_ROW
    B, H, cap = 2, 2, 300
    q = torch.zeros(B, H, D, dtype=torch.bfloat16)
    kv = workloads.randn_bf16(B * cap, D, seed=14, stream=2)
    kvf = _f64(kv)
    d_pos = torch.tensor([299, 136], dtype=torch.int32)
    off = torch.tensor([0, cap], dtype=torch.int64)
    out, lse = oracle.decode(q, kv, scale=workloads.SCALE, d_pos=d_pos, row_offset=off, lib=lib)
    for b, rows in enumerate(_attended("dense", B, d_pos=d_pos, row_offset=off)):
        n = len(rows)
        mean = np.array([float(sum(Fraction(float(kvf[r, f])) for r in rows) / n) for f in range(512)])
        for h in range(H):
            assert abs(lse[b, h] - math.log(n)) <= 1e-13 * math.log(n), "uniform dense lse != ln n"
            assert np.abs(out[b, h] - mean).max() <= 1e-13, "uniform dense out != mean row"
    lens = torch.tensor([1000, 37], dtype=torch.int32)
    off2 = torch.tensor([0, 1000], dtype=torch.int64)
    kv2 = workloads.randn_bf16(1037, D, seed=14, stream=5)
    kv2f = _f64(kv2)
    idx = torch.stack([workloads.unique_indices(1000, 30, seed=14, stream=3, chunk=0),
                       workloads.unique_indices(37, 30, seed=14, stream=3, chunk=1)])
    idx[0, 5] = -3          # masked entries shrink n
    idx[1, 2] = 37
    out, lse = oracle.decode(q, kv2, scale=workloads.SCALE, indices=idx, cache_len=lens, row_offset=off2,
                             lib=lib)
    for b, rows in enumerate(_attended("sparse", B, row_offset=off2, indices=idx, cache_len=lens)):
        n = len(rows)
        assert n == 29
        mean = np.array([float(sum(Fraction(float(kv2f[r, f])) for r in rows) / n) for f in range(512)])
        for h in range(H):
            assert abs(lse[b, h] - math.log(n)) <= 1e-13 * math.log(n), "uniform sparse lse != ln n"
            assert np.abs(out[b, h] - mean).max() <= 1e-13, "uniform sparse out != mean row"


def pin_single_row(lib=None):
    D = workloads.D_ROW
    H = 3
    q = workloads.randn_bf16(H, D, seed=15, stream=1).view(1, H, D)
    kv = workloads.randn_bf16(4, D, seed=15, stream=2)
    d_pos = torch.tensor([0], dtype=torch.int32)
    out, lse = oracle.decode(q, kv, scale=workloads.SCALE, d_pos=d_pos, lib=lib)
    kvf = _f64(kv)
    qf = _f64(q)
    for h in range(H):
        assert np.array_equal(out[0, h], kvf[0, :512]), "T=1: out must equal the row's latent"
        s = float(np.dot(qf[0, h], kvf[0])) * workloads.SCALE
        assert abs(lse[0, h] - s) <= 1e-12 * max(1.0, abs(s)), "T=1: lse must equal the score"


def pin_identical_rows(lib=None):
    D = workloads.D_ROW
    T = 64
    q = workloads.randn_bf16(2, D, seed=16, stream=1).view(1, 2, D)
    kv = workloads.randn_bf16(T, D, seed=16, stream=2)
    kv[:, :512] = kv[0, :512]           # same latent everywhere, different rope parts
    out, _ = oracle.decode(q, kv, scale=workloads.SCALE, d_pos=torch.tensor([T - 1], dtype=torch.int32),
                           lib=lib)
    v = _f64(kv)[0, :512]
    assert np.abs(out[0] - v[None]).max() <= 1e-13 * max(1.0, np.abs(v).max()), "identical rows: out != v"


def pin_split_invariance(lib=None):
    D = workloads.D_ROW
    T = 517
    q = workloads.randn_bf16(2, D, seed=17, stream=1).view(1, 2, D)
    kv = workloads.randn_bf16(T, D, seed=17, stream=2)
    d_pos = torch.tensor([T - 1], dtype=torch.int32)
    ref_o, ref_l = oracle.decode(q, kv, scale=workloads.SCALE, d_pos=d_pos, lib=lib)
    for S in (1, 2, 3, 5, 8, 16, 64):
        for g in (1, 32):
            o, l = oracle.decode_split(q, kv, scale=workloads.SCALE, splits=S, granule=g, d_pos=d_pos, lib=lib)
            _close(l, ref_l, 1e-12, f"split S={S} g={g} lse")
            _close(o, ref_o, 1e-12, f"split S={S} g={g} out")
    # sparse list with masked entries
    lens = torch.tensor([T], dtype=torch.int32)
    off = torch.tensor([0], dtype=torch.int64)
    idx = workloads.unique_indices(T, 300, seed=17, stream=3).view(1, -1).clone()
    idx[0, 10] = -1
    idx[0, 250] = T
    ref_o, ref_l = oracle.decode(q, kv, scale=workloads.SCALE, indices=idx, cache_len=lens, row_offset=off,
                                 lib=lib)
    for S in (1, 4, 7, 64):
        o, l = oracle.decode_split(q, kv, scale=workloads.SCALE, splits=S, granule=32, indices=idx,
                                   cache_len=lens, row_offset=off, lib=lib)
        _close(l, ref_l, 1e-12, f"sparse split S={S} lse")
        _close(o, ref_o, 1e-12, f"sparse split S={S} out")
    # a single slice reproduces the whole computation as its own partial
    o, l, op, lp = oracle.decode_split(q, kv, scale=workloads.SCALE, splits=1, d_pos=d_pos,
                                       return_partials=True, lib=lib)
    _close(op[:, :, 0], o, 1e-15, "S=1 partial out")
    _close(lp[:, :, 0], l, 1e-15, "S=1 partial lse")
    # more slices than rows: trailing slices are empty (lse_s = -inf, o_s = 0)
    small_pos = torch.tensor([4], dtype=torch.int32)
    o, l, op, lp = oracle.decode_split(q, kv, scale=workloads.SCALE, splits=8, d_pos=small_pos,
                                       return_partials=True, lib=lib)
    assert np.all(np.isneginf(lp[0, :, 5:])) and np.all(op[0, :, 5:] == 0.0), "empty slices"
    o1, l1 = oracle.decode(q, kv, scale=workloads.SCALE, d_pos=small_pos, lib=lib)
    _close(l, l1, 1e-13, "empty-slice lse")
    _close(o, o1, 1e-13, "empty-slice out")


def pin_sparse_is_dense(lib=None):
    D = workloads.D_ROW
    T = 400
    q = workloads.randn_bf16(3, D, seed=18, stream=1).view(1, 3, D)
    kv = workloads.randn_bf16(T, D, seed=18, stream=2)
    dense_o, dense_l = oracle.decode(q, kv, scale=workloads.SCALE, d_pos=torch.tensor([T - 1], dtype=torch.int32),
                                     lib=lib)
    idx = workloads.unique_indices(T, T, seed=18, stream=3).view(1, -1)
    so, sl = oracle.decode(q, kv, scale=workloads.SCALE, indices=idx, cache_len=torch.tensor([T], dtype=torch.int32),
                           row_offset=torch.tensor([0], dtype=torch.int64), lib=lib)
    _close(sl, dense_l, 1e-12, "sparse(all ids) lse vs dense")
    _close(so, dense_o, 1e-12, "sparse(all ids) out vs dense")


def pin_permutation(lib=None):
    D = workloads.D_ROW
    T = 2000
    q = workloads.randn_bf16(2, D, seed=19, stream=1).view(1, 2, D)
    kv = workloads.randn_bf16(T, D, seed=19, stream=2)
    lens = torch.tensor([T], dtype=torch.int32)
    off = torch.tensor([0], dtype=torch.int64)
    idx = workloads.unique_indices(T, 256, seed=19, stream=3).view(1, -1)
    perm = workloads.unique_indices(256, 256, seed=19, stream=4).long()
    a_o, a_l = oracle.decode(q, kv, scale=workloads.SCALE, indices=idx, cache_len=lens, row_offset=off, lib=lib)
    b_o, b_l = oracle.decode(q, kv, scale=workloads.SCALE, indices=idx[:, perm], cache_len=lens, row_offset=off,
                             lib=lib)
    _close(b_l, a_l, 1e-13, "permuted ids lse")
    _close(b_o, a_o, 1e-13, "permuted ids out")


def pin_argmax_limit(lib=None):
    D = workloads.D_ROW
    T = 128
    q = workloads.randn_bf16(2, D, seed=20, stream=1).view(1, 2, D)
    kv = workloads.randn_bf16(T, D, seed=20, stream=2)
    big = (q.float() * 1024.0).to(torch.bfloat16)      # exact: power-of-two scaling
    out, _ = oracle.decode(big, kv, scale=workloads.SCALE, d_pos=torch.tensor([T - 1], dtype=torch.int32), lib=lib)
    s = _f64(big)[0] @ _f64(kv).T
    for h in range(2):
        top = int(np.argmax(s[h]))
        gap = np.sort(s[h])[-1] - np.sort(s[h])[-2]
        assert gap * workloads.SCALE > 40, "fixture: top score must dominate"
        assert np.abs(out[0, h] - _f64(kv)[top, :512]).max() <= 1e-9, "large q: out must be the arg-max row"


def _torch_e4m3(b: np.ndarray) -> np.ndarray:
    """PyTorch's float8_e4m3fn widening of E4M3 bytes (independent of the oracle)."""
    return torch.from_numpy(np.ascontiguousarray(b)).view(torch.float8_e4m3fn).double().numpy()


def pin_e4m3_decoding(lib=None):
    every = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_values(every, lib=lib)
    ref = _torch_e4m3(every)
    assert np.array_equal(np.isnan(v), np.isnan(ref)), "E4M3: NaN patterns"
    fin = ~np.isnan(ref)
    assert np.array_equal(v[fin], ref[fin]), "E4M3: byte values differ from float8_e4m3fn"
    assert v[0x01] == 2.0 ** -9 and v[0x38] == 1.0 and v[0x7E] == 448.0, "E4M3: special values"


def pin_e4m3_decode(lib=None):
    """The FP8-cache decode at the real dims against numpy float64 softmax over
    the cache dequantised by PyTorch's float8 widening times the scale."""
    rng = np.random.default_rng(31)
    T = 90
    kv8 = rng.integers(0, 256, size=(T, 576), dtype=np.uint8)
    kv8[(kv8 & 0x7F) == 0x7F] = 0x30
    q = workloads.randn_bf16(3, 576, seed=31, stream=1).view(1, 3, 576)
    vals = _torch_e4m3(kv8)
    for kv_scale in (1.0, 0.37):
        out, lse = oracle.decode_e4m3(q, kv8, kv_scale=kv_scale, scale=workloads.SCALE,
                                      d_pos=np.array([T - 1], np.int32), lib=lib)
        v = vals * kv_scale
        s = (_f64(q)[0] @ v.T) * workloads.SCALE
        m = s.max(axis=1, keepdims=True)
        w = np.exp(s - m)
        ref_lse = (m + np.log(w.sum(axis=1, keepdims=True)))[:, 0]
        ref = (w / w.sum(axis=1, keepdims=True)) @ v[:, :512]
        _close(out[0], ref, 1e-9 * max(1.0, np.abs(ref).max()), f"E4M3 decode out (scale {kv_scale})")
        _close(lse[0], ref_lse, 1e-11, f"E4M3 decode lse (scale {kv_scale})")


ALL_PINS = [pin_bruteforce_dense, pin_bruteforce_sparse, pin_numpy_reference, pin_uniform_scores,
            pin_single_row, pin_identical_rows, pin_split_invariance, pin_sparse_is_dense,
            pin_permutation, pin_argmax_limit, pin_e4m3_decoding, pin_e4m3_decode]
