"""fp64 CPU oracle for split-KV MLA decode (ctypes binding to ``liboracle.so``).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``decode_attention_mla_gb300``) never imports it and shares no code with it.

The oracle computes, per request b and head h, over the attended rows R_b
(dense: ``0..d_pos[b]``; sparse: the in-range entries of the index list)::

    s_t    = (q_lat . c_t + q_rope . k_rope_t) * scale
    lse    = m + ln sum_t exp(s_t - m),   m = max_t s_t
    out[f] = sum_t exp(s_t - lse) * c_t[f]

in float64 from the exact widening of the stored bf16 values, in plain
sequential loops (two passes: max, then sum).  ``decode_split`` emulates the
split-KV partials and their log-sum-exp merge in float64.  Passages followed:
"Graph-resident decode" (Lecture 08) s.2 (n_ctx = *d_pos + 1; row address
cache + pos * key_length) and s.6 (normalised merge of per-slice partials, slice
sum in ascending order); "Launch Geometry" (Lecture 04) s.8 (a split count only
re-associates the combine); "The Commit That Changed Direction" (sparse gather
of indexed latent rows).  ``decode_e4m3`` takes an FP8 (OCP E4M3) cache with
one scale and dequantises it (``e4m3(byte) * kv_scale``, exact in float64)
before the same definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out_path: str) -> str:
    """Compile one C source file into a shared library (portable flags only)."""
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source if it is missing or stale."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


SOURCE_PATH = _SRC


def _bind(path: str):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    LL = ctypes.c_longlong
    D = ctypes.c_double
    lib.oracle_mla_decode_f64.restype = I
    lib.oracle_mla_decode_f64.argtypes = [P, P, LL, LL, I, I, I, I, D, I, P, P, P, P, I, P, P, I]
    lib.oracle_mla_decode_split_f64.restype = I
    lib.oracle_mla_decode_split_f64.argtypes = [P, P, LL, LL, I, I, I, I, D, I, P, P, P, P, I, I, I,
                                                P, P, P, P, I]
    lib.oracle_hardware_threads.restype = I
    lib.oracle_hardware_threads.argtypes = []
    lib.oracle_mla_project_f64.restype = I
    lib.oracle_mla_project_f64.argtypes = [P, P, I, I, I, I, P]
    lib.oracle_mla_decode_e4m3_f64.restype = I
    lib.oracle_mla_decode_e4m3_f64.argtypes = [P, P, D, LL, LL, I, I, I, I, D, I, P, P, P, P, I, I, I,
                                               P, P, P, P, I]
    lib.oracle_e4m3_to_f64.restype = I
    lib.oracle_e4m3_to_f64.argtypes = [P, LL, P]
    return lib


def bind(path: str):
    """Load another build of ``mla_oracle.c`` (e.g. a copy with a planted mistake)."""
    return _bind(path)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB_PATH)
        return _lib


def hardware_threads() -> int:
    return int(_load().oracle_hardware_threads())


def _u16(a) -> np.ndarray:
    """bf16 data as a contiguous uint16 numpy array (accepts torch bf16 tensors)."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        a = a.contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs must be torch.bfloat16 or uint16 bit patterns")
    return a


def _np(a, dtype):
    if a is None:
        return None
    if hasattr(a, "numpy") and not isinstance(a, np.ndarray):
        a = a.contiguous().numpy()
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _common(q, kv, d_latent, d_rope, row_stride):
    q16 = _u16(q)
    kv16 = _u16(kv)
    D = d_latent + d_rope
    if q16.shape[-1] != D:
        raise ValueError(f"q last dim {q16.shape[-1]} != d_latent + d_rope = {D}")
    if q16.ndim != 3:
        raise ValueError("q must be [B, H, d_latent + d_rope]")
    if row_stride is None:
        row_stride = kv16.shape[-1]
    kv_rows = kv16.size // row_stride if kv16.size else 0
    return q16, kv16, int(row_stride), int(kv_rows)


def decode(q, kv, *, scale: float, d_latent: int = 512, d_rope: int = 64, d_pos=None,
           indices=None, cache_len=None, row_offset=None, row_stride=None, n_threads: int = 0, lib=None):
    """Two-pass fp64 MLA decode.  Dense when ``indices`` is None.

    Returns ``(out[B,H,d_latent] float64, lse[B,H] float64)``.  ``lib`` selects
    another build of the same source (used by the tests that plant mistakes).
    """
    q16, kv16, row_stride, kv_rows = _common(q, kv, d_latent, d_rope, row_stride)
    B, H, _ = q16.shape
    sparse = indices is not None
    d_pos_a = _np(d_pos, np.int32)
    idx_a = _np(indices, np.int32)
    len_a = _np(cache_len, np.int32)
    off_a = _np(row_offset, np.int64)
    topk = int(idx_a.shape[-1]) if sparse else 0
    out = np.zeros((B, H, d_latent), np.float64)
    lse = np.zeros((B, H), np.float64)
    rc = (lib or _load()).oracle_mla_decode_f64(
        _ptr(q16), _ptr(kv16), kv_rows, row_stride, B, H, d_latent, d_rope, float(scale), int(sparse),
        _ptr(d_pos_a), _ptr(off_a), _ptr(len_a), _ptr(idx_a), topk, _ptr(out), _ptr(lse), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_mla_decode_f64 failed with status {rc}")
    return out, lse


def decode_split(q, kv, *, scale: float, splits: int, granule: int = 1, d_latent: int = 512,
                 d_rope: int = 64, d_pos=None, indices=None, cache_len=None, row_offset=None,
                 row_stride=None, n_threads: int = 0, return_partials: bool = False, lib=None):
    """fp64 emulation of split-KV partials plus the log-sum-exp merge.

    The attended entries (dense positions, or sparse list entries) are cut into
    ``splits`` contiguous slices of ``ceil(n / splits)`` entries rounded up to
    ``granule``; trailing slices may be empty (lse_s = -inf, o_s = 0).
    """
    q16, kv16, row_stride, kv_rows = _common(q, kv, d_latent, d_rope, row_stride)
    B, H, _ = q16.shape
    sparse = indices is not None
    d_pos_a = _np(d_pos, np.int32)
    idx_a = _np(indices, np.int32)
    len_a = _np(cache_len, np.int32)
    off_a = _np(row_offset, np.int64)
    topk = int(idx_a.shape[-1]) if sparse else 0
    out = np.zeros((B, H, d_latent), np.float64)
    lse = np.zeros((B, H), np.float64)
    o_part = np.zeros((B, H, splits, d_latent), np.float64) if return_partials else None
    lse_part = np.zeros((B, H, splits), np.float64) if return_partials else None
    rc = (lib or _load()).oracle_mla_decode_split_f64(
        _ptr(q16), _ptr(kv16), kv_rows, row_stride, B, H, d_latent, d_rope, float(scale), int(sparse),
        _ptr(d_pos_a), _ptr(off_a), _ptr(len_a), _ptr(idx_a), topk, int(splits), int(granule),
        _ptr(out), _ptr(lse), _ptr(o_part), _ptr(lse_part), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_mla_decode_split_f64 failed with status {rc}")
    if return_partials:
        return out, lse, o_part, lse_part
    return out, lse


def _u8(a) -> np.ndarray:
    """E4M3 bytes as a contiguous uint8 numpy array (accepts torch uint8 / float8_e4m3fn tensors)."""
    if hasattr(a, "dtype") and str(a.dtype) in ("torch.float8_e4m3fn", "torch.uint8"):
        import torch
        a = a.contiguous().view(torch.uint8).numpy()
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError("E4M3 inputs must be torch.float8_e4m3fn / uint8 tensors or uint8 arrays")
    return a


def e4m3_values(data, *, lib=None) -> np.ndarray:
    """The value of every E4M3 byte of ``data`` (float64, same shape): the
    dequantisation step with scale 1."""
    b = _u8(data)
    out = np.zeros(b.shape, np.float64)
    rc = (lib or _load()).oracle_e4m3_to_f64(_ptr(b), int(b.size), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle_e4m3_to_f64 failed with status {rc}")
    return out


def decode_e4m3(q, kv, *, kv_scale: float, scale: float, d_latent: int = 512, d_rope: int = 64, d_pos=None,
                indices=None, cache_len=None, row_offset=None, row_stride=None, splits: int = 0, granule: int = 1,
                n_threads: int = 0, return_partials: bool = False, lib=None):
    """As :func:`decode` (``splits`` >= 1: as :func:`decode_split`) over an
    E4M3 cache: ``kv`` holds the bytes of rows of ``d_latent + d_rope``
    values, each value ``e4m3(byte) * kv_scale``; q stays bf16."""
    q16 = _u16(q)
    kv8 = _u8(kv)
    D = d_latent + d_rope
    if q16.ndim != 3 or q16.shape[-1] != D:
        raise ValueError("q must be [B, H, d_latent + d_rope]")
    if row_stride is None:
        row_stride = kv8.shape[-1]
    kv_rows = kv8.size // row_stride if kv8.size else 0
    B, H, _ = q16.shape
    sparse = indices is not None
    d_pos_a = _np(d_pos, np.int32)
    idx_a = _np(indices, np.int32)
    len_a = _np(cache_len, np.int32)
    off_a = _np(row_offset, np.int64)
    topk = int(idx_a.shape[-1]) if sparse else 0
    out = np.zeros((B, H, d_latent), np.float64)
    lse = np.zeros((B, H), np.float64)
    o_part = np.zeros((B, H, splits, d_latent), np.float64) if return_partials else None
    lse_part = np.zeros((B, H, splits), np.float64) if return_partials else None
    rc = (lib or _load()).oracle_mla_decode_e4m3_f64(
        _ptr(q16), _ptr(kv8), float(kv_scale), int(kv_rows), int(row_stride), B, H, d_latent, d_rope, float(scale),
        int(sparse), _ptr(d_pos_a), _ptr(off_a), _ptr(len_a), _ptr(idx_a), topk, int(splits), int(granule),
        _ptr(out), _ptr(lse), _ptr(o_part), _ptr(lse_part), int(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_mla_decode_e4m3_f64 failed with status {rc}")
    if return_partials:
        return out, lse, o_part, lse_part
    return out, lse


def project(latent, wv_b, *, lib=None):
    """fp64 projection of a merged latent through wv_b, per head:
    ``y[b,h,v] = sum_r latent[b,h,r] * wv_b[h,v,r]``.

    ``latent`` [B, H, d_latent] (any float dtype, taken exactly as double),
    ``wv_b`` bf16 [H, v_dim, d_latent]; returns y [B, H, v_dim] float64."""
    lat = _np(latent, np.float64)
    w16 = _u16(wv_b)
    if lat.ndim != 3 or w16.ndim != 3 or w16.shape[0] != lat.shape[1] or w16.shape[2] != lat.shape[2]:
        raise ValueError("latent must be [B, H, d] and wv_b [H, v_dim, d]")
    B, H, d = lat.shape
    v_dim = w16.shape[1]
    y = np.zeros((B, H, v_dim), np.float64)
    rc = (lib or _load()).oracle_mla_project_f64(_ptr(lat), _ptr(w16), B, H, d, v_dim, _ptr(y))
    if rc != 0:
        raise ValueError(f"oracle_mla_project_f64 failed with status {rc}")
    return y
