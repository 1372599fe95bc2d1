"""Python binding of ``libmla_decode.so`` (split-KV MLA decode on GB300).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/mla_decode.h``.  Tensors are
PyTorch CUDA tensors; the binding passes their device pointers, sizes and the
current CUDA stream.  If the library is not built, importing works but every
call raises ``RuntimeError`` -- there is no fallback path.

Typical use::

    import decode_attention_mla_gb300 as mla
    plan = mla.plan(batch=1, heads=16, max_ctx=8192, scale=1/24)
    scratch = mla.alloc_scratch(plan)           # before any graph capture
    mla.forward(plan, q, kv, out, lse, scratch, d_pos=d_pos)
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_decode.so")

D_LATENT = 512
D_ROPE = 64
D_ROW = 576
MAX_SPLITS = 256

OK, EINVAL, EUNSUPPORTED, ESCRATCH, EALIGN, ECUDA, EDEVICE, ENOTREADY = 0, -1, -2, -3, -4, -5, -6, -7
ESTATICLIMIT = -8
STATIC_SCRATCH_BYTES = 8 << 20      # scratch of mla_decode_forward_static


class Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int), ("heads", ctypes.c_int), ("d_latent", ctypes.c_int),
                ("d_rope", ctypes.c_int), ("sparse", ctypes.c_int), ("max_ctx", ctypes.c_int),
                ("topk", ctypes.c_int), ("scale", ctypes.c_float), ("num_sms", ctypes.c_int),
                ("splits_override", ctypes.c_int), ("variant", ctypes.c_int), ("pdl", ctypes.c_int),
                ("stall_test", ctypes.c_int), ("kv_fp8", ctypes.c_int)]


class Plan(ctypes.Structure):
    _fields_ = [("shape", Shape), ("magic", ctypes.c_int), ("variant", ctypes.c_int),
                ("splits", ctypes.c_int), ("entries_per_split", ctypes.c_int), ("head_group", ctypes.c_int),
                ("n_head_groups", ctypes.c_int), ("ctas_per_sm", ctypes.c_int), ("num_sms", ctypes.c_int),
                ("grid_x", ctypes.c_int), ("grid_y", ctypes.c_int), ("grid_z", ctypes.c_int),
                ("block", ctypes.c_int), ("smem_bytes", ctypes.c_int), ("combine_grid_x", ctypes.c_int),
                ("combine_grid_y", ctypes.c_int), ("combine_block", ctypes.c_int),
                ("scratch_bytes", ctypes.c_size_t), ("o_part_offset", ctypes.c_size_t),
                ("lse_part_offset", ctypes.c_size_t), ("status_offset", ctypes.c_size_t),
                ("flat_ranges", ctypes.c_int)]

    def as_dict(self) -> dict:
        d = {k: getattr(self, k) for k, _ in self._fields_ if k != "shape"}
        d["shape"] = {k: getattr(self.shape, k) for k, _ in Shape._fields_}
        return d


class Args(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("kv", ctypes.c_void_p), ("kv_rows", ctypes.c_longlong),
                ("row_stride", ctypes.c_longlong), ("d_pos", ctypes.c_void_p), ("row_offset", ctypes.c_void_p),
                ("cache_len", ctypes.c_void_p), ("indices", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("lse", ctypes.c_void_p), ("kv_scale", ctypes.c_float)]


class MLADecodeError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {strerror(status)} (status {status})")


_lock = threading.Lock()
_lib = None

EXPORTED = ("mla_decode_abi_version", "mla_decode_plan", "mla_decode_run", "mla_decode_combine",
            "mla_decode_forward", "mla_decode_append", "mla_decode_advance", "mla_decode_scratch_init",
            "mla_decode_strerror", "mla_decode_forward_static", "mla_decode_project", "mla_decode_forward_step",
            "mla_floor_empty_pair", "mla_floor_read", "mla_floor_gather", "mla_decode_static_status", "mla_decode_static_reset")


def lib():
    """The loaded library; raises RuntimeError if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -m decode_attention_mla_gb300.build` "
                               "(or __graft_entry__.build()); there is no fallback implementation")
        L = ctypes.CDLL(LIB_PATH)
        P, I, SZ, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_longlong
        L.mla_decode_abi_version.restype = I
        L.mla_decode_abi_version.argtypes = []
        L.mla_decode_plan.restype = I
        L.mla_decode_plan.argtypes = [ctypes.POINTER(Shape), ctypes.POINTER(Plan)]
        for name in ("mla_decode_run", "mla_decode_combine", "mla_decode_forward"):
            fn = getattr(L, name)
            fn.restype = I
            fn.argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(Args), P, SZ, P]
        L.mla_decode_forward_step.restype = I
        L.mla_decode_forward_step.argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(Args), P, SZ, P, I, P]
        L.mla_decode_forward_static.restype = I
        L.mla_decode_forward_static.argtypes = [ctypes.POINTER(Plan), ctypes.POINTER(Args), P]
        L.mla_decode_append.restype = I
        L.mla_decode_append.argtypes = [P, LL, LL, P, P, P, I, P]
        L.mla_decode_project.restype = I
        L.mla_decode_project.argtypes = [P, P, I, I, I, P, I, P]
        L.mla_decode_advance.restype = I
        L.mla_decode_advance.argtypes = [P, I, P]
        L.mla_decode_scratch_init.restype = I
        L.mla_decode_scratch_init.argtypes = [P, SZ, P]
        L.mla_decode_strerror.restype = ctypes.c_char_p
        L.mla_decode_strerror.argtypes = [I]
        L.mla_decode_static_status.restype = I
        L.mla_decode_static_status.argtypes = [P, P]
        L.mla_decode_static_reset.restype = I
        L.mla_decode_static_reset.argtypes = [P]
        L.mla_floor_empty_pair.restype = I
        L.mla_floor_empty_pair.argtypes = [I, I, I, I, I, I, I, P]
        L.mla_floor_read.restype = I
        L.mla_floor_read.argtypes = [P, SZ, I, P, P, I, P]
        L.mla_floor_gather.restype = I
        L.mla_floor_gather.argtypes = [P, LL, LL, I, P, LL, I, P, P, I, P]
        _lib = L
        return L


def strerror(status: int) -> str:
    try:
        return lib().mla_decode_strerror(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _check(rc: int, what: str) -> None:
    if rc != OK:
        raise MLADecodeError(rc, what)


def _ptr(t):
    if t is None:
        return None
    if not getattr(t, "is_cuda", False):
        raise ValueError("tensors passed to the MLA decode kernels must be CUDA tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def plan(*, batch: int, heads: int, scale: float, max_ctx: int = 0, topk: int = 0, sparse: bool = False,
         num_sms: int = 0, splits: int = 0, variant: int = 0, pdl: bool = False, stall_test: bool = False,
         kv_fp8: bool = False) -> Plan:
    """``mla_decode_plan``: derive the split count, grid and scratch layout.

    ``num_sms=0`` queries the current CUDA device and prepares the kernels on it
    (do this before capturing a graph).  ``kv_fp8``: the cache holds E4M3 bytes
    (pass the cache's scale as ``kv_scale`` to :func:`make_args` / :func:`forward`)."""
    s = Shape(batch=batch, heads=heads, d_latent=D_LATENT, d_rope=D_ROPE, sparse=int(bool(sparse)),
              max_ctx=max_ctx, topk=topk, scale=scale, num_sms=num_sms, splits_override=splits,
              variant=variant, pdl=int(bool(pdl)), stall_test=int(bool(stall_test)), kv_fp8=int(bool(kv_fp8)))
    p = Plan()
    _check(lib().mla_decode_plan(ctypes.byref(s), ctypes.byref(p)), "mla_decode_plan")
    return p


def alloc_scratch(p: Plan, device=None):
    """Allocate and zero the caller-owned scratch the plan needs (outside capture)."""
    import torch
    n = (int(p.scratch_bytes) + 255) // 256 * 256
    buf = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    scratch_init(buf)
    return buf


def scratch_init(scratch, stream=None) -> None:
    _check(lib().mla_decode_scratch_init(_ptr(scratch), scratch.numel() * scratch.element_size(), _stream(stream)),
           "mla_decode_scratch_init")


def status_word(p: Plan, scratch) -> int:
    """The device status word of a scratch region (0 = healthy); synchronises."""
    import torch
    off = int(p.status_offset)
    return int(scratch[off:off + 4].view(torch.int32).item())


def make_args(q, kv, out, lse, *, d_pos=None, row_offset=None, cache_len=None, indices=None,
              kv_rows: int | None = None, row_stride: int | None = None, kv_scale: float = 1.0) -> Args:
    """Per-call arguments.  ``kv``: bf16 rows, or E4M3 bytes (uint8 / float8_e4m3fn) for plans made
    with ``kv_fp8`` (then ``row_stride`` counts bytes and ``kv_scale`` is the cache's scale)."""
    if row_stride is None:
        row_stride = kv.stride(0) if kv.dim() == 2 else D_ROW
    if kv_rows is None:
        kv_rows = kv.shape[0] if kv.dim() == 2 else kv.numel() // row_stride
    return Args(q=_ptr(q), kv=_ptr(kv), kv_rows=int(kv_rows), row_stride=int(row_stride), d_pos=_ptr(d_pos),
                row_offset=_ptr(row_offset), cache_len=_ptr(cache_len), indices=_ptr(indices), out=_ptr(out),
                lse=_ptr(lse), kv_scale=float(kv_scale))


def _scratch_args(scratch):
    return _ptr(scratch), scratch.numel() * scratch.element_size()


def run(p: Plan, args: Args, scratch, stream=None) -> None:
    """``mla_decode_run``: launch the split partial kernel."""
    sp, sb = _scratch_args(scratch)
    _check(lib().mla_decode_run(ctypes.byref(p), ctypes.byref(args), sp, sb, _stream(stream)), "mla_decode_run")


def combine(p: Plan, args: Args, scratch, stream=None) -> None:
    """``mla_decode_combine``: launch the log-sum-exp merge kernel."""
    sp, sb = _scratch_args(scratch)
    _check(lib().mla_decode_combine(ctypes.byref(p), ctypes.byref(args), sp, sb, _stream(stream)),
           "mla_decode_combine")


def forward_args(p: Plan, args: Args, scratch, stream=None) -> None:
    """``mla_decode_forward``: partial + combine with prebuilt arguments."""
    sp, sb = _scratch_args(scratch)
    _check(lib().mla_decode_forward(ctypes.byref(p), ctypes.byref(args), sp, sb, _stream(stream)),
           "mla_decode_forward")


def forward_step_args(p: Plan, args: Args, scratch, new_rows, *, advance: bool = True, stream=None) -> None:
    """``mla_decode_forward_step``: append ``new_rows`` at d_pos, partial + combine, then (if ``advance``)
    d_pos += 1, in two launches (dense plans)."""
    sp, sb = _scratch_args(scratch)
    _check(lib().mla_decode_forward_step(ctypes.byref(p), ctypes.byref(args), sp, sb, _ptr(new_rows),
                                         int(bool(advance)), _stream(stream)), "mla_decode_forward_step")


def forward_step(p: Plan, q, kv, out, lse, scratch, new_rows, *, d_pos, row_offset=None, advance: bool = True,
                 kv_rows=None, row_stride=None, stream=None) -> None:
    """As :func:`forward`, with the cache append before it and the position advance after it folded in."""
    a = make_args(q, kv, out, lse, d_pos=d_pos, row_offset=row_offset, kv_rows=kv_rows, row_stride=row_stride)
    forward_step_args(p, a, scratch, new_rows, advance=advance, stream=stream)


def forward(p: Plan, q, kv, out, lse, scratch, *, d_pos=None, row_offset=None, cache_len=None, indices=None,
            kv_rows=None, row_stride=None, kv_scale: float = 1.0, stream=None) -> None:
    """Partial + combine: ``out[B,H,512]`` and ``lse[B,H]`` (fp32) from bf16 ``q`` and ``kv``
    (bf16 rows, or E4M3 bytes with ``kv_scale`` for ``kv_fp8`` plans)."""
    a = make_args(q, kv, out, lse, d_pos=d_pos, row_offset=row_offset, cache_len=cache_len, indices=indices,
                  kv_rows=kv_rows, row_stride=row_stride, kv_scale=kv_scale)
    forward_args(p, a, scratch, stream)


def forward_static(p: Plan, q, kv, out, lse, *, d_pos=None, row_offset=None, cache_len=None, indices=None,
                   kv_rows=None, row_stride=None, stream=None) -> None:
    """``mla_decode_forward_static``: as :func:`forward`, with the library's own 8 MiB static scratch."""
    a = make_args(q, kv, out, lse, d_pos=d_pos, row_offset=row_offset, cache_len=cache_len, indices=indices,
                  kv_rows=kv_rows, row_stride=row_stride)
    _check(lib().mla_decode_forward_static(ctypes.byref(p), ctypes.byref(a), _stream(stream)),
           "mla_decode_forward_static")


def static_status(dst, stream=None) -> None:
    """``mla_decode_static_status``: stream-ordered copy of the static scratch's status word into
    ``dst`` (a CUDA int32 tensor of at least one element)."""
    _check(lib().mla_decode_static_status(_ptr(dst), _stream(stream)), "mla_decode_static_status")


def static_reset(stream=None) -> None:
    """``mla_decode_static_reset``: clear the static scratch's status word."""
    _check(lib().mla_decode_static_reset(_stream(stream)), "mla_decode_static_reset")


def append(kv, new_rows, d_pos, *, row_offset=None, kv_rows=None, row_stride=None, stream=None) -> None:
    """``mla_decode_append``: write new_rows[b] at cache row base_b + d_pos[b] (on the device)."""
    if row_stride is None:
        row_stride = kv.stride(0)
    if kv_rows is None:
        kv_rows = kv.shape[0]
    batch = int(d_pos.numel())
    _check(lib().mla_decode_append(_ptr(kv), int(kv_rows), int(row_stride), _ptr(new_rows), _ptr(d_pos),
                                   _ptr(row_offset), batch, _stream(stream)), "mla_decode_append")


def project(latent, wv_b, y, *, pdl: bool = False, stream=None) -> None:
    """``mla_decode_project``: y[B,H,v] = latent[B,H,512] . wv_b[H,v,512]^T per head (fp32 out)."""
    B, H, r = latent.shape
    if r != D_LATENT or tuple(wv_b.shape[:1]) != (H,) or wv_b.shape[-1] != D_LATENT:
        raise ValueError("latent must be [B, H, 512] and wv_b [H, v_dim, 512]")
    v_dim = int(wv_b.shape[1])
    _check(lib().mla_decode_project(_ptr(latent), _ptr(wv_b), int(B), int(H), v_dim, _ptr(y), int(bool(pdl)),
                                    _stream(stream)), "mla_decode_project")


def advance(d_pos, stream=None) -> None:
    """``mla_decode_advance``: d_pos += 1 on the device."""
    _check(lib().mla_decode_advance(_ptr(d_pos), int(d_pos.numel()), _stream(stream)), "mla_decode_advance")


def floor_empty_pair(a, b, *, pdl: bool = True, stream=None) -> None:
    """``mla_floor_empty_pair``: two empty kernels with launch shapes a and b,
    each a (grid, block, dynamic shared bytes) triple."""
    _check(lib().mla_floor_empty_pair(int(a[0]), int(a[1]), int(a[2]), int(b[0]), int(b[1]), int(b[2]),
                                      int(bool(pdl)), _stream(stream)), "mla_floor_empty_pair")


def floor_read(src, nbytes: int, ctas: int, sink, status, *, pdl: bool = True, stream=None) -> None:
    """``mla_floor_read``: one kernel of ``ctas`` CTAs reading ``nbytes`` of ``src`` with bulk copies;
    ``sink``: uint32/int32 [ctas], ``status``: int32 [1] (zeroed by the caller)."""
    _check(lib().mla_floor_read(_ptr(src), int(nbytes), int(ctas), _ptr(sink), _ptr(status), int(bool(pdl)),
                                _stream(stream)), "mla_floor_read")


def floor_gather(kv, rows, ctas: int, sink, status, *, row_bytes: int | None = None, pdl: bool = True,
                 stream=None) -> None:
    """``mla_floor_gather``: one kernel of ``ctas`` CTAs gathering the cache rows listed in ``rows``
    (int64) with one bulk copy per row; ``kv``: [kv_rows, row_stride] (bf16 or bytes)."""
    stride = kv.stride(0) * kv.element_size()
    rb = int(row_bytes) if row_bytes is not None else kv.shape[1] * kv.element_size()
    _check(lib().mla_floor_gather(_ptr(kv), int(kv.shape[0]), int(stride), rb, _ptr(rows), int(rows.numel()),
                                  int(ctas), _ptr(sink), _ptr(status), int(bool(pdl)), _stream(stream)),
           "mla_floor_gather")


def abi_version() -> int:
    return int(lib().mla_decode_abi_version())
