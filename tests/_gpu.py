"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare with the fp64 oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import decode_attention_mla_gb300 as mla
import oracle

# Parity bar for floating point: bf16 inputs, fp32 accumulation.
OUT_ATOL = 2e-3       # max |out - out_ref|
LSE_RTOL = 1e-4       # max |lse - lse_ref| / max(|lse_ref|, 1)


def dev():
    return torch.device("cuda:0")


VARIANTS = [1, 2]      # warp-MMA kernel, tcgen05 kernel (dense and sparse)
# dense bf16 decode also runs on the warp-MMA kernel with P . V on tcgen05
DENSE_VARIANTS = [1, 2, 5]
GRANULE = {1: 32, 2: 16, 5: 32}


def run_dense(x, *, splits=0, pdl=False, num_sms=0, heads=None, scratch=None, plan=None, max_ctx=None, variant=0,
              kv_dev=None):
    """Dense decode of workloads.DenseInputs on the GPU; returns (out, lse, plan, scratch)."""
    d = dev()
    B, H, _ = x.q.shape
    if plan is None:
        mc = max_ctx or int(x.d_pos.max()) + 1
        plan = mla.plan(batch=B, heads=H, max_ctx=mc, scale=x.scale, splits=splits, pdl=pdl, num_sms=num_sms,
                        variant=variant)
    if scratch is None:
        scratch = mla.alloc_scratch(plan)
    out = torch.full((B, H, 512), float("nan"), device=d)
    lse = torch.full((B, H), float("nan"), device=d)
    kv = kv_dev if kv_dev is not None else x.kv.to(d)
    mla.forward(plan, x.q.to(d), kv, out, lse, scratch, d_pos=x.d_pos.to(d),
                row_offset=x.row_offset.to(d) if B > 1 else None)
    torch.cuda.synchronize()
    return out, lse, plan, scratch


def run_sparse(x, *, splits=0, pdl=False, scratch=None, plan=None, kv_dev=None, variant=0, num_sms=0):
    d = dev()
    B, H, _ = x.q.shape
    topk = x.indices.shape[1]
    if plan is None:
        plan = mla.plan(batch=B, heads=H, sparse=True, topk=topk, scale=x.scale, splits=splits, pdl=pdl,
                        variant=variant, num_sms=num_sms)
    if scratch is None:
        scratch = mla.alloc_scratch(plan)
    out = torch.full((B, H, 512), float("nan"), device=d)
    lse = torch.full((B, H), float("nan"), device=d)
    kv = kv_dev if kv_dev is not None else x.kv.to(d)
    mla.forward(plan, x.q.to(d), kv, out, lse, scratch, indices=x.indices.to(d), cache_len=x.cache_len.to(d),
                row_offset=x.row_offset.to(d))
    torch.cuda.synchronize()
    return out, lse, plan, scratch


def oracle_dense(x, **kw):
    return oracle.decode(x.q, x.kv, scale=x.scale, d_pos=x.d_pos, row_offset=x.row_offset, **kw)


def oracle_sparse(x, **kw):
    return oracle.decode(x.q, x.kv, scale=x.scale, indices=x.indices, cache_len=x.cache_len,
                         row_offset=x.row_offset, **kw)


def errors(out, lse, ref_o, ref_l):
    o = out.double().cpu().numpy() if isinstance(out, torch.Tensor) else out
    l = lse.double().cpu().numpy() if isinstance(lse, torch.Tensor) else lse
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isfinite(l), fin), "finiteness of lse differs from the oracle"
    err_l = float((np.abs(l[fin] - ref_l[fin]) / np.maximum(np.abs(ref_l[fin]), 1.0)).max()) if fin.any() else 0.0
    assert np.isfinite(o).all(), "non-finite output"
    err_o = float(np.abs(o - ref_o).max())
    return err_o, err_l


def assert_parity(out, lse, ref_o, ref_l, what=""):
    err_o, err_l = errors(out, lse, ref_o, ref_l)
    assert err_o <= OUT_ATOL, f"{what}: max|out - oracle| = {err_o:.3e} > {OUT_ATOL}"
    assert err_l <= LSE_RTOL, f"{what}: max rel lse err = {err_l:.3e} > {LSE_RTOL}"
    return err_o, err_l


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view(torch.int32)
