"""GPU parity of the wv_b projection of the merged latent ("Graph-resident
decode", Lecture 08, s.6) against the fp64 oracle, alone and after a full
decode, inside a captured graph, and bit-identical across runs."""
import numpy as np
import pytest
import torch

import _gpu
import decode_attention_mla_gb300 as mla
import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()
    torch.cuda.set_device(0)
    yield


def _inputs(B, H, V, seed):
    g = torch.Generator().manual_seed(seed)
    lat = torch.randn(B, H, 512, generator=g)
    w = (torch.randn(H, V, 512, generator=g) / 512 ** 0.5).to(torch.bfloat16)
    return lat, w


def _run(lat, w, pdl=False):
    d = _gpu.dev()
    B, H, _ = lat.shape
    y = torch.full((B, H, w.shape[1]), float("nan"), device=d)
    mla.project(lat.to(d), w.to(d), y, pdl=pdl)
    torch.cuda.synchronize()
    return y


def _bound(lat, w, lat_err=0.0):
    """|y_gpu - y_ref| bound per output: fp32 accumulation over 512 products
    (relative 2^-18 of the sum of magnitudes, generous) plus the propagated
    error of the latent (lat_err per entry)."""
    a = np.abs(lat.double().numpy())
    wa = np.abs(w.double().numpy())
    mag = np.einsum("bhr,hvr->bhv", a, wa)
    return mag * 2.0 ** -18 + lat_err * wa.sum(axis=2)[None] + 1e-7


@pytest.mark.parametrize("B,H,V", [(1, 16, 128), (3, 16, 16), (9, 32, 512), (1, 128, 128), (17, 4, 64)])
def test_project_matches_oracle(B, H, V):
    lat, w = _inputs(B, H, V, seed=B * 1000 + H + V)
    y = _run(lat, w).double().cpu().numpy()
    ref = oracle.project(lat.double().numpy(), w)
    assert np.isfinite(y).all()
    assert (np.abs(y - ref) <= _bound(lat, w)).all(), float(np.abs(y - ref).max())


def test_project_bit_identical_across_runs():
    lat, w = _inputs(5, 16, 128, seed=7)
    y0 = _run(lat, w)
    for _ in range(4):
        assert torch.equal(_run(lat, w), y0)


def test_decode_then_project_matches_oracle():
    """out of the full decode (within 2e-3 of the oracle per entry), projected:
    within the propagated bound of the oracle's projection of its own out."""
    x = workloads.dense(1, 16, 3000, seed=71)
    out, lse, plan, _ = _gpu.run_dense(x)
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, "decode before projection")
    _, w = _inputs(1, 16, 128, seed=72)
    d = _gpu.dev()
    y = torch.empty(1, 16, 128, device=d)
    mla.project(out, w.to(d), y)
    torch.cuda.synchronize()
    ref = oracle.project(ro, w)
    bound = _bound(torch.as_tensor(ro), w, lat_err=_gpu.OUT_ATOL)
    assert (np.abs(y.double().cpu().numpy() - ref) <= bound).all()


def test_project_in_a_graph_after_the_combine():
    """partial + combine + projection (PDL) captured once and replayed: the
    projection of every replay equals the eager one, bit for bit."""
    x = workloads.dense(1, 16, 2000, seed=73)
    d = _gpu.dev()
    plan = mla.plan(batch=1, heads=16, max_ctx=2000, scale=x.scale, pdl=True)
    scratch = mla.alloc_scratch(plan)
    q, kv, dp = x.q.to(d), x.kv.to(d), x.d_pos.to(d)
    out = torch.empty(1, 16, 512, device=d)
    lse = torch.empty(1, 16, device=d)
    _, w = _inputs(1, 16, 128, seed=74)
    wd = w.to(d)
    y = torch.empty(1, 16, 128, device=d)
    mla.forward(plan, q, kv, out, lse, scratch, d_pos=dp)
    mla.project(out, wd, y, pdl=True)
    torch.cuda.synchronize()
    y_eager = y.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mla.forward(plan, q, kv, out, lse, scratch, d_pos=dp)
        mla.project(out, wd, y, pdl=True)
    for _ in range(3):
        y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, y_eager)
