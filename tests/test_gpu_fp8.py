"""GPU parity of the E4M3 (FP8) cache path (dense decode, warp-MMA kernel:
E4M3 rows staged by TMA and widened to f16 in shared memory, f16 products,
the cache's scale folded into the scores and the output) against the fp64
oracle over the same bytes and scale; the same bar as the bf16 cache.  Every
test runs on both forms of the kernel: P . V on the warps (variant 1) and on
tcgen05 (variant 5)."""
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


_VARIANT = [1]          # the kernel form under test (set per test by the fixture below)


@pytest.fixture(params=[1, 5], autouse=True)
def _variant(request):
    _VARIANT[0] = request.param
    yield request.param


def _run(x, kv8, kv_scale, *, splits=0, max_ctx=None, plan=None, scratch=None, num_sms=0, kv_dev=None):
    d = _gpu.dev()
    B, H, _ = x.q.shape
    if plan is None:
        mc = max_ctx or int(x.d_pos.max()) + 1
        plan = mla.plan(batch=B, heads=H, max_ctx=mc, scale=x.scale, splits=splits, kv_fp8=True, num_sms=num_sms,
                        variant=_VARIANT[0])
    if scratch is None:
        scratch = mla.alloc_scratch(plan)
    out = torch.full((B, H, 512), float("nan"), device=d)
    lse = torch.full((B, H), float("nan"), device=d)
    kv = kv_dev if kv_dev is not None else kv8.to(d)
    mla.forward(plan, x.q.to(d), kv, out, lse, scratch, d_pos=x.d_pos.to(d),
                row_offset=x.row_offset.to(d) if B > 1 else None, kv_scale=kv_scale)
    torch.cuda.synchronize()
    return out, lse, plan, scratch


def _oracle(x, kv8, kv_scale, **kw):
    return oracle.decode_e4m3(x.q, kv8, kv_scale=kv_scale, scale=x.scale, d_pos=x.d_pos,
                              row_offset=x.row_offset if x.q.shape[0] > 1 else None, **kw)


@pytest.mark.parametrize("T", [1, 5, 31, 32, 33, 100, 1000, 8192])
@pytest.mark.parametrize("splits", [0, 3])
def test_fp8_dense_matches_oracle(T, splits):
    x = workloads.dense(1, 16, T, seed=700 + T)
    kv8, kv_scale = workloads.to_e4m3(x.kv)
    out, lse, plan, scratch = _run(x, kv8, kv_scale, splits=splits)
    assert plan.variant == _VARIANT[0]
    ro, rl = _oracle(x, kv8, kv_scale)
    _gpu.assert_parity(out, lse, ro, rl, f"E4M3 T={T} S={plan.splits}")
    assert mla.status_word(plan, scratch) == 0


@pytest.mark.parametrize("H", [32, 64, 128])
def test_fp8_more_heads(H):
    x = workloads.dense(1, H, 3000, seed=710 + H)
    kv8, kv_scale = workloads.to_e4m3(x.kv)
    out, lse, plan, _ = _run(x, kv8, kv_scale)
    ro, rl = _oracle(x, kv8, kv_scale)
    _gpu.assert_parity(out, lse, ro, rl, f"E4M3 H={H}")


@pytest.mark.parametrize("T", [32768, 131072])
def test_fp8_context_sweep_workloads(T):
    """The E4M3 rows of the bench at full size (the planner's S, PDL on)."""
    x = workloads.dense(1, 16, T, seed=T + 13)
    kv8, kv_scale = workloads.to_e4m3(x.kv)
    d = _gpu.dev()
    plan = mla.plan(batch=1, heads=16, max_ctx=T, scale=x.scale, kv_fp8=True, pdl=True, variant=_VARIANT[0])
    scratch = mla.alloc_scratch(plan)
    out = torch.full((1, 16, 512), float("nan"), device=d)
    lse = torch.full((1, 16), float("nan"), device=d)
    mla.forward(plan, x.q.to(d), kv8.to(d), out, lse, scratch, d_pos=x.d_pos.to(d), kv_scale=kv_scale)
    torch.cuda.synchronize()
    ro, rl = _oracle(x, kv8, kv_scale)
    _gpu.assert_parity(out, lse, ro, rl, f"E4M3 T={T} S={plan.splits}")
    assert mla.status_word(plan, scratch) == 0


def test_fp8_partials_match_oracle_split_emulation():
    x = workloads.dense(1, 16, 2000, seed=720)
    kv8, kv_scale = workloads.to_e4m3(x.kv)
    out, lse, plan, scratch = _run(x, kv8, kv_scale, splits=5)
    S = plan.splits
    _, _, op, lp = _oracle(x, kv8, kv_scale, splits=S, granule=32, return_partials=True)
    o_off, l_off = plan.o_part_offset, plan.lse_part_offset
    o_gpu = scratch[o_off:o_off + 16 * S * 512 * 4].view(torch.float32).view(1, 16, S, 512).double().cpu().numpy()
    l_gpu = scratch[l_off:l_off + 16 * S * 4].view(torch.float32).view(1, 16, S).double().cpu().numpy()
    assert np.abs(o_gpu - op).max() <= _gpu.OUT_ATOL
    fin = np.isfinite(lp)
    assert np.array_equal(np.isfinite(l_gpu), fin)
    assert (np.abs(l_gpu[fin] - lp[fin]) / np.maximum(np.abs(lp[fin]), 1)).max() <= _gpu.LSE_RTOL


def test_fp8_batch_ragged_and_few_ctas():
    B, H, cap = 3, 16, 2500
    x = workloads.dense(B, H, cap, seed=730)
    x.d_pos = torch.tensor([2499, 40, 1111], dtype=torch.int32)
    kv8, kv_scale = workloads.to_e4m3(x.kv)
    ro, rl = _oracle(x, kv8, kv_scale)
    for s, sms in ((0, 0), (7, 0), (9, 3)):
        out, lse, plan, _ = _run(x, kv8, kv_scale, splits=s, max_ctx=cap, num_sms=sms)
        _gpu.assert_parity(out, lse, ro, rl, f"E4M3 B=3 ragged S={plan.splits} grid={plan.grid_x}")


@pytest.mark.parametrize("factor", [1.0, 0.37, 2.0 ** -3, 3.0])
def test_fp8_scale_values(factor):
    """The same bytes under other scales (multiples of the quantiser's, so the
    values stay near the N(0, 1) magnitudes the absolute bar is stated for)."""
    x = workloads.dense(1, 16, 700, seed=740)
    kv8, s0 = workloads.to_e4m3(x.kv)
    kv_scale = s0 * factor
    out, lse, _, _ = _run(x, kv8, kv_scale)
    ro, rl = _oracle(x, kv8, kv_scale)
    _gpu.assert_parity(out, lse, ro, rl, f"E4M3 kv_scale={kv_scale}")


def test_fp8_uniform_scores_closed_form():
    T = 999
    x = workloads.dense(1, 16, T, seed=750)
    x.q = torch.zeros_like(x.q)
    kv8, kv_scale = workloads.to_e4m3(x.kv)
    out, lse, _, _ = _run(x, kv8, kv_scale, splits=4)
    mean = (oracle.e4m3_values(kv8)[:, :512] * kv_scale).mean(0)
    assert np.abs(out.double().cpu().numpy() - mean[None, None]).max() <= _gpu.OUT_ATOL
    assert np.abs(lse.double().cpu().numpy() - np.log(T)).max() <= _gpu.LSE_RTOL * np.log(T)


def test_fp8_bit_identical_across_runs():
    x = workloads.dense(1, 16, 5000, seed=760)
    kv8, kv_scale = workloads.to_e4m3(x.kv)
    out0, lse0, plan, scratch = _run(x, kv8, kv_scale, splits=11)
    for _ in range(4):
        out, lse, _, _ = _run(x, kv8, kv_scale, plan=plan, scratch=scratch)
        assert torch.equal(_gpu.bits(out), _gpu.bits(out0)) and torch.equal(_gpu.bits(lse), _gpu.bits(lse0))


@pytest.mark.parametrize("T", [37, 1000])
def test_fp8_rows_past_the_context_may_hold_nan(T):
    """E4M3 NaN bytes (0x7F) fill the cache past the context: never attended."""
    x = workloads.dense(1, 16, T, seed=770 + T)
    kv8, kv_scale = workloads.to_e4m3(x.kv)
    full = torch.full((T + 300, 576), 0x7F, dtype=torch.uint8)
    full[:T] = kv8
    out, lse, _, _ = _run(x, kv8, kv_scale, max_ctx=T + 300, kv_dev=full.to(_gpu.dev()))
    ro, rl = _oracle(x, kv8, kv_scale)
    _gpu.assert_parity(out, lse, ro, rl, f"E4M3 NaN past the context, T={T}")


def test_fp8_padded_row_stride():
    """Rows 640 bytes apart (a padded cache): the same result as packed rows."""
    T = 1500
    x = workloads.dense(1, 16, T, seed=780)
    kv8, kv_scale = workloads.to_e4m3(x.kv)
    padded = torch.zeros((T, 640), dtype=torch.uint8)
    padded[:, :576] = kv8
    d = _gpu.dev()
    plan = mla.plan(batch=1, heads=16, max_ctx=T, scale=x.scale, kv_fp8=True, variant=_VARIANT[0])
    scratch = mla.alloc_scratch(plan)
    out = torch.empty(1, 16, 512, device=d)
    lse = torch.empty(1, 16, device=d)
    kvp = padded.to(d)
    mla.forward(plan, x.q.to(d), kvp, out, lse, scratch, d_pos=x.d_pos.to(d), kv_rows=T, row_stride=640,
                kv_scale=kv_scale)
    torch.cuda.synchronize()
    ro, rl = _oracle(x, kv8, kv_scale)
    _gpu.assert_parity(out, lse, ro, rl, "E4M3 padded rows")
