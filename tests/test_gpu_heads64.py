"""GPU parity of the tcgen05 kernel with 64 heads per CTA (variant 4, dense
decode, H a multiple of 64: scores with the heads on the M side, one softmax
thread per head, P as a bf16 pair along K) against the fp64 oracle; the same
bar as every other kernel."""
import numpy as np
import pytest
import torch

import _gpu
import decode_attention_mla_gb300 as mla
import oracle
import workloads

pytestmark = pytest.mark.gpu

V64 = 4


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()
    torch.cuda.set_device(0)
    yield


@pytest.mark.parametrize("H", [64, 128])
@pytest.mark.parametrize("T", [1, 2, 5, 15, 16, 17, 63, 64, 65, 100, 1000, 2049])
@pytest.mark.parametrize("splits", [0, 3])
def test_dense_heads64(H, T, splits):
    x = workloads.dense(1, H, T, seed=T + H + 7)
    out, lse, plan, scratch = _gpu.run_dense(x, splits=splits, variant=V64)
    assert plan.variant == V64 and plan.head_group == 64
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, f"H={H} T={T} S={plan.splits}")
    assert mla.status_word(plan, scratch) == 0


def test_heads64_partials_match_oracle_split_emulation():
    x = workloads.dense(1, 64, 1000, seed=153)
    out, lse, plan, scratch = _gpu.run_dense(x, splits=5, variant=V64)
    S = plan.splits
    _, _, op, lp = oracle.decode_split(x.q, x.kv, scale=x.scale, splits=S, granule=16, d_pos=x.d_pos,
                                       return_partials=True)
    o_off, l_off = plan.o_part_offset, plan.lse_part_offset
    o_gpu = scratch[o_off:o_off + 64 * S * 512 * 4].view(torch.float32).view(1, 64, S, 512).double().cpu().numpy()
    l_gpu = scratch[l_off:l_off + 64 * S * 4].view(torch.float32).view(1, 64, S).double().cpu().numpy()
    assert np.abs(o_gpu - op).max() <= _gpu.OUT_ATOL
    fin = np.isfinite(lp)
    assert np.array_equal(np.isfinite(l_gpu), fin)
    assert (np.abs(l_gpu[fin] - lp[fin]) / np.maximum(np.abs(lp[fin]), 1)).max() <= _gpu.LSE_RTOL


def test_heads64_batch_ragged_and_many_items():
    """Three requests of different lengths, two head groups each; with 7 and
    200 slices a CTA walks several items (and empty slices are written)."""
    B, H, cap = 3, 128, 1500
    x = workloads.dense(B, H, cap, seed=154)
    x.d_pos = torch.tensor([1499, 17, 640], dtype=torch.int32)
    ro, rl = _gpu.oracle_dense(x)
    for s in (0, 7, 200):
        out, lse, plan, _ = _gpu.run_dense(x, max_ctx=cap, splits=s, variant=V64)
        _gpu.assert_parity(out, lse, ro, rl, f"dense B=3 H=128 ragged S={plan.splits}")


def test_heads64_few_ctas_walk_many_items():
    """A grid of 3 CTAs over 2 head groups x 11 slices: every CTA runs several
    items in a row, so the query tile, tensor memory and the P_lo buffer are
    handed from one item to the next."""
    x = workloads.dense(1, 128, 3000, seed=155)
    out, lse, plan, _ = _gpu.run_dense(x, splits=11, num_sms=3, variant=V64)
    assert plan.grid_x == 3
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, "H=128, 3 CTAs, 22 items")


def test_heads64_bit_identical_across_runs():
    x = workloads.dense(1, 128, 3000, seed=156)
    out0, lse0, plan, scratch = _gpu.run_dense(x, splits=9, variant=V64)
    for _ in range(5):
        out, lse, _, _ = _gpu.run_dense(x, plan=plan, scratch=scratch)
        assert torch.equal(_gpu.bits(out), _gpu.bits(out0)) and torch.equal(_gpu.bits(lse), _gpu.bits(lse0))


def test_heads64_agrees_with_heads32():
    x = workloads.dense(1, 128, 5000, seed=157)
    a = _gpu.run_dense(x, variant=3)
    b = _gpu.run_dense(x, variant=V64)
    assert (a[0] - b[0]).abs().max().item() <= 2 * _gpu.OUT_ATOL
    assert ((a[1] - b[1]).abs() / a[1].abs().clamp(min=1)).max().item() <= 2 * _gpu.LSE_RTOL


def test_heads64_rescale_path():
    """Scores that grow along the context move the reference of every head
    (and rescale O in tensor memory) many times within one slice."""
    T = 4000
    x = workloads.dense(1, 64, T, seed=158)
    ramp = torch.linspace(0.0, 12.0, T).unsqueeze(1)
    kv = x.kv.float()
    kv[:, :512] = kv[:, :512] + ramp * x.q[0, 0, :512].float().sign().unsqueeze(0) * 0.05
    x.kv = kv.to(torch.bfloat16)
    x.q = (x.q.float() * 4.0).to(torch.bfloat16)
    ro, rl = _gpu.oracle_dense(x)
    out, lse, plan, _ = _gpu.run_dense(x, splits=1, variant=V64)
    _gpu.assert_parity(out, lse, ro, rl, "growing scores, 64 heads per CTA")


def test_heads64_single_head_rescales():
    """Only head 37's scores grow (its query row scaled up): one thread moves
    its reference while the other 63 do not, so O is rescaled by a factor
    that is 1 for every other head."""
    T = 3000
    x = workloads.dense(1, 64, T, seed=159)
    ramp = torch.linspace(0.0, 10.0, T).unsqueeze(1)
    kv = x.kv.float()
    kv[:, :512] = kv[:, :512] + ramp * x.q[0, 37, :512].float().sign().unsqueeze(0) * 0.05
    x.kv = kv.to(torch.bfloat16)
    q = x.q.float()
    q[0, 37] *= 5.0
    x.q = q.to(torch.bfloat16)
    ro, rl = _gpu.oracle_dense(x)
    out, lse, _, _ = _gpu.run_dense(x, splits=2, variant=V64)
    _gpu.assert_parity(out, lse, ro, rl, "one head's scores grow")


def test_heads64_uniform_scores_closed_form():
    T = 777
    x = workloads.dense(1, 64, T, seed=160)
    x.q = torch.zeros_like(x.q)
    out, lse, _, _ = _gpu.run_dense(x, splits=6, variant=V64)
    mean = x.kv[:, :512].double().mean(0).numpy()
    assert np.abs(out.double().cpu().numpy() - mean[None, None]).max() <= _gpu.OUT_ATOL
    assert np.abs(lse.double().cpu().numpy() - np.log(T)).max() <= _gpu.LSE_RTOL * np.log(T)


@pytest.mark.parametrize("T", [37, 1000, 4097])
def test_heads64_rows_past_the_context_may_hold_nan(T):
    x = workloads.dense(1, 64, T, seed=195 + T)
    d = _gpu.dev()
    kv = torch.full((T + 300, 576), float("nan"), dtype=torch.bfloat16)
    kv[:T] = x.kv
    out, lse, plan, _ = _gpu.run_dense(x, max_ctx=T + 300, variant=V64, kv_dev=kv.to(d))
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, f"NaN past the context, 64 heads per CTA, T={T}")
