"""mla_decode_forward_static: the forward pass on the library's own static
scratch array (no caller buffer, no allocation), against mla_decode_forward
on the same plan and inputs.  The file name sorts last, so in a full run it
follows every other GPU test; it also passes on its own."""
import ctypes

import pytest
import torch

import _gpu
import decode_attention_mla_gb300 as mla
import workloads


def _fake_args(**kw):
    base = dict(q=0x10000, kv=0x20000, kv_rows=100, row_stride=576, d_pos=0x30000, row_offset=0x60000,
                cache_len=None, indices=None, out=0x40000, lse=0x50000)
    base.update(kw)
    return mla.Args(**base)


def _static(p, a):
    return mla.lib().mla_decode_forward_static(ctypes.byref(p) if p is not None else None,
                                               ctypes.byref(a) if a is not None else None, None)


def test_static_rejects_plans_beyond_the_limit():
    """Checked on the host before any CUDA call: argument errors, then the size limit."""
    big = mla.plan(batch=8, heads=128, max_ctx=131072, scale=0.05, splits=64, num_sms=152)
    assert big.scratch_bytes > mla.STATIC_SCRATCH_BYTES
    assert _static(big, _fake_args()) == mla.ESTATICLIMIT
    assert "8 MiB" in mla.strerror(mla.ESTATICLIMIT)
    assert _static(None, _fake_args()) == mla.EINVAL
    assert _static(big, None) == mla.EINVAL
    assert _static(big, _fake_args(q=None)) == mla.EINVAL
    assert _static(big, _fake_args(q=0x10002)) == mla.EALIGN


def test_static_limit_boundary():
    """256 + align256(B*H*S*2048) + align256(B*H*S*4) bytes: B = 1, H = 16 fits up
    to S = 255; S = 256 is refused on the host, before any CUDA call."""
    fits = mla.plan(batch=1, heads=16, max_ctx=131072, scale=0.05, splits=255, num_sms=152)
    over = mla.plan(batch=1, heads=16, max_ctx=131072, scale=0.05, splits=256, num_sms=152)
    assert fits.scratch_bytes == 256 + 255 * 16 * 2048 + -(-255 * 16 * 4 // 256) * 256
    assert fits.scratch_bytes <= mla.STATIC_SCRATCH_BYTES < over.scratch_bytes
    assert _static(over, _fake_args()) == mla.ESTATICLIMIT
    h128 = [mla.plan(batch=1, heads=128, max_ctx=131072, scale=0.05, splits=s, num_sms=152, variant=1)
            for s in (31, 32)]
    assert h128[0].scratch_bytes <= mla.STATIC_SCRATCH_BYTES < h128[1].scratch_bytes
    assert _static(h128[1], _fake_args()) == mla.ESTATICLIMIT


def test_static_rejects_a_stale_plan_layout():
    """A plan whose split count (and grids) grew while scratch_bytes stayed as
    planned is refused before the size check could let it write past the array."""
    small = mla.plan(batch=1, heads=16, max_ctx=8192, scale=0.05, splits=64, num_sms=152)
    big = mla.plan(batch=1, heads=16, max_ctx=8192, scale=0.05, splits=256, num_sms=152)
    bad = mla.Plan.from_buffer_copy(small)
    bad.splits, bad.grid_x, bad.combine_grid_x = big.splits, big.grid_x, big.combine_grid_x
    assert bad.scratch_bytes <= mla.STATIC_SCRATCH_BYTES < big.scratch_bytes
    assert _static(bad, _fake_args()) == mla.EINVAL


def test_static_limit_matches_the_header():
    import re
    from pathlib import Path
    text = (Path(__file__).resolve().parents[1] / "include" / "mla_decode.h").read_text()
    m = re.search(r"#define MLA_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == mla.STATIC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def _nan_like(out, lse):
    return torch.full_like(out, float("nan")), torch.full_like(lse, float("nan"))


@pytest.mark.gpu
@pytest.mark.parametrize("variant", _gpu.DENSE_VARIANTS)
def test_static_dense_matches_forward_twice(gpu, variant):
    x = workloads.dense(3, 16, 1000, seed=21)
    x.d_pos = torch.tensor([999, 76, 512], dtype=torch.int32)
    out_ref, lse_ref, plan, _ = _gpu.run_dense(x, max_ctx=1000, variant=variant)
    assert plan.scratch_bytes <= mla.STATIC_SCRATCH_BYTES
    q, kv, d_pos, ro = x.q.to(gpu), x.kv.to(gpu), x.d_pos.to(gpu), x.row_offset.to(gpu)
    for call in range(2):
        out, lse = _nan_like(out_ref, lse_ref)
        free0 = torch.cuda.mem_get_info()[0] if call == 1 else None
        mla.forward_static(plan, q, kv, out, lse, d_pos=d_pos, row_offset=ro)
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free0, "free device memory changed during a call made after set-up"
        assert torch.equal(_gpu.bits(out), _gpu.bits(out_ref)), f"call {call}: out differs from mla_decode_forward"
        assert torch.equal(_gpu.bits(lse), _gpu.bits(lse_ref)), f"call {call}: lse differs from mla_decode_forward"
    ro_, rl_ = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro_, rl_, "forward_static dense")


@pytest.mark.gpu
@pytest.mark.parametrize("variant", _gpu.VARIANTS)
def test_static_sparse_matches_forward_twice(gpu, variant):
    x = workloads.sparse(2, 16, [5000, 300], 300, seed=5)
    out_ref, lse_ref, plan, _ = _gpu.run_sparse(x, variant=variant)
    q, kv = x.q.to(gpu), x.kv.to(gpu)
    idx, cl, ro = x.indices.to(gpu), x.cache_len.to(gpu), x.row_offset.to(gpu)
    for call in range(2):
        out, lse = _nan_like(out_ref, lse_ref)
        mla.forward_static(plan, q, kv, out, lse, indices=idx, cache_len=cl, row_offset=ro)
        torch.cuda.synchronize()
        assert torch.equal(_gpu.bits(out), _gpu.bits(out_ref)), f"call {call}: out differs from mla_decode_forward"
        assert torch.equal(_gpu.bits(lse), _gpu.bits(lse_ref)), f"call {call}: lse differs from mla_decode_forward"
    ro_, rl_ = _gpu.oracle_sparse(x)
    _gpu.assert_parity(out, lse, ro_, rl_, "forward_static sparse")


@pytest.mark.gpu
def test_static_near_limit_plan(gpu):
    """dense T=8192 (the timed workload's shape): a plan of several MiB of partials."""
    x = workloads.make("dense_t8192")
    out_ref, lse_ref, plan, _ = _gpu.run_dense(x)
    assert 1 << 20 < plan.scratch_bytes <= mla.STATIC_SCRATCH_BYTES
    out, lse = _nan_like(out_ref, lse_ref)
    for _ in range(2):
        mla.forward_static(plan, x.q.to(gpu), x.kv.to(gpu), out, lse, d_pos=x.d_pos.to(gpu))
    torch.cuda.synchronize()
    assert torch.equal(_gpu.bits(out), _gpu.bits(out_ref))
    assert torch.equal(_gpu.bits(lse), _gpu.bits(lse_ref))


def test_static_status_rejects_bad_arguments():
    """Checked on the host before any CUDA call."""
    L = mla.lib()
    assert L.mla_decode_static_status(None, None) == mla.EINVAL
    assert L.mla_decode_static_status(ctypes.c_void_p(0x10002), None) == mla.EALIGN


@pytest.mark.gpu
def test_static_status_reports_a_timeout_until_reset(gpu):
    """A wait timeout inside mla_decode_forward_static is visible through
    mla_decode_static_status until mla_decode_static_reset clears it; the next
    healthy call still matches mla_decode_forward."""
    x = workloads.dense(1, 16, 4000, seed=62)
    q, kv, dp = x.q.to(gpu), x.kv.to(gpu), x.d_pos.to(gpu)
    out = torch.zeros(1, 16, 512, device=gpu)
    lse = torch.zeros(1, 16, device=gpu)
    st = torch.full((1,), -99, dtype=torch.int32, device=gpu)
    pinned = torch.full((1,), -99, dtype=torch.int32).pin_memory()

    mla.static_reset()
    mla.static_status(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    stalled = mla.plan(batch=1, heads=16, max_ctx=4000, scale=x.scale, variant=1, stall_test=True)
    mla.forward_static(stalled, q, kv, out, lse, d_pos=dp)
    mla.static_status(st)
    mla.lib().mla_decode_static_status(ctypes.c_void_p(pinned.data_ptr()),
                                       mla._stream(torch.cuda.current_stream()))
    torch.cuda.synchronize()
    assert int(st.item()) == mla.EDEVICE
    assert int(pinned.item()) == mla.EDEVICE

    mla.static_reset()
    healthy = mla.plan(batch=1, heads=16, max_ctx=4000, scale=x.scale, variant=1)
    out_ref, lse_ref, _, _ = _gpu.run_dense(x, plan=healthy)
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    mla.forward_static(healthy, q, kv, out, lse, d_pos=dp)
    mla.static_status(st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(_gpu.bits(out), _gpu.bits(out_ref))
    assert torch.equal(_gpu.bits(lse), _gpu.bits(lse_ref))
