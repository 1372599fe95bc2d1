"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs.  Bar: max|out - oracle| <= 2e-3 and relative LSE error
<= 1e-4; byte identity across runs at a fixed split count."""
import math

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


# ---- dense, small shapes: several stages, ragged tails, many split counts ----
@pytest.mark.parametrize("variant", _gpu.DENSE_VARIANTS)
@pytest.mark.parametrize("T", [1, 5, 31, 32, 33, 79, 80, 81, 100, 160, 256, 1000, 2049])
@pytest.mark.parametrize("splits", [0, 1, 3, 8])
def test_dense_small(T, splits, variant):
    x = workloads.dense(1, 16, T, seed=T)
    out, lse, plan, scratch = _gpu.run_dense(x, splits=splits, variant=variant)
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, f"dense T={T} S={plan.splits}")
    assert mla.status_word(plan, scratch) == 0


def test_dense_t256_workload():
    x = workloads.make("dense_t256")
    out, lse, plan, _ = _gpu.run_dense(x)
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, "dense_t256")


@pytest.mark.parametrize("variant", _gpu.DENSE_VARIANTS)
def test_dense_t8192_split_sweep(variant):
    x = workloads.make("dense_t8192")
    ro, rl = _gpu.oracle_dense(x)
    results = {}
    for s in (1, 2, 4, 8, 16, 32, 64, 128, 0):
        out, lse, plan, _ = _gpu.run_dense(x, splits=s, variant=variant)
        _gpu.assert_parity(out, lse, ro, rl, f"dense_t8192 S={plan.splits}")
        results[plan.splits] = (out.double().cpu().numpy(), lse.double().cpu().numpy())
    keys = sorted(results)
    for a in keys:
        for b in keys:
            assert np.abs(results[a][0] - results[b][0]).max() <= 2 * _gpu.OUT_ATOL
            assert (np.abs(results[a][1] - results[b][1]) / np.maximum(np.abs(rl), 1)).max() <= 2 * _gpu.LSE_RTOL


@pytest.mark.parametrize("splits", [17, 20, 21, 40, 41, 80, 81, 160, 161, 256])
def test_combine_unit_and_batch_shapes(splits):
    """Split counts around every change of the combine's unit (1, 2, 4, 8
    warps) and of its load batch (one batch of up to 20 slices per warp, or
    two of 16), on the timed workload's shape, against the oracle."""
    x = workloads.make("dense_t8192")
    ro, rl = _gpu.oracle_dense(x)
    out, lse, plan, _ = _gpu.run_dense(x, splits=splits, variant=1)
    assert plan.splits == splits
    _gpu.assert_parity(out, lse, ro, rl, f"dense_t8192 S={splits}")


@pytest.mark.parametrize("T", [16384, 32768, 65536, 131072])
def test_dense_context_sweep_workloads(T):
    """The H = 16 context sweep at full size, in the launch configuration the
    bench times (the planner's S and kernel, PDL on): every output against the
    fp64 oracle.  At T = 32768 and 65536 (S = 147, 7 slots per CTA) the two
    MMA groups hold 4 and 3 slots of an item."""
    x = workloads.dense(1, 16, T, seed=T + 11)
    out, lse, plan, scratch = _gpu.run_dense(x, pdl=True)
    assert plan.variant == 1
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, f"dense H=16 T={T} S={plan.splits}")
    assert mla.status_word(plan, scratch) == 0


@pytest.mark.parametrize("variant", _gpu.DENSE_VARIANTS)
def test_dense_partials_match_oracle_split_emulation(variant):
    """The partial kernel's scratch (o_s, lse_s) against the oracle's fp64 emulation
    of the same slices (cut at the kernel's granule, as the plan cuts them)."""
    x = workloads.dense(1, 16, 1000, seed=3)
    out, lse, plan, scratch = _gpu.run_dense(x, splits=5, variant=variant)
    S = plan.splits
    _, _, op, lp = oracle.decode_split(x.q, x.kv, scale=x.scale, splits=S, granule=_gpu.GRANULE[variant],
                                       d_pos=x.d_pos, return_partials=True)
    o_off, l_off = plan.o_part_offset, plan.lse_part_offset
    o_gpu = scratch[o_off:o_off + 16 * S * 512 * 4].view(torch.float32).view(1, 16, S, 512).double().cpu().numpy()
    l_gpu = scratch[l_off:l_off + 16 * S * 4].view(torch.float32).view(1, 16, S).double().cpu().numpy()
    assert np.abs(o_gpu - op).max() <= _gpu.OUT_ATOL
    fin = np.isfinite(lp)
    assert np.array_equal(np.isfinite(l_gpu), fin)
    assert (np.abs(l_gpu[fin] - lp[fin]) / np.maximum(np.abs(lp[fin]), 1)).max() <= _gpu.LSE_RTOL


@pytest.mark.parametrize("variant", _gpu.DENSE_VARIANTS)
def test_dense_batch_ragged(variant):
    B, H, cap = 3, 16, 1500
    x = workloads.dense(B, H, cap, seed=21)
    x.d_pos = torch.tensor([1499, 17, 640], dtype=torch.int32)
    out, lse, plan, _ = _gpu.run_dense(x, max_ctx=cap, variant=variant)
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, "dense batch 3 ragged")


@pytest.mark.parametrize("variant", _gpu.DENSE_VARIANTS)
@pytest.mark.parametrize("H", [32, 64, 128])
def test_dense_more_heads(H, variant):
    x = workloads.dense(1, H, 2000, seed=H)
    out, lse, plan, _ = _gpu.run_dense(x, variant=variant)
    assert plan.n_head_groups == H // 16
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, f"dense H={H}")


@pytest.mark.parametrize("variant", _gpu.DENSE_VARIANTS)
def test_dense_row_stride_and_capacity(variant):
    """Rows padded to a 640-element stride; d_pos beyond the cache is clamped."""
    T = 700
    x = workloads.dense(1, 16, T, seed=5)
    d = _gpu.dev()
    padded = torch.zeros(T, 640, dtype=torch.bfloat16)
    padded[:, :576] = x.kv
    plan = mla.plan(batch=1, heads=16, max_ctx=T, scale=x.scale, variant=variant)
    scratch = mla.alloc_scratch(plan)
    out = torch.empty(1, 16, 512, device=d)
    lse = torch.empty(1, 16, device=d)
    mla.forward(plan, x.q.to(d), padded.to(d), out, lse, scratch, d_pos=x.d_pos.to(d))
    torch.cuda.synchronize()
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, "row stride 640")
    # d_pos past the last row: only the rows that exist are attended
    big = torch.tensor([T + 50], dtype=torch.int32)
    mla.forward(plan, x.q.to(d), x.kv.to(d), out, lse, scratch, d_pos=big.to(d))
    torch.cuda.synchronize()
    _gpu.assert_parity(out, lse, ro, rl, "d_pos clamped to the cache")


@pytest.mark.parametrize("variant", _gpu.DENSE_VARIANTS)
def test_uniform_scores_closed_form(variant):
    """q = 0: every score is 0, so out = mean of the attended latent rows and lse = ln n."""
    T = 777
    x = workloads.dense(1, 16, T, seed=9)
    x.q = torch.zeros_like(x.q)
    out, lse, _, _ = _gpu.run_dense(x, splits=6, variant=variant)
    mean = x.kv[:, :512].double().mean(0).numpy()
    assert np.abs(out.double().cpu().numpy() - mean[None, None]).max() <= _gpu.OUT_ATOL
    assert np.abs(lse.double().cpu().numpy() - math.log(T)).max() <= _gpu.LSE_RTOL * math.log(T)


# ---- sparse ------------------------------------------------------------------
@pytest.mark.parametrize("variant", _gpu.VARIANTS)
def test_sparse_k2048_workload(variant):
    x = workloads.make("sparse_k2048")
    ro, rl = _gpu.oracle_sparse(x)
    for s in (0, 1, 7, 64):
        out, lse, plan, _ = _gpu.run_sparse(x, splits=s, variant=variant)
        _gpu.assert_parity(out, lse, ro, rl, f"sparse_k2048 S={plan.splits}")


@pytest.mark.parametrize("variant", _gpu.VARIANTS)
@pytest.mark.parametrize("topk", [1, 17, 64, 80, 81, 300])
def test_sparse_small(topk, variant):
    x = workloads.sparse(2, 16, [5000, 300], topk, seed=topk)
    out, lse, plan, _ = _gpu.run_sparse(x, variant=variant)
    ro, rl = _gpu.oracle_sparse(x)
    _gpu.assert_parity(out, lse, ro, rl, f"sparse k={topk}")


@pytest.mark.parametrize("variant", _gpu.VARIANTS)
def test_sparse_masking_out_of_range_ids(variant):
    x = workloads.sparse(2, 16, [4000, 900], 256, seed=31)
    idx = x.indices.clone()
    idx[0, 3] = -1
    idx[0, 100] = 4000          # == cache_len: masked
    idx[1, 0] = 900
    idx[1, 7] = 2 ** 31 - 1
    idx[1, 255] = -(2 ** 31)
    x.indices = idx
    out, lse, plan, _ = _gpu.run_sparse(x, splits=3, variant=variant)
    ro, rl = _gpu.oracle_sparse(x)
    _gpu.assert_parity(out, lse, ro, rl, "sparse masked ids")


@pytest.mark.parametrize("variant", _gpu.VARIANTS)
def test_sparse_all_masked_is_empty(variant):
    x = workloads.sparse(1, 16, 100, 40, seed=32)
    x.indices = torch.full_like(x.indices, -7)
    out, lse, _, _ = _gpu.run_sparse(x, splits=2, variant=variant)
    assert torch.isneginf(lse).all()
    assert (out == 0).all()


def test_sparse_equals_dense_on_permutation():
    T = 3000
    xd = workloads.dense(1, 16, T, seed=33)
    perm = workloads.unique_indices(T, T, seed=33, stream=9).view(1, -1)
    xs = workloads.SparseInputs(q=xd.q, kv=xd.kv, indices=perm, cache_len=torch.tensor([T], dtype=torch.int32),
                                row_offset=torch.tensor([0], dtype=torch.int64))
    od, ld, _, _ = _gpu.run_dense(xd)
    os_, ls, _, _ = _gpu.run_sparse(xs)
    assert (od - os_).abs().max().item() <= 2 * _gpu.OUT_ATOL
    assert ((ld - ls).abs() / ld.abs().clamp(min=1)).max().item() <= 2 * _gpu.LSE_RTOL


def test_sparse_b64_workload_all_requests():
    """Full-size ragged batch (~5 GB cache, 64 requests of top-2048 lists) on the
    GPU, every request of the batch against the oracle, element by element, for
    each kernel variant."""
    x = workloads.make("sparse_b64")
    d = _gpu.dev()
    kv_dev = x.kv.to(d)
    ro, rl = _gpu.oracle_sparse(x)
    assert ro.shape == (64, 16, 512)
    for variant in _gpu.VARIANTS:
        out, lse, plan, scratch = _gpu.run_sparse(x, kv_dev=kv_dev, variant=variant)
        assert mla.status_word(plan, scratch) == 0
        _gpu.assert_parity(out, lse, ro, rl, f"sparse_b64 all 64 requests, variant {variant}")
    del kv_dev


# ---- determinism, A/A, PDL, guards -------------------------------------------
@pytest.mark.parametrize("variant", _gpu.DENSE_VARIANTS)
def test_fixed_split_is_bit_identical_across_runs(variant):
    x = workloads.dense(1, 16, 8192, seed=41)
    ref = None
    for _ in range(10):
        out, lse, plan, _ = _gpu.run_dense(x, splits=32, variant=variant)
        cur = (_gpu.bits(out).clone(), _gpu.bits(lse).clone())
        if ref is None:
            ref = cur
        else:
            assert torch.equal(cur[0], ref[0]) and torch.equal(cur[1], ref[1])


@pytest.mark.parametrize("variant", _gpu.VARIANTS)
def test_aa_control_sparse(variant):
    """Two independent runs of the same arm (fresh scratch each) must match byte for byte."""
    x = workloads.sparse(4, 16, [9000, 7000, 12000, 4096], 512, seed=42)
    a = _gpu.run_sparse(x, splits=4, variant=variant)
    b = _gpu.run_sparse(x, splits=4, variant=variant)
    assert torch.equal(_gpu.bits(a[0]), _gpu.bits(b[0])) and torch.equal(_gpu.bits(a[1]), _gpu.bits(b[1]))


@pytest.mark.parametrize("variant", _gpu.DENSE_VARIANTS)
def test_pdl_on_off_bit_identical(variant):
    x = workloads.dense(1, 16, 4096, seed=43)
    a = _gpu.run_dense(x, splits=16, pdl=False, variant=variant)
    b = _gpu.run_dense(x, splits=16, pdl=True, variant=variant)
    assert torch.equal(_gpu.bits(a[0]), _gpu.bits(b[0])) and torch.equal(_gpu.bits(a[1]), _gpu.bits(b[1]))


def test_guard_regions_untouched():
    """out, lse and scratch live inside larger buffers; the bytes around them must not change."""
    x = workloads.dense(1, 16, 2000, seed=44)
    d = _gpu.dev()
    plan = mla.plan(batch=1, heads=16, max_ctx=2000, scale=x.scale, splits=9)
    G = 1024
    sbuf = torch.full((plan.scratch_bytes + 2 * G * 4,), 0xA5, dtype=torch.uint8, device=d)
    scratch = sbuf[G * 4:G * 4 + plan.scratch_bytes]
    mla.scratch_init(scratch)
    obuf = torch.full((16 * 512 + 2 * G,), 7.0, device=d)
    lbuf = torch.full((16 + 2 * G,), 7.0, device=d)
    out = obuf[G:G + 16 * 512].view(1, 16, 512)
    lse = lbuf[G:G + 16].view(1, 16)
    mla.forward(plan, x.q.to(d), x.kv.to(d), out, lse, scratch, d_pos=x.d_pos.to(d))
    torch.cuda.synchronize()
    assert (sbuf[:G * 4] == 0xA5).all() and (sbuf[G * 4 + plan.scratch_bytes:] == 0xA5).all()
    assert (obuf[:G] == 7.0).all() and (obuf[G + 16 * 512:] == 7.0).all()
    assert (lbuf[:G] == 7.0).all() and (lbuf[G + 16:] == 7.0).all()
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, "guarded buffers")


def test_plan_on_device_matches_occupancy_target():
    p = mla.plan(batch=1, heads=16, max_ctx=131072, scale=workloads.SCALE)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert p.num_sms == sms
    assert p.ctas_per_sm == 1 and p.grid_x == min(p.splits, sms)


@pytest.mark.parametrize("variant", _gpu.VARIANTS)
def test_persistent_grid_walks_many_items(variant):
    """Forced split counts far above the SM count: each CTA walks several items."""
    x = workloads.dense(2, 32, 3000, seed=45)
    ro, rl = _gpu.oracle_dense(x)
    for s in (150, 256):
        out, lse, plan, _ = _gpu.run_dense(x, splits=s, variant=variant)
        assert plan.grid_x < 2 * 2 * s
        _gpu.assert_parity(out, lse, ro, rl, f"dense B=2 H=32 S={s}")


def test_variants_agree():
    """The warp-MMA and tcgen05 kernels on the same inputs: both within the bar of the
    oracle, and within twice the bar of each other."""
    x = workloads.dense(1, 16, 5000, seed=46)
    a = _gpu.run_dense(x, variant=1)
    b = _gpu.run_dense(x, variant=2)
    assert (a[0] - b[0]).abs().max().item() <= 2 * _gpu.OUT_ATOL
    assert ((a[1] - b[1]).abs() / a[1].abs().clamp(min=1)).max().item() <= 2 * _gpu.LSE_RTOL


def test_tcgen05_rescale_path():
    """Scores that keep growing along the context force the softmax reference to
    move (and O to be rescaled in tensor memory) many times within one slice."""
    T = 4000
    x = workloads.dense(1, 16, T, seed=47)
    ramp = torch.linspace(0.0, 12.0, T).unsqueeze(1)
    kv = x.kv.float()
    kv[:, :512] = kv[:, :512] + ramp * x.q[0, 0, :512].float().sign().unsqueeze(0) * 0.05
    x.kv = kv.to(torch.bfloat16)
    x.q = (x.q.float() * 4.0).to(torch.bfloat16)
    ro, rl = _gpu.oracle_dense(x)
    for variant in _gpu.VARIANTS:
        out, lse, plan, _ = _gpu.run_dense(x, splits=1, variant=variant)
        _gpu.assert_parity(out, lse, ro, rl, f"growing scores, variant {variant}")


@pytest.mark.parametrize("variant", _gpu.VARIANTS)
@pytest.mark.parametrize("T,splits", [(37, 0), (100, 3), (1000, 0), (1000, 7), (4097, 0)])
def test_dense_rows_past_the_context_may_hold_nan(T, splits, variant):
    """A cache allocated for max_ctx rows holds anything past the context
    (here NaN): the attended rows alone decide the result, including the rows
    a kernel loads past a slice's end inside its last tile."""
    x = workloads.dense(1, 16, T, seed=90 + T)
    d = _gpu.dev()
    cap = T + 300
    kv = torch.full((cap, 576), float("nan"), dtype=torch.bfloat16)
    kv[:T] = x.kv
    out, lse, plan, _ = _gpu.run_dense(x, splits=splits, max_ctx=cap, variant=variant, kv_dev=kv.to(d))
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, f"NaN past the context, T={T} S={plan.splits}")


@pytest.mark.parametrize("variant", _gpu.VARIANTS)
@pytest.mark.parametrize("topk", [17, 81, 300])
def test_sparse_unlisted_rows_may_hold_nan(topk, variant):
    """Rows no list names (and the rows masked ids would point at) hold NaN:
    only the listed rows may reach the result."""
    x = workloads.sparse(2, 16, [5000, 300], topk, seed=200 + topk)
    idx = x.indices.clone()
    idx[0, 0] = -1
    idx[1, topk - 1] = 300           # == cache_len: masked
    x.indices = idx
    kv = torch.full_like(x.kv, float("nan"))
    for b in range(2):
        ids = x.indices[b]
        ok = (ids >= 0) & (ids < x.cache_len[b])
        rows = x.row_offset[b] + ids[ok].long()
        kv[rows] = x.kv[rows]
    out, lse, plan, _ = _gpu.run_sparse(x, splits=3, variant=variant, kv_dev=kv.to(_gpu.dev()))
    ro, rl = _gpu.oracle_sparse(x)
    _gpu.assert_parity(out, lse, ro, rl, f"sparse k={topk}, NaN outside the lists")


@pytest.mark.parametrize("variant", _gpu.VARIANTS)
@pytest.mark.parametrize("splits", [1, 3, 5])
def test_few_ctas_walk_many_slot_items(variant, splits):
    """A grid planned for 3 SMs: each CTA walks several items of many slots
    (odd and even slot counts, ragged requests), carrying its ring of slots
    and its query tiles from item to item."""
    x = workloads.dense(2, 32, 3000, seed=46)
    x.d_pos = torch.tensor([2999, 1234], dtype=torch.int32)
    ro, rl = _gpu.oracle_dense(x)
    out, lse, plan, _ = _gpu.run_dense(x, splits=splits, num_sms=3, variant=variant)
    assert plan.grid_x <= 3 and 2 * plan.n_head_groups * plan.splits > plan.grid_x
    _gpu.assert_parity(out, lse, ro, rl, f"dense B=2 H=32 S={plan.splits} on {plan.grid_x} CTAs")


@pytest.mark.parametrize("variant", _gpu.VARIANTS)
def test_sparse_few_ctas_walk_many_items(variant):
    x = workloads.sparse(3, 16, [5000, 800, 9000], 700, seed=47)
    ro, rl = _gpu.oracle_sparse(x)
    for s in (1, 2, 5):
        out, lse, plan, _ = _gpu.run_sparse(x, splits=s, num_sms=4, variant=variant)
        assert plan.grid_x <= 4
        _gpu.assert_parity(out, lse, ro, rl, f"sparse B=3 S={plan.splits} on 4 CTAs")
