"""The fused decode step (mla_decode_forward_step: the cache append folded
into the partial kernel, the cache write and the position advance into the
combine) against the separate launches it replaces (append, forward,
advance), bit for bit, and against the fp64 oracle: every dense kernel
variant, several steps in a row, ragged batches, the edge of the cache, and
a captured graph."""
import numpy as np
import pytest
import torch

import _gpu
import decode_attention_mla_gb300 as mla
import workloads

pytestmark = pytest.mark.gpu

# (variant, heads): warp-MMA, tcgen05 with 16, 32 and 64 heads per CTA, warp-MMA
# with P . V on tcgen05
KERNELS = [(1, 16), (2, 16), (3, 32), (4, 64), (4, 128), (5, 16), (5, 64)]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()
    torch.cuda.set_device(0)
    yield


def _bits16(t):
    return t.contiguous().view(torch.int16)


class Pair:
    """Two copies of the same decode state; `fused` steps one with
    mla_decode_forward_step, `separate` the other with append + forward (+ advance)."""

    def __init__(self, q, kv, d_pos, plan, row_offset=None):
        d = _gpu.dev()
        self.plan = plan
        self.q = q.to(d)
        self.kv = [kv.to(d), kv.to(d)]
        self.d_pos = [d_pos.to(d), d_pos.to(d)]
        self.row_offset = row_offset.to(d) if row_offset is not None else None
        B, H, _ = q.shape
        self.out = [torch.full((B, H, 512), float("nan"), device=d) for _ in range(2)]
        self.lse = [torch.full((B, H), float("nan"), device=d) for _ in range(2)]
        self.scratch = [mla.alloc_scratch(plan), mla.alloc_scratch(plan)]

    def fused(self, new_rows, advance=True):
        mla.forward_step(self.plan, self.q, self.kv[0], self.out[0], self.lse[0], self.scratch[0], new_rows,
                         d_pos=self.d_pos[0], row_offset=self.row_offset, advance=advance)

    def separate(self, new_rows, advance=True):
        mla.append(self.kv[1], new_rows, self.d_pos[1], row_offset=self.row_offset)
        mla.forward(self.plan, self.q, self.kv[1], self.out[1], self.lse[1], self.scratch[1], d_pos=self.d_pos[1],
                    row_offset=self.row_offset)
        if advance:
            mla.advance(self.d_pos[1])

    def assert_same(self, what):
        torch.cuda.synchronize()
        assert torch.equal(_gpu.bits(self.out[0]), _gpu.bits(self.out[1])), f"{what}: out"
        assert torch.equal(_gpu.bits(self.lse[0]), _gpu.bits(self.lse[1])), f"{what}: lse"
        assert torch.equal(_bits16(self.kv[0]), _bits16(self.kv[1])), f"{what}: cache"
        assert torch.equal(self.d_pos[0], self.d_pos[1]), f"{what}: d_pos"


def _one_step_case(variant, H, T, seed):
    """Cache of T + 8 rows: rows 0..T-2 attended history, row T-1 (the new row's
    place) and the rest NaN, so a step that failed to take the new row would
    leave NaN in the output."""
    x = workloads.dense(1, H, T, seed=seed)
    cap = T + 8
    kv = torch.full((cap, 576), float("nan"), dtype=torch.bfloat16)
    kv[:T - 1] = x.kv[:T - 1]
    new_row = x.kv[T - 1:T].clone()
    d_pos = torch.tensor([T - 1], dtype=torch.int32)
    plan = mla.plan(batch=1, heads=H, max_ctx=cap, scale=x.scale, variant=variant, pdl=True)
    return x, kv, new_row, d_pos, plan


@pytest.mark.parametrize("variant,H", KERNELS)
@pytest.mark.parametrize("T", [1, 2, 31, 33, 100, 3000])
def test_fused_step_equals_separate_launches(variant, H, T):
    x, kv, new_row, d_pos, plan = _one_step_case(variant, H, T, seed=300 + T + H)
    pair = Pair(x.q, kv, d_pos, plan)
    nr = new_row.to(_gpu.dev())
    pair.fused(nr)
    pair.separate(nr)
    pair.assert_same(f"variant {variant} H={H} T={T}")
    assert int(pair.d_pos[0].item()) == T
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(pair.out[0], pair.lse[0], ro, rl, f"fused step, variant {variant} H={H} T={T}")
    assert mla.status_word(plan, pair.scratch[0]) == 0


@pytest.mark.parametrize("variant,H", KERNELS)
def test_fused_steps_in_a_row(variant, H):
    """Six steps: each appends the next row and attends one more row; the two
    copies stay identical in every byte of out, lse, cache and position."""
    T0, steps = 500, 6
    x = workloads.dense(1, H, T0 + steps, seed=410 + H)
    cap = T0 + steps + 4
    kv = torch.full((cap, 576), float("nan"), dtype=torch.bfloat16)
    kv[:T0] = x.kv[:T0]
    plan = mla.plan(batch=1, heads=H, max_ctx=cap, scale=x.scale, variant=variant, pdl=True)
    pair = Pair(x.q, kv, torch.tensor([T0], dtype=torch.int32), plan)
    d = _gpu.dev()
    for k in range(steps):
        nr = x.kv[T0 + k:T0 + k + 1].to(d)
        pair.fused(nr)
        pair.separate(nr)
        pair.assert_same(f"variant {variant} step {k}")
    x.d_pos = torch.tensor([T0 + steps - 1], dtype=torch.int32)
    ro, rl = _gpu.oracle_dense(x)
    _gpu.assert_parity(pair.out[0], pair.lse[0], ro, rl, "after six fused steps")


@pytest.mark.parametrize("variant,H", [(1, 16), (4, 128)])
def test_fused_step_ragged_batch_and_cache_edge(variant, H):
    """Three packed requests: one mid-segment, one whose new row is the last
    row of the whole cache, one whose position lies past the cache (nothing
    written there, the rows that exist attended, the position still advanced)."""
    lens = [700, 90, 1200]
    offsets = [0, 700, 790]
    total = 1990
    g = torch.Generator().manual_seed(77)
    kv = torch.randn(total, 576, generator=g).to(torch.bfloat16)
    q = torch.randn(3, H, 576, generator=g).to(torch.bfloat16)
    new_rows = torch.randn(3, 576, generator=g).to(torch.bfloat16)
    d_pos = torch.tensor([400, 89, 1200 + 5], dtype=torch.int32)     # request 2: past the end of the cache
    row_offset = torch.tensor(offsets, dtype=torch.int64)
    plan = mla.plan(batch=3, heads=H, max_ctx=max(lens) + 8, scale=1.0 / 24.0, variant=variant, pdl=True)
    pair = Pair(q, kv, d_pos, plan, row_offset=row_offset)
    nr = new_rows.to(_gpu.dev())
    pair.fused(nr)
    pair.separate(nr)
    pair.assert_same(f"ragged, variant {variant}")
    assert pair.d_pos[0].cpu().tolist() == [401, 90, 1206]


@pytest.mark.parametrize("variant,H", [(1, 16), (4, 64)])
def test_fused_step_without_advance(variant, H):
    x, kv, new_row, d_pos, plan = _one_step_case(variant, H, 257, seed=520 + H)
    pair = Pair(x.q, kv, d_pos, plan)
    nr = new_row.to(_gpu.dev())
    pair.fused(nr, advance=False)
    pair.separate(nr, advance=False)
    pair.assert_same("advance = 0")
    assert int(pair.d_pos[0].item()) == 256


@pytest.mark.parametrize("variant,H", [(1, 16), (4, 128)])
def test_fused_steps_captured_in_a_graph(variant, H):
    """Eight fused steps captured once and replayed (the position reset before
    each replay) give the bytes of eight eager separate steps."""
    T0, steps = 2000, 8
    x = workloads.dense(1, H, T0 + steps, seed=630 + H)
    cap = T0 + steps
    kv0 = torch.full((cap, 576), float("nan"), dtype=torch.bfloat16)
    kv0[:T0] = x.kv[:T0]
    d = _gpu.dev()
    plan = mla.plan(batch=1, heads=H, max_ctx=cap, scale=x.scale, variant=variant, pdl=True)
    new_rows = x.kv[T0:T0 + steps].to(d)
    q = x.q.to(d)
    # eager, separate launches
    kv_e = kv0.to(d)
    dp_e = torch.tensor([T0], dtype=torch.int32, device=d)
    out_e = torch.empty(steps, 1, H, 512, device=d)
    lse_e = torch.empty(steps, 1, H, device=d)
    sc_e = mla.alloc_scratch(plan)
    for k in range(steps):
        mla.append(kv_e, new_rows[k:k + 1], dp_e)
        mla.forward(plan, q, kv_e, out_e[k], lse_e[k], sc_e, d_pos=dp_e)
        mla.advance(dp_e)
    torch.cuda.synchronize()
    # fused, captured
    kv_g = kv0.to(d)
    dp_g = torch.tensor([T0], dtype=torch.int32, device=d)
    out_g = torch.empty_like(out_e)
    lse_g = torch.empty_like(lse_e)
    sc_g = mla.alloc_scratch(plan)
    args = [mla.make_args(q, kv_g, out_g[k], lse_g[k], d_pos=dp_g) for k in range(steps)]
    mla.forward_step_args(plan, args[0], sc_g, new_rows[0:1], advance=False)   # first use outside capture
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for k in range(steps):
            mla.forward_step_args(plan, args[k], sc_g, new_rows[k:k + 1], advance=True)
    for r in range(3):
        kv_g.copy_(kv0.to(d))
        dp_g.fill_(T0)
        out_g.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(_gpu.bits(out_g), _gpu.bits(out_e)), f"replay {r}: out"
        assert torch.equal(_gpu.bits(lse_g), _gpu.bits(lse_e)), f"replay {r}: lse"
        assert torch.equal(_bits16(kv_g), _bits16(kv_e)), f"replay {r}: cache"
        assert int(dp_g.item()) == T0 + steps
