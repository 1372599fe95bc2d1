"""Graph-resident multi-step decode: 64 steps of [append row at d_pos -> partial
-> combine -> d_pos += 1] captured as one CUDA graph and replayed.  Checks:
every step against the fp64 oracle (all 64 steps at full size), replays byte
identical to each other and to the eager run, and a deliberately frozen row
position that is right on step 0 and wrong from step 1 on (so a single-step
check would not have caught it)."""
import numpy as np
import pytest
import torch

import _gpu
import decode_attention_mla_gb300 as mla
import workloads
from _steps import oracle_all_steps as _oracle_all_steps, oracle_step as _oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()
    torch.cuda.set_device(0)
    yield


class Loop:
    """Device state of the multi-step workload and the per-step call sequence."""

    def __init__(self, g: workloads.GraphInputs, H: int, pdl: bool = False, splits: int = 0, variant: int = 0):
        d = _gpu.dev()
        self.g = g
        self.H = H
        self.kv = g.kv.to(d)
        self.kv_init = self.kv.clone()
        self.new_rows = g.new_rows.to(d)
        self.q = g.q_steps.to(d)
        self.d_pos = torch.tensor([g.d_pos0], dtype=torch.int32, device=d)
        self.d_pos_init = self.d_pos.clone()
        self.frozen = self.d_pos.clone()
        self.out = torch.zeros(g.steps, 1, H, 512, device=d)
        self.lse = torch.zeros(g.steps, 1, H, device=d)
        self.plan = mla.plan(batch=1, heads=H, max_ctx=g.d_pos0 + g.steps, scale=g.scale, pdl=pdl, splits=splits,
                             variant=variant)
        self.scratch = mla.alloc_scratch(self.plan)

    def reset(self):
        self.kv.copy_(self.kv_init)
        self.d_pos.copy_(self.d_pos_init)
        self.frozen.copy_(self.d_pos_init)

    def steps(self, freeze_append=False):
        self.d_pos.copy_(self.d_pos_init)
        for k in range(self.g.steps):
            mla.append(self.kv, self.new_rows[k], self.frozen if freeze_append else self.d_pos)
            mla.forward(self.plan, self.q[k], self.kv, self.out[k], self.lse[k], self.scratch, d_pos=self.d_pos)
            mla.advance(self.d_pos)


_H128_ORACLE = {}


def _capture(loop, freeze_append=False):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):          # warm-up outside capture, then restore the initial state
        loop.steps(freeze_append)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    loop.reset()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        loop.steps(freeze_append)
    torch.cuda.synchronize()
    return graph


@pytest.mark.parametrize("pdl", [False, True])
def test_graph_small_all_steps(pdl):
    """Short context, 16 steps, every step checked against the oracle."""
    g = workloads.graph(128, 500, 16, seed=1)
    loop = Loop(g, 128, pdl=pdl)
    loop.reset()
    loop.steps()                                            # eager reference run
    torch.cuda.synchronize()
    eager_out, eager_lse = loop.out.clone(), loop.lse.clone()
    graph = _capture(loop)
    for r in range(4):                                      # one replay proves nothing
        loop.reset()
        loop.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(_gpu.bits(loop.out), _gpu.bits(eager_out)), f"replay {r} out != eager"
        assert torch.equal(_gpu.bits(loop.lse), _gpu.bits(eager_lse)), f"replay {r} lse != eager"
        assert int(loop.d_pos.item()) == 500 + 16
    for k in range(16):
        ro, rl = _oracle_step(g, k)
        _gpu.assert_parity(loop.out[k], loop.lse[k], ro, rl, f"graph step {k}")
    assert mla.status_word(loop.plan, loop.scratch) == 0


def test_graph_frozen_position_fails_from_step_one():
    """A cache-row write whose position never advances is right on step 0 and
    wrong afterwards: the multi-step check must see it."""
    g = workloads.graph(16, 300, 4, seed=2)
    loop = Loop(g, 16)
    graph = _capture(loop, freeze_append=True)
    loop.reset()
    graph.replay()
    torch.cuda.synchronize()
    ro, rl = _oracle_step(g, 0)
    _gpu.assert_parity(loop.out[0], loop.lse[0], ro, rl, "frozen step 0")
    for k in (1, 2, 3):
        ro, rl = _oracle_step(g, k)
        err_o, _ = _gpu.errors(loop.out[k], loop.lse[k], ro, rl)
        assert err_o > 10 * _gpu.OUT_ATOL, f"frozen append went unnoticed at step {k}"


@pytest.mark.parametrize("variant", [0, 3])
def test_graph_h128_workload(variant):
    """The 64-step, H=128, 32k-context workload: replays byte identical to eager;
    every one of the 64 steps against the oracle.
    Run with the planner's kernel (64 heads per CTA here) and with the
    32-heads-per-CTA tcgen05 kernel forced."""
    g = workloads.make("graph_h128")
    loop = Loop(g, 128, variant=variant)
    loop.reset()
    loop.steps()
    torch.cuda.synchronize()
    eager_out, eager_lse = loop.out.clone(), loop.lse.clone()
    graph = _capture(loop)
    for r in range(3):
        loop.reset()
        loop.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(_gpu.bits(loop.out), _gpu.bits(eager_out)), f"replay {r}"
        assert torch.equal(_gpu.bits(loop.lse), _gpu.bits(eager_lse)), f"replay {r}"
    assert torch.isfinite(loop.out).all() and torch.isfinite(loop.lse).all()
    if "ref" not in _H128_ORACLE:
        _H128_ORACLE["ref"] = _oracle_all_steps(g)
    ro, rl = _H128_ORACLE["ref"]
    for k in range(g.steps):
        _gpu.assert_parity(loop.out[k], loop.lse[k], ro[k:k + 1], rl[k:k + 1], f"graph_h128 step {k}")
    assert mla.status_word(loop.plan, loop.scratch) == 0
