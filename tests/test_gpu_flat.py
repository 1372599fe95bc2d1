"""GPU parity of the flat split of batched sparse decode (the B * topk list
entries cut into one range per CTA, pieces of at most two requests per range,
missing slices written empty) against the fp64 oracle, and against the
uniform split of the same inputs."""
import pytest
import torch

import _gpu
import decode_attention_mla_gb300 as mla
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


@pytest.mark.parametrize("B,lens,topk,sms", [
    (40, 1500, 1024, 0),                     # 143 ranges of 288 entries, up to 5 pieces per request
    (100, [600 + 7 * b for b in range(100)], 512, 0),   # 146 ranges of 352
    (3, [5000, 800, 9000], 700, 4),          # four CTAs, ranges of 544 crossing request boundaries
    (5, 2500, 1024, 7),                      # seven ranges of 736
    (7, 3000, 2000, 10),                     # ten ranges of 1408
])
def test_flat_split_matches_oracle(B, lens, topk, sms):
    x = workloads.sparse(B, 16, lens, topk, seed=900 + B)
    out, lse, plan, scratch = _gpu.run_sparse(x, num_sms=sms)
    assert plan.flat_ranges > 0, "this shape takes the flat split"
    ro, rl = _gpu.oracle_sparse(x)
    _gpu.assert_parity(out, lse, ro, rl, f"flat split B={B} topk={topk} ranges={plan.flat_ranges} S={plan.splits}")
    assert mla.status_word(plan, scratch) == 0


def test_flat_split_agrees_with_uniform_split():
    x = workloads.sparse(64, 16, 3000, 1024, seed=910)
    a = _gpu.run_sparse(x)
    b = _gpu.run_sparse(x, splits=3)                 # an explicit split count keeps the uniform split
    assert a[2].flat_ranges > 0 and b[2].flat_ranges == 0
    assert (a[0] - b[0]).abs().max().item() <= 2 * _gpu.OUT_ATOL
    assert ((a[1] - b[1]).abs() / a[1].abs().clamp(min=1)).max().item() <= 2 * _gpu.LSE_RTOL


def test_flat_split_masked_and_duplicate_ids():
    """Out-of-range ids and a request whose list is masked entirely, under
    the flat split (its pieces attend nothing: lse = -inf, out = 0)."""
    B, topk = 40, 1024
    x = workloads.sparse(B, 16, 2000, topk, seed=920)
    idx = x.indices.clone()
    idx[1, ::7] = -5
    idx[2, 3::11] = 2000 + 9                         # past the segment
    idx[4, :] = -1                                   # nothing attended
    idx[6, 10:20] = idx[6, 0]                        # duplicates count once per entry
    x.indices = idx
    out, lse, plan, _ = _gpu.run_sparse(x)
    assert plan.flat_ranges > 0
    ro, rl = _gpu.oracle_sparse(x)
    _gpu.assert_parity(out, lse, ro, rl, "flat split, masked ids")
    assert torch.isinf(lse[4]).all() and (out[4] == 0).all()


def test_flat_split_bit_identical_across_runs():
    x = workloads.sparse(100, 16, 700, 512, seed=930)
    out0, lse0, plan, scratch = _gpu.run_sparse(x)
    assert plan.flat_ranges > 0
    for _ in range(4):
        out, lse, _, _ = _gpu.run_sparse(x, plan=plan, scratch=scratch)
        assert torch.equal(_gpu.bits(out), _gpu.bits(out0)) and torch.equal(_gpu.bits(lse), _gpu.bits(lse0))
