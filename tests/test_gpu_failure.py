"""Failure detection without a GPU fault: the stall-test hook makes one thread
of the partial kernel wait (about 1 ms) on a barrier nothing arrives at.  The
timeout path must run end to end: every role leaves through its bounded
waits, the CTA drains its copies and MMAs, the status word reads
MLA_EDEVICE, and the context stays usable for the next, healthy call."""
import time

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


@pytest.mark.parametrize("variant,heads,sparse", [(1, 16, False), (1, 16, True), (2, 16, False), (2, 16, True),
                                                  (3, 32, False), (4, 64, False), (5, 16, False)])
def test_wait_timeout_sets_status_and_context_survives(variant, heads, sparse):
    d = _gpu.dev()
    if sparse:
        x = workloads.sparse(2, heads, [5000, 3000], 700, seed=61)
        kw = dict(sparse=True, topk=700)
        io = dict(indices=x.indices.to(d), cache_len=x.cache_len.to(d), row_offset=x.row_offset.to(d))
    else:
        x = workloads.dense(1, heads, 4000, seed=61)
        kw = dict(max_ctx=4000)
        io = dict(d_pos=x.d_pos.to(d))
    q, kv = x.q.to(d), x.kv.to(d)
    B = q.shape[0]
    out = torch.zeros(B, heads, 512, device=d)
    lse = torch.zeros(B, heads, device=d)

    stalled = mla.plan(batch=B, heads=heads, scale=x.scale, variant=variant, stall_test=True, **kw)
    scratch = mla.alloc_scratch(stalled)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    mla.forward(stalled, q, kv, out, lse, scratch, **io)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert mla.status_word(stalled, scratch) == mla.EDEVICE
    assert elapsed < 1.0, f"the abort path took {elapsed:.3f} s"

    # the same context, a healthy plan: correct results and a clean status word
    healthy = mla.plan(batch=B, heads=heads, scale=x.scale, variant=variant, **kw)
    scratch2 = mla.alloc_scratch(healthy)
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    mla.forward(healthy, q, kv, out, lse, scratch2, **io)
    torch.cuda.synchronize()
    assert mla.status_word(healthy, scratch2) == 0
    ro, rl = _gpu.oracle_sparse(x) if sparse else _gpu.oracle_dense(x)
    _gpu.assert_parity(out, lse, ro, rl, f"after a stalled call, variant {variant}")
