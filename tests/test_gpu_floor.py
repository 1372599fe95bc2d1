"""The floor probes on the GPU: the empty pair runs with and without PDL, and
the read kernel reads exactly its piece of the region (checked through the
word each CTA writes back, recomputed here from the same bytes)."""
import numpy as np
import pytest
import torch

import decode_attention_mla_gb300 as mla

pytestmark = pytest.mark.gpu

ROUND = 6 * 32 * 1024       # bytes a CTA reads per round (six 32 KiB bulk copies)


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from __graft_entry__ import build
    build()
    torch.cuda.set_device(0)
    yield


@pytest.mark.parametrize("pdl", [True, False])
def test_empty_pair_runs(pdl):
    for _ in range(3):
        mla.floor_empty_pair((128, 384, 200000), (64, 256, 120 * 1024), pdl=pdl)
        mla.floor_empty_pair((1, 32, 0), (152, 1024, 0), pdl=pdl)
    torch.cuda.synchronize()


def _expected_sink(data: np.ndarray, nbytes: int, ctas: int) -> np.ndarray:
    per = (nbytes // 16 + ctas - 1) // ctas * 16
    out = np.zeros(ctas, dtype=np.uint64)
    for i in range(ctas):
        lo, hi = i * per, min(nbytes, i * per + per)
        for off in range(lo, hi, ROUND):
            out[i] += int(data[off:off + 4].view(np.uint32)[0])
    return (out % (1 << 32)).astype(np.uint32)


@pytest.mark.parametrize("nbytes,ctas", [(16, 1), (4096, 8), (9437184, 152), (9437184, 128),
                                         (3 * ROUND + 48, 2), (1 << 20, 300)])
def test_read_covers_its_piece(nbytes, ctas):
    g = torch.Generator().manual_seed(nbytes ^ ctas)
    host = torch.randint(0, 256, (nbytes + 64,), dtype=torch.uint8, generator=g)
    src = host.cuda()
    sink = torch.full((ctas,), -1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.floor_read(src, nbytes, ctas, sink, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    want = _expected_sink(host.numpy(), nbytes, ctas)
    got = sink.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, want)


def _expected_gather(rows: np.ndarray, n: int, ctas: int, per_round: int) -> np.ndarray:
    """The word each CTA writes: the first word of every round's first row up to
    the round before last, plus that of the last even round (left in half 0)."""
    per = -(-n // ctas)
    out = np.zeros(ctas, dtype=np.uint64)
    for i in range(ctas):
        lo, hi = i * per, min(n, i * per + per)
        if hi <= lo:
            continue
        firsts = [int(rows[s]) for s in range(lo, hi, per_round)]
        R = len(firsts)
        acc = sum(firsts[:max(0, R - 2)]) + firsts[(R - 1) // 2 * 2]
        out[i] = acc
    return (out % (1 << 32)).astype(np.uint32)


@pytest.mark.parametrize("kv_rows,stride,row_bytes,n,ctas", [
    (5000, 1152, 1152, 4096, 152), (5000, 1152, 1152, 1, 1), (70000, 1152, 1152, 131072, 152),
    (3000, 1152, 576, 2000, 7), (3000, 1168, 1152, 999, 300), (100, 32, 16, 1000, 3)])
def test_gather_reads_the_listed_rows(kv_rows, stride, row_bytes, n, ctas):
    g = torch.Generator().manual_seed(n + ctas)
    kv = torch.zeros(kv_rows, stride, dtype=torch.uint8)
    kv[:, :4] = torch.arange(kv_rows, dtype=torch.int32).view(-1, 1).view(torch.uint8).view(kv_rows, 4)
    rows = torch.randint(0, kv_rows, (n,), dtype=torch.int64, generator=g)
    sink = torch.full((ctas,), -1, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvd, rowsd = kv.cuda(), rows.cuda()
    mla.floor_gather(kvd, rowsd, ctas, sink, status, row_bytes=row_bytes)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    per_round = min((6 * 32 * 1024 // 2) // row_bytes, 128)
    want = _expected_gather(rows.numpy(), n, ctas, per_round)
    assert np.array_equal(sink.cpu().numpy().view(np.uint32), want)


def test_gather_skips_rows_outside_the_cache():
    kv = torch.zeros(64, 1152, dtype=torch.uint8, device="cuda")
    rows = torch.tensor([3, -1, 64, 1 << 40, 5, 63], dtype=torch.int64, device="cuda")
    sink = torch.zeros(2, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.floor_gather(kv, rows, 2, sink, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
