"""The seeded input generators: shapes, determinism, ranges, uniqueness."""
import torch

import workloads


def test_randn_deterministic_and_thread_independent():
    a = workloads.randn_bf16(20000, 576, seed=3, stream=2, threads=1)
    b = workloads.randn_bf16(20000, 576, seed=3, stream=2, threads=4)
    assert a.dtype == torch.bfloat16 and a.shape == (20000, 576)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    c = workloads.randn_bf16(20000, 576, seed=4, stream=2)
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))
    m, s = a.float().mean().item(), a.float().std().item()
    assert abs(m) < 0.01 and abs(s - 1.0) < 0.01


def test_unique_indices():
    idx = workloads.unique_indices(65536, 2048, seed=0, stream=3)
    assert idx.dtype == torch.int32 and idx.numel() == 2048
    assert torch.unique(idx).numel() == 2048
    assert int(idx.min()) >= 0 and int(idx.max()) < 65536
    assert not torch.equal(idx, torch.sort(idx).values)      # unsorted


def test_named_small_workloads():
    d = workloads.make("dense_t256")
    assert d.q.shape == (1, 16, 576) and d.kv.shape == (256, 576) and int(d.d_pos[0]) == 255
    s = workloads.make("sparse_k2048")
    assert s.kv.shape == (65536, 576) and s.indices.shape == (1, 2048)
    g = workloads.graph(128, 64, 4)
    assert g.q_steps.shape == (4, 1, 128, 576) and g.kv.shape == (68, 576)
    assert torch.count_nonzero(g.kv[64:].float()) == 0


def test_ragged_lengths_range():
    lens = workloads.ragged_lengths(64, 4096, 131072, seed=0)
    assert lens.shape == (64,) and int(lens.min()) >= 4096 and int(lens.max()) <= 131072
    assert torch.equal(lens, workloads.ragged_lengths(64, 4096, 131072, seed=0))
