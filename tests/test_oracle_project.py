"""Pins of the oracle's projection of the merged latent through wv_b
("Graph-resident decode", Lecture 08, s.6: after the merge, the latent is
projected through wv_b per head): checked against facts other than the oracle
itself -- selection by one-hot weight rows (exact), and exact rational
arithmetic on small inputs."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle


def _bf16(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def test_one_hot_rows_select_latent_entries():
    """wv_b[h][v] = e_{p_h(v)} selects latent[b][h][p_h(v)] exactly (catches a
    transposed or mis-indexed weight, a wrong head or request offset)."""
    rng = np.random.default_rng(1)
    B, H, d, V = 3, 4, 512, 128
    lat = rng.standard_normal((B, H, d))
    w = np.zeros((H, V, d), np.float32)
    perms = [rng.permutation(d)[:V] for _ in range(H)]
    for h in range(H):
        w[h, np.arange(V), perms[h]] = 1.0
    y = oracle.project(lat, _bf16(w))
    for h in range(H):
        assert np.array_equal(y[:, h, :], lat[:, h, perms[h]])


def test_exact_rationals_small():
    """Dyadic latents times bf16 weights, summed exactly: the double result is
    within a few units in the last place of the exact value."""
    rng = np.random.default_rng(2)
    B, H, d, V = 2, 3, 9, 5
    lat = rng.integers(-64, 64, (B, H, d)) / 8.0
    w = _bf16(rng.standard_normal((H, V, d)))
    wd = w.float().numpy()               # the bf16 values, exact in float32
    y = oracle.project(lat, w)
    for b in range(B):
        for h in range(H):
            for v in range(V):
                exact = sum(Fraction(float(lat[b, h, r])) * Fraction(float(wd[h, v, r])) for r in range(d))
                scale = sum(abs(Fraction(float(lat[b, h, r])) * Fraction(float(wd[h, v, r]))) for r in range(d))
                assert abs(Fraction(float(y[b, h, v])) - exact) <= scale * Fraction(1, 2 ** 48)


def test_zero_latent_and_shape_checks():
    w = _bf16(np.ones((2, 16, 512)))
    assert (oracle.project(np.zeros((1, 2, 512)), w) == 0).all()
    with pytest.raises(ValueError):
        oracle.project(np.zeros((1, 3, 512)), w)
