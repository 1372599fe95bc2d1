"""Pins of the oracle's FP8 (OCP E4M3) cache path: the byte decoding against
the format's definition (special values, order, sign) and PyTorch's own
float8_e4m3fn conversion, and the dequantised decode against the bf16 decode
on values both formats hold exactly."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads


def _values():
    return oracle.e4m3_values(np.arange(256, dtype=np.uint8))


def test_e4m3_special_values():
    v = _values()
    assert v[0x00] == 0.0 and math.copysign(1.0, v[0x00]) == 1.0
    assert v[0x80] == 0.0 and math.copysign(1.0, v[0x80]) == -1.0
    assert v[0x01] == 2.0 ** -9                      # smallest subnormal
    assert v[0x07] == 7 * 2.0 ** -9                  # largest subnormal
    assert v[0x08] == 2.0 ** -6                      # smallest normal
    assert v[0x38] == 1.0                            # exponent field 7 = bias
    assert v[0x39] == 1.125                          # one mantissa step
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0    # largest finite
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF]) and np.isnan(v).sum() == 2
    assert np.isfinite(v[np.arange(256) % 128 != 0x7F]).all()


def test_e4m3_order_and_sign():
    v = _values()
    pos = v[:0x7F]
    assert (np.diff(pos) > 0).all()                  # 0x00 .. 0x7E strictly increasing
    for b in range(0x7F):
        assert v[b | 0x80] == -v[b]


def test_e4m3_matches_torch_float8():
    """PyTorch's float8_e4m3fn widening of every byte equals the oracle's."""
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    v = _values()
    assert np.array_equal(np.isnan(ref), np.isnan(v))
    fin = ~np.isnan(v)
    assert np.array_equal(ref[fin], v[fin])


def _random_e4m3(shape, seed):
    """Random finite E4M3 bytes (NaN patterns replaced)."""
    g = np.random.default_rng(seed)
    b = g.integers(0, 256, size=shape, dtype=np.uint8)
    b[(b & 0x7F) == 0x7F] = 0x38
    return b


def _as_bf16(vals):
    t = torch.from_numpy(vals.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(t.double().numpy(), vals)  # every E4M3 value is a bf16 value
    return t


@pytest.mark.parametrize("sparse", [False, True])
@pytest.mark.parametrize("splits", [0, 3])
def test_e4m3_decode_equals_bf16_decode_on_the_same_values(sparse, splits):
    B, H, rows = 2, 4, 300
    kv8 = _random_e4m3((rows, 576), seed=5)
    kvb = _as_bf16(oracle.e4m3_values(kv8))
    g = torch.Generator().manual_seed(6)
    q = torch.randn(B, H, 576, generator=g).to(torch.bfloat16)
    scale = 1.0 / 24.0
    kw = dict(row_offset=np.array([0, 150], np.int64))
    if sparse:
        kw.update(indices=np.array([[3, 140, 7, -1, 99], [0, 149, 200, 12, 5]], np.int32),
                  cache_len=np.array([150, 150], np.int32))
    else:
        kw.update(d_pos=np.array([120, 140], np.int32))
    if splits:
        o8, l8 = oracle.decode_e4m3(q, kv8, kv_scale=1.0, scale=scale, splits=splits, granule=16, **kw)
        ob, lb = oracle.decode_split(q, kvb, scale=scale, splits=splits, granule=16, **kw)
    else:
        o8, l8 = oracle.decode_e4m3(q, kv8, kv_scale=1.0, scale=scale, **kw)
        ob, lb = oracle.decode(q, kvb, scale=scale, **kw)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_e4m3_scale_multiplies_values():
    """With kv_scale = 4 every value is 4x: the scores are those of scale 4 * scale
    over the unscaled values and the output is 4x that decode's output."""
    kv8 = _random_e4m3((200, 576), seed=8)
    kvb = _as_bf16(oracle.e4m3_values(kv8))
    g = torch.Generator().manual_seed(9)
    q = torch.randn(1, 8, 576, generator=g).to(torch.bfloat16)
    d_pos = np.array([199], np.int32)
    o8, l8 = oracle.decode_e4m3(q, kv8, kv_scale=4.0, scale=0.01, d_pos=d_pos)
    ob, lb = oracle.decode(q, kvb, scale=0.04, d_pos=d_pos)
    assert np.array_equal(o8, 4.0 * ob) and np.array_equal(l8, lb)


def test_e4m3_workload_quantisation_round_trip():
    """The input recipe's quantiser: every byte decodes (times the scale) to
    within half an E4M3 step of the bf16 value it came from."""
    x = workloads.dense(1, 16, 64, seed=3)
    kv8, kv_scale = workloads.to_e4m3(x.kv)
    vals = oracle.e4m3_values(kv8) * kv_scale
    src = x.kv.double().numpy()
    assert np.isfinite(vals).all()
    rel = np.abs(vals - src) / np.maximum(np.abs(src), 2.0 ** -6 * kv_scale)
    assert rel.max() <= 2.0 ** -4 + 1e-12
