"""Stored tiny fixtures (tests/golden/tiny_cases.json, written by
tests/golden/make_golden.py from the oracle): the oracle built here must
reproduce them, and they must agree with the 50-digit evaluation of the
definition."""
import json
import os

import numpy as np
import torch

import _pins
import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _bf16(bits, shape):
    return torch.tensor(bits, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).view(*shape)


def _load():
    with open(os.path.join(HERE, "tiny_cases.json")) as f:
        return json.load(f)["cases"]


def test_golden_cases():
    for c in _load():
        q = _bf16(c["q_bits"], c["q_shape"])
        kv = _bf16(c["kv_bits"], c["kv_shape"])
        kw = dict(scale=c["scale"], d_latent=c["d_latent"], d_rope=c["d_rope"],
                  row_offset=torch.tensor(c["row_offset"], dtype=torch.int64))
        if c["kind"] == "dense":
            kw["d_pos"] = torch.tensor(c["d_pos"], dtype=torch.int32)
            rows = _pins._attended("dense", q.shape[0], d_pos=kw["d_pos"], row_offset=kw["row_offset"])
        else:
            kw["indices"] = torch.tensor(c["indices"], dtype=torch.int32)
            kw["cache_len"] = torch.tensor(c["cache_len"], dtype=torch.int32)
            rows = _pins._attended("sparse", q.shape[0], row_offset=kw["row_offset"], indices=kw["indices"],
                                   cache_len=kw["cache_len"])
        out, lse = oracle.decode(q, kv, **kw)
        want_o = np.array(c["out"])
        want_l = np.array(c["lse"])
        assert np.abs(out - want_o).max() <= 1e-14
        assert np.abs(lse - want_l).max() <= 1e-14
        ref_o, ref_l = _pins._decimal_reference(q, kv, rows, c["scale"], c["d_latent"])
        _pins._close(want_l, ref_l, 1e-13, "golden lse vs definition")
        _pins._close(want_o, ref_o, 1e-13, "golden out vs definition")
