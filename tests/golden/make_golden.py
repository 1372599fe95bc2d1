"""Write tests/golden/tiny_cases.json: small seeded inputs and the fp64 oracle's
outputs for them.  Calls only the oracle and the seeded input generators.

The pages print no worked MLA example, so these stored values are regression
fixtures of the oracle (the same build on another machine must reproduce them),
and the test that reads them also checks them against the 50-digit evaluation
of the definition softmax((q_lat.c + q_rope.k_rope) * scale) . c.

Usage:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import torch  # noqa: E402

import oracle  # noqa: E402
import workloads  # noqa: E402


def _bits(t):
    return t.contiguous().view(torch.int16).to(torch.int32).bitwise_and(0xFFFF).flatten().tolist()


def main():
    dc, dr = 8, 4
    cases = []
    # dense, batch 2, ragged contexts
    q = workloads.randn_bf16(6, dc + dr, seed=101, stream=1).view(2, 3, dc + dr)
    kv = workloads.randn_bf16(20, dc + dr, seed=101, stream=2)
    d_pos = torch.tensor([9, 3], dtype=torch.int32)
    off = torch.tensor([0, 10], dtype=torch.int64)
    out, lse = oracle.decode(q, kv, scale=0.25, d_latent=dc, d_rope=dr, d_pos=d_pos, row_offset=off)
    cases.append(dict(kind="dense", d_latent=dc, d_rope=dr, scale=0.25, q_shape=list(q.shape), q_bits=_bits(q),
                      kv_shape=list(kv.shape), kv_bits=_bits(kv), d_pos=d_pos.tolist(), row_offset=off.tolist(),
                      out=out.tolist(), lse=lse.tolist()))
    # sparse, batch 2, with out-of-range ids
    q = workloads.randn_bf16(4, dc + dr, seed=102, stream=1).view(2, 2, dc + dr)
    kv = workloads.randn_bf16(15, dc + dr, seed=102, stream=2)
    lens = torch.tensor([11, 4], dtype=torch.int32)
    off = torch.tensor([0, 11], dtype=torch.int64)
    idx = torch.tensor([[10, 0, 5, -2, 11], [3, 1, 4, 0, 2]], dtype=torch.int32)
    out, lse = oracle.decode(q, kv, scale=0.3, d_latent=dc, d_rope=dr, indices=idx, cache_len=lens,
                             row_offset=off)
    cases.append(dict(kind="sparse", d_latent=dc, d_rope=dr, scale=0.3, q_shape=list(q.shape), q_bits=_bits(q),
                      kv_shape=list(kv.shape), kv_bits=_bits(kv), indices=idx.tolist(), cache_len=lens.tolist(),
                      row_offset=off.tolist(), out=out.tolist(), lse=lse.tolist()))
    with open(os.path.join(HERE, "tiny_cases.json"), "w") as f:
        json.dump({"generator": "tests/golden/make_golden.py", "cases": cases}, f, indent=1)


if __name__ == "__main__":
    main()
