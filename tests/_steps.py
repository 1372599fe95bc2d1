"""Oracle of a multi-step dense decode workload (workloads.graph): step k
writes new row k at d_pos0 + k, attends rows 0 .. d_pos0 + k, then advances."""
import oracle
import torch


def oracle_step(g, k, heads=None):
    kv = g.kv.clone()
    kv[g.d_pos0:g.d_pos0 + k + 1] = g.new_rows[:k + 1, 0]
    q = g.q_steps[k] if heads is None else g.q_steps[k][:, heads]
    return oracle.decode(q, kv, scale=g.scale, d_pos=torch.tensor([g.d_pos0 + k], dtype=torch.int32))


def oracle_all_steps(g):
    """The oracle for every step of a multi-step workload in one batched call:
    step k attends rows 0 .. d_pos0 + k of the cache after k + 1 appends, which
    are the same rows in the cache after all appends (rows past d_pos0 + k are
    not attended), so the steps become the requests of one batch that share
    one cache segment."""
    kv = g.kv.clone()
    kv[g.d_pos0:g.d_pos0 + g.steps] = g.new_rows[:, 0]
    q = torch.cat([g.q_steps[k] for k in range(g.steps)], dim=0)
    d_pos = torch.arange(g.d_pos0, g.d_pos0 + g.steps, dtype=torch.int32)
    return oracle.decode(q, kv, scale=g.scale, d_pos=d_pos, row_offset=torch.zeros(g.steps, dtype=torch.int64))
