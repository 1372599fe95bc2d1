"""The fp64 oracle against facts fixed by the mathematics (no GPU needed)."""
import pytest

import _pins


@pytest.mark.parametrize("pin", _pins.ALL_PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()


def test_batched_steps_oracle_equals_step_by_step():
    """The full-size graph test checks its 64 steps with one batched oracle
    call (the steps as requests sharing the cache after all appends); that
    reading must give, step for step, the oracle of the cache as it stood
    at that step, bit for bit (the same rows are summed in the same order)."""
    import numpy as np
    import workloads
    from _steps import oracle_all_steps, oracle_step
    g = workloads.graph(16, 300, 7, seed=3)
    ro, rl = oracle_all_steps(g)
    for k in range(g.steps):
        o1, l1 = oracle_step(g, k)
        assert np.array_equal(ro[k:k + 1], o1) and np.array_equal(rl[k:k + 1], l1), f"step {k}"
    # control: step 0 with the last step's context bound would attend the later rows and differ
    import oracle
    import torch
    kv = g.kv.clone()
    kv[g.d_pos0:g.d_pos0 + g.steps] = g.new_rows[:, 0]
    o_late, _ = oracle.decode(g.q_steps[0], kv, scale=g.scale,
                              d_pos=torch.tensor([g.d_pos0 + g.steps - 1], dtype=torch.int32))
    assert np.abs(o_late - ro[0:1]).max() > 1e-6
