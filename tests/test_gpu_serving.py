"""Closed-loop continuous batching on the GPU: the scheduler plans, one
pa_mixed_step runs each step, the scheduler commits.  At sampled steps the
step's output and pools are checked against the oracle's mixed step on the
same inputs; every request finishes and its blocks come back."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from paged_kv_cache_continuous_gb300 import workload as wl
from paged_kv_cache_continuous_gb300.serving import ServingLoop

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("chunking", [False, True])
def test_serving_loop_matches_oracle(cuda_lib, chunking):
    shape = wl.Shape(num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16, num_blocks=600)
    loop = ServingLoop(shape, seed=5, max_batch_prefill_tokens=512, max_waiting_tokens=4, chunking=chunking)
    rng = np.random.default_rng(7)
    nid, checked = 0, 0
    for step in range(60):
        for _ in range(int(rng.poisson(1.0)) if step < 40 else 0):
            loop.submit(nid, int(rng.integers(1, 600 if chunking else 500)), int(rng.integers(1, 40)))
            nid += 1
        check = step % 7 == 3
        plan = loop.step(keep_inputs=check)
        if not check or plan is None:
            continue
        L = loop.last
        out, ek, ev = oracle.mixed_step(bits(L["q"]), bits(L["k"]), bits(L["v"]), plan["q_start_loc"], plan["seq_lens"],
                                        plan["slot_mapping"], plan["block_table"], plan["num_decode"],
                                        bits(L["kp_before"]), bits(L["vp_before"]))
        assert np.array_equal(bits(loop.kp), ek) and np.array_equal(bits(loop.vp), ev), f"pools at step {step}"
        assert_close(L["out"], out, f"mixed step {step}")
        checked += 1
    for _ in range(2000):
        if loop.step() is None:
            break
    assert checked >= 5
    assert sorted(loop.finished) == list(range(nid))
    assert loop.sched.stats() == {"queued": 0, "running": 0, "free_blocks": shape.num_blocks, "waiting_steps":
                                  loop.sched.stats()["waiting_steps"]}
