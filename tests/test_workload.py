"""Seeded generators and the free-list allocator (host only)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_continuous_gb300 import workload as wl


def test_allocator_lifo_no_dup_no_leak():
    a = wl.BlockAllocator(10, 4, [3, 1, 4, 0, 5, 9, 2, 6, 8, 7])
    a.ensure(0, 5)            # 2 blocks: 3, 1
    a.ensure(1, 4)            # 1 block: 4
    assert a.tables == {0: [3, 1], 1: [4]}
    a.ensure(0, 9)            # grows by one: 0
    assert a.tables[0] == [3, 1, 0]
    a.release(0)              # pushed 3, 1, 0 -> next handed out is 0
    a.ensure(2, 8)
    assert a.tables[2] == [0, 1]
    assert a.num_free() == 10 - 3
    with pytest.raises(wl.NoBlocks):
        a.ensure(3, 4 * 8)
    a.release(1); a.release(2)
    assert sorted(a.free) == list(range(10))


def test_slot_identity():
    a = wl.BlockAllocator(6, 4, [5, 2, 0, 1, 3, 4])
    a.ensure(7, 10)
    assert [a.slot(7, p) for p in (0, 3, 4, 9)] == [20, 23, 8, 1]


def test_workloads_shapes_and_budgets():
    shape, kp, vp, st = wl.mixed(pool_device=None)
    n = st.q_start_loc[1:] - st.q_start_loc[:-1]
    assert st.num_decode == 120 and np.all(n[:120] == 1)
    assert n[120:].sum() <= 4096 and n[120:].min() >= 64 and n[120:].max() <= 1024
    assert shape.num_q_heads == 32 and shape.num_kv_heads == 8 and shape.block_size == 16
    # every live slot distinct and consistent with the table
    assert len(set(st.slot_mapping.tolist())) == st.num_tokens
    exp = oracle.expected_slots(st.q_start_loc, st.seq_lens, st.block_table, shape.block_size)
    assert np.array_equal(exp, st.slot_mapping)
    shape2, _, _, st2 = wl.llama7b_decode(pool_device=None)
    assert st2.num_seqs == 128 and 2 <= st2.seq_lens.min() and st2.seq_lens.max() <= 2049
    used = sum(-(-int(L) // 16) for L in st2.seq_lens)
    assert shape2.num_blocks == int(np.ceil(1.1 * used))


def test_churn_steps_reuse_blocks():
    ch = wl.Churn(num_seqs=40, steps=6, max_context=300, prompt_range=(5, 40), block_size=8,
                  num_q_heads=4, num_kv_heads=2, head_dim=16)
    seen_free = []
    for _ in range(6):
        st = ch.step()
        assert st.num_seqs == 40
        assert st.num_decode == (40 if not seen_free else 36)
        live = [b for t in ch.alloc.tables.values() for b in t]
        assert len(live) == len(set(live))
        assert len(live) + ch.alloc.num_free() == ch.shape.num_blocks
        exp = oracle.expected_slots(st.q_start_loc, st.seq_lens, st.block_table, 8)
        assert np.array_equal(exp, st.slot_mapping)
        seen_free.append(ch.alloc.num_free())


def test_seeded_determinism():
    a = wl.tiny()
    b = wl.tiny()
    assert torch.equal(a[1], b[1]) and torch.equal(a[4].q, b[4].q)
    assert np.array_equal(a[3].block_table, b[3].block_table)
