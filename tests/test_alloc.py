"""The library's host block allocator against the seeded generator's
free-list allocator: identical block tables and slots, bit for bit (CPU)."""
import numpy as np
import pytest
import torch

from paged_kv_cache_continuous_gb300 import binding, build
from paged_kv_cache_continuous_gb300 import workload as wl


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def test_bad_initial_order():
    with pytest.raises(binding.PagedAttnError):
        binding.BlockAllocator(4, 16, [0, 1, 1, 2])


def test_exhaustion_changes_nothing():
    a = binding.BlockAllocator(4, 16)
    a.ensure(1, 40)
    with pytest.raises(binding.PagedAttnError) as e:
        a.ensure(2, 33)
    assert e.value.code == binding.ERR_NO_BLOCKS
    assert a.num_free() == 1 and a.num_blocks_of(2) == 0


def test_churn_matches_reference_allocator():
    g = torch.Generator().manual_seed(17)
    N, B = 300, 16
    order = torch.randperm(N, generator=g).tolist()
    ref = wl.BlockAllocator(N, B, order)
    lib = binding.BlockAllocator(N, B, order)
    rng = np.random.default_rng(5)
    live = {}
    next_id = 0
    for step in range(200):
        op = rng.integers(0, 3)
        if op < 2 or not live:
            sid = next_id if (op == 0 or not live) else int(rng.choice(list(live)))
            if sid == next_id:
                next_id += 1
            n = live.get(sid, 0) + int(rng.integers(1, 90))
            try:
                ref.ensure(sid, n)
                ok = True
            except wl.NoBlocks:
                ok = False
            if ok:
                lib.ensure(sid, n)
                live[sid] = n
            else:
                with pytest.raises(binding.PagedAttnError):
                    lib.ensure(sid, n)
        else:
            sid = int(rng.choice(list(live)))
            ref.release(sid)
            lib.release(sid)
            del live[sid]
        assert lib.num_free() == ref.num_free()
        if live:
            seqs = sorted(live)
            width = max(-(-live[s] // B) for s in seqs) + 2
            assert np.array_equal(lib.block_table(seqs, width), ref.table_rows(seqs, width))
            n_new = [min(3, live[s]) for s in seqs]
            tot = [live[s] for s in seqs]
            exp = [ref.slot(s, t - k + j) for s, k, t in zip(seqs, n_new, tot) for j in range(k)]
            assert np.array_equal(lib.slot_mapping(seqs, n_new, tot), np.array(exp, dtype=np.int32))
