"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: their device memory is
planned once at start-up and nothing may be allocated while requests are
served.  pa_decode_noalloc runs the same split-K decode with the partials in
a fixed 16 MiB buffer inside the library.  These tests call it through the C
ABI and compare it with pa_decode (caller workspace) on the same inputs, with
the tolerance the other decode tests use; the file is collected last so a
stop-at-first-failure run has already run everything else.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import MAX_ABS, MEAN_ABS, dev
from paged_kv_cache_continuous_gb300 import binding as pa
from paged_kv_cache_continuous_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _batch(seed, lens, Hq=32, Hkv=8, d=128, B=16):
    g = torch.Generator().manual_seed(seed)
    N = sum(-(-L // B) for L in lens) + 4
    shape = wl.Shape(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B, num_blocks=N)
    alloc = wl.BlockAllocator(N, B, torch.randperm(N, generator=g).tolist())
    st = wl.make_step(alloc, shape, list(range(len(lens))), [1] * len(lens), lens, len(lens), g)
    kp, vp = wl.new_pool(shape, seed + 77, "cuda")
    pa.kv_append(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kp, vp)
    return shape, kp, vp, st


def _agree(a, b):
    err = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS


def test_noalloc_matches_decode_on_two_calls_in_a_row(cuda_lib):
    pa.set_decode_split(0)
    lens = [1, 17, 300, 1025, 2049, 4000, 64, 511]
    shape, kp, vp, st = _batch(101, lens)
    args = (shape, dev(st.q), kp, vp, dev(st.block_table), dev(st.seq_lens), st.max_seq_len)
    assert pa.workspace_size(shape, st.num_seqs, st.max_seq_len) <= (16 << 20)
    ref = pa.decode(*args)
    first = pa.decode_noalloc(*args)
    second = pa.decode_noalloc(*args)
    pa.check_device_error()
    _agree(first, ref)
    _agree(second, ref)


def test_noalloc_reuses_its_buffer_across_batches(cuda_lib):
    """The buffer keeps the previous call's partials; a different batch (other
    lengths, heads and split counts) must not see them."""
    pa.set_decode_split(0)
    for seed, lens, hq, hkv in ((102, [3000, 5, 800], 64, 8), (103, [70, 2600, 1, 1300, 999], 16, 16)):
        shape, kp, vp, st = _batch(seed, lens, Hq=hq, Hkv=hkv)
        args = (shape, dev(st.q), kp, vp, dev(st.block_table), dev(st.seq_lens), st.max_seq_len)
        ref = pa.decode(*args)
        out = pa.decode_noalloc(*args)
        pa.check_device_error()
        _agree(out, ref)


def test_noalloc_rejects_a_batch_larger_than_its_buffer(cuda_lib):
    """32 sequences of 32 769 tokens with 64 query heads need ~69 MB of
    partials: rejected on the host with a clear message, nothing enqueued."""
    shape = wl.Shape(num_q_heads=64, num_kv_heads=8, head_dim=128, block_size=16, num_blocks=4)
    S, L = 32, 32769
    q = torch.zeros(S, 64, 128, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(4, 8, 16, 128, dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros(S, -(-L // 16), dtype=torch.int32, device="cuda")
    lens = torch.full((S,), L, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PagedAttnError) as e:
        pa.decode_noalloc(shape, q, pool, pool, bt, lens, L)
    assert e.value.code == pa.ERR_WORKSPACE and "built-in buffer" in str(e.value)
