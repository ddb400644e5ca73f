"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot hand the library a workspace: their device memory is
planned once at start-up and nothing may be allocated while requests are
served.  pa_decode_noalloc runs the same split-K decode with the partials in
a fixed 16 MiB buffer inside the library.  These tests call it through the C
ABI on inputs drawn on the host, compare every output element with the fp64
oracle (the tolerance of the other decode tests) and with pa_decode (caller
workspace) on the same inputs; the file is collected last so a
stop-at-first-failure run has already run everything else.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import MAX_ABS, MEAN_ABS, assert_close, bits, dev
from paged_kv_cache_continuous_gb300 import binding as pa
from paged_kv_cache_continuous_gb300 import workload as wl

pytestmark = pytest.mark.gpu

SCRATCH = 16 << 20


def _batch(seed, lens, Hq=32, Hkv=8, d=128, B=16):
    """A decode step drawn on the host; the device pools get the GPU append,
    the oracle's host mirror the oracle's append."""
    g = torch.Generator().manual_seed(seed)
    N = sum(-(-L // B) for L in lens) + 4
    shape = wl.Shape(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B, num_blocks=N)
    alloc = wl.BlockAllocator(N, B, torch.randperm(N, generator=g).tolist())
    st = wl.make_step(alloc, shape, list(range(len(lens))), [1] * len(lens), lens, len(lens), g)
    kh, vh = wl.new_pool(shape, seed + 77)
    kp, vp = dev(kh), dev(vh)
    pa.kv_append(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kp, vp)
    kq, vq = oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, bits(kh), bits(vh))
    ref = oracle.decode(bits(st.q), kq, vq, st.block_table, st.seq_lens)
    return shape, kp, vp, st, ref


def _agree(a, b):
    err = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS


def test_noalloc_matches_oracle_and_decode_on_two_calls_in_a_row(cuda_lib):
    pa.set_decode_split(0)
    lens = [1, 17, 300, 1025, 2049, 4000, 64, 511]
    shape, kp, vp, st, ref = _batch(101, lens)
    args = (shape, dev(st.q), kp, vp, dev(st.block_table), dev(st.seq_lens), st.max_seq_len)
    assert pa.workspace_size(shape, st.num_seqs, st.max_seq_len) <= SCRATCH
    with_ws = pa.decode(*args)
    first = pa.decode_noalloc(*args)
    second = pa.decode_noalloc(*args)
    pa.check_device_error()
    assert_close(first, ref, "noalloc, first call")
    assert_close(second, ref, "noalloc, second call")
    _agree(first, with_ws)
    _agree(second, with_ws)


def test_noalloc_reuses_its_buffer_across_batches(cuda_lib):
    """The buffer keeps the previous call's partials; a different batch (other
    lengths, heads and split counts) must not see them."""
    pa.set_decode_split(0)
    for seed, lens, hq, hkv in ((102, [3000, 5, 800], 64, 8), (103, [70, 2600, 1, 1300, 999], 16, 16)):
        shape, kp, vp, st, ref = _batch(seed, lens, Hq=hq, Hkv=hkv)
        args = (shape, dev(st.q), kp, vp, dev(st.block_table), dev(st.seq_lens), st.max_seq_len)
        out = pa.decode_noalloc(*args)
        with_ws = pa.decode(*args)
        pa.check_device_error()
        assert_close(out, ref, f"noalloc Hq={hq} Hkv={hkv}")
        _agree(out, with_ws)


def test_noalloc_accepts_a_batch_above_the_workspace_bound(cuda_lib):
    """pa_workspace_size is an upper bound (it assumes the shortest split);
    the call checks the exact need of the plan it runs.  48 sequences of up
    to 4096 tokens with 64 query heads / 8 KV heads: the bound is ~26 MB, the
    plan's need (512-token splits: partials and work items) ~13 MB, so the
    call is accepted and must be right."""
    pa.set_decode_split(0)
    rng = np.random.default_rng(104)
    lens = [4096] + rng.integers(1, 4097, size=47).tolist()
    shape, kp, vp, st, ref = _batch(104, lens, Hq=64, Hkv=8)
    split, max_splits = pa.decode_plan(shape, st.num_seqs, st.max_seq_len)
    partials = st.num_seqs * 64 * max_splits * (128 + 2) * 4 if max_splits > 1 else 0
    need = -(-partials // 16) * 16 + st.num_seqs * (max(max_splits, 1) * 8 * 16 + 8) + 16  # + the plan
    assert pa.workspace_size(shape, st.num_seqs, st.max_seq_len) > SCRATCH >= need, (split, max_splits)
    out = pa.decode_noalloc(shape, dev(st.q), kp, vp, dev(st.block_table), dev(st.seq_lens), st.max_seq_len)
    pa.check_device_error()
    assert_close(out, ref, "noalloc above the workspace bound")


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
