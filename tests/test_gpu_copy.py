"""Whole-block copies (fork, migration, swap) on the GPU against the oracle:
bit-exact, since a copy is byte work."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bits, dev
from paged_kv_cache_continuous_gb300 import binding as pa
from paged_kv_cache_continuous_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _pools(shape, n, seed):
    kp, vp = wl.new_pool(wl.Shape(shape.num_q_heads, shape.num_kv_heads, shape.head_dim, shape.block_size, n),
                         seed)
    return kp, vp


def _ids(n, k, rng):
    return rng.choice(n, size=k, replace=False).astype(np.int32)


@pytest.mark.parametrize("Hkv,d,B,pairs", [
    (8, 128, 16, 300),    # 32 KB blocks (Llama-3-8B-shaped KV heads)
    (32, 128, 32, 40),    # 256 KB blocks: several CTAs per block, two vectors in flight
    (1, 64, 16, 5000),    # 2 KB blocks, more pairs than the grid has rows
    (2, 64, 32, 1),       # one pair
])
def test_copy_device_to_device(cuda_lib, Hkv, d, B, pairs):
    shape = wl.Shape(num_q_heads=Hkv, num_kv_heads=Hkv, head_dim=d, block_size=B, num_blocks=1)
    rng = np.random.default_rng(Hkv * 1000 + pairs)
    ns, nd = pairs + 17, pairs + 5
    sk, sv = _pools(shape, ns, 1)
    dk, dv = _pools(shape, nd, 2)
    si, di = _ids(ns, pairs, rng), _ids(nd, pairs, rng)
    gdk, gdv = dev(dk), dev(dv)
    pa.copy_blocks(shape, dev(sk), dev(sv), gdk, gdv, dev(si), dev(di))
    pa.check_device_error()
    ek, ev = oracle.copy_blocks(bits(sk), bits(sv), bits(dk), bits(dv), si, di)
    assert np.array_equal(bits(gdk), ek) and np.array_equal(bits(gdv), ev)


def test_fork_in_pool_then_decode(cuda_lib):
    """Copy one sequence's blocks to free blocks of the same pool; decode over
    the copy equals decode over the original bit for bit, and the pool equals
    the oracle's."""
    g = torch.Generator().manual_seed(5)
    shape = wl.Shape(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16, num_blocks=160)
    alloc = wl.BlockAllocator(shape.num_blocks, shape.block_size,
                              torch.randperm(shape.num_blocks, generator=g).tolist())
    L = 1000
    st = wl.make_step(alloc, shape, [0], [L], [L], 0, g)
    kp, vp = wl.new_pool(shape, 77)
    kd, vd = dev(kp), dev(vp)
    pa.kv_append(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kd, vd)
    nb = -(-L // 16)
    src = st.block_table[0, :nb].astype(np.int32)
    free = np.array([b for b in range(shape.num_blocks) if b not in set(src.tolist())], dtype=np.int32)
    dst = np.random.default_rng(3).permutation(free)[:nb].astype(np.int32)
    before_k, before_v = bits(kd), bits(vd)
    pa.copy_blocks(shape, kd, vd, kd, vd, dev(src), dev(dst))
    pa.check_device_error()
    ek, ev = oracle.copy_blocks(before_k, before_v, before_k.copy(), before_v.copy(), src, dst)
    assert np.array_equal(bits(kd), ek) and np.array_equal(bits(vd), ev)
    q = wl.bf16_randn((1, 32, 128), g)
    bt2 = st.block_table.copy()
    bt2[0, :nb] = dst
    lens = dev(np.array([L], dtype=np.int32))
    a = pa.decode(shape, dev(q), kd, vd, dev(st.block_table), lens, L)
    b = pa.decode(shape, dev(q), kd, vd, dev(bt2), lens, L)
    pa.check_device_error()
    assert torch.equal(a, b)


def test_swap_out_and_in_through_pinned_host(cuda_lib):
    """Device -> pinned host pool -> other device blocks, each leg bit-exact."""
    shape = wl.Shape(num_q_heads=8, num_kv_heads=8, head_dim=128, block_size=16, num_blocks=1)
    rng = np.random.default_rng(11)
    nd, nh, k = 400, 150, 120
    gk, gv = _pools(shape, nd, 3)
    hk0, hv0 = _pools(shape, nh, 4)
    kd, vd = dev(gk), dev(gv)
    hk, hv = hk0.clone().pin_memory(), hv0.clone().pin_memory()
    out_src, host_slots = _ids(nd, k, rng), _ids(nh, k, rng)
    pa.copy_blocks(shape, kd, vd, hk, hv, dev(out_src), dev(host_slots))
    pa.check_device_error()
    ek, ev = oracle.copy_blocks(bits(gk), bits(gv), bits(hk0), bits(hv0), out_src, host_slots)
    assert np.array_equal(bits(hk), ek) and np.array_equal(bits(hv), ev)
    in_dst = rng.permutation(np.setdiff1d(np.arange(nd), out_src))[:k].astype(np.int32)
    before_k, before_v = bits(kd), bits(vd)
    pa.copy_blocks(shape, hk, hv, kd, vd, dev(host_slots), dev(in_dst))
    pa.check_device_error()
    ek2, ev2 = oracle.copy_blocks(ek, ev, before_k, before_v, host_slots, in_dst)
    assert np.array_equal(bits(kd), ek2) and np.array_equal(bits(vd), ev2)
    assert np.array_equal(bits(kd)[in_dst], bits(gk)[out_src])


def test_copy_bad_ids_flag_error(cuda_lib):
    """An id outside its pool records PA_ERR_BAD_INDEX; that pair is skipped
    and every other pair still lands."""
    shape = wl.Shape(num_q_heads=4, num_kv_heads=4, head_dim=64, block_size=16, num_blocks=1)
    sk, sv = _pools(shape, 30, 5)
    dk, dv = _pools(shape, 20, 6)
    si = np.array([3, 30, 7, 9, -1], dtype=np.int32)
    di = np.array([0, 1, 20, 4, 5], dtype=np.int32)
    gdk, gdv = dev(dk), dev(dv)
    pa.copy_blocks(shape, dev(sk), dev(sv), gdk, gdv, dev(si), dev(di))
    with pytest.raises(pa.PagedAttnError) as e:
        pa.check_device_error()
    assert e.value.code == pa.ERR_BAD_INDEX
    ok = np.array([0, 3])
    ek, ev = oracle.copy_blocks(bits(sk), bits(sv), bits(dk), bits(dv), si[ok], di[ok])
    assert np.array_equal(bits(gdk), ek) and np.array_equal(bits(gdv), ev)
