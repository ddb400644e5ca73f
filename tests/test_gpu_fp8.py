"""fp8 (e4m3) KV cache on the GPU against the oracle: the quantising append
bit-exact (the code is an integer decision, taken in float on both sides),
decode over fp8 pools within the attention tolerance."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits, dev
from paged_kv_cache_continuous_gb300 import binding as pa
from paged_kv_cache_continuous_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _scales(Hkv, seed):
    rng = np.random.default_rng(seed)
    return (rng.uniform(0.01, 0.03, Hkv).astype(np.float32), rng.uniform(0.01, 0.03, Hkv).astype(np.float32))


def _case(seed, lens, Hq, Hkv, B, d=128):
    g = torch.Generator().manual_seed(seed)
    N = sum(-(-L // B) for L in lens) + 5
    shape = wl.Shape(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B, num_blocks=N)
    alloc = wl.BlockAllocator(N, B, torch.randperm(N, generator=g).tolist())
    st = wl.make_step(alloc, shape, list(range(len(lens))), list(lens), list(lens), 0, g,
                      width=max(-(-L // B) for L in lens) + 2)
    rng = np.random.default_rng(seed)
    kp0 = rng.integers(0, 126, size=(N, Hkv, B, d)).astype(np.uint8)  # stale codes (finite)
    vp0 = rng.integers(0, 126, size=(N, Hkv, B, d)).astype(np.uint8)
    q = wl.bf16_randn((len(lens), Hq, d), g)
    return shape, st, kp0, vp0, q


@pytest.mark.parametrize("Hq,Hkv,B,d", [(32, 8, 16, 128), (32, 32, 16, 128), (64, 4, 32, 128), (64, 8, 16, 128),
                                        (16, 8, 32, 128), (40, 8, 16, 128), (24, 8, 32, 128),
                                        (32, 8, 16, 64), (32, 32, 32, 64), (64, 4, 16, 64), (24, 8, 16, 64)])
def test_fp8_append_and_decode(cuda_lib, Hq, Hkv, B, d):
    lens = [1, 15, 16, 17, 255, 700, 2049]
    shape, st, kp0, vp0, q = _case(Hq + B + d, lens, Hq, Hkv, B, d)
    ks, vs = _scales(Hkv, Hq)
    kd, vd = dev(kp0), dev(vp0)
    pa.kv_append_fp8(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), dev(ks), dev(vs), kd, vd)
    pa.check_device_error()
    ek, ev = oracle.kv_append_fp8(bits(st.k_new), bits(st.v_new), st.slot_mapping, ks, vs, kp0, vp0)
    assert np.array_equal(kd.cpu().numpy(), ek) and np.array_equal(vd.cpu().numpy(), ev), "pools differ"
    lens_a = np.array(lens, np.int32)
    out = pa.decode_fp8(shape, dev(q), kd, vd, dev(ks), dev(vs), dev(st.block_table), dev(lens_a), max(lens))
    pa.check_device_error()
    ref = oracle.decode_fp8(bits(q), ek, ev, ks, vs, st.block_table, lens_a)
    assert_close(out, ref, f"fp8 decode Hq={Hq} Hkv={Hkv} B={B} d={d}")


@pytest.mark.parametrize("d", [128, 64])
def test_fp8_decode_split_vs_single(cuda_lib, d):
    """Split-K over fp8 pools agrees with one split (merge path)."""
    lens = [3000, 64, 1234]
    shape, st, kp0, vp0, q = _case(3, lens, 32, 8, 16, d)
    ks, vs = _scales(8, 4)
    kd, vd = dev(kp0), dev(vp0)
    pa.kv_append_fp8(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), dev(ks), dev(vs), kd, vd)
    args = (shape, dev(q), kd, vd, dev(ks), dev(vs), dev(st.block_table), dev(np.array(lens, np.int32)), max(lens))
    pa.set_decode_split(256)
    try:
        a = pa.decode_fp8(*args)
    finally:
        pa.set_decode_split(4096)
    try:
        b = pa.decode_fp8(*args)
    finally:
        pa.set_decode_split(0)
    pa.check_device_error()
    assert (a.float() - b.float()).abs().max().item() <= 1e-2


def test_fp8_append_bad_slot_flags_error(cuda_lib):
    shape, st, kp0, vp0, q = _case(7, [40], 8, 2, 16)
    ks, vs = _scales(2, 7)
    slots = st.slot_mapping.copy()
    slots[3] = shape.num_blocks * shape.block_size
    kd, vd = dev(kp0), dev(vp0)
    pa.kv_append_fp8(shape, dev(st.k_new), dev(st.v_new), dev(slots), dev(ks), dev(vs), kd, vd)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.check_device_error()
    assert e.value.code == pa.ERR_BAD_INDEX
    slots_ok = slots.copy()
    slots_ok[3] = -1
    ek, ev = oracle.kv_append_fp8(bits(st.k_new), bits(st.v_new), slots_ok, ks, vs, kp0, vp0)
    assert np.array_equal(kd.cpu().numpy(), ek) and np.array_equal(vd.cpu().numpy(), ev)
