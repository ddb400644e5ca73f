"""Rotary embedding fused with the KV append on the GPU against the oracle:
rotated values within one bf16 unit in the last place of the fp64 oracle's
(+ 2^-20 absolute: the GPU rotates in fp32, then rounds to bf16),
values and untouched pool slots bit-exact, attention over the rotated inputs
within the attention tolerance."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits, dev
from paged_kv_cache_continuous_gb300 import binding as pa
from paged_kv_cache_continuous_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _f64(b):
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _within_ulp(gpu_bits, ref, what):
    """Within one bf16 ulp of the fp64 value, plus 2^-20 absolute: the kernel
    rotates in fp32, and x cos - y sin of inputs of size ~1 that nearly cancel
    carries fp32's absolute error (~1e-7) into a result far smaller than 1."""
    g = _f64(gpu_bits)
    mag = np.maximum(np.abs(ref), 2.0 ** -126)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    bad = np.abs(g - ref) > ulp + 2.0 ** -20
    assert not bad.any(), f"{what}: {int(bad.sum())} values off by more than one bf16 ulp, max {np.abs(g - ref).max():.3g}"


def _case(seed, T, Hq, Hkv, d, B, positions):
    g = torch.Generator().manual_seed(seed)
    nb = T + 4
    shape = wl.Shape(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B, num_blocks=nb)
    q, k, v = wl.bf16_randn((T, Hq, d), g), wl.bf16_randn((T, Hkv, d), g), wl.bf16_randn((T, Hkv, d), g)
    perm = torch.randperm(nb * B, generator=g)[:T].to(torch.int32).numpy()
    slots = perm.copy()
    slots[1::7] = -1  # some tokens are not appended
    kp, vp = wl.new_pool(shape, seed + 1)
    return shape, q, k, v, np.asarray(positions, dtype=np.int32), slots, kp, vp


@pytest.mark.parametrize("Hq,Hkv,d,B", [(32, 8, 128, 16), (4, 2, 64, 32), (12, 12, 128, 32)])
def test_rope_append_matches_oracle(cuda_lib, Hq, Hkv, d, B):
    T = 50
    rng = np.random.default_rng(Hq)
    pos = rng.integers(0, 40000, size=T)
    pos[:4] = [0, 1, 2, 32767]
    shape, q, k, v, pos, slots, kp, vp = _case(Hq + d, T, Hq, Hkv, d, B, pos)
    kd, vd = dev(kp), dev(vp)
    q_out = pa.rope_append(shape, dev(q), dev(k), dev(v), dev(pos), dev(slots), kd, vd)
    pa.check_device_error()
    q_rot, k_rot, ek, ev = oracle.rope_append(bits(q), bits(k), bits(v), pos, slots, bits(kp), bits(vp))
    _within_ulp(bits(q_out), q_rot, "q")
    gk, gv = bits(kd), bits(vd)
    assert np.array_equal(gv, ev), "values must be copied bit for bit"
    written = np.zeros(gk.shape[0] * B, dtype=bool)
    for i, sl in enumerate(slots):
        if sl < 0:
            continue
        written[sl] = True
        _within_ulp(gk[sl // B, :, sl % B], k_rot[i], f"k of token {i}")
    mask = np.repeat(~written.reshape(-1, B)[:, None, :, None], Hkv, axis=1).repeat(d, axis=3)
    assert np.array_equal(gk[mask], ek[mask]), "slots not appended to must be untouched"


def test_rope_in_place_and_then_decode(cuda_lib):
    """q rotated in place; decode over the rotated pool equals the oracle's
    decode over its own rotated (bf16-rounded) queries and keys."""
    g = torch.Generator().manual_seed(9)
    shape = wl.Shape(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16, num_blocks=200)
    alloc = wl.BlockAllocator(shape.num_blocks, shape.block_size,
                              torch.randperm(shape.num_blocks, generator=g).tolist())
    lens = [300, 1, 57, 1024]
    pre = wl.make_step(alloc, shape, [0, 1, 2, 3], lens, lens, 0, g)
    kp, vp = wl.new_pool(shape, 3)
    pos = np.concatenate([np.arange(L) for L in lens]).astype(np.int32)
    kd, vd = dev(kp), dev(vp)
    qd = dev(pre.q)
    pa.rope_append(shape, qd, dev(pre.k_new), dev(pre.v_new), dev(pos), dev(pre.slot_mapping), kd, vd, q_out=qd)
    # decode: the last token of every sequence attends over the whole sequence
    last = np.cumsum(lens) - 1
    qdec = qd[torch.as_tensor(last, device=qd.device)].contiguous()
    out = pa.decode(shape, qdec, kd, vd, dev(pre.block_table), dev(np.array(lens, np.int32)), max(lens))
    pa.check_device_error()
    q_rot, k_rot, ek, ev = oracle.rope_append(bits(pre.q), bits(pre.k_new), bits(pre.v_new), pos,
                                              pre.slot_mapping, bits(kp), bits(vp))
    qref = oracle.to_bf16(q_rot[last])
    ref = oracle.decode(qref, ek, ev, pre.block_table, np.array(lens, np.int32))
    assert_close(out, ref, "decode after rope")
    # prefill over the same rotated data
    pout = pa.prefill(shape, qd, kd, vd, dev(pre.q_start_loc), max(lens), block_table=dev(pre.block_table))
    pa.check_device_error()
    rows = np.sort(np.random.default_rng(0).choice(int(sum(lens)), 64, replace=False))
    pairs = np.array([(r, h) for r in rows for h in range(shape.num_q_heads)], dtype=np.int32)
    pref = oracle.prefill(oracle.to_bf16(q_rot), ek, ev, pre.q_start_loc, block_table=pre.block_table, pairs=pairs)
    got = pout[torch.as_tensor(pairs[:, 0], device=pout.device).long(), torch.as_tensor(pairs[:, 1], device=pout.device).long()]
    assert_close(got, pref, "prefill after rope")


def test_rope_bad_position_flags_error(cuda_lib):
    shape, q, k, v, pos, slots, kp, vp = _case(5, 8, 4, 2, 64, 16, np.arange(8))
    pos[3] = -2
    kd, vd = dev(kp), dev(vp)
    q_out = pa.rope_append(shape, dev(q), dev(k), dev(v), dev(pos), dev(slots), kd, vd)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.check_device_error()
    assert e.value.code == pa.ERR_BAD_INDEX
    ok = np.array([i for i in range(8) if i != 3])
    q_rot = oracle.rope(bits(q)[ok], pos[ok])
    _within_ulp(bits(q_out)[ok], q_rot, "q of the valid tokens")
