"""KV append on the GPU against the oracle: pool contents bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import bits, dev
from paged_kv_cache_continuous_gb300 import binding as pa
from paged_kv_cache_continuous_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _append_and_compare(shape, kp, vp, step, slots=None):
    slots = step.slot_mapping if slots is None else slots
    kd, vd = dev(kp), dev(vp)
    pa.kv_append(shape, dev(step.k_new), dev(step.v_new), dev(slots), kd, vd)
    pa.check_device_error()
    ek, ev = oracle.kv_append(bits(step.k_new), bits(step.v_new), slots, bits(kp), bits(vp))
    assert np.array_equal(bits(kd), ek) and np.array_equal(bits(vd), ev)
    return kd, vd


def test_append_tiny_prefill_then_decode(cuda_lib):
    shape, kp, vp, pre, dec, _ = wl.tiny()
    kd, vd = _append_and_compare(shape, kp, vp, pre)
    _append_and_compare(shape, kd.cpu(), vd.cpu(), dec)


def test_append_padding_slots_skipped(cuda_lib):
    shape, kp, vp, pre, _, _ = wl.tiny()
    slots = pre.slot_mapping.copy()
    slots[::3] = -1
    _append_and_compare(shape, kp, vp, pre, slots)


@pytest.mark.parametrize("B", [16, 32])
def test_append_mixed_batch_full_size(cuda_lib, B):
    """The mixed-step batch (120 decode rows + 8 prompts, up to 4216 rows, 8 KV
    heads, d 128), and the same with 32-token blocks."""
    if B == 16:
        shape, kp, vp, st = wl.mixed()
    else:
        shape, kp, vp, st = wl.prefill_only(31, [300, 17, 1, 64, 129], block_size=32)
    _append_and_compare(shape, kp, vp, st)


def test_append_out_of_range_slot_flags_error(cuda_lib):
    shape, kp, vp, pre, _, _ = wl.tiny()
    slots = pre.slot_mapping.copy()
    slots[5] = shape.num_blocks * shape.block_size  # one past the pool
    kd, vd = dev(kp), dev(vp)
    pa.kv_append(shape, dev(pre.k_new), dev(pre.v_new), dev(slots), kd, vd)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.check_device_error()
    assert e.value.code == pa.ERR_BAD_INDEX
    # every other row still landed, nothing else was touched
    slots_ok = slots.copy()
    slots_ok[5] = -1
    ek, ev = oracle.kv_append(bits(pre.k_new), bits(pre.v_new), slots_ok, bits(kp), bits(vp))
    assert np.array_equal(bits(kd), ek) and np.array_equal(bits(vd), ev)
    pa.check_device_error()  # the word was cleared


def test_append_is_idempotent(cuda_lib):
    shape, kp, vp, pre, _, _ = wl.tiny()
    kd, vd = _append_and_compare(shape, kp, vp, pre)
    k1, v1 = kd.clone(), vd.clone()
    pa.kv_append(shape, dev(pre.k_new), dev(pre.v_new), dev(pre.slot_mapping), kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(kd, k1) and torch.equal(vd, v1)
