"""Split-K GQA decode on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_appended, assert_close, bits, compact_pool, dev, sample
from paged_kv_cache_continuous_gb300 import binding as pa
from paged_kv_cache_continuous_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _decode_gpu(shape, kd, vd, st, max_len=None):
    return pa.decode(shape, dev(st.q), kd, vd, dev(st.block_table), dev(st.seq_lens),
                     max_len or st.max_seq_len)


def _append_gpu(shape, kp, vp, st):
    kd, vd = dev(kp), dev(vp)
    pa.kv_append(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kd, vd)
    return kd, vd


def _ragged(seed, lens, Hq, Hkv, d, B, stale="fill"):
    g = torch.Generator().manual_seed(seed)
    lens = [int(x) for x in lens]
    N = sum(-(-L // B) for L in lens) + 7
    shape = wl.Shape(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B, num_blocks=N)
    alloc = wl.BlockAllocator(N, B, torch.randperm(N, generator=g).tolist())
    sg = np.random.default_rng(seed) if stale == "junk" else None
    st = wl.make_step(alloc, shape, list(range(len(lens))), [1] * len(lens), lens, len(lens), g,
                      width=max(-(-L // B) for L in lens) + 3, stale_gen=sg)
    kp, vp = wl.new_pool(shape, seed + 1000)
    return shape, kp, vp, st


def _check_full(shape, kp, vp, st, what, split=0):
    pa.set_decode_split(split)
    try:
        kd, vd = _append_gpu(shape, kp, vp, st)
        out = _decode_gpu(shape, kd, vd, st)
        pa.check_device_error()
    finally:
        pa.set_decode_split(0)
    kq, vq = oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, bits(kp), bits(vp))
    ref = oracle.decode(bits(st.q), kq, vq, st.block_table, st.seq_lens)
    assert_close(out, ref, what)
    return out, kd, vd


def test_decode_tiny(cuda_lib):
    shape, kp, vp, pre, dec, _ = wl.tiny()
    kd, vd = _append_gpu(shape, kp, vp, pre)
    kq, vq = oracle.kv_append(bits(pre.k_new), bits(pre.v_new), pre.slot_mapping, bits(kp), bits(vp))
    _check_full(shape, kd.cpu(), vd.cpu(), dec, "tiny decode")


LENS = [1, 15, 16, 17, 255, 256, 257, 700, 1500, 2049]


@pytest.mark.parametrize("Hq,Hkv,d,B", [
    (32, 32, 128, 16),   # G = 1 (Llama-7B heads)
    (32, 8, 128, 16),    # G = 4
    (64, 8, 128, 16),    # G = 8 (70B-shaped)
    (32, 2, 128, 32),    # G = 16, 32-token blocks
    (8, 4, 64, 16),      # d = 64
    (12, 4, 64, 32),     # G = 3, d = 64, B = 32
])
@pytest.mark.parametrize("split", [0, 64])
def test_decode_ragged(cuda_lib, Hq, Hkv, d, B, split):
    shape, kp, vp, st = _ragged(7, LENS, Hq, Hkv, d, B)
    _check_full(shape, kp, vp, st, f"G={Hq // Hkv} d={d} B={B} split={split}", split)


@pytest.mark.parametrize("Hq,Hkv,d,B", [(32, 8, 128, 16), (64, 8, 128, 32), (8, 8, 64, 16)])
def test_short_last_split_joins(cuda_lib, Hq, Hkv, d, B):
    """With 256-token splits, a last split of at most 32 tokens joins the one
    before (lengths k * 256 + 1 .. + 32), one of 33 or more is an item of its
    own; every case, merged or not, against the oracle."""
    lens = [257, 256 + 32, 256 + 33, 512 + 1, 512 + 16, 512 + 32, 512 + 33, 3 * 256 + 1, 256, 33]
    shape, kp, vp, st = _ragged(12, lens, Hq, Hkv, d, B)
    _check_full(shape, kp, vp, st, f"joined last split G={Hq // Hkv} d={d} B={B}", 256)


def test_split_and_unsplit_agree(cuda_lib):
    shape, kp, vp, st = _ragged(8, [3000, 900, 64], 32, 8, 128, 16)
    outs = []
    for split in (4096, 256, 16):
        pa.set_decode_split(split)
        kd, vd = _append_gpu(shape, kp, vp, st)
        outs.append(_decode_gpu(shape, kd, vd, st).float())
    pa.set_decode_split(0)
    # Different splits move the running maximum, so the bf16 rounding of the
    # weights (relative 2^-9) differs between them: they agree to far better
    # than the oracle tolerance, but not bit for bit.
    for o in outs[1:]:
        d = (o - outs[0]).abs()
        assert d.max().item() <= 4e-3 and d.mean().item() <= 2e-4


def test_stale_table_entries_never_read(cuda_lib):
    shape, kp, vp, st = _ragged(9, LENS, 32, 8, 128, 16, stale="junk")
    _check_full(shape, kp, vp, st, "junk past the last block")


def test_block_permutation_invariance(cuda_lib):
    """(a) relabelling physical blocks leaves the output bit-identical."""
    shape, kp, vp, st = _ragged(10, LENS, 32, 8, 128, 16)
    out, kd, vd = _check_full(shape, kp, vp, st, "before relabel")
    perm = torch.randperm(shape.num_blocks, generator=torch.Generator().manual_seed(3))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(shape.num_blocks)
    kq, vq = torch.empty_like(kd), torch.empty_like(vd)
    kq[perm.cuda()] = kd
    vq[perm.cuda()] = vd
    bt = st.block_table.copy()
    m = bt >= 0
    bt[m] = perm.numpy()[bt[m]]
    out2 = pa.decode(shape, dev(st.q), kq, vq, dev(bt), dev(st.seq_lens), st.max_seq_len)
    assert torch.equal(out, out2)


def test_constant_v_and_single_token(cuda_lib):
    """(b) constant V -> that constant (to within one bf16 rounding step);
    (c) a one-token context -> exactly its V row."""
    shape, kp, vp, st = _ragged(11, [1, 40, 1, 333], 16, 4, 128, 16)
    c = torch.randn(128, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    st_c = wl.Step(**{**st.__dict__, "v_new": c.expand_as(st.v_new).clone()})
    kd, vd = _append_gpu(shape, kp, c.expand_as(vp).clone(), st_c)
    out = _decode_gpu(shape, kd, vd, st_c).float().cpu()
    cf = c.float().expand(16, 128)
    assert torch.all((out[[1, 3]] - cf).abs() <= cf.abs() * 2 ** -8), "constant V"
    out, _, _ = _check_full(shape, kp, vp, st, "one-token rows")
    out = out.cpu()
    for s in (0, 2):
        for h in range(16):
            assert torch.equal(out[s, h], st.v_new[s, h // 4]), "one-token context"


def test_empty_context_gives_zeros(cuda_lib):
    shape, kp, vp, st = _ragged(12, [5, 7], 8, 2, 128, 16)
    lens = np.array([0, 7], dtype=np.int32)
    kd, vd = dev(kp), dev(vp)
    out = pa.decode(shape, dev(st.q), kd, vd, dev(st.block_table), dev(lens), 7)
    pa.check_device_error()
    assert torch.all(out[0] == 0)


def test_bad_block_id_flags_error(cuda_lib):
    shape, kp, vp, st = _ragged(13, [40, 70], 8, 2, 128, 16)
    bt = st.block_table.copy()
    bt[1, 2] = shape.num_blocks + 5
    kd, vd = dev(kp), dev(vp)
    pa.decode(shape, dev(st.q), kd, vd, dev(bt), dev(st.seq_lens), 70)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.check_device_error()
    assert e.value.code == pa.ERR_BAD_INDEX


def test_validation_mode_skips_work(cuda_lib):
    shape, kp, vp, st = _ragged(14, [40, 70], 8, 2, 128, 16)
    bt = st.block_table.copy()
    bt[0, 1] = -3
    kd, vd = dev(kp), dev(vp)
    out = torch.full((2, 8, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    pa.set_validation(True)
    try:
        pa.decode(shape, dev(st.q), kd, vd, dev(bt), dev(st.seq_lens), 70, out=out)
        with pytest.raises(pa.PagedAttnError):
            pa.check_device_error()
    finally:
        pa.set_validation(False)
    assert torch.all(out == 7.0)


def _sampled_full_size(shape, kp_d, vp_d, st, rng, n_pairs, what):
    """Full-size step: the initial pools are drawn on the device (a seeded
    generator) and copied to the host before the GPU append; the oracle then
    appends on that host mirror, and the whole device pool must equal it bit
    for bit before the oracle decodes sampled (sequence, head) pairs from it."""
    kd, vd = kp_d, vp_d
    kh, vh = bits(kd), bits(vd)
    pa.kv_append(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kd, vd)
    out = _decode_gpu(shape, kd, vd, st)
    pa.check_device_error()
    assert_appended(kd, vd, st, shape.block_size, what)
    oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, kh, vh, inplace=True)
    assert np.array_equal(bits(kd), kh) and np.array_equal(bits(vd), vh), f"{what}: pools after the append"
    S, Hq = st.num_seqs, shape.num_q_heads
    seqs = sample(rng, S, 12)
    kc, vc, bt = compact_pool(kh, vh, st.block_table, st.seq_lens, seqs, shape.block_size)
    pairs = np.array([(i, int(h)) for i in range(len(seqs)) for h in rng.choice(Hq, 4, replace=False)],
                     dtype=np.int32)
    q = bits(st.q)[seqs]
    ref = oracle.decode(q, kc, vc, bt, st.seq_lens[seqs], pairs=pairs)
    got = out[torch.tensor(seqs[pairs[:, 0]]), torch.tensor(pairs[:, 1])]
    assert_close(got, ref, what)


def test_llama7b_decode_full_size_sampled(cuda_lib):
    shape, kp, vp, st = wl.llama7b_decode(pool_device="cuda")
    _sampled_full_size(shape, kp, vp, st, np.random.default_rng(0), 48, "Llama-7B decode")


def test_long_context_full_size_sampled(cuda_lib):
    shape, kp, vp, st = wl.long_context(pool_device="cuda")
    _sampled_full_size(shape, kp, vp, st, np.random.default_rng(1), 48, "32 x 32K decode")


# ------------------------------------------------ decode with fused append --
@pytest.mark.parametrize("Hq,Hkv,d,B", [(32, 32, 128, 16), (32, 8, 128, 16), (64, 8, 128, 16), (32, 2, 128, 32),
                                         (8, 4, 64, 16), (12, 4, 64, 32)])
@pytest.mark.parametrize("split", [0, 64])
def test_decode_append_matches_oracle(cuda_lib, Hq, Hkv, d, B, split):
    """pa_decode_append = pa_kv_append of the step's rows, then pa_decode:
    the pools bit for bit against the oracle's append, the outputs against
    the oracle's decode over those pools."""
    shape, kp, vp, st = _ragged(15, LENS, Hq, Hkv, d, B)
    kd, vd = dev(kp), dev(vp)
    pa.set_decode_split(split)
    try:
        out = pa.decode_append(shape, dev(st.q), dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kd, vd,
                               dev(st.block_table), dev(st.seq_lens), st.max_seq_len)
        pa.check_device_error()
    finally:
        pa.set_decode_split(0)
    kq, vq = oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, bits(kp), bits(vp))
    assert np.array_equal(bits(kd), kq) and np.array_equal(bits(vd), vq), "pools after the fused append"
    ref = oracle.decode(bits(st.q), kq, vq, st.block_table, st.seq_lens)
    assert_close(out, ref, f"decode_append G={Hq // Hkv} d={d} B={B} split={split}")


def test_decode_append_padding_and_bad_slot(cuda_lib):
    """Padding slots (< 0) write nothing; a slot past the pool is skipped and
    flagged, every other row still lands and decodes."""
    shape, kp, vp, st = _ragged(16, [40, 1, 300, 77], 16, 4, 128, 16)
    slots = st.slot_mapping.copy()
    slots[1] = -1
    kd, vd = dev(kp), dev(vp)
    pa.decode_append(shape, dev(st.q), dev(st.k_new), dev(st.v_new), dev(slots), kd, vd,
                     dev(st.block_table), dev(st.seq_lens), st.max_seq_len)
    pa.check_device_error()
    kq, vq = oracle.kv_append(bits(st.k_new), bits(st.v_new), slots, bits(kp), bits(vp))
    assert np.array_equal(bits(kd), kq) and np.array_equal(bits(vd), vq), "padding slot"
    bad = st.slot_mapping.copy()
    bad[2] = shape.num_blocks * shape.block_size + 3
    kd2, vd2 = dev(kp), dev(vp)
    pa.decode_append(shape, dev(st.q), dev(st.k_new), dev(st.v_new), dev(bad), kd2, vd2,
                     dev(st.block_table), dev(st.seq_lens), st.max_seq_len)
    with pytest.raises(pa.PagedAttnError) as e:
        pa.check_device_error()
    assert e.value.code == pa.ERR_BAD_INDEX
    bad[2] = -1
    kq2, vq2 = oracle.kv_append(bits(st.k_new), bits(st.v_new), bad, bits(kp), bits(vp))
    assert np.array_equal(bits(kd2), kq2) and np.array_equal(bits(vd2), vq2), "rows beside a bad slot"


def test_decode_append_is_append_then_decode_for_any_slots(cuda_lib):
    """The rows go in before anything is read, so any distinct slots give
    exactly pa_kv_append + pa_decode: here two sequences' new rows are
    written into each other's last positions (the oracle appends the same)."""
    shape, kp, vp, st = _ragged(17, [40, 70, 5], 8, 2, 128, 16)
    slots = st.slot_mapping.copy()
    slots[0], slots[1] = slots[1], slots[0]
    kd, vd = dev(kp), dev(vp)
    out = pa.decode_append(shape, dev(st.q), dev(st.k_new), dev(st.v_new), dev(slots), kd, vd,
                           dev(st.block_table), dev(st.seq_lens), st.max_seq_len)
    pa.check_device_error()
    kq, vq = oracle.kv_append(bits(st.k_new), bits(st.v_new), slots, bits(kp), bits(vp))
    assert np.array_equal(bits(kd), kq) and np.array_equal(bits(vd), vq)
    ref = oracle.decode(bits(st.q), kq, vq, st.block_table, st.seq_lens)
    assert_close(out, ref, "decode_append with exchanged slots")


def test_decode_append_validation_mode_writes_nothing_on_a_bad_table(cuda_lib):
    shape, kp, vp, st = _ragged(18, [40, 70, 5], 8, 2, 128, 16)
    bt = st.block_table.copy()
    bt[1, 1] = -4
    kd, vd = dev(kp), dev(vp)
    out = torch.full((3, 8, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    pa.set_validation(True)
    try:
        pa.decode_append(shape, dev(st.q), dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kd, vd,
                         dev(bt), dev(st.seq_lens), st.max_seq_len, out=out)
        with pytest.raises(pa.PagedAttnError) as e:
            pa.check_device_error()
    finally:
        pa.set_validation(False)
    assert e.value.code == pa.ERR_BAD_INDEX
    assert torch.all(out == 7.0)
    assert np.array_equal(bits(kd), bits(kp)) and np.array_equal(bits(vd), bits(vp)), "nothing written"


def test_llama7b_decode_append_full_size_sampled(cuda_lib):
    """The bench's step through pa_decode_append at full size: whole pools
    against the oracle's append on a host snapshot, sampled outputs."""
    shape, kd, vd, st = wl.llama7b_decode(pool_device="cuda")
    kh, vh = bits(kd), bits(vd)
    out = pa.decode_append(shape, dev(st.q), dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kd, vd,
                           dev(st.block_table), dev(st.seq_lens), st.max_seq_len)
    pa.check_device_error()
    oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, kh, vh, inplace=True)
    assert np.array_equal(bits(kd), kh) and np.array_equal(bits(vd), vh), "pools after the fused append"
    rng = np.random.default_rng(6)
    seqs = sample(rng, st.num_seqs, 12)
    kc, vc, bt = compact_pool(kh, vh, st.block_table, st.seq_lens, seqs, shape.block_size)
    pairs = np.array([(i, int(h)) for i in range(len(seqs)) for h in rng.choice(32, 4, replace=False)],
                     dtype=np.int32)
    ref = oracle.decode(bits(st.q)[seqs], kc, vc, bt, st.seq_lens[seqs], pairs=pairs)
    got = out[torch.tensor(seqs[pairs[:, 0]]), torch.tensor(pairs[:, 1])]
    assert_close(got, ref, "Llama-7B decode_append")


@pytest.mark.parametrize("split", [0, 64])
def test_decode_bitwise_repeatable(cuda_lib, split):
    """An item's result depends on the item alone (its warps merge by
    item-local role; a split sequence's partials are merged in split order),
    so repeated calls -- whose plans may order equal-length items
    differently -- give the same bits."""
    shape, kp, vp, st = _ragged(13, LENS * 6, 32, 8, 128, 16)
    kd, vd = _append_gpu(shape, kp, vp, st)
    pa.set_decode_split(split)
    try:
        outs = [_decode_gpu(shape, kd, vd, st).clone() for _ in range(5)]
        pa.check_device_error()
    finally:
        pa.set_decode_split(0)
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
