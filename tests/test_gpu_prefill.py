"""tcgen05 causal prefill (dense and paged, with prefixes) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_appended, assert_close, bits, compact_pool, dev, prefill_spread, sample
from paged_kv_cache_continuous_gb300 import binding as pa
from paged_kv_cache_continuous_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _dense_case(seed, lens, Hq, Hkv, d):
    g = torch.Generator().manual_seed(seed)
    T = sum(lens)
    shape = wl.Shape(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=16, num_blocks=1)
    q = wl.bf16_randn((T, Hq, d), g)
    k = wl.bf16_randn((T, Hkv, d), g)
    v = wl.bf16_randn((T, Hkv, d), g)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    return shape, q, k, v, cu


def test_prefill_dense_tiny(cuda_lib):
    shape, _, _, _, _, full = wl.tiny()
    out = pa.prefill(shape, dev(full.q), dev(full.k_new), dev(full.v_new), dev(full.q_start_loc),
                     full.max_q_len)
    pa.check_device_error()
    ref = oracle.prefill(bits(full.q), bits(full.k_new), bits(full.v_new), full.q_start_loc)
    assert_close(out, ref, "tiny dense prefill")


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (16, 16, 128), (8, 4, 128), (24, 8, 128), (16, 2, 64)])
def test_prefill_dense_ragged(cuda_lib, Hq, Hkv, d):
    lens = [1, 7, 127, 128, 129, 300, 513]
    shape, q, k, v, cu = _dense_case(21, lens, Hq, Hkv, d)
    out = pa.prefill(shape, dev(q), dev(k), dev(v), dev(cu), max(lens))
    pa.check_device_error()
    ref = oracle.prefill(bits(q), bits(k), bits(v), cu)
    assert_close(out, ref, f"dense ragged Hq={Hq} Hkv={Hkv} d={d}")


@pytest.mark.parametrize("slope", [1.0, 0.1, -0.1])
def test_prefill_growing_scores(cuda_lib, slope):
    """Scores that grow (or shrink) steadily along the keys: q . k_j ~ 8 slope j.
    slope 1 moves every row's running maximum by ~2^130 per 128-key tile, 0.1 by
    ~2^13 (a move past 2^64 every few tiles), -0.1 keeps the first key the
    largest -- the paths where the kernel moves its running maximum and
    rescales O.  V ~ N(0,1) as everywhere else.  With weights halving per
    key at slope 1, an output is dominated by a few values: its bf16 rounding
    (up to 2^-7 for magnitudes in [2, 4), 2^-6 in [4, 8)) plus the bf16
    rounding of the dominant weights can pass 1e-2.  Such elements are held
    to the bound of that arithmetic (bf16 weights, consistent normalisation,
    bf16 output) computed from their exact softmax weights, and printed."""
    g = torch.Generator().manual_seed(23)
    lens = [1000, 700, 129]
    T, Hq, Hkv, d = sum(lens), 32, 8, 128
    shape = wl.Shape(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=16, num_blocks=1)
    q = (torch.randn(T, Hq, d, generator=g) * 0.1)
    q[:, :, 0] = 8.0
    k = (torch.randn(T, Hkv, d, generator=g) * 0.1)
    pos = torch.cat([torch.arange(L, dtype=torch.float32) for L in lens])
    k[:, :, 0] = slope * pos[:, None]
    v = torch.randn(T, Hkv, d, generator=g)
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    out = pa.prefill(shape, dev(q), dev(k), dev(v), dev(cu), max(lens))
    pa.check_device_error()
    ref = oracle.prefill(bits(q), bits(k), bits(v), cu)
    f64 = lambda t: t.double().numpy()
    assert_close(out, ref, f"growing scores slope={slope}", spread=prefill_spread(f64(q), f64(k), f64(v), cu, ref))


def _paged_case(seed, prefix_and_new, Hq, Hkv, d, B):
    """Sequences with `prefix` cached tokens (already in the pool) and `new`
    prompt rows; the new rows are appended on the GPU first."""
    g = torch.Generator().manual_seed(seed)
    tot = [p + n for p, n in prefix_and_new]
    N = sum(-(-L // B) for L in tot) + 5
    shape = wl.Shape(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=B, num_blocks=N)
    alloc = wl.BlockAllocator(N, B, torch.randperm(N, generator=g).tolist())
    st = wl.make_step(alloc, shape, list(range(len(tot))), [n for _, n in prefix_and_new], tot, 0, g,
                      width=max(-(-L // B) for L in tot) + 2)
    kp, vp = wl.new_pool(shape, seed + 500)
    return shape, kp, vp, st, np.array([p for p, _ in prefix_and_new], dtype=np.int32)


@pytest.mark.parametrize("Hq,Hkv,d,B", [(32, 8, 128, 16), (32, 8, 128, 32), (16, 8, 128, 16), (12, 12, 128, 32),
                                         (8, 8, 64, 16), (64, 8, 128, 16)])
def test_prefill_paged_with_prefix(cuda_lib, Hq, Hkv, d, B):
    case = [(0, 1), (5, 200), (130, 129), (1000, 64), (17, 300), (0, 256)]
    shape, kp, vp, st, pre = _paged_case(22, case, Hq, Hkv, d, B)
    kd, vd = dev(kp), dev(vp)
    pa.kv_append(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kd, vd)
    out = pa.prefill(shape, dev(st.q), kd, vd, dev(st.q_start_loc), st.max_q_len,
                     prefix_lens=dev(pre), block_table=dev(st.block_table))
    pa.check_device_error()
    kq, vq = oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, bits(kp), bits(vp))
    ref = oracle.prefill(bits(st.q), kq, vq, st.q_start_loc, prefix_lens=pre, block_table=st.block_table)
    assert_close(out, ref, f"paged prefill Hq={Hq} Hkv={Hkv} d={d} B={B}")


@pytest.mark.parametrize("pairs", [1, 3])
@pytest.mark.parametrize("Hq,Hkv", [(24, 8), (32, 8), (16, 16), (16, 8)])
def test_prefill_few_pairs(cuda_lib, pairs, Hq, Hkv):
    """One or three CTA pairs: every pair walks dozens of work units in turn,
    most with idle sub-tiles (short prompts), so each hand-off between
    consecutive units -- a Q buffer reused two units later, the K/V ring,
    output staging, the last V tile's tail -- is crossed many times in one
    launch.  Idle warps that ran ahead once freed a Q buffer still in use."""
    lens = [1, 7, 127, 128, 129, 300, 513, 40, 1000, 65]
    shape, q, k, v, cu = _dense_case(29, lens, Hq, Hkv, 128)
    pa.set_prefill_pairs(pairs)
    try:
        out = pa.prefill(shape, dev(q), dev(k), dev(v), dev(cu), max(lens))
        pa.check_device_error()
    finally:
        pa.set_prefill_pairs(0)
    ref = oracle.prefill(bits(q), bits(k), bits(v), cu)
    assert_close(out, ref, f"dense prefill on {pairs} pair(s) Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("pairs", [1, 2])
def test_prefill_paged_few_pairs(cuda_lib, pairs):
    case = [(0, 1), (5, 200), (130, 129), (1000, 64), (17, 300), (0, 256), (64, 3), (0, 700)]
    shape, kp, vp, st, pre = _paged_case(24, case, 24, 8, 128, 16)
    kd, vd = dev(kp), dev(vp)
    pa.kv_append(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kd, vd)
    pa.set_prefill_pairs(pairs)
    try:
        out = pa.prefill(shape, dev(st.q), kd, vd, dev(st.q_start_loc), st.max_q_len,
                         prefix_lens=dev(pre), block_table=dev(st.block_table))
        pa.check_device_error()
    finally:
        pa.set_prefill_pairs(0)
    kq, vq = oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, bits(kp), bits(vp))
    ref = oracle.prefill(bits(st.q), kq, vq, st.q_start_loc, prefix_lens=pre, block_table=st.block_table)
    assert_close(out, ref, f"paged prefill on {pairs} pair(s)")


def test_decode_equals_last_prefill_row(cuda_lib):
    """(d) decode of token t equals row t of causal prefill over the sequence."""
    shape, kp, vp, pre, dec, full = wl.tiny()
    kd, vd = dev(kp), dev(vp)
    for st in (pre, dec, full):
        pa.kv_append(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kd, vd)
    dout = pa.decode(shape, dev(dec.q), kd, vd, dev(dec.block_table), dev(dec.seq_lens), dec.max_seq_len)
    pout = pa.prefill(shape, dev(full.q), kd, vd, dev(full.q_start_loc), full.max_q_len,
                      block_table=dev(full.block_table))
    pa.check_device_error()
    last = torch.tensor(full.q_start_loc[1:] - 1)
    diff = (dout.float() - pout[last.cuda()].float()).abs().max().item()
    assert diff <= 1e-2


def test_prefill_bad_block_flags_error(cuda_lib):
    shape, kp, vp, st, pre = _paged_case(23, [(10, 100), (0, 50)], 8, 2, 128, 16)
    bt = st.block_table.copy()
    bt[0, 3] = -7
    kd, vd = dev(kp), dev(vp)
    pa.prefill(shape, dev(st.q), kd, vd, dev(st.q_start_loc), st.max_q_len, prefix_lens=dev(pre),
               block_table=dev(bt))
    with pytest.raises(pa.PagedAttnError) as e:
        pa.check_device_error()
    assert e.value.code == pa.ERR_BAD_INDEX


@pytest.mark.parametrize("prompts", [[1024] * 4, [4096]], ids=["4x1024", "1x4096"])
def test_prefill_full_size_sampled(cuda_lib, prompts):
    shape, kp, vp, st = wl.prefill_only(40 + len(prompts), prompts, pool_device="cuda")
    kd, vd = kp, vp
    kh, vh = bits(kd), bits(vd)  # the drawn initial pools, before the GPU append
    pa.kv_append(shape, dev(st.k_new), dev(st.v_new), dev(st.slot_mapping), kd, vd)
    out = pa.prefill(shape, dev(st.q), kd, vd, dev(st.q_start_loc), st.max_q_len,
                     block_table=dev(st.block_table))
    pa.check_device_error()
    assert_appended(kd, vd, st, shape.block_size, f"prefill {prompts}")
    oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, kh, vh, inplace=True)
    assert np.array_equal(bits(kd), kh) and np.array_equal(bits(vd), vh), "pools after the append"
    rng = np.random.default_rng(2)
    rows = np.concatenate([sample(rng, st.num_tokens, 40), st.q_start_loc[1:] - 1, st.q_start_loc[:-1]])
    pairs = np.array([(int(r), int(h)) for r in rows for h in rng.choice(shape.num_q_heads, 3, replace=False)],
                     dtype=np.int32)
    kc, vc, bt = compact_pool(kh, vh, st.block_table, st.seq_lens, range(st.num_seqs), shape.block_size)
    ref = oracle.prefill(bits(st.q), kc, vc, st.q_start_loc, block_table=bt, pairs=pairs)
    got = out[torch.tensor(pairs[:, 0]), torch.tensor(pairs[:, 1])]
    assert_close(got, ref, f"prefill {prompts}")
