"""The mixed continuous-batching step and the 64-step churn on the GPU,
checked against the oracle at every step."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits, compact_pool, dev, sample
from paged_kv_cache_continuous_gb300 import binding as pa
from paged_kv_cache_continuous_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _mixed_gpu(shape, st, kd, vd, ws=None):
    return pa.mixed_step(shape, dev(st.q), dev(st.k_new), dev(st.v_new), dev(st.q_start_loc),
                         dev(st.seq_lens), dev(st.slot_mapping), dev(st.block_table), st.num_decode,
                         st.max_seq_len, st.max_q_len, kd, vd, ws=ws)


def test_tiny_three_steps(cuda_lib):
    """Prefill {5,17,33,64}, one decode token each, then the full sequences in
    fresh blocks: pools bit-exact and outputs within tolerance at every step."""
    shape, kp, vp, pre, dec, full = wl.tiny()
    kd, vd = dev(kp), dev(vp)
    kh, vh = bits(kp), bits(vp)
    for st in (pre, dec, full):
        out = _mixed_gpu(shape, st, kd, vd)
        pa.check_device_error()
        ref, kh, vh = oracle.mixed_step(bits(st.q), bits(st.k_new), bits(st.v_new), st.q_start_loc,
                                        st.seq_lens, st.slot_mapping, st.block_table, st.num_decode, kh, vh)
        assert np.array_equal(bits(kd), kh) and np.array_equal(bits(vd), vh)
        assert_close(out, ref, f"tiny step num_decode={st.num_decode}")


def test_mixed_small_all_rows(cuda_lib):
    shape, kp, vp, st = wl.mixed(seed=33, num_decode=20, num_prompts=5, prompt_range=(1, 300),
                                 prefill_budget=900, max_context=700)
    kd, vd = dev(kp), dev(vp)
    out = _mixed_gpu(shape, st, kd, vd)
    pa.check_device_error()
    ref, kh, vh = oracle.mixed_step(bits(st.q), bits(st.k_new), bits(st.v_new), st.q_start_loc, st.seq_lens,
                                    st.slot_mapping, st.block_table, st.num_decode, bits(kp), bits(vp))
    assert np.array_equal(bits(kd), kh) and np.array_equal(bits(vd), vh)
    assert_close(out, ref, "mixed small")


def _sampled_step_check(shape, st, out, kd, vd, rng, what, host_pool=None):
    """Sampled decode pairs and prefill rows of one step vs the oracle."""
    nd = st.num_decode
    H = shape.num_q_heads
    if host_pool is None:
        seqs = np.unique(np.concatenate([sample(rng, nd, 8), nd + sample(rng, st.num_seqs - nd, 4)]))
        kc, vc, bt = compact_pool(kd, vd, st.block_table, st.seq_lens, seqs, shape.block_size)
    else:
        seqs = np.unique(np.concatenate([sample(rng, nd, 8), nd + sample(rng, st.num_seqs - nd, 4)]))
        kc, vc = host_pool
        bt = st.block_table[seqs]
    dec = seqs[seqs < nd]
    if len(dec):
        i = np.arange(len(dec))
        pairs = np.array([(int(j), int(h)) for j in i for h in rng.choice(H, 3, replace=False)], dtype=np.int32)
        ref = oracle.decode(bits(st.q)[dec], kc, vc, bt[: len(dec)], st.seq_lens[dec], pairs=pairs)
        got = out[torch.tensor(dec[pairs[:, 0]]), torch.tensor(pairs[:, 1])]
        assert_close(got, ref, what + " decode rows")
    pf = seqs[seqs >= nd]
    if len(pf):
        qs = st.q_start_loc
        n = qs[pf + 1] - qs[pf]
        cu = np.zeros(len(pf) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(n)
        rows_idx = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in pf])
        local = []
        for j, s in enumerate(pf):
            for r in {0, int(n[j]) - 1, int(rng.integers(0, n[j]))}:
                local += [(int(cu[j] + r), int(h)) for h in rng.choice(H, 2, replace=False)]
        pairs = np.array(local, dtype=np.int32)
        ref = oracle.prefill(bits(st.q)[rows_idx], kc, vc, cu, prefix_lens=st.seq_lens[pf] - n,
                             block_table=bt[len(dec):], pairs=pairs)
        got = out[torch.tensor(rows_idx[pairs[:, 0]]), torch.tensor(pairs[:, 1])]
        assert_close(got, ref, what + " prefill rows")


def test_mixed_full_size(cuda_lib):
    """120 decode sequences + 8 prompts (<= 4096 rows), Hq 32 / Hkv 8."""
    shape, kp, vp, st = wl.mixed()
    kd, vd = dev(kp), dev(vp)
    out = _mixed_gpu(shape, st, kd, vd)
    pa.check_device_error()
    kh, vh = oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, bits(kp), bits(vp))
    assert np.array_equal(bits(kd), kh) and np.array_equal(bits(vd), vh)
    _sampled_step_check(shape, st, out, kd, vd, np.random.default_rng(4), "mixed full", host_pool=(kh, vh))


def test_churn_64_steps(cuda_lib):
    """512 sequences, log-uniform contexts, B = 32; 10 % replaced by prompts
    each step.  Every step: the rows written at the step's slots and sampled
    outputs vs the oracle; the whole pools bit-exact at three steps."""
    ch = wl.Churn(pool_device="cuda")
    shape = ch.shape
    kd, vd = ch.initial_pool()
    kh, vh = bits(kd), bits(vd)  # the oracle's host mirror of the pools
    rng = np.random.default_rng(5)
    ws = pa.workspace(shape, 512, 8192 + 80)
    for step in range(ch.steps):
        st = ch.step()
        out = _mixed_gpu(shape, st, kd, vd, ws)
        pa.check_device_error()
        oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, kh, vh, inplace=True)
        sl = torch.tensor(st.slot_mapping, dtype=torch.long, device="cuda")
        blk, off = sl // shape.block_size, sl % shape.block_size
        for pool, new in ((kd, st.k_new), (vd, st.v_new)):
            got = pool[blk, :, off, :].cpu()
            assert torch.equal(got, new), f"step {step}: appended rows differ"
        _sampled_step_check(shape, st, out, kd, vd, rng, f"churn step {step}", host_pool=(kh, vh))
        if step in (0, 31, ch.steps - 1):
            assert np.array_equal(bits(kd), kh) and np.array_equal(bits(vd), vh), f"pool differs at {step}"


@pytest.mark.parametrize("pairs", [1, 7, "planned", 75, 76, 1000])
def test_mixed_split_small(cuda_lib, pairs):
    """pa_mixed_step_split at several prefill pair counts (76 and above: no
    room left for the decode, so the step runs unsplit): pools bit-exact,
    every output row within tolerance of the oracle, prefill rows bit-exact
    with the unsplit step's."""
    shape, kp, vp, st = wl.mixed(seed=34, num_decode=24, num_prompts=5, prompt_range=(1, 400),
                                 prefill_budget=1200, max_context=900)
    nd = st.num_decode
    if pairs == "planned":
        rows = np.diff(st.q_start_loc)[nd:]
        pairs = pa.mixed_prefill_pairs(shape, st.seq_lens[:nd], rows, st.seq_lens[nd:] - rows)
        assert pairs >= 1
    kd, vd = dev(kp), dev(vp)
    args = (shape, dev(st.q), dev(st.k_new), dev(st.v_new), dev(st.q_start_loc), dev(st.seq_lens),
            dev(st.slot_mapping), dev(st.block_table), nd, st.max_seq_len, st.max_q_len)
    out = pa.mixed_step(*args, kd, vd, prefill_pairs=pairs)
    pa.check_device_error()
    ref, kh, vh = oracle.mixed_step(bits(st.q), bits(st.k_new), bits(st.v_new), st.q_start_loc, st.seq_lens,
                                    st.slot_mapping, st.block_table, nd, bits(kp), bits(vp))
    assert np.array_equal(bits(kd), kh) and np.array_equal(bits(vd), vh)
    assert_close(out, ref, f"mixed split {pairs}")
    kd2, vd2 = dev(kp), dev(vp)
    out2 = pa.mixed_step(*args, kd2, vd2)
    pa.check_device_error()
    r0 = int(st.q_start_loc[nd])
    assert torch.equal(out[r0:], out2[r0:]), "prefill rows differ from the unsplit step"


def test_mixed_split_full_size_planned(cuda_lib):
    """The 120-decode + 8-prompt step on the planned partition: pools
    bit-exact, sampled outputs vs the oracle."""
    shape, kp, vp, st = wl.mixed()
    nd = st.num_decode
    rows = np.diff(st.q_start_loc)[nd:]
    pairs = pa.mixed_prefill_pairs(shape, st.seq_lens[:nd], rows, st.seq_lens[nd:] - rows)
    assert 1 <= pairs < torch.cuda.get_device_properties(0).multi_processor_count // 2
    kd, vd = dev(kp), dev(vp)
    out = pa.mixed_step(shape, dev(st.q), dev(st.k_new), dev(st.v_new), dev(st.q_start_loc), dev(st.seq_lens),
                        dev(st.slot_mapping), dev(st.block_table), nd, st.max_seq_len, st.max_q_len, kd, vd,
                        prefill_pairs=pairs)
    pa.check_device_error()
    kh, vh = oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, bits(kp), bits(vp))
    assert np.array_equal(bits(kd), kh) and np.array_equal(bits(vd), vh)
    _sampled_step_check(shape, st, out, kd, vd, np.random.default_rng(6), "mixed split full", host_pool=(kh, vh))


def test_mixed_split_decode_rows_bitexact(cuda_lib):
    """With the decode split fixed, the partitioned step's decode rows equal
    the undivided step's bit for bit: the decode grid differs (fewer CTAs)
    but an item's result does not depend on the CTA that runs it."""
    shape, kp, vp, st = wl.mixed(seed=35, num_decode=40, num_prompts=4, prompt_range=(100, 500),
                                 prefill_budget=1600, max_context=1500)
    nd = st.num_decode
    args = (shape, dev(st.q), dev(st.k_new), dev(st.v_new), dev(st.q_start_loc), dev(st.seq_lens),
            dev(st.slot_mapping), dev(st.block_table), nd, st.max_seq_len, st.max_q_len)
    pa.set_decode_split(256)
    try:
        kd, vd = dev(kp), dev(vp)
        out1 = pa.mixed_step(*args, kd, vd, prefill_pairs=20)
        kd2, vd2 = dev(kp), dev(vp)
        out2 = pa.mixed_step(*args, kd2, vd2)
        pa.check_device_error()
    finally:
        pa.set_decode_split(0)
    assert torch.equal(out1, out2)
