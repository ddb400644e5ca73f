"""Pins for the fp64 oracle: checks against things other than itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with
what the mathematics or a library routine fixes.  They are collected as tests
in test_oracle_pins.py and re-run against deliberately broken copies of the
oracle in test_oracle_mutations.py (each broken copy must fail one of them).

The library routine is torch's ``scaled_dot_product_attention`` in float64 on
the CPU, applied to keys/values laid out densely in their original token
order (no paging involved), with KV head h // G repeated for query head h.
"""
from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from paged_kv_cache_continuous_gb300 import workload as wl

GOLDEN = Path(__file__).resolve().parent / "golden"


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sdpa_rows(q, k, v, mask=None):
    """q [n, Hq, d], k/v [L, Hkv, d] (bf16 tensors) -> float64 [n, Hq, d] via torch SDPA."""
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    qf = q.to(torch.float64).permute(1, 0, 2)[None]
    kf = k.to(torch.float64).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vf = v.to(torch.float64).repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(qf, kf, vf, attn_mask=mask)
    return o[0].permute(1, 0, 2).numpy()


def bottom_right_causal(n: int, L: int) -> torch.Tensor:
    """Row i (absolute position L - n + i) may see keys 0 .. L - n + i."""
    i = torch.arange(n)[:, None]
    j = torch.arange(L)[None, :]
    return j <= (L - n + i)


def _tiny_after_steps():
    shape, kp, vp, pre, dec, full = wl.tiny()
    kp1, vp1 = oracle.kv_append(bits(pre.k_new), bits(pre.v_new), pre.slot_mapping, bits(kp), bits(vp))
    kp2, vp2 = oracle.kv_append(bits(dec.k_new), bits(dec.v_new), dec.slot_mapping, kp1, vp1)
    return shape, (kp, vp), (kp1, vp1), (kp2, vp2), pre, dec, full


def _token_rows(pre, dec, s):
    """Original token order of sequence s: its prompt rows then its decode row."""
    a, b = int(pre.q_start_loc[s]), int(pre.q_start_loc[s + 1])
    k = torch.cat([pre.k_new[a:b], dec.k_new[s:s + 1]])
    v = torch.cat([pre.v_new[a:b], dec.v_new[s:s + 1]])
    return k, v


# ---------------------------------------------------------------------------
# Library-routine pins (dense, unpaged, original token order)
# ---------------------------------------------------------------------------

def pin_decode_vs_sdpa():
    shape, _, _, (kp2, vp2), pre, dec, _ = _tiny_after_steps()
    out = oracle.decode(bits(dec.q), kp2, vp2, dec.block_table, dec.seq_lens)
    for s in range(dec.num_seqs):
        k, v = _token_rows(pre, dec, s)
        ref = sdpa_rows(dec.q[s:s + 1], k, v)[0]
        np.testing.assert_allclose(out[s], ref, rtol=0, atol=1e-12)


def pin_prefill_dense_vs_sdpa():
    shape, _, _, _, pre, dec, full = _tiny_after_steps()
    out = oracle.prefill(bits(full.q), bits(full.k_new), bits(full.v_new), full.q_start_loc)
    for s in range(full.num_seqs):
        a, b = int(full.q_start_loc[s]), int(full.q_start_loc[s + 1])
        n = b - a
        ref = sdpa_rows(full.q[a:b], full.k_new[a:b], full.v_new[a:b], bottom_right_causal(n, n))
        np.testing.assert_allclose(out[a:b], ref, rtol=0, atol=1e-12)


def pin_prefill_paged_vs_sdpa():
    """Prompt rows read through the block table after their append."""
    shape, _, (kp1, vp1), _, pre, dec, _ = _tiny_after_steps()
    out = oracle.prefill(bits(pre.q), kp1, vp1, pre.q_start_loc, block_table=pre.block_table)
    for s in range(pre.num_seqs):
        a, b = int(pre.q_start_loc[s]), int(pre.q_start_loc[s + 1])
        n = b - a
        ref = sdpa_rows(pre.q[a:b], pre.k_new[a:b], pre.v_new[a:b], bottom_right_causal(n, n))
        np.testing.assert_allclose(out[a:b], ref, rtol=0, atol=1e-12)


def pin_chunked_prefill_vs_sdpa():
    """A 70-token sequence whose first 29 tokens are cached (prefix) and whose
    last 41 arrive as one chunk: rows of the chunk must equal the last 41 rows
    of full causal attention (bottom-right alignment)."""
    shape = wl.Shape(num_q_heads=6, num_kv_heads=3, head_dim=32, block_size=16, num_blocks=12)
    g = torch.Generator().manual_seed(11)
    alloc = wl.BlockAllocator(shape.num_blocks, shape.block_size,
                              torch.randperm(shape.num_blocks, generator=g).tolist())
    first = wl.make_step(alloc, shape, [0], [29], [29], 0, g)
    chunk = wl.make_step(alloc, shape, [0], [41], [70], 0, g)
    kp, vp = wl.new_pool(shape, 5)
    kp, vp = oracle.kv_append(bits(first.k_new), bits(first.v_new), first.slot_mapping, bits(kp), bits(vp))
    kp, vp = oracle.kv_append(bits(chunk.k_new), bits(chunk.v_new), chunk.slot_mapping, kp, vp)
    out = oracle.prefill(bits(chunk.q), kp, vp, chunk.q_start_loc, prefix_lens=[29],
                         block_table=chunk.block_table)
    k = torch.cat([first.k_new, chunk.k_new])
    v = torch.cat([first.v_new, chunk.v_new])
    ref = sdpa_rows(chunk.q, k, v, bottom_right_causal(41, 70))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Layout contract and indexing
# ---------------------------------------------------------------------------

def pin_append_layout():
    """Token i with slot (blk*B + off) lands at pool[blk, h, off, :] for every
    KV head h, K and V kept apart; every other element keeps its bits; slot -1
    is skipped."""
    N, H, B, d = 5, 3, 4, 8
    rng = np.random.default_rng(3)
    kp = rng.integers(0, 2 ** 16, size=(N, H, B, d), dtype=np.uint16)
    vp = rng.integers(0, 2 ** 16, size=(N, H, B, d), dtype=np.uint16)
    kn = rng.integers(0, 2 ** 16, size=(4, H, d), dtype=np.uint16)
    vn = rng.integers(0, 2 ** 16, size=(4, H, d), dtype=np.uint16)
    slots = np.array([2 * B + 1, -1, 4 * B + 3, 0], dtype=np.int32)
    k2, v2 = oracle.kv_append(kn, vn, slots, kp, vp)
    ek, ev = kp.copy(), vp.copy()
    for i, s in enumerate(slots):
        if s < 0:
            continue
        ek[s // B, :, s % B, :] = kn[i]
        ev[s // B, :, s % B, :] = vn[i]
    assert np.array_equal(k2, ek) and np.array_equal(v2, ev)
    # spot values written by hand, independent of the loop above
    assert np.array_equal(k2[2, :, 1, :], kn[0]) and np.array_equal(v2[4, :, 3, :], vn[2])
    assert np.array_equal(k2[1], kp[1]) and np.array_equal(v2[3], vp[3])


def pin_append_errors():
    N, H, B, d = 2, 1, 4, 2
    z = np.zeros((N, H, B, d), dtype=np.uint16)
    kn = np.ones((2, H, d), dtype=np.uint16)
    for slots, err in (([1, 1], "duplicate"), ([0, N * B], "range")):
        try:
            oracle.kv_append(kn, kn, np.array(slots, dtype=np.int32), z, z)
        except oracle.OracleError as e:
            assert err in str(e)
        else:
            raise AssertionError(f"slots {slots} accepted")


def pin_expected_slots_vs_allocator():
    """The oracle's slot formula against the allocator's own bookkeeping."""
    for st in (wl.tiny()[3], wl.tiny()[4], wl.mixed(num_decode=6, num_prompts=3,
                                                    prompt_range=(20, 70), prefill_budget=200)[3]):
        exp = oracle.expected_slots(st.q_start_loc, st.seq_lens, st.block_table, st.shape.block_size)
        assert np.array_equal(exp, st.slot_mapping)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

def _single_seq_pool(L, d=16, H=2, G=2, B=4, seed=0, kfn=None, vfn=None, qfn=None):
    """Pool holding one sequence of L tokens in shuffled blocks; returns
    (q bits [1,Hq,d], kp, vp, bt, lens, k_rows, v_rows) with k_rows/v_rows
    float64 [L, H, d] in token order (values are exact bf16)."""
    nb = -(-L // B)
    N = nb + 3
    rng = np.random.default_rng(seed)
    perm = rng.permutation(N)[:nb]
    k = torch.randn(L, H, d, generator=torch.Generator().manual_seed(seed)).to(torch.bfloat16)
    v = torch.randn(L, H, d, generator=torch.Generator().manual_seed(seed + 1)).to(torch.bfloat16)
    q = torch.randn(1, H * G, d, generator=torch.Generator().manual_seed(seed + 2)).to(torch.bfloat16)
    if kfn: k = kfn(k)
    if vfn: v = vfn(v)
    if qfn: q = qfn(q, k)
    kp = np.zeros((N, H, B, d), dtype=np.uint16)
    vp = np.zeros((N, H, B, d), dtype=np.uint16)
    slots = np.array([perm[j // B] * B + j % B for j in range(L)], dtype=np.int32)
    kp, vp = oracle.kv_append(bits(k), bits(v), slots, kp, vp)
    bt = np.full((1, nb + 2), -1, dtype=np.int32)
    bt[0, :nb] = perm
    return bits(q), kp, vp, bt, np.array([L], dtype=np.int32), k.double().numpy(), v.double().numpy()


def pin_constant_v():
    c = torch.tensor([0.5, -1.25, 3.0, 0.0] * 4, dtype=torch.bfloat16)
    q, kp, vp, bt, lens, _, _ = _single_seq_pool(37, vfn=lambda v: c.expand_as(v).clone())
    out = oracle.decode(q, kp, vp, bt, lens)
    np.testing.assert_allclose(out[0], np.broadcast_to(c.double().numpy(), out[0].shape),
                               rtol=0, atol=1e-14)


def pin_one_token_context():
    q, kp, vp, bt, lens, _, v = _single_seq_pool(1)
    out = oracle.decode(q, kp, vp, bt, lens)
    G = out.shape[1] // v.shape[1]
    for h in range(out.shape[1]):
        assert np.array_equal(out[0, h], v[0, h // G])


def pin_zero_query_is_mean():
    q, kp, vp, bt, lens, _, v = _single_seq_pool(23, qfn=lambda q, k: torch.zeros_like(q))
    out = oracle.decode(q, kp, vp, bt, lens)
    G = out.shape[1] // v.shape[1]
    for h in range(out.shape[1]):
        np.testing.assert_allclose(out[0, h], v[:, h // G].mean(axis=0), rtol=0, atol=1e-13)


def pin_dominant_key():
    """q = alpha * k_j with alpha large: the weight of key j -> 1, out -> v_j."""
    j = 9

    def kfn(k):
        k = k.clone()
        k[:, :, :] = k[:, :, :] * 0.05  # all keys small ...
        k[j] = torch.sign(k[j]) * 1.0    # ... except key j, a +-1 vector
        return k.to(torch.bfloat16)

    def qfn(q, k):
        return (k[j].repeat_interleave(2, dim=0)[None] * 64.0).to(torch.bfloat16)

    q, kp, vp, bt, lens, _, v = _single_seq_pool(20, kfn=kfn, qfn=qfn)
    out = oracle.decode(q, kp, vp, bt, lens)
    for h in range(out.shape[1]):
        np.testing.assert_allclose(out[0, h], v[j, h // 2], rtol=0, atol=1e-9)


def pin_two_key_golden():
    """Hand-derived values (tests/golden/two_key_softmax.json)."""
    gd = json.loads((GOLDEN / "two_key_softmax.json").read_text())
    d = gd["head_dim"]
    to_bits = lambda a: bits(torch.tensor(a, dtype=torch.float32).to(torch.bfloat16))
    q = to_bits(gd["q"])[None, None, :]
    k = to_bits(gd["k"])[:, None, :]
    v = to_bits(gd["v"])[:, None, :]
    kp = np.zeros((1, 1, 2, d), dtype=np.uint16)
    vp = np.zeros((1, 1, 2, d), dtype=np.uint16)
    kp, vp = oracle.kv_append(k, v, np.array([0, 1], dtype=np.int32), kp, vp)
    out = oracle.decode(q, kp, vp, np.array([[0]], dtype=np.int32), np.array([2], dtype=np.int32))
    np.testing.assert_allclose(out[0, 0], gd["out"], rtol=0, atol=1e-15)
    # explicit scale override: scale 1 doubles the logit gap to 2
    out1 = oracle.decode(q, kp, vp, np.array([[0]], dtype=np.int32), np.array([2], dtype=np.int32),
                         scale=1.0)
    np.testing.assert_allclose(out1[0, 0], gd["out_scale_1"], rtol=0, atol=1e-15)


# ---------------------------------------------------------------------------
# Invariants
# ---------------------------------------------------------------------------

def pin_block_permutation_invariance():
    """(a) Relabelling physical blocks (pool and tables together) leaves every
    output bit-identical."""
    shape, _, _, (kp2, vp2), pre, dec, _ = _tiny_after_steps()
    out = oracle.decode(bits(dec.q), kp2, vp2, dec.block_table, dec.seq_lens)
    perm = np.random.default_rng(9).permutation(shape.num_blocks)  # new id of old block b
    kq, vq = np.empty_like(kp2), np.empty_like(vp2)
    kq[perm], vq[perm] = kp2, vp2
    bt = dec.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    out2 = oracle.decode(bits(dec.q), kq, vq, bt, dec.seq_lens)
    assert np.array_equal(out, out2)


def pin_decode_equals_prefill_row():
    """(d) Decode of token t equals row t of causal prefill over the same
    sequence (the full sequences are prefilled again in fresh blocks)."""
    shape, _, _, (kp2, vp2), pre, dec, full = _tiny_after_steps()
    dout = oracle.decode(bits(dec.q), kp2, vp2, dec.block_table, dec.seq_lens)
    kp3, vp3 = oracle.kv_append(bits(full.k_new), bits(full.v_new), full.slot_mapping, kp2, vp2)
    pout = oracle.prefill(bits(full.q), kp3, vp3, full.q_start_loc, block_table=full.block_table)
    for s in range(dec.num_seqs):
        last = int(full.q_start_loc[s + 1]) - 1
        np.testing.assert_allclose(dout[s], pout[last], rtol=0, atol=1e-13)


def pin_mixed_step_composition():
    """mixed_step = append, then decode rows and prefill rows, on a step that
    holds both (3 decode sequences, 2 prompts): each row equals SDPA over the
    sequence's tokens in original order."""
    shape = wl.Shape(num_q_heads=4, num_kv_heads=2, head_dim=16, block_size=4, num_blocks=40)
    g = torch.Generator().manual_seed(21)
    alloc = wl.BlockAllocator(shape.num_blocks, shape.block_size,
                              torch.randperm(shape.num_blocks, generator=g).tolist())
    hist = wl.make_step(alloc, shape, [0, 1, 2], [7, 13, 2], [7, 13, 2], 0, g)
    kp, vp = wl.new_pool(shape, 77)
    kp, vp = oracle.kv_append(bits(hist.k_new), bits(hist.v_new), hist.slot_mapping, bits(kp), bits(vp))
    st = wl.make_step(alloc, shape, [0, 1, 2, 3, 4], [1, 1, 1, 9, 5], [8, 14, 3, 9, 5], 3, g)
    out, kq, vq = oracle.mixed_step(bits(st.q), bits(st.k_new), bits(st.v_new), st.q_start_loc,
                                    st.seq_lens, st.slot_mapping, st.block_table, st.num_decode,
                                    kp, vp)
    for s in range(5):
        a, b = int(st.q_start_loc[s]), int(st.q_start_loc[s + 1])
        if s < 3:
            ha, hb = int(hist.q_start_loc[s]), int(hist.q_start_loc[s + 1])
            k = torch.cat([hist.k_new[ha:hb], st.k_new[a:b]])
            v = torch.cat([hist.v_new[ha:hb], st.v_new[a:b]])
        else:
            k, v = st.k_new[a:b], st.v_new[a:b]
        ref = sdpa_rows(st.q[a:b], k, v, bottom_right_causal(b - a, k.shape[0]))
        np.testing.assert_allclose(out[a:b], ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# Whole-block copies (fork, migration, swap)
# ---------------------------------------------------------------------------

def _fork_case():
    """One 23-token sequence (B = 4: 6 blocks) in a 24-block pool; the 6
    lowest free block ids receive the copies."""
    shape = wl.Shape(num_q_heads=4, num_kv_heads=2, head_dim=16, block_size=4, num_blocks=24)
    g = torch.Generator().manual_seed(31)
    alloc = wl.BlockAllocator(shape.num_blocks, shape.block_size,
                              torch.randperm(shape.num_blocks, generator=g).tolist())
    st = wl.make_step(alloc, shape, [0], [23], [23], 0, g)
    kp, vp = wl.new_pool(shape, 99)
    kp, vp = oracle.kv_append(bits(st.k_new), bits(st.v_new), st.slot_mapping, bits(kp), bits(vp))
    src = st.block_table[0, :6].astype(np.int32)
    dst = np.array([b for b in range(shape.num_blocks) if b not in set(src.tolist())][:6], dtype=np.int32)
    q = wl.bf16_randn((1, 4, 16), g)
    return shape, st, kp, vp, src, dst, q


def pin_copy_blocks_fork_vs_sdpa():
    """A sequence forked by copying its blocks inside the pool and pointing a
    second table at the copies: decode over the fork equals SDPA over the
    sequence's tokens in original order, the source blocks are untouched and
    decode over the original table is unchanged."""
    shape, st, kp, vp, src, dst, q = _fork_case()
    kf, vf = oracle.copy_blocks(kp, vp, kp, vp, src, dst)
    assert np.array_equal(kf[src], kp[src]) and np.array_equal(vf[src], vp[src])
    bt2 = st.block_table.copy()
    bt2[0, :6] = dst
    lens = np.array([23], dtype=np.int32)
    out_fork = oracle.decode(bits(q), kf, vf, bt2, lens)
    ref = sdpa_rows(q, st.k_new, st.v_new)
    np.testing.assert_allclose(out_fork, ref, rtol=0, atol=1e-12)
    assert np.array_equal(out_fork, oracle.decode(bits(q), kf, vf, st.block_table, lens))


def pin_copy_blocks_swap_round_trip():
    """Swap out to a 10-block host pool and back into other device blocks: the
    host pool holds token t of the sequence at [t // B][h][t % B] (the layout
    written as numpy indexing), and decode through the swapped-in blocks equals
    decode through the originals bit for bit."""
    shape, st, kp, vp, src, dst, q = _fork_case()
    zk = np.zeros((10,) + kp.shape[1:], dtype=np.uint16)
    kh, vh = oracle.copy_blocks(kp, vp, zk, zk.copy(), src, np.arange(6, dtype=np.int32))
    kn, vn = bits(st.k_new), bits(st.v_new)
    for t in range(23):
        assert np.array_equal(kh[t // 4, :, t % 4], kn[t]) and np.array_equal(vh[t // 4, :, t % 4], vn[t])
    assert not kh[6:].any() and not vh[6:].any()
    kd, vd = oracle.copy_blocks(kh, vh, kp, vp, np.arange(6, dtype=np.int32), dst)
    bt2 = st.block_table.copy()
    bt2[0, :6] = dst
    lens = np.array([23], dtype=np.int32)
    assert np.array_equal(oracle.decode(bits(q), kd, vd, bt2, lens),
                          oracle.decode(bits(q), kp, vp, st.block_table, lens))


def pin_copy_blocks_errors():
    """Ids outside either pool and a destination that is also a source (same
    pool) are rejected."""
    shape, st, kp, vp, src, dst, q = _fork_case()
    for bad_src, bad_dst in ((np.array([24], np.int32), np.array([0], np.int32)),
                             (np.array([-1], np.int32), np.array([0], np.int32)),
                             (np.array([0], np.int32), np.array([24], np.int32))):
        try:
            oracle.copy_blocks(kp, vp, kp.copy(), vp.copy(), bad_src, bad_dst)
        except ValueError:
            continue
        raise AssertionError("out-of-range block id accepted")
    try:
        oracle.copy_blocks(kp, vp, kp, vp, src[:2], np.array([src[1], dst[0]], dtype=np.int32))
    except ValueError:
        return
    raise AssertionError("overlapping source and destination accepted")


# ---------------------------------------------------------------------------
# Rotary position embedding (RoFormer; Llama / GPT-NeoX pairing) and bf16 rounding
# ---------------------------------------------------------------------------

def _rope_case(seed, T=5, H=3, d=16):
    g = torch.Generator().manual_seed(seed)
    x = wl.bf16_randn((T, H, d), g)
    pos = np.array([0, 1, 7, 1000, 32767][:T], dtype=np.int32)
    return bits(x), pos


def _f64(b):
    """bf16 bit patterns -> float64 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_rope_identity_at_position_zero():
    """Position 0 rotates by nothing: the result is the input, exactly."""
    xb, _ = _rope_case(1)
    out = oracle.rope(xb, np.zeros(xb.shape[0], dtype=np.int32))
    assert np.array_equal(out, _f64(xb))


def pin_rope_is_complex_rotation():
    """Pair (i, i + d/2) as the complex number x_i + j x_{i+d/2}: the embedding
    multiplies it by exp(j p theta^(-2i/d)) (numpy complex arithmetic)."""
    xb, pos = _rope_case(2)
    T, H, d = xb.shape
    x = _f64(xb)
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    ang = pos[:, None].astype(np.float64) * np.power(10000.0, -np.arange(half) * 2.0 / d)[None, :]
    w = z * np.exp(1j * ang)[:, None, :]
    ref = np.concatenate([w.real, w.imag], axis=-1)
    np.testing.assert_allclose(oracle.rope(xb, pos), ref, rtol=0, atol=1e-12)


def pin_rope_relative_position():
    """The defining property: <R(m) q, R(n) k> depends on m - n only."""
    g = torch.Generator().manual_seed(3)
    q, k = bits(wl.bf16_randn((1, 1, 64), g)), bits(wl.bf16_randn((1, 1, 64), g))
    dots = []
    for shift in (0, 5, 1234):
        qr = oracle.rope(q, np.array([17 + shift], np.int32))
        kr = oracle.rope(k, np.array([9 + shift], np.int32))
        dots.append(float((qr * kr).sum()))
    assert max(dots) - min(dots) < 1e-9, dots


def pin_to_bf16_rounding():
    """Round to nearest, ties to the even significand: every value is checked
    against the nearest of all bf16 numbers near it, in exact rational
    arithmetic (brute force)."""
    from fractions import Fraction
    vals = [1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8 + 2.0 ** -20), 3.14159, 1e-30,
            -7.5e5, 2.0 ** -126 * 1.5, 0.0, 255.5, 256.5]
    got = oracle.to_bf16(np.array(vals))
    for v, b in zip(vals, got):
        if v == 0.0:
            assert b == 0
            continue
        fv = abs(Fraction(v))
        e = fv.numerator.bit_length() - fv.denominator.bit_length()
        # candidates m * 2^(ee - 7), significand m in [128, 256)
        cands = [(Fraction(m) * Fraction(2) ** (ee - 7), m) for ee in range(e - 2, e + 3) for m in range(128, 256)]
        dist = min(abs(c - fv) for c, _ in cands)
        near = [(c, m) for c, m in cands if abs(c - fv) == dist]
        best = near[0][0] if len(near) == 1 else [c for c, m in near if m % 2 == 0][0]
        want = int(np.float32(float(best)).view(np.uint32)) >> 16 | (0x8000 if v < 0 else 0)
        assert int(b) == want, (v, hex(int(b)), hex(want))


def pin_rope_append_pool():
    """The pool receives the rotated keys rounded to bf16 and the values bit
    for bit; the rotated queries are returned unrounded."""
    shape = wl.Shape(num_q_heads=4, num_kv_heads=2, head_dim=16, block_size=4, num_blocks=8)
    g = torch.Generator().manual_seed(4)
    q, k, v = (bits(wl.bf16_randn((3, h, 16), g)) for h in (4, 2, 2))
    kp, vp = wl.new_pool(shape, 5)
    slots = np.array([5, 0, 13], np.int32)
    pos = np.array([2, 3, 40], np.int32)
    q_rot, k_rot, kp2, vp2 = oracle.rope_append(q, k, v, pos, slots, bits(kp), bits(vp))
    np.testing.assert_allclose(q_rot, oracle.rope(q, pos), rtol=0, atol=0)
    for i, sl in enumerate(slots):
        assert np.array_equal(kp2[sl // 4, :, sl % 4], oracle.to_bf16(k_rot[i]))
        assert np.array_equal(vp2[sl // 4, :, sl % 4], v[i])


# ---------------------------------------------------------------------------
# fp8 (e4m3) KV cache: one scale per KV head
# ---------------------------------------------------------------------------

def pin_e4m3_codes_match_torch():
    """Every e4m3 code decodes as torch's float8_e4m3fn does; float32 values
    in range encode as torch rounds them (nearest, ties to even); beyond 448
    the code saturates."""
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_to_double(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])
    g = torch.Generator().manual_seed(8)
    x = torch.cat([(torch.randn(20000, generator=g) * 40).clamp(-447, 447),
                   torch.randn(2000, generator=g) * 1e-3])
    assert np.array_equal(oracle.e4m3_from_float(x.numpy()), x.to(torch.float8_e4m3fn).view(torch.uint8).numpy())
    assert list(oracle.e4m3_from_float(np.array([1e4, -1e4, 449.0], np.float32))) == [0x7e, 0xfe, 0x7e]


def _fp8_case(seed):
    shape = wl.Shape(num_q_heads=8, num_kv_heads=2, head_dim=16, block_size=4, num_blocks=12)
    g = torch.Generator().manual_seed(seed)
    alloc = wl.BlockAllocator(shape.num_blocks, shape.block_size,
                              torch.randperm(shape.num_blocks, generator=g).tolist())
    st = wl.make_step(alloc, shape, [0, 1], [21, 9], [21, 9], 0, g)
    ks = np.array([0.05, 0.02], np.float32)
    vs = np.array([0.03, 0.07], np.float32)
    kp0 = np.random.default_rng(seed).integers(0, 126, size=(12, 2, 4, 16)).astype(np.uint8)
    vp0 = np.random.default_rng(seed + 1).integers(0, 126, size=(12, 2, 4, 16)).astype(np.uint8)
    return shape, st, ks, vs, kp0, vp0


def pin_kv_append_fp8_codes():
    """A key element x of KV head h lands as the e4m3 code of float(x) / scale[h]
    (torch's float32 division and float8 cast); untouched bytes keep theirs."""
    shape, st, ks, vs, kp0, vp0 = _fp8_case(12)
    kp, vp = oracle.kv_append_fp8(bits(st.k_new), bits(st.v_new), st.slot_mapping, ks, vs, kp0, vp0)
    kq = (st.k_new.float() / torch.from_numpy(ks)[None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    vq = (st.v_new.float() / torch.from_numpy(vs)[None, :, None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    touched = np.zeros(kp.shape[0] * 4, dtype=bool)
    for i, sl in enumerate(st.slot_mapping):
        assert np.array_equal(kp[sl // 4, :, sl % 4], kq[i]) and np.array_equal(vp[sl // 4, :, sl % 4], vq[i])
        touched[sl] = True
    keep = ~np.repeat(touched.reshape(-1, 4)[:, None, :, None], 2, axis=1).repeat(16, axis=3)
    assert np.array_equal(kp[keep], kp0[keep]) and np.array_equal(vp[keep], vp0[keep])


def pin_decode_fp8_vs_sdpa():
    """Decode over fp8 pools equals torch's float64 SDPA over the dequantized
    keys and values (code * scale), gathered in token order."""
    shape, st, ks, vs, kp0, vp0 = _fp8_case(13)
    kp, vp = oracle.kv_append_fp8(bits(st.k_new), bits(st.v_new), st.slot_mapping, ks, vs, kp0, vp0)
    g = torch.Generator().manual_seed(14)
    q = wl.bf16_randn((2, 8, 16), g)
    lens = np.array([21, 9], np.int32)
    out = oracle.decode_fp8(bits(q), kp, vp, ks, vs, st.block_table, lens)
    deq = lambda pool, sc: torch.from_numpy(pool).view(torch.float8_e4m3fn).double() * torch.from_numpy(sc).double()[None, :, None, None]
    kd, vd = deq(kp, ks), deq(vp, vs)
    for s_, L in enumerate(lens):
        idx = [(int(st.block_table[s_, j // 4]), j % 4) for j in range(L)]
        K = torch.stack([kd[b, :, o] for b, o in idx])  # [L, Hkv, d]
        V = torch.stack([vd[b, :, o] for b, o in idx])
        Kx = K.repeat_interleave(4, dim=1).permute(1, 0, 2)
        Vx = V.repeat_interleave(4, dim=1).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(q[s_].double()[:, None, :], Kx, Vx)[:, 0, :]
        np.testing.assert_allclose(out[s_], ref.numpy(), rtol=0, atol=1e-12)


ALL_PINS = [
    pin_decode_vs_sdpa, pin_prefill_dense_vs_sdpa, pin_prefill_paged_vs_sdpa,
    pin_chunked_prefill_vs_sdpa, pin_append_layout, pin_append_errors,
    pin_expected_slots_vs_allocator, pin_constant_v, pin_one_token_context,
    pin_zero_query_is_mean, pin_dominant_key, pin_two_key_golden,
    pin_block_permutation_invariance, pin_decode_equals_prefill_row,
    pin_mixed_step_composition, pin_copy_blocks_fork_vs_sdpa, pin_copy_blocks_swap_round_trip,
    pin_copy_blocks_errors, pin_rope_identity_at_position_zero, pin_rope_is_complex_rotation,
    pin_rope_relative_position, pin_to_bf16_rounding, pin_rope_append_pool,
    pin_e4m3_codes_match_torch, pin_kv_append_fp8_codes, pin_decode_fp8_vs_sdpa,
]
