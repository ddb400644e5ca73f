"""Single-kernel cases for profiling (ncu) and quick timing.

    python -m paged_kv_cache_continuous_gb300.profile_cases decode [num_seqs] [llama7b|long]
    python -m paged_kv_cache_continuous_gb300.profile_cases decode_append [num_seqs]
    python -m paged_kv_cache_continuous_gb300.profile_cases prefill 4096 | 1024,1024,1024,1024
    python -m paged_kv_cache_continuous_gb300.profile_cases append [mixed|churn]
    python -m paged_kv_cache_continuous_gb300.profile_cases decode_fp8 [num_seqs]
    python -m paged_kv_cache_continuous_gb300.profile_cases rope [num_tokens]
    python -m paged_kv_cache_continuous_gb300.profile_cases copy [num_pairs]

Each case builds its seeded workload on cuda:0, makes three warm-up calls and
then one more, so `ncu -k regex:<kernel> -s 3 -c 1` captures a warm launch.
"""
from __future__ import annotations

import sys

import numpy as np
import torch

from . import binding as pa
from . import workload as wl


def _d(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda() if isinstance(x, np.ndarray) else x.cuda()


def decode(num_seqs: int = 128, which: str = "llama7b"):
    if which == "long":
        shape, kp, vp, st = wl.long_context(pool_device="cuda", num_seqs=num_seqs)
    else:
        shape, kp, vp, st = wl.llama7b_decode(pool_device="cuda", num_seqs=num_seqs)
    pa.kv_append(shape, _d(st.k_new), _d(st.v_new), _d(st.slot_mapping), kp, vp)
    q, bt, lens = _d(st.q), _d(st.block_table), _d(st.seq_lens)
    ws = pa.workspace(shape, st.num_seqs, st.max_seq_len)
    out = torch.empty_like(q)
    for _ in range(4):
        pa.decode(shape, q, kp, vp, bt, lens, st.max_seq_len, out=out, ws=ws)
    pa.check_device_error()
    split, nsplit = pa.decode_plan(shape, st.num_seqs, st.max_seq_len)
    kv = int(st.seq_lens.astype(np.int64).sum()) * shape.num_kv_heads * shape.head_dim * 4
    print(f"decode {which} seqs={st.num_seqs} split={split} max_splits={nsplit} kv_bytes={kv}")


def decode_append(num_seqs: int = 128):
    """The Llama-7B-shaped decode step with its append fused (the bench's step)."""
    shape, kp, vp, st = wl.llama7b_decode(pool_device="cuda", num_seqs=num_seqs)
    q, kn, vn, sl = _d(st.q), _d(st.k_new), _d(st.v_new), _d(st.slot_mapping)
    bt, lens = _d(st.block_table), _d(st.seq_lens)
    ws = pa.workspace(shape, st.num_seqs, st.max_seq_len)
    out = torch.empty_like(q)
    for _ in range(4):
        pa.decode_append(shape, q, kn, vn, sl, kp, vp, bt, lens, st.max_seq_len, out=out, ws=ws)
    pa.check_device_error()
    print(f"decode_append seqs={st.num_seqs}")


def decode_fp8(num_seqs: int = 128):
    """The Llama-7B-shaped decode step over fp8 (e4m3) pools."""
    shape, _, _, st = wl.llama7b_decode(pool_device=None, num_seqs=num_seqs)
    N, H, B, d = shape.num_blocks, shape.num_kv_heads, shape.block_size, shape.head_dim
    g = torch.Generator(device="cuda").manual_seed(1)
    kp = torch.randint(0, 126, (N, H, B, d), dtype=torch.uint8, device="cuda", generator=g)
    vp = torch.randint(0, 126, (N, H, B, d), dtype=torch.uint8, device="cuda", generator=g)
    ks = torch.full((H,), 0.02, dtype=torch.float32, device="cuda")
    q, bt, lens = _d(st.q), _d(st.block_table), _d(st.seq_lens)
    ws = pa.workspace(shape, st.num_seqs, st.max_seq_len)
    out = torch.empty_like(q)
    for _ in range(4):
        pa.decode_fp8(shape, q, kp, vp, ks, ks, bt, lens, st.max_seq_len, out=out, ws=ws)
    pa.check_device_error()
    print(f"decode_fp8 seqs={st.num_seqs}")


def prefill(prompts):
    shape, kp, vp, st = wl.prefill_only(64, prompts, pool_device="cuda")
    pa.kv_append(shape, _d(st.k_new), _d(st.v_new), _d(st.slot_mapping), kp, vp)
    q, bt, cu = _d(st.q), _d(st.block_table), _d(st.q_start_loc)
    out = torch.empty_like(q)
    for _ in range(4):
        pa.prefill(shape, q, kp, vp, cu, st.max_q_len, block_table=bt, out=out)
    pa.check_device_error()
    print(f"prefill prompts={prompts}")


def append(which: str = "mixed"):
    """The mixed step's rows (3196), or one churn step's (~13.6 K rows, B = 32)."""
    if which == "churn":
        ch = wl.Churn(pool_device="cuda", draw_values=False)
        st = [ch.step() for _ in range(6)][-1]
        shape = ch.shape
        kp, vp = ch.initial_pool()
        g = torch.Generator(device="cuda").manual_seed(3)
        T = st.num_tokens
        kn = torch.randn(T, shape.num_kv_heads, shape.head_dim, generator=g, device="cuda").to(torch.bfloat16)
        vn = torch.randn_like(kn)
        sl = _d(st.slot_mapping)
    else:
        shape, kp, vp, st = wl.mixed(pool_device="cuda")
        kn, vn, sl = _d(st.k_new), _d(st.v_new), _d(st.slot_mapping)
    for _ in range(4):
        pa.kv_append(shape, kn, vn, sl, kp, vp)
    pa.check_device_error()
    print(f"append tokens={st.num_tokens}")


def rope(T: int = 4096, Hq: int = 32, Hkv: int = 8):
    """Rotary embedding fused with the append, the bench's prompt step shape."""
    g = torch.Generator().manual_seed(23)
    nb = T // 16 + 16
    shape = wl.Shape(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, block_size=16, num_blocks=nb)
    q = wl.bf16_randn((T, Hq, 128), g).cuda()
    k, v = wl.bf16_randn((T, Hkv, 128), g).cuda(), wl.bf16_randn((T, Hkv, 128), g).cuda()
    kp = torch.zeros((nb, Hkv, 16, 128), dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    pos = torch.arange(T, dtype=torch.int32, device="cuda")
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int32).cuda()
    q_out = torch.empty_like(q)
    for _ in range(4):
        pa.rope_append(shape, q, k, v, pos, slots, kp, vp, q_out=q_out)
    pa.check_device_error()
    print(f"rope tokens={T} Hq={Hq} Hkv={Hkv}")


def copy(num_pairs: int = 1024):
    """A block fork inside one pool pair (the bench's block shape: 32 KV heads x
    16 tokens x 128 dims, 128 KB per block and pool)."""
    N = 2 * num_pairs
    shape = wl.Shape(num_q_heads=32, num_kv_heads=32, head_dim=128, block_size=16, num_blocks=N)
    kp = torch.empty((N, 32, 16, 128), dtype=torch.bfloat16, device="cuda").normal_()
    vp = torch.empty_like(kp).normal_()
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(17)).to(torch.int32)
    src, dst = perm[:num_pairs].cuda(), perm[num_pairs:].cuda()
    for _ in range(4):
        pa.copy_blocks(shape, kp, vp, kp, vp, src, dst)
    pa.check_device_error()
    print(f"copy pairs={num_pairs} bytes={4 * num_pairs * 32 * 16 * 128 * 2}")


def main(argv):
    pa.load()
    torch.cuda.set_device(0)
    case = argv[1] if len(argv) > 1 else "decode"
    if case == "decode":
        decode(int(argv[2]) if len(argv) > 2 else 128, argv[3] if len(argv) > 3 else "llama7b")
    elif case == "decode_append":
        decode_append(int(argv[2]) if len(argv) > 2 else 128)
    elif case == "prefill":
        prefill([int(x) for x in (argv[2] if len(argv) > 2 else "4096").split(",")])
    elif case == "append":
        append(argv[2] if len(argv) > 2 else "mixed")
    elif case == "decode_fp8":
        decode_fp8(int(argv[2]) if len(argv) > 2 else 128)
    elif case == "rope":
        rope(int(argv[2]) if len(argv) > 2 else 4096)
    elif case == "copy":
        copy(int(argv[2]) if len(argv) > 2 else 1024)
    else:
        raise SystemExit(f"unknown case {case}")


if __name__ == "__main__":
    main(sys.argv)
