"""Shared helpers of the GPU parity tests (device transfer, comparison,
sampling).  Expected values come only from the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle

MAX_ABS = 1e-2   # attention outputs (bf16, fp32 accumulation) vs the fp64 oracle
MEAN_ABS = 1e-3


def dev(x, device="cuda"):
    if isinstance(x, np.ndarray):
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)
    return x.contiguous().to(device)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_close(gpu_bf16: torch.Tensor, ref: np.ndarray, what: str = "",
                 max_abs: float = MAX_ABS, mean_abs: float = MEAN_ABS):
    g = gpu_bf16.detach().float().cpu().double().numpy().reshape(ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= max_abs and mean <= mean_abs, f"{what}: max abs {mx:.3g}, mean abs {mean:.3g}"
    return mx, mean


def compact_pool(k_pool: torch.Tensor, v_pool: torch.Tensor, block_table: np.ndarray,
                 seq_lens: np.ndarray, rows, block_size: int):
    """Host copies of only the blocks that sequences `rows` use, with their
    table rows renumbered to the compact pool (a block relabelling, which
    leaves attention unchanged)."""
    used = []
    for r in rows:
        nb = -(-int(seq_lens[r]) // block_size)
        used += block_table[r, :nb].tolist()
    uniq = sorted(set(used))
    remap = {b: i for i, b in enumerate(uniq)}
    idx = torch.tensor(uniq if uniq else [0], dtype=torch.long, device=k_pool.device)
    kc = bits(k_pool.index_select(0, idx))
    vc = bits(v_pool.index_select(0, idx))
    width = block_table.shape[1]
    bt = np.full((len(rows), width), -1, dtype=np.int32)
    for i, r in enumerate(rows):
        nb = -(-int(seq_lens[r]) // block_size)
        bt[i, :nb] = [remap[b] for b in block_table[r, :nb]]
    return kc, vc, bt


def sample(rng: np.random.Generator, n_total: int, k: int) -> np.ndarray:
    k = min(k, n_total)
    return np.sort(rng.choice(n_total, size=k, replace=False))
