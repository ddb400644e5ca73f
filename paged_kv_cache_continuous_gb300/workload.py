"""Seeded synthetic inputs for paged KV-cache attention steps.

This module is shared by the tests, the benchmark and the oracle checks.  It
holds none of the attention arithmetic: it draws lengths, plays the router's
block allocator (fixed-size blocks handed out from a free list and returned
when a request finishes -- TGI architecture wiki, data-sketchers.com, section
"The Router"; Blitzscale docs, "used blocks" accounting), and fills tensors
with seeded N(0, 1) values rounded to bf16.

Workloads, shaped like the serving parameters the pages list as router
defaults (128 concurrent requests, 1024 input tokens, 2048 total tokens, 4096
batch prefill tokens; head_dim 128):

* ``tiny``       4 prompts {5,17,33,64}, Hq 4 / Hkv 2, d 64, B 16, 32 blocks:
                 a prefill step, a decode step, and a prefill of the full
                 sequences in fresh blocks.
* ``llama7b_decode``  128 sequences, cached context U[1,2048], Hq = Hkv = 32,
                 d 128, B 16, pool = total blocks + 10 %, shuffled blocks.
* ``mixed``      120 decode sequences (context U[1,2048]) + 8 prompts
                 U[64,1024] with sum <= 4096, Hq 32 / Hkv 8, d 128, B 16.
* ``long_context``  32 sequences with 32768 cached tokens, Hq 64 / Hkv 8.
* ``churn``      512 sequences, log-uniform context in [1,8192], B 32,
                 Hq 32 / Hkv 8; 64 decode steps, 10 % of sequences finish
                 each step and are replaced by prompts U[16,512].

Draw order inside one workload: lengths, block permutation, q, k_new, v_new,
initial pool contents.  Large pools may be drawn on the GPU (``pool_device``),
from a seeded CUDA generator; everything else is drawn on the host.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch


class NoBlocks(RuntimeError):
    """The free list cannot satisfy a reservation."""


@dataclass
class Shape:
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float = 0.0  # 0 -> 1/sqrt(head_dim)


class BlockAllocator:
    """Free-list block allocator (last freed, first reused).

    ``initial_order`` is the order in which never-used blocks are handed out;
    a seeded permutation gives a shuffled physical assignment.
    """

    def __init__(self, num_blocks: int, block_size: int, initial_order=None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = list(range(num_blocks)) if initial_order is None else [int(b) for b in initial_order]
        assert sorted(order) == list(range(num_blocks))
        self.free = order[::-1]  # stack: pop() hands out order[0] first
        self.tables: dict[int, list[int]] = {}

    def num_free(self) -> int:
        return len(self.free)

    def ensure(self, seq: int, num_tokens: int) -> None:
        """Make sequence ``seq`` own enough blocks for ``num_tokens`` tokens."""
        table = self.tables.setdefault(seq, [])
        need = -(-int(num_tokens) // self.block_size) - len(table)
        if need > len(self.free):
            raise NoBlocks(f"need {need} blocks, {len(self.free)} free")
        for _ in range(max(need, 0)):
            table.append(self.free.pop())

    def release(self, seq: int) -> None:
        """Return every block of ``seq`` to the free list, in table order."""
        for b in self.tables.pop(seq):
            self.free.append(b)

    def slot(self, seq: int, pos: int) -> int:
        return self.tables[seq][pos // self.block_size] * self.block_size + pos % self.block_size

    def table_rows(self, seqs, width: int, fill: int = -1) -> np.ndarray:
        out = np.full((len(seqs), width), fill, dtype=np.int32)
        for r, s in enumerate(seqs):
            t = self.tables[s]
            out[r, :len(t)] = t
        return out


@dataclass
class Step:
    """Inputs of one continuous-batching step (everything on the host).

    The first ``num_decode`` sequences have one query row each; the rest are
    prompts (or prompt chunks).  ``seq_lens`` counts tokens after this step's
    append.  Rows of q/k_new/v_new are packed by ``q_start_loc``.
    """
    shape: Shape
    q: torch.Tensor            # bf16 [T, Hq, d]
    k_new: torch.Tensor        # bf16 [T, Hkv, d]
    v_new: torch.Tensor        # bf16 [T, Hkv, d]
    q_start_loc: np.ndarray    # int32 [S + 1]
    seq_lens: np.ndarray       # int32 [S]
    slot_mapping: np.ndarray   # int32 [T]
    block_table: np.ndarray    # int32 [S, max_blocks]
    num_decode: int
    seq_ids: list = field(default_factory=list)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q_start_loc[-1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def max_q_len(self) -> int:
        n = self.q_start_loc[1:] - self.q_start_loc[:-1]
        return int(n[self.num_decode:].max()) if self.num_seqs > self.num_decode else 0


def bf16_randn(shape, gen: torch.Generator, device="cpu") -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(torch.bfloat16)


def new_pool(shape: Shape, seed: int, device="cpu"):
    """Seeded N(0,1) bf16 K and V pools [N, Hkv, B, d] (the initial cache contents).
    ``device=None`` skips the pools (index-only use)."""
    if device is None:
        return None, None
    dims = (shape.num_blocks, shape.num_kv_heads, shape.block_size, shape.head_dim)
    if torch.device(device).type == "cuda":
        g = torch.Generator(device=device)
    else:
        g = torch.Generator()
    g.manual_seed(seed)
    k = bf16_randn(dims, g, device)
    v = bf16_randn(dims, g, device)
    return k, v


def make_step(alloc: BlockAllocator, shape: Shape, seqs, n_new, total_after,
              num_decode: int, gen: torch.Generator, width: int | None = None,
              stale_fill: int = -1, stale_gen: np.random.Generator | None = None,
              value_gen: torch.Generator | None = None, draw_values: bool = True) -> Step:
    """Reserve blocks and draw q/k_new/v_new for one step.

    seqs[i] gets n_new[i] new tokens at positions total_after[i]-n_new[i] ..
    total_after[i]-1.  Block-table entries past a sequence's last block are
    ``stale_fill`` (or seeded junk when ``stale_gen`` is given).  The values
    come from ``value_gen`` (default ``gen``); with ``draw_values=False`` they
    are not drawn (q/k_new/v_new are None: index-only use, e.g. when the
    values are drawn on the device)."""
    n_new = [int(n) for n in n_new]
    total_after = [int(t) for t in total_after]
    for s, L in zip(seqs, total_after):
        alloc.ensure(s, L)
    q_start = np.zeros(len(seqs) + 1, dtype=np.int32)
    q_start[1:] = np.cumsum(n_new)
    T = int(q_start[-1])
    slots = np.empty(T, dtype=np.int32)
    for i, (s, n, L) in enumerate(zip(seqs, n_new, total_after)):
        for j in range(n):
            slots[q_start[i] + j] = alloc.slot(s, L - n + j)
    B = shape.block_size
    need = max([-(-L // B) for L in total_after] + [1])
    width = need if width is None else max(width, need)
    bt = alloc.table_rows(seqs, width, stale_fill)
    if stale_gen is not None:
        for r, L in enumerate(total_after):
            used = -(-L // B)
            junk = stale_gen.integers(-(2 ** 31), 2 ** 31 - 1, size=width - used, dtype=np.int64)
            bt[r, used:] = junk.astype(np.int32)
    q = k = v = None
    if draw_values:
        vg = gen if value_gen is None else value_gen
        q = bf16_randn((T, shape.num_q_heads, shape.head_dim), vg)
        k = bf16_randn((T, shape.num_kv_heads, shape.head_dim), vg)
        v = bf16_randn((T, shape.num_kv_heads, shape.head_dim), vg)
    return Step(shape=shape, q=q, k_new=k, v_new=v, q_start_loc=q_start,
                seq_lens=np.asarray(total_after, dtype=np.int32), slot_mapping=slots,
                block_table=bt, num_decode=int(num_decode), seq_ids=list(seqs))


def _permutation(n: int, gen: torch.Generator) -> list[int]:
    return torch.randperm(n, generator=gen).tolist()


# --------------------------------------------------------------------------
# Named workloads
# --------------------------------------------------------------------------

TINY_PROMPTS = (5, 17, 33, 64)


def tiny(seed: int = 1):
    """Tiny paged step: prompts {5,17,33,64} prefilled, one decode token each,
    then the full sequences {6,18,34,65} prefilled again in fresh blocks.

    Returns (shape, k_pool, v_pool, prefill_step, decode_step, full_step)."""
    shape = Shape(num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16, num_blocks=32)
    g = torch.Generator().manual_seed(seed)
    perm = _permutation(shape.num_blocks, g)
    alloc = BlockAllocator(shape.num_blocks, shape.block_size, perm)
    S = len(TINY_PROMPTS)
    pre = make_step(alloc, shape, list(range(S)), TINY_PROMPTS, TINY_PROMPTS, 0, g)
    dec = make_step(alloc, shape, list(range(S)), [1] * S, [n + 1 for n in TINY_PROMPTS], S, g)
    # The same tokens again, as one prompt per sequence, in fresh blocks.
    full_lens = [n + 1 for n in TINY_PROMPTS]
    qs, ks, vs = [], [], []
    for s in range(S):
        a, b = int(pre.q_start_loc[s]), int(pre.q_start_loc[s + 1])
        qs += [pre.q[a:b], dec.q[s:s + 1]]
        ks += [pre.k_new[a:b], dec.k_new[s:s + 1]]
        vs += [pre.v_new[a:b], dec.v_new[s:s + 1]]
    full = make_step(alloc, shape, list(range(S, 2 * S)), full_lens, full_lens, 0, g)
    full.q, full.k_new, full.v_new = torch.cat(qs), torch.cat(ks), torch.cat(vs)
    kp, vp = new_pool(shape, seed * 1000 + 7)
    return shape, kp, vp, pre, dec, full


def _decode_workload(seed, contexts, shape_kw, pool_device="cpu", stale="fill"):
    g = torch.Generator().manual_seed(seed)
    contexts = [int(c) for c in contexts]
    B = shape_kw["block_size"]
    lens = [c + 1 for c in contexts]
    total_blocks = sum(-(-L // B) for L in lens)
    N = math.ceil(1.1 * total_blocks)
    shape = Shape(num_blocks=N, **shape_kw)
    alloc = BlockAllocator(N, B, _permutation(N, g))
    S = len(lens)
    sg = np.random.default_rng(seed) if stale == "junk" else None
    step = make_step(alloc, shape, list(range(S)), [1] * S, lens, S, g, stale_gen=sg)
    kp, vp = new_pool(shape, seed * 1000 + 7, pool_device)
    return shape, kp, vp, step


def llama7b_decode(seed: int = 2, pool_device="cpu", num_seqs: int = 128, max_context: int = 2048,
                   stale="fill"):
    """128 running sequences, cached context U[1, 2048]; one new token each."""
    g = torch.Generator().manual_seed(seed)
    contexts = torch.randint(1, max_context + 1, (num_seqs,), generator=g).tolist()
    return _decode_workload(seed + 100, contexts,
                            dict(num_q_heads=32, num_kv_heads=32, head_dim=128, block_size=16),
                            pool_device, stale)


def long_context(seed: int = 4, pool_device="cpu", num_seqs: int = 32, context: int = 32768):
    """32 sequences with 32768 cached tokens each, 64 query / 8 KV heads."""
    return _decode_workload(seed + 100, [context] * num_seqs,
                            dict(num_q_heads=64, num_kv_heads=8, head_dim=128, block_size=16),
                            pool_device)


def mixed(seed: int = 3, pool_device="cpu", num_decode: int = 120, num_prompts: int = 8,
          prompt_range=(64, 1024), prefill_budget: int = 4096, max_context: int = 2048):
    """120 decode sequences (context U[1,2048]) merged with 8 new prompts
    U[64,1024] whose sum is <= 4096 (all 8 redrawn until it is)."""
    g = torch.Generator().manual_seed(seed)
    contexts = torch.randint(1, max_context + 1, (num_decode,), generator=g).tolist()
    while True:
        prompts = torch.randint(prompt_range[0], prompt_range[1] + 1, (num_prompts,),
                                generator=g).tolist()
        if sum(prompts) <= prefill_budget:
            break
    B = 16
    lens = [c + 1 for c in contexts] + prompts
    N = math.ceil(1.1 * sum(-(-L // B) for L in lens))
    shape = Shape(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=B, num_blocks=N)
    alloc = BlockAllocator(N, B, _permutation(N, g))
    S = len(lens)
    step = make_step(alloc, shape, list(range(S)), [1] * num_decode + prompts, lens,
                     num_decode, g)
    kp, vp = new_pool(shape, seed * 1000 + 7, pool_device)
    return shape, kp, vp, step


def prefill_only(seed: int, prompts, num_q_heads=32, num_kv_heads=8, head_dim=128,
                 block_size=16, pool_device="cpu"):
    """Fresh prompts only (no decode rows), e.g. 4 x 1024 or 1 x 4096."""
    g = torch.Generator().manual_seed(seed)
    prompts = [int(p) for p in prompts]
    N = math.ceil(1.1 * sum(-(-L // block_size) for L in prompts))
    shape = Shape(num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                  block_size=block_size, num_blocks=N)
    alloc = BlockAllocator(N, block_size, _permutation(N, g))
    step = make_step(alloc, shape, list(range(len(prompts))), prompts, prompts, 0, g)
    kp, vp = new_pool(shape, seed * 1000 + 7, pool_device)
    return shape, kp, vp, step


def chunked_prefill(seed: int = 6, num_seqs: int = 4, prefix: int = 3072, chunk: int = 1024,
                    num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16, pool_device="cpu"):
    """Chunked prefill over a cached prefix: each sequence already holds
    ``prefix`` tokens in the pool (initial contents) and brings its next
    ``chunk`` prompt rows, appended at positions prefix .. prefix + chunk - 1.
    Returns (shape, k_pool, v_pool, step, prefix_lens)."""
    g = torch.Generator().manual_seed(seed)
    L = prefix + chunk
    N = math.ceil(1.1 * num_seqs * -(-L // block_size))
    shape = Shape(num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                  block_size=block_size, num_blocks=N)
    alloc = BlockAllocator(N, block_size, _permutation(N, g))
    step = make_step(alloc, shape, list(range(num_seqs)), [chunk] * num_seqs, [L] * num_seqs, 0, g)
    kp, vp = new_pool(shape, seed * 1000 + 7, pool_device)
    return shape, kp, vp, step, np.full(num_seqs, prefix, dtype=np.int32)


def log_uniform_context(g: torch.Generator, n: int, hi: int = 8192) -> list[int]:
    """L = clamp(floor(exp(U(0, ln(hi + 1)))), 1, hi)."""
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return [min(max(int(math.floor(math.exp(x * math.log(hi + 1)))), 1), hi) for x in u.tolist()]


class Churn:
    """Fragmented serving stress: 512 sequences (log-uniform context in
    [1, 8192], B = 32), 64 steps.  Every step each running sequence decodes
    one token; after the step round(0.1 * S) sequences finish (sampled without
    replacement), their blocks go back on the free list, and as many new
    prompts U[16, 512] join the next step as prefills.

    Lengths, block assignment and finishing are drawn from one generator and
    the step's q/k/v rows from a second (seed + 1), so ``draw_values=False``
    gives the same trace of indices without drawing the values."""

    def __init__(self, seed: int = 5, num_seqs: int = 512, steps: int = 64,
                 max_context: int = 8192, prompt_range=(16, 512), finish_frac: float = 0.1,
                 pool_device="cpu", num_q_heads=32, num_kv_heads=8, head_dim=128,
                 block_size=32, draw_values: bool = True):
        self.g = torch.Generator().manual_seed(seed)
        self.gv = torch.Generator().manual_seed(seed + 1)
        self.draw_values = draw_values
        self.steps = steps
        self.prompt_range = prompt_range
        self.num_finish = int(round(finish_frac * num_seqs))
        ctx = log_uniform_context(self.g, num_seqs, max_context)
        B = block_size
        initial = sum(-(-c // B) for c in ctx)
        N = math.ceil(1.1 * initial) + 2 * num_seqs
        self.shape = Shape(num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                           head_dim=head_dim, block_size=B, num_blocks=N)
        self.alloc = BlockAllocator(N, B, _permutation(N, self.g))
        # Cached contexts already hold their tokens (initial pool contents).
        self.ctx = {}
        for s, c in enumerate(ctx):
            self.alloc.ensure(s, c)
            self.ctx[s] = c
        self.next_id = num_seqs
        self.pending_prompts: list[int] = []  # seq ids admitted for the next step
        self.prompt_len: dict[int, int] = {}
        self.pool_seed = seed * 1000 + 7
        self.pool_device = pool_device
        self.width = -(-(max_context + steps + 1) // B) + 1

    def initial_pool(self):
        return new_pool(self.shape, self.pool_seed, self.pool_device)

    def step(self) -> Step:
        decode_ids = sorted(s for s in self.ctx if s not in self.prompt_len)
        prompt_ids = list(self.pending_prompts)
        seqs = decode_ids + prompt_ids
        n_new = [1] * len(decode_ids) + [self.prompt_len[s] for s in prompt_ids]
        after = [self.ctx[s] + 1 for s in decode_ids] + [self.prompt_len[s] for s in prompt_ids]
        st = make_step(self.alloc, self.shape, seqs, n_new, after, len(decode_ids), self.g,
                       width=self.width, value_gen=self.gv, draw_values=self.draw_values)
        for s, L in zip(seqs, after):
            self.ctx[s] = L
        for s in prompt_ids:
            del self.prompt_len[s]
        self.pending_prompts = []
        # Finish a seeded 10 % and admit as many prompts for the next step.
        alive = sorted(self.ctx)
        pick = torch.randperm(len(alive), generator=self.g)[: self.num_finish].tolist()
        for i in sorted(pick):
            s = alive[i]
            self.alloc.release(s)
            del self.ctx[s]
        lo, hi = self.prompt_range
        for _ in range(self.num_finish):
            s = self.next_id
            self.next_id += 1
            self.prompt_len[s] = int(torch.randint(lo, hi + 1, (1,), generator=self.g).item())
            self.ctx[s] = 0
            self.pending_prompts.append(s)
        return st
