"""Closed-loop continuous batching: the host scheduler (include/pa_sched.h)
plans each step, one pa_mixed_step_split runs it on the GPU (prefill and
decode side by side on a planned division of the SMs), the scheduler commits
it.  Mock mode: there is no model, so each step's queries, keys and values
are seeded random bf16 rows (the attention path sees the shapes, ragged
lengths and pool traffic of a served batch); requests arrive from a
synthetic trace.

What it follows: the scheduling loop of text-generation-inference's router
(Router/Webserver deep dive, section "Scheduling loop from the source"): the
loop keeps taking the next batch from the queue within the token budgets,
prefills the new requests and decodes the running ones, and filters out the
requests that are done (their blocks return to the allocator).
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as pa
from . import workload as wl


class ServingLoop:
    def __init__(self, shape: wl.Shape, device="cuda", seed: int = 0, **sched_kw):
        self.shape = shape
        self.device = torch.device(device)
        width = sched_kw.pop("width", None) or -(-sched_kw.get("max_total_tokens", 2048) // shape.block_size) + 1
        self.sched = pa.Scheduler(shape.num_blocks, shape.block_size, width=width, **sched_kw)
        self.kp, self.vp = wl.new_pool(shape, seed, device=self.device)
        self.gen = torch.Generator(device=self.device).manual_seed(seed + 1)
        self.steps = 0
        self.generated = 0
        self.finished = []
        self.prompt_len = {}
        self.last = None  # the last step's inputs (host numpy / device tensors), for checking
        self.gpu_events = []  # (start, end) CUDA events around each step's pa_mixed_step, if timed (adds a GPU sleep per step)
        self.time_gpu = False
        self.partition = True  # pa_mixed_step_split on the planned pair count (False: pa_mixed_step)

    def submit(self, request_id: int, input_tokens: int, max_new_tokens: int):
        self.sched.submit(request_id, input_tokens, max_new_tokens)
        self.prompt_len[request_id] = input_tokens

    def step(self, keep_inputs: bool = False):
        """Plan, run and commit one step; returns the step's plan (None when
        nothing is queued or running)."""
        plan = self.sched.plan()
        if plan is None:
            self.sched.commit()
            return None
        sh, dev = self.shape, self.device
        T = plan["num_tokens"]
        randn = lambda *s: torch.randn(*s, generator=self.gen, device=dev, dtype=torch.float32).to(torch.bfloat16)
        q = randn(T, sh.num_q_heads, sh.head_dim)
        kn, vn = randn(T, sh.num_kv_heads, sh.head_dim), randn(T, sh.num_kv_heads, sh.head_dim)
        tod = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev, non_blocking=True)
        qs, lens = tod(plan["q_start_loc"]), tod(plan["seq_lens"])
        slots, bt = tod(plan["slot_mapping"]), tod(plan["block_table"])
        nd = plan["num_decode"]
        rows = np.diff(plan["q_start_loc"])
        max_q = int(rows[nd:].max()) if len(rows) > nd else 1
        max_len = int(plan["seq_lens"].max())
        if keep_inputs:
            self.last = dict(plan=plan, q=q, k=kn, v=vn, kp_before=self.kp.clone(), vp_before=self.vp.clone())
        # The GPU's SMs are divided between the step's prefill and decode by
        # the cost model, from the lengths the plan already holds on the host
        # (only for steps that have both).
        lens_h = plan["seq_lens"]
        pairs = None
        if self.partition and 0 < nd < len(rows):
            pairs = pa.mixed_prefill_pairs(sh, lens_h[:nd], rows[nd:], lens_h[nd:] - rows[nd:])
        if self.time_gpu:
            # A GPU sleep first, so that the step's launches are all queued
            # when the start event is reached: the events then bracket the
            # step's device time, not the host's enqueue of it.
            torch.cuda._sleep(1_000_000)
            ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            ev[0].record()
        out = pa.mixed_step(sh, q, kn, vn, qs, lens, slots, bt, nd, max_len, max_q, self.kp, self.vp,
                            prefill_pairs=pairs)
        if self.time_gpu:
            ev[1].record()
            self.gpu_events.append(ev)
        if keep_inputs:
            self.last["out"] = out
        done = self.sched.commit()
        self.finished += done
        self.steps += 1
        # tokens produced: one per decode row, one per prompt completed this step
        ids, lens_h = plan["seq_ids"], plan["seq_lens"]
        self.generated += nd + sum(1 for i in range(nd, len(ids)) if lens_h[i] == self.prompt_len[int(ids[i])])
        for rid in done:
            self.prompt_len.pop(rid, None)
        return plan

    def gpu_ms(self) -> list[float]:
        """Device time of each timed step's pa_mixed_step (synchronises)."""
        torch.cuda.synchronize(self.device)
        return [a.elapsed_time(b) for a, b in self.gpu_events]
