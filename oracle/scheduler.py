"""Reference of the host continuous-batching scheduler (test infrastructure
only: the tests compare the library's decisions with this one's).

Written from the text-generation-inference Router/Webserver deep dive,
section "Scheduling loop from the source" (the loop takes the next batch
from a FIFO queue against a token budget for the running batch and one for
a prefill; max_waiting_tokens forces admission after that many steps;
waiting_served_ratio sets the least batch worth admitting, running size x
ratio; with prefill chunking both are ignored and new prompts are prefilled
together with the running batch's step), with the launcher defaults of the
TGI architecture wiki, section "Router".  Where the page is silent, this
reference takes the plainest reading of the loop it describes, each stated
here and nowhere derived from the code under test:
  - one step is one forward pass: every running request whose prompt is done
    decodes one token, and the step's admitted prompt rows are prefilled in
    the same pass (the page prefills new prompts with the running batch);
  - a request's reservation against the total-token budget is its prompt
    plus its max_new tokens, rounded up to whole blocks (the router's block
    allocator hands out whole blocks, TGI architecture wiki, "Router");
  - the queue is FIFO: admission takes requests in arrival order and stops
    at the first that does not fit (no request overtakes another);
  - with chunking, a step's prefill rows plus its decode rows stay within
    max_batch_prefill_tokens, and prompts already under way go first;
  - a request's first token comes at the end of its prompt, and it leaves
    once it has produced max_new tokens.

Plain Python: lists, dicts and integer arithmetic, step by step.  Block ids
are not modelled (only counts): where several block assignments are valid,
the tests check validity instead of equality.
"""
from __future__ import annotations

import math


class RefScheduler:
    def __init__(self, num_blocks, block_size, max_batch_prefill_tokens=4096, max_batch_total_tokens=0,
                 max_waiting_tokens=20, waiting_served_ratio=1.2, max_batch_size=0, chunking=False,
                 max_input_tokens=1024, max_total_tokens=2048):
        self.B = block_size
        self.pool_tokens = num_blocks * block_size
        cap = max_batch_total_tokens
        self.total_cap = self.pool_tokens if cap == 0 or cap > self.pool_tokens else cap
        self.prefill_cap = max_batch_prefill_tokens
        self.max_wait = max_waiting_tokens
        self.ratio = waiting_served_ratio
        self.max_batch = max_batch_size
        self.chunking = chunking
        self.max_in = max_input_tokens
        self.max_tot = max_total_tokens
        self.queue = []      # dicts, FIFO
        self.running = []    # dicts, admission order
        self.waiting = 0
        self.planned = None
        self.free_blocks = num_blocks
        self.blocks = {}     # id -> blocks held

    def _reserve(self, r):
        return -(-(r["n"] + r["m"]) // self.B) * self.B

    def submit(self, rid, n, m):
        known = {r["id"] for r in self.queue + self.running}
        if rid in known or n < 1 or m < 1 or n > self.max_in or n + m > self.max_tot:
            raise ValueError("rejected")
        if not self.chunking and n > self.prefill_cap:  # a whole prompt must fit one prefill
            raise ValueError("rejected")
        r = {"id": rid, "n": n, "m": m, "pre": 0, "gen": 0}
        if self._reserve(r) > self.total_cap:
            raise ValueError("rejected")
        self.queue.append(r)

    def cancel(self, rid):
        for lst in (self.queue, self.running):
            for i, r in enumerate(lst):
                if r["id"] == rid:
                    del lst[i]
                    self.free_blocks += self.blocks.pop(rid, 0)
                    return
        raise ValueError("unknown")

    def plan(self):
        """[(id, rows, len_after, is_decode)] of the next step, decode rows first."""
        steps = [(r["id"], 1, r["n"] + r["gen"], True) for r in self.running if r["pre"] == r["n"]]
        n_decode = len(steps)
        budget_total = self.total_cap - sum(self._reserve(r) for r in self.running)
        room = self.max_batch - len(self.running) if self.max_batch > 0 else len(self.queue)
        admitted = []
        if self.chunking:
            budget = self.prefill_cap - n_decode
            for r in self.running:
                if r["pre"] < r["n"] and budget > 0:
                    c = min(r["n"] - r["pre"], budget)
                    steps.append((r["id"], c, r["pre"] + c, False))
                    budget -= c
            reserved = 0
            for e in self.queue:
                if budget <= 0 or len(admitted) >= room or reserved + self._reserve(e) > budget_total:
                    break
                c = min(e["n"], budget)
                steps.append((e["id"], c, c, False))
                budget -= c
                reserved += self._reserve(e)
                admitted.append(e)
        else:
            if not self.running or self.waiting >= self.max_wait:
                min_size = 0
            else:
                min_size = math.floor(len(self.running) * self.ratio)
            if len(self.queue) >= min_size:
                pre = reserved = 0
                for e in self.queue:
                    if len(admitted) >= room or pre + e["n"] > self.prefill_cap or \
                            reserved + self._reserve(e) > budget_total:
                        break
                    pre += e["n"]
                    reserved += self._reserve(e)
                    admitted.append(e)
                if len(admitted) < min_size:
                    admitted = []
            steps += [(e["id"], e["n"], e["n"], False) for e in admitted]
        for rid, rows, after, _ in steps:
            need = -(-after // self.B) - self.blocks.get(rid, 0)
            if need > 0:
                assert need <= self.free_blocks, "reservations keep the pool large enough"
                self.free_blocks -= need
                self.blocks[rid] = self.blocks.get(rid, 0) + need
        for e in admitted:
            self.queue.remove(e)
            self.running.append(e)
        if admitted:
            self.waiting = 0
        elif self.running:
            self.waiting += 1
        self.planned = steps
        return steps, n_decode

    def commit(self):
        done = []
        rows = {rid: (r, dec) for rid, r, _, dec in (self.planned or [])}
        keep = []
        for r in self.running:
            if r["id"] in rows:
                n_rows, dec = rows[r["id"]]
                if dec:
                    r["gen"] += 1
                else:
                    r["pre"] += n_rows
                    if r["pre"] == r["n"]:
                        r["gen"] = 1
            if r["gen"] >= r["m"]:
                done.append(r["id"])
                self.free_blocks += self.blocks.pop(r["id"], 0)
            else:
                keep.append(r)
        self.running = keep
        self.planned = None
        return done
