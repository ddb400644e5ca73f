"""Benchmark of the paged-attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one continuous-batching decode step of the Llama-7B-shaped
workload (128 running sequences, cached context U[1, 2048], 32 query / 32 KV
heads, head_dim 128, 16-token blocks, shuffled physical blocks): append each
sequence's new K/V row into the block pool and run split-K decode attention
(partial + merge) -- one pa_decode_append call, the append fused into the
decode launch.  Inputs are resident in HBM when the timed region starts;
the pools (2.4 GB) exceed the 129 MB L2, so no flush is needed between steps.

`value` is the step's algorithmic HBM traffic per second (GB/s): the K/V
bytes decode must read (sum over sequences of L * Hkv * d * 2 B, K and V),
q, out, block-table entries and lengths, the split-K partials (written and
read back), and the append's reads and writes.  The prefill half of the
metric is measured in the same run on causal prompt batches (the mixed
step's 8 prompts, 4 x 1024, 1 x 4096; Hq 32 / Hkv 8) and reported in
TFLOP/s over the unmasked causal pairs only (4 d flops per query head and
(row, key) pair).

With --impl reference the fp64 CPU oracle runs the same step on the host
cores (a bounded sample of the sequences per step) and reports the same
metric.  Under torchrun (N > 1) every rank runs an independent replica
(weak scaling, no collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np
import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "paged decode KV-read GB/s (% of HBM peak); prefill attn TFLOP/s (% of peak)"
WORKLOAD = ("Llama-7B-shaped decode step: 128 running sequences, context U[1,2048] (+1 appended), "
            "Hq 32 / Hkv 32, head_dim 128, block 16, pool = blocks + 10%, shuffled blocks")


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


# ---------------------------------------------------------------- workload --
def decode_step_bytes(shape, seq_lens: np.ndarray, split: int, block_size: int) -> dict:
    """Algorithmic bytes of one append + decode step."""
    Hq, Hkv, d = shape.num_q_heads, shape.num_kv_heads, shape.head_dim
    S = len(seq_lens)
    L = seq_lens.astype(np.int64)
    kv = int(L.sum()) * Hkv * d * 2 * 2
    qo = 2 * S * Hq * d * 2
    tables = int(np.ceil(L / block_size).sum()) * 4 + S * 4
    nsplit = np.maximum(1, -(-L // split))
    # a last split of at most split / 8 tokens joins the one before
    nsplit = np.where((nsplit > 1) & (L - (nsplit - 1) * split <= split // 8), nsplit - 1, nsplit)
    multi = nsplit > 1
    partials = int((nsplit[multi]).sum()) * Hq * (d + 2) * 4 * 2
    append = S * Hkv * d * 2 * 2 * 2 + S * 4  # read k_new, v_new; write the rows; slots
    decode = kv + qo + tables + partials
    return {"kv": kv, "decode": decode, "append": append, "step": decode + append}


def causal_flops(prompts, prefix, Hq, d) -> float:
    tot = 0
    for n, p in zip(prompts, prefix):
        tot += n * p + n * (n + 1) // 2  # unmasked (row, key) pairs
    return 4.0 * d * Hq * tot


def time_each(dev, fn, iters, flush=None, warmup=3):
    """Median device time (s) of fn() over `iters` launches, each bracketed by
    CUDA events on the current stream, with the L2 flushed before each one
    when `flush` (a buffer larger than L2) is given.  Without a flush, a GPU
    sleep queued first lets the host enqueue every launch before the GPU
    reaches it, so a launch shorter than the host's per-call time is not
    timed waiting for its own enqueue (the flush does the same per launch)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(dev)
    ts = []
    if flush is None:
        torch.cuda._sleep(int(2e6 + 2e5 * iters))  # ~1 ms + 0.1 ms per launch of GPU clock cycles
    for _ in range(iters):
        if flush is not None:
            flush.add_(1.0)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize(dev)
    return float(np.median([x.elapsed_time(y) for x, y in ts])) / 1e3


def l2_flush_buffer(dev):
    return torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.15)
        except FileNotFoundError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, f in enumerate(flags) if f == "Active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- distributed --
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max_sum(t_local: float, units_local: float, world: int, device):
    """Max of the ranks' elapsed times and sum of their units."""
    if world == 1:
        return t_local, units_local
    import torch.distributed as dist
    t = torch.tensor([t_local], dtype=torch.float64, device=device)
    u = torch.tensor([units_local], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------- our arm --
def run_ours(args, world, rank, local):
    from paged_kv_cache_continuous_gb300 import binding as pa
    from paged_kv_cache_continuous_gb300 import workload as wl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.load()
    hbm_peak, bf16_peak, peak_src = peaks()

    shape, kp, vp, st = wl.llama7b_decode(pool_device=dev)
    tod = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev) if isinstance(x, np.ndarray) else x.to(dev)
    q, kn, vn = tod(st.q), tod(st.k_new), tod(st.v_new)
    slots, bt, lens = tod(st.slot_mapping), tod(st.block_table), tod(st.seq_lens)
    max_len = st.max_seq_len
    ws = pa.workspace(shape, st.num_seqs, max_len, dev)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)

    def step():
        # the step's append fused into the decode launch (pa_decode_append)
        pa.decode_append(shape, q, kn, vn, slots, kp, vp, bt, lens, max_len, out=out, ws=ws)

    for _ in range(args.warmup):
        step()
    pa.check_device_error()

    _, max_splits = pa.decode_plan(shape, st.num_seqs, max_len)
    split = pa.planned_split(ws, shape, st.num_seqs, max_len)  # the split the plan launch took
    nbytes = decode_step_bytes(shape, st.seq_lens, split, shape.block_size)
    launches_per_step = 2  # the plan launch (with the append) and the decode kernel

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for i in range(K):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    barrier(world)
    pa.check_device_error()
    t_local = e0.elapsed_time(e1) / 1e3
    t_dec = float(np.mean([a[0].elapsed_time(a[1]) for a in ev])) / 1e3
    # The standalone append (pa_kv_append) and decode (pa_decode) of the same
    # step, outside the timed region, for comparison with the fused launch.
    t_app = time_each(dev, lambda: pa.kv_append(shape, kn, vn, slots, kp, vp), max(20, min(K, 200)))
    t_dec_alone = time_each(dev, lambda: pa.decode(shape, q, kp, vp, bt, lens, max_len, out=out, ws=ws),
                            max(20, min(K, 200)))
    t_max, bytes_all = reduce_max_sum(t_local, nbytes["step"] * K, world, dev)
    value = bytes_all / t_max / 1e9

    # ---- end to end through the public API with host buffers
    host = {k: v.cpu().pin_memory() for k, v in dict(q=q, kn=kn, vn=vn, slots=slots, bt=bt, lens=lens).items()}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    dbuf = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = out.numel() * out.element_size()
    Ke = max(20, min(K, 500))

    def e2e_step():
        for k, v in host.items():
            dbuf[k].copy_(v, non_blocking=True)
        pa.decode_append(shape, dbuf["q"], dbuf["kn"], dbuf["vn"], dbuf["slots"], kp, vp, dbuf["bt"], dbuf["lens"],
                         max_len, out=out, ws=ws)
        out_h.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(Ke):
        e2e_step()
    s1.record(stream)
    torch.cuda.synchronize(dev)
    t_e2e_serial, _ = reduce_max_sum(s0.elapsed_time(s1) / 1e3, nbytes["step"] * Ke, world, dev)

    # The same steps pipelined the way a serving loop runs them: every step
    # still copies its own inputs in and its output out, but on two copy
    # streams, into double-buffered device inputs and outputs, so that step
    # i + 1's inputs cross the host link and step i - 1's output returns
    # while step i's kernels run.
    ref_h = out_h.clone()
    hs, ds = torch.cuda.Stream(dev), torch.cuda.Stream(dev)  # host->device, device->host
    bufs = [dbuf, {k: torch.empty_like(v) for k, v in dbuf.items()}]
    outs = [out, torch.empty_like(out)]
    outs_h = [out_h, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def h2d_of(i):
        b = i % 2
        with torch.cuda.stream(hs):
            if i >= 2:
                hs.wait_event(ev_comp[b])  # step i - 2 has read buffer b
            for k, v in host.items():
                bufs[b][k].copy_(v, non_blocking=True)
            ev_in[b].record(hs)

    def run_pipelined(n):
        h2d_of(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:
                h2d_of(i + 1)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # step i - 2's output has left buffer b
            d = bufs[b]
            pa.decode_append(shape, d["q"], d["kn"], d["vn"], d["slots"], kp, vp, d["bt"], d["lens"], max_len,
                             out=outs[b], ws=ws)
            ev_comp[b].record(stream)
            with torch.cuda.stream(ds):
                ds.wait_event(ev_comp[b])
                outs_h[b].copy_(outs[b], non_blocking=True)
                ev_out[b].record(ds)
        stream.wait_event(ev_out[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(ev_out[(n - 2) % 2])

    run_pipelined(4)
    torch.cuda.synchronize(dev)
    barrier(world)
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p0.record(stream)
    hs.wait_event(p0)
    ds.wait_event(p0)
    run_pipelined(Ke)
    p1.record(stream)
    torch.cuda.synchronize(dev)
    t_e2e, bytes_e2e = reduce_max_sum(p0.elapsed_time(p1) / 1e3, nbytes["step"] * Ke, world, dev)
    # every step has the same inputs: both output buffers hold the serial run's result
    assert torch.equal(outs_h[0], ref_h) and torch.equal(outs_h[1], ref_h), "pipelined e2e output differs"

    # ---- prefill half of the metric (tensor cores), timed alone with L2 flushed
    prefill = measure_prefill(pa, wl, dev, bf16_peak, peak_src, args.prefill_iters) if rank == 0 else None
    copy = measure_copy(pa, wl, dev, hbm_peak, args.prefill_iters) if rank == 0 else None
    rope = measure_rope(pa, wl, dev, hbm_peak, args.prefill_iters) if rank == 0 else None
    fp8 = measure_fp8_decode(pa, wl, dev, hbm_peak, max(20, min(args.steps, 500))) if rank == 0 else None
    serving = [measure_serving(dev, c) for c in (False, True)] if rank == 0 else None
    long_ctx = measure_long_context(pa, wl, dev, hbm_peak, max(20, min(args.steps, 200))) if rank == 0 else None
    mixed = measure_mixed_step(pa, wl, dev, hbm_peak, bf16_peak, args.prefill_iters) if rank == 0 else None
    churn = measure_churn(pa, wl, dev, hbm_peak, bf16_peak, args.warmup) if rank == 0 else None
    chunked = measure_chunked_prefill(pa, wl, dev, bf16_peak, args.prefill_iters) if rank == 0 else None

    clocks = clk.summary()
    traffic = load_traffic("decode_splitk", nbytes, st.num_seqs)
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(t_max / K * 1e3, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "num_seqs": st.num_seqs, "num_q_heads": shape.num_q_heads,
                   "num_kv_heads": shape.num_kv_heads, "head_dim": shape.head_dim,
                   "block_size": shape.block_size, "num_blocks": shape.num_blocks,
                   "context_tokens": int(st.seq_lens.sum()), "decode_split_tokens": split,
                   "l2": "inputs larger than L2 (KV pools 2.4 GB > 129 MB); no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm",
                     "kernel": "decode with the append fused (decode_plan_kernel + decode_splitk_kernel, splits merged in-kernel)",
                     "achieved": round(nbytes["step"] / t_dec / 1e9, 1), "peak": hbm_peak,
                     "unit": "GB/s", "frac": round(nbytes["step"] / t_dec / 1e9 / hbm_peak, 4),
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs copy)",
                     "frac_of_nominal_8TBps": round(nbytes["step"] / t_dec / 1e9 / 8000.0, 4),
                     "traffic": traffic, "algorithmic_bytes": nbytes["step"],
                     "kernel_ms": round(t_dec * 1e3, 5)},
        "unfused": {"append_ms": round(t_app * 1e3, 5), "append_GBps": round(nbytes["append"] / t_app / 1e9, 1),
                    "decode_ms": round(t_dec_alone * 1e3, 5),
                    "decode_GBps": round(nbytes["decode"] / t_dec_alone / 1e9, 1),
                    "note": "pa_kv_append and pa_decode of the same step as two calls (outside the timed region)"},
        "e2e": {"value": round(bytes_e2e / t_e2e / 1e9, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke,
                "how": "every step copies its inputs from pinned host memory and its output back, on two copy "
                       "streams with double-buffered device buffers, overlapped with the neighbouring steps' "
                       "kernels (pa_decode_append on the main stream); one event pair around all steps (the "
                       "device-timed loop of `value` records an event pair around every step as well)",
                "serial": {"value": round(bytes_e2e / t_e2e_serial / 1e9, 2), "unit": "GB/s",
                           "how": "copy in, pa_decode_append, copy out, all on one stream"}},
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "prefill": prefill,
        "block_copy": copy,
        "rope_append": rope,
        "fp8_decode": fp8,
        "serving_loop": serving,
        "long_context": long_ctx,
        "mixed_step": mixed,
        "churn": churn,
        "chunked_prefill": chunked,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(shape, kp, vp, st, split, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_other_workload(args, local):
    """One secondary measurement alone (the same leg the contract line
    carries): long_context, mixed, churn or chunked_prefill."""
    from paged_kv_cache_continuous_gb300 import binding as pa
    from paged_kv_cache_continuous_gb300 import workload as wl
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.load()
    hbm_peak, bf16_peak, _ = peaks()
    legs = {
        "long_context": lambda: measure_long_context(pa, wl, dev, hbm_peak, args.steps),
        "mixed": lambda: measure_mixed_step(pa, wl, dev, hbm_peak, bf16_peak, args.prefill_iters),
        "churn": lambda: measure_churn(pa, wl, dev, hbm_peak, bf16_peak, args.warmup),
        "chunked_prefill": lambda: measure_chunked_prefill(pa, wl, dev, bf16_peak, args.prefill_iters),
    }
    print(json.dumps({"workload": args.workload, **legs[args.workload]()}), flush=True)


def load_traffic(kernel: str, nbytes, num_seqs):
    """DRAM bytes per launch from the committed ncu summary, if it matches the
    current kernel build (profiles/decode_llama7b_traffic.json)."""
    p = ROOT / "profiles" / "decode_llama7b_traffic.json"
    if not p.exists():
        return None
    try:
        d = json.loads(p.read_text())
        import hashlib
        csrc = ROOT / "paged_kv_cache_continuous_gb300" / "csrc"
        for name, key in (("decode.cu", "decode_cu_sha256"), ("pa_common.cuh", "pa_common_cuh_sha256")):
            if d.get(key) != hashlib.sha256((csrc / name).read_bytes()).hexdigest():
                return None  # the kernel changed since the counters were taken
        # the call's three launches: the decode kernel and the plan and merge
        # launches beside it
        other = sum(v.get("dram_bytes", 0) for v in d.get("other_launches_of_the_call", {}).values())
        return d.get("dram_bytes_per_launch") + other
    except Exception:
        return None


def measure_prefill(pa, wl, dev, bf16_peak, peak_src, iters):
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    res = {}
    cases = {"mixed-step prompts": None, "4x1024": [1024] * 4, "1x4096": [4096]}
    for name, prompts in cases.items():
        if prompts is None:
            shape, kp, vp, st_m = wl.mixed(pool_device=dev)
            nd = st_m.num_decode
            qs = st_m.q_start_loc[nd:] - st_m.q_start_loc[nd]
            rows = slice(int(st_m.q_start_loc[nd]), int(st_m.q_start_loc[-1]))
            n = (qs[1:] - qs[:-1]).tolist()
            q = st_m.q[rows].to(dev)
            kn, vn = st_m.k_new[rows].to(dev), st_m.v_new[rows].to(dev)
            slots = torch.from_numpy(st_m.slot_mapping[rows]).to(dev)
            bt = torch.from_numpy(np.ascontiguousarray(st_m.block_table[nd:])).to(dev)
            cu = torch.from_numpy(np.ascontiguousarray(qs)).to(dev)
        else:
            shape, kp, vp, st_p = wl.prefill_only(60 + len(prompts), prompts, pool_device=dev)
            n = prompts
            q, kn, vn = st_p.q.to(dev), st_p.k_new.to(dev), st_p.v_new.to(dev)
            slots = torch.from_numpy(st_p.slot_mapping).to(dev)
            bt = torch.from_numpy(st_p.block_table).to(dev)
            cu = torch.from_numpy(st_p.q_start_loc).to(dev)
        pa.kv_append(shape, kn, vn, slots, kp, vp)
        out = torch.empty_like(q)
        for _ in range(3):
            pa.prefill(shape, q, kp, vp, cu, max(n), block_table=bt, out=out)
        pa.check_device_error()
        times = []
        for _ in range(iters):
            flush.add_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            pa.prefill(shape, q, kp, vp, cu, max(n), block_table=bt, out=out)
            b.record()
            times.append((a, b))
        torch.cuda.synchronize(dev)
        t = float(np.median([x.elapsed_time(y) for x, y in times])) / 1e3
        fl = causal_flops(n, [0] * len(n), shape.num_q_heads, shape.head_dim)
        res[name] = {"prompts": n if len(n) <= 8 else len(n), "ms": round(t * 1e3, 4),
                     "tflops": round(fl / t / 1e12, 1), "frac": round(fl / t / 1e12 / bf16_peak, 4)}
        del kp, vp
        # Back to back: the same prompt lengths in four input sets of their
        # own (fresh pools, queries and outputs: ~86 MB each for 4096 rows, so
        # four exceed L2 and every launch reads its inputs from DRAM), one
        # launch after another with no flush between, one event pair around
        # them all: the rate a stream of prefills runs at, without the
        # launch latency a lone launch after a flush is timed with.
        sets = []
        for j in range(4):
            shp, kpj, vpj, stj = wl.prefill_only(200 + 10 * j + len(n), n, pool_device=dev)
            qj = stj.q.to(dev)
            pa.kv_append(shp, stj.k_new.to(dev), stj.v_new.to(dev), torch.from_numpy(stj.slot_mapping).to(dev),
                         kpj, vpj)
            sets.append((shp, qj, kpj, vpj, torch.from_numpy(stj.q_start_loc).to(dev),
                         torch.from_numpy(stj.block_table).to(dev), torch.empty_like(qj)))
        for shp, qj, kpj, vpj, cuj, btj, oj in sets:
            pa.prefill(shp, qj, kpj, vpj, cuj, max(n), block_table=btj, out=oj)
        torch.cuda.synchronize(dev)
        n_l = 4 * max(iters // 2, 10)
        torch.cuda._sleep(int(2e6 + 2e5 * n_l))  # the launches queue up before the GPU reaches them
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for j in range(n_l):
            shp, qj, kpj, vpj, cuj, btj, oj = sets[j % 4]
            pa.prefill(shp, qj, kpj, vpj, cuj, max(n), block_table=btj, out=oj)
        b.record()
        torch.cuda.synchronize(dev)
        pa.check_device_error()
        t2 = a.elapsed_time(b) / 1e3 / n_l
        res[name]["back_to_back"] = {"ms": round(t2 * 1e3, 4), "tflops": round(fl / t2 / 1e12, 1),
                                     "frac": round(fl / t2 / 1e12 / bf16_peak, 4), "launches": n_l,
                                     "l2": "four input sets in turn (inputs larger than L2); no flush"}
        del sets
    best = max(res.values(), key=lambda r: r["tflops"])
    return {"bound": "tensor", "kernel": "prefill_pair_kernel (tcgen05 cta_group::2, P in TMEM; head_dim 128)", "unit": "TFLOP/s",
            "peak": bf16_peak, "peak_source": f"{peak_src} (MEASURED_PEAKS.json bf16_tflops burst)",
            "workloads": res, "achieved_best": best["tflops"], "frac_best": best["frac"],
            "flops_counted": "4*d*Hq per unmasked causal (row, key) pair",
            "l2": "flushed (256 MB write) before each launch (back_to_back: see its own l2 key)"}


def measure_copy(pa, wl, dev, hbm_peak, iters):
    """Whole-block copies with the decode workload's block shape (32 KV heads x
    16 tokens x 128 dims: 128 KB per block and pool): a 4096-block fork
    inside a 1 GB device pool pair, and 1024-block swaps to and from pinned
    host pools.  Bytes counted: K and V, read once and written once."""
    shape = wl.Shape(num_q_heads=32, num_kv_heads=32, head_dim=128, block_size=16, num_blocks=8192)
    blk = shape.num_kv_heads * shape.block_size * shape.head_dim * 2
    kp = torch.empty((8192, 32, 16, 128), dtype=torch.bfloat16, device=dev).normal_()
    vp = torch.empty_like(kp).normal_()
    g = torch.Generator().manual_seed(17)
    perm = torch.randperm(8192, generator=g).to(torch.int32)
    src, dst = perm[:4096].to(dev), perm[4096:].to(dev)
    hk = torch.empty((1024, 32, 16, 128), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    hids = torch.arange(1024, dtype=torch.int32, device=dev)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(iters):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            ts.append((a, b))
        torch.cuda.synchronize(dev)
        pa.check_device_error()
        return float(np.median([x.elapsed_time(y) for x, y in ts])) / 1e3

    t_fork = timed(lambda: pa.copy_blocks(shape, kp, vp, kp, vp, src, dst))
    t_out = timed(lambda: pa.copy_blocks(shape, kp, vp, hk, hv, src[:1024], hids))
    t_in = timed(lambda: pa.copy_blocks(shape, hk, hv, kp, vp, hids, dst[:1024]))
    fork_b, swap_b = 2 * 2 * 4096 * blk, 2 * 1024 * blk
    # The host link's own rate: one plain pinned copy of the same bytes (both
    # pools, 256 MB) in each direction, as a denominator for the swaps.
    dflat, hflat = kp[:2048].view(-1), hk.view(-1)
    hflat2 = torch.empty(2 * hflat.numel(), dtype=hflat.dtype).pin_memory()
    t_link_out = timed(lambda: hflat2.copy_(dflat, non_blocking=True))
    t_link_in = timed(lambda: dflat.copy_(hflat2, non_blocking=True))
    link_out, link_in = swap_b / t_link_out / 1e9, swap_b / t_link_in / 1e9
    return {"kernel": "copy_blocks_kernel", "block_bytes_per_pool": blk,
            "fork_4096_blocks": {"ms": round(t_fork * 1e3, 4), "GBps": round(fork_b / t_fork / 1e9, 1),
                                 "frac_hbm": round(fork_b / t_fork / 1e9 / hbm_peak, 4),
                                 "bytes": "K+V read + written"},
            "swap_out_1024_blocks": {"ms": round(t_out * 1e3, 4), "GBps": round(swap_b / t_out / 1e9, 1),
                                     "bytes": "K+V moved to pinned host",
                                     "frac_link": round(swap_b / t_out / 1e9 / link_out, 4)},
            "swap_in_1024_blocks": {"ms": round(t_in * 1e3, 4), "GBps": round(swap_b / t_in / 1e9, 1),
                                    "bytes": "K+V moved from pinned host",
                                    "frac_link": round(swap_b / t_in / 1e9 / link_in, 4)},
            "link_peak": {"d2h_GBps": round(link_out, 1), "h2d_GBps": round(link_in, 1),
                          "how": "one cudaMemcpyAsync of 256 MB between device and pinned host memory"}}


def measure_rope(pa, wl, dev, hbm_peak, iters):
    """Rotary embedding fused with the append (pa_rope_append), L2 flushed
    before each launch: a 4096-token prompt step (Hq 32, Hkv 8, d 128) and the
    decode step's 128 tokens (Hq = Hkv = 32).  Bytes: q read and written, k and
    v read and written to the pool, positions and slots read."""
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    res = {}
    for name, T, Hq, Hkv in (("prompt_4096", 4096, 32, 8), ("decode_step_128", 128, 32, 32)):
        g = torch.Generator().manual_seed(23)
        nb = T // 16 + 16
        shape = wl.Shape(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, block_size=16, num_blocks=nb)
        q = wl.bf16_randn((T, Hq, 128), g).to(dev)
        k, v = wl.bf16_randn((T, Hkv, 128), g).to(dev), wl.bf16_randn((T, Hkv, 128), g).to(dev)
        kp = torch.zeros((nb, Hkv, 16, 128), dtype=torch.bfloat16, device=dev)
        vp = torch.zeros_like(kp)
        pos = torch.arange(T, dtype=torch.int32, device=dev)
        slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int32).to(dev)
        q_out = torch.empty_like(q)
        for _ in range(3):
            pa.rope_append(shape, q, k, v, pos, slots, kp, vp, q_out=q_out)
        pa.check_device_error()
        ts = []
        for _ in range(iters):
            flush.add_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            pa.rope_append(shape, q, k, v, pos, slots, kp, vp, q_out=q_out)
            b.record()
            ts.append((a, b))
        torch.cuda.synchronize(dev)
        t = float(np.median([x.elapsed_time(y) for x, y in ts])) / 1e3
        nbytes = T * (Hq + 2 * Hkv) * 128 * 2 * 2 + 8 * T
        res[name] = {"tokens": T, "ms": round(t * 1e3, 4), "GBps": round(nbytes / t / 1e9, 1),
                     "frac_hbm": round(nbytes / t / 1e9 / hbm_peak, 4)}
        if name == "prompt_4096":
            # Back to back over four input sets (4 x ~100 MB > L2, so every
            # launch reads and writes DRAM), one event pair around all launches:
            # the rate a serving loop's consecutive steps see, launch gaps
            # included, without the per-launch flush and events.
            sets = [(q, k, v, pos, slots, kp, vp, q_out)]
            for j in range(3):
                g2 = torch.Generator().manual_seed(31 + j)
                sets.append((wl.bf16_randn((T, Hq, 128), g2).to(dev), wl.bf16_randn((T, Hkv, 128), g2).to(dev),
                             wl.bf16_randn((T, Hkv, 128), g2).to(dev), pos,
                             torch.randperm(nb * 16, generator=g2)[:T].to(torch.int32).to(dev),
                             torch.zeros_like(kp), torch.zeros_like(vp), torch.empty_like(q)))
            for st_ in sets:
                pa.rope_append(shape, *st_[:5], st_[5], st_[6], q_out=st_[7])
            torch.cuda.synchronize(dev)
            n_l = max(4 * iters, 40)
            torch.cuda._sleep(int(2e6 + 2e5 * n_l))  # the launches queue up before the GPU reaches them
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for j in range(n_l):
                st_ = sets[j % 4]
                pa.rope_append(shape, *st_[:5], st_[5], st_[6], q_out=st_[7])
            b.record()
            torch.cuda.synchronize(dev)
            pa.check_device_error()
            t2 = a.elapsed_time(b) / 1e3 / n_l
            res["prompt_4096_back_to_back"] = {
                "tokens": T, "ms": round(t2 * 1e3, 4), "GBps": round(nbytes / t2 / 1e9, 1),
                "frac_hbm": round(nbytes / t2 / 1e9 / hbm_peak, 4), "launches": n_l,
                "l2": "four input sets of ~100 MB in turn (inputs larger than L2); no flush"}
            del sets
    return {"kernel": "rope_append_kernel", "l2": "flushed (256 MB write) before each launch", **res}


def measure_fp8_decode(pa, wl, dev, hbm_peak, steps):
    """The decode step's attention (Llama-7B shape, 128 sequences) over fp8
    (e4m3) pools with per-KV-head scales: pa_decode_fp8.  Bytes counted: the
    fp8 K/V (one byte per element), q, out, tables, lengths and split
    partials; the rate in sequences decoded per second as well."""
    shape, _, _, st = wl.llama7b_decode(pool_device=None)
    N, H, B, d = shape.num_blocks, shape.num_kv_heads, shape.block_size, shape.head_dim
    kp = torch.randint(0, 126, (N, H, B, d), dtype=torch.uint8, device=dev)
    vp = torch.randint(0, 126, (N, H, B, d), dtype=torch.uint8, device=dev)
    ks = torch.full((H,), 0.02, dtype=torch.float32, device=dev)
    vs = torch.full((H,), 0.02, dtype=torch.float32, device=dev)
    tod = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev) if isinstance(x, np.ndarray) else x.to(dev)
    q, bt, lens = tod(st.q), tod(st.block_table), tod(st.seq_lens)
    ws = pa.workspace(shape, st.num_seqs, st.max_seq_len, dev)
    out = torch.empty_like(q)
    for _ in range(5):
        pa.decode_fp8(shape, q, kp, vp, ks, vs, bt, lens, st.max_seq_len, out=out, ws=ws)
    pa.check_device_error()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        pa.decode_fp8(shape, q, kp, vp, ks, vs, bt, lens, st.max_seq_len, out=out, ws=ws)
    b.record()
    torch.cuda.synchronize(dev)
    pa.check_device_error()
    t = a.elapsed_time(b) / 1e3 / steps
    split = pa.planned_split(ws, shape, st.num_seqs, st.max_seq_len)
    nb = decode_step_bytes(shape, st.seq_lens, split, shape.block_size)
    fp8_bytes = nb["decode"] - nb["kv"] // 2
    return {"kernel": "decode_splitk_kernel<128,16,*,fp8> (splits merged in-kernel)", "ms": round(t * 1e3, 5),
            "GBps": round(fp8_bytes / t / 1e9, 1), "frac_hbm": round(fp8_bytes / t / 1e9 / hbm_peak, 4),
            "algorithmic_bytes": int(fp8_bytes), "sequences_per_s": round(st.num_seqs / t, 1),
            "l2": "inputs larger than L2 (fp8 pools 1.2 GB)"}


def measure_serving(dev, chunking: bool):
    """Closed-loop continuous batching (host scheduler + one pa_mixed_step_split
    per step, the SMs divided by the planned pair count when a step has both
    prompts and decode rows; mock activations): 512 requests arrive at once,
    prompts U[16, 512], U[64, 256] new tokens each, Hq 32 / Hkv 8 / d 128,
    B 16; run until all are done.  Wall-clock over the whole run (host
    planning, H2D of the step's index arrays and the GPU step), and the GPU
    time of the steps alone (a second identical run, each step queued behind
    a GPU sleep so that its events bracket device time only)."""
    from paged_kv_cache_continuous_gb300 import workload as wl
    from paged_kv_cache_continuous_gb300.serving import ServingLoop
    import time
    def run(time_gpu):
        shape = wl.Shape(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16, num_blocks=26000)
        loop = ServingLoop(shape, device=dev, seed=11, max_batch_prefill_tokens=4096, chunking=chunking,
                           max_input_tokens=1024, max_total_tokens=2048, max_seqs=1024, max_tokens=8192)
        rng = np.random.default_rng(12)
        for i in range(512):
            loop.submit(i, int(rng.integers(16, 513)), int(rng.integers(64, 257)))
        torch.cuda.synchronize(dev)
        loop.time_gpu = time_gpu
        t0 = time.perf_counter()
        while loop.step() is not None:
            pass
        torch.cuda.synchronize(dev)
        return loop, time.perf_counter() - t0

    # wall clock from a plain run; the device time of the steps from a second,
    # identical (seeded) run that queues each step behind a GPU sleep
    loop, wall = run(False)
    loop_t, _ = run(True)
    gpu = np.array(loop_t.gpu_ms())
    return {"requests": 512, "steps": loop.steps, "generated_tokens": loop.generated, "wall_s": round(wall, 4),
            "tokens_per_s": round(loop.generated / wall, 1), "ms_per_step": round(wall / loop.steps * 1e3, 4),
            "gpu_ms_per_step": round(float(gpu.mean()), 4), "gpu_s": round(float(gpu.sum()) / 1e3, 4),
            "tokens_per_gpu_s": round(loop.generated / (float(gpu.sum()) / 1e3), 1),
            "chunking": chunking,
            "note": "wall clock includes host planning and Python marshalling; gpu_* is the step's device "
                    "time (CUDA events around each pa_mixed_step queued behind a GPU sleep) alone"}


def measure_long_context(pa, wl, dev, hbm_peak, iters):
    """Long-context decode: 32 sequences of 32 768 cached tokens (+1 appended),
    Hq 64 / Hkv 8 (70B-shaped GQA), B 16: append, then split-K decode + merge.
    The pools (4.7 GB) exceed L2, so launches run back to back."""
    shape, kp, vp, st = wl.long_context(pool_device=dev)
    tod = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev) if isinstance(x, np.ndarray) else x.to(dev)
    q, kn, vn = tod(st.q), tod(st.k_new), tod(st.v_new)
    slots, bt, lens = tod(st.slot_mapping), tod(st.block_table), tod(st.seq_lens)
    ws = pa.workspace(shape, st.num_seqs, st.max_seq_len, dev)
    out = torch.empty_like(q)
    t_app = time_each(dev, lambda: pa.kv_append(shape, kn, vn, slots, kp, vp), iters)
    t_dec = time_each(dev, lambda: pa.decode(shape, q, kp, vp, bt, lens, st.max_seq_len, out=out, ws=ws), iters)
    pa.check_device_error()
    split = pa.planned_split(ws, shape, st.num_seqs, st.max_seq_len)
    nsplit = -(-int(st.max_seq_len) // split)
    if nsplit > 1 and int(st.max_seq_len) - (nsplit - 1) * split <= split // 8:
        nsplit -= 1
    nb = decode_step_bytes(shape, st.seq_lens, split, shape.block_size)
    del kp, vp
    return {"workload": "32 x 32768 cached tokens (+1), Hq 64 / Hkv 8, d 128, B 16",
            "kernel": "decode_splitk_kernel (splits merged in-kernel)", "split_tokens": split, "splits": nsplit,
            "decode_ms": round(t_dec * 1e3, 5), "algorithmic_bytes": nb["decode"],
            "GBps": round(nb["decode"] / t_dec / 1e9, 1), "frac_hbm": round(nb["decode"] / t_dec / 1e9 / hbm_peak, 4),
            "append_ms": round(t_app * 1e3, 5), "l2": "inputs larger than L2 (pools 4.7 GB); no flush"}


def measure_mixed_step(pa, wl, dev, hbm_peak, bf16_peak, iters):
    """The mixed continuous-batching step: 120 decode sequences (context
    U[1,2048]) + 8 prompts U[64,1024] (sum <= 4096), Hq 32 / Hkv 8, d 128,
    B 16, through one pa_mixed_step_split (append, then decode and prefill
    on two streams, the prefill on the CTA pairs pa_mixed_prefill_pairs
    plans from the host lengths, the decode on the other SMs); the
    unpartitioned pa_mixed_step, decode and prefill alone beside it.  L2
    flushed before each launch.  frac: the step's lower bound with decode (and append) on HBM
    and prefill on the tensor cores perfectly overlapped, over its time."""
    shape, kp, vp, st = wl.mixed(pool_device=dev)
    tod = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev) if isinstance(x, np.ndarray) else x.to(dev)
    q, kn, vn = tod(st.q), tod(st.k_new), tod(st.v_new)
    qs, lens, slots, bt = tod(st.q_start_loc), tod(st.seq_lens), tod(st.slot_mapping), tod(st.block_table)
    nd = st.num_decode
    ws = pa.workspace(shape, nd, st.max_seq_len, dev)
    out = torch.empty_like(q)
    flush = l2_flush_buffer(dev)
    rows_h = np.diff(st.q_start_loc)[nd:]
    pairs = pa.mixed_prefill_pairs(shape, st.seq_lens[:nd], rows_h, st.seq_lens[nd:] - rows_h)
    t_step = time_each(dev, lambda: pa.mixed_step(shape, q, kn, vn, qs, lens, slots, bt, nd, st.max_seq_len,
                                                  st.max_q_len, kp, vp, out=out, ws=ws, prefill_pairs=pairs),
                       iters, flush)
    t_shared = time_each(dev, lambda: pa.mixed_step(shape, q, kn, vn, qs, lens, slots, bt, nd, st.max_seq_len,
                                                    st.max_q_len, kp, vp, out=out, ws=ws), iters, flush)
    dmax = int(st.seq_lens[:nd].max())
    qd, btd, lensd = q[:nd], bt[:nd].contiguous(), lens[:nd].contiguous()
    outd = torch.empty_like(qd)
    t_dec = time_each(dev, lambda: pa.decode(shape, qd, kp, vp, btd, lensd, dmax, out=outd, ws=ws), iters, flush)
    r0 = int(st.q_start_loc[nd])
    qp = q[r0:].contiguous()
    cup = (qs[nd:] - r0).contiguous()
    btp = bt[nd:].contiguous()
    outp = torch.empty_like(qp)
    t_pre = time_each(dev, lambda: pa.prefill(shape, qp, kp, vp, cup, st.max_q_len, block_table=btp, out=outp),
                      iters, flush)
    pa.check_device_error()
    split = pa.planned_split(ws, shape, nd, dmax)
    nb = decode_step_bytes(shape, st.seq_lens[:nd], split, shape.block_size)
    T = int(st.q_start_loc[-1])
    append_b = T * shape.num_kv_heads * shape.head_dim * 2 * 2 * 2 + 4 * T
    n = np.diff(st.q_start_loc[nd:]).tolist()
    fl = causal_flops(n, [0] * len(n), shape.num_q_heads, shape.head_dim)
    bound = max((nb["decode"] + append_b) / (hbm_peak * 1e9), fl / (bf16_peak * 1e12))
    del kp, vp
    return {"workload": "120 decode (context U[1,2048]) + 8 prompts U[64,1024] (sum <= 4096), Hq 32 / Hkv 8, "
                        "d 128, B 16", "prompts": n,
            "step_ms": round(t_step * 1e3, 5), "prefill_pairs": pairs,
            "step_ms_unpartitioned": round(t_shared * 1e3, 5), "decode_alone_ms": round(t_dec * 1e3, 5),
            "prefill_alone_ms": round(t_pre * 1e3, 5),
            "decode_bytes": nb["decode"], "append_bytes": append_b, "prefill_flops": fl,
            "decode_alone_GBps": round(nb["decode"] / t_dec / 1e9, 1),
            "decode_alone_frac_hbm": round(nb["decode"] / t_dec / 1e9 / hbm_peak, 4),
            "prefill_alone_tflops": round(fl / t_pre / 1e12, 1),
            "prefill_alone_frac_bf16": round(fl / t_pre / 1e12 / bf16_peak, 4),
            "step_bound_ms": round(bound * 1e3, 5), "frac": round(bound / t_step, 4),
            "l2": "flushed (256 MB write) before each launch"}


def measure_churn(pa, wl, dev, hbm_peak, bf16_peak, warmup):
    """Fragmented serving stress: 512 sequences (log-uniform context in
    [1, 8192]), Hq 32 / Hkv 8, d 128, B 32, 64 consecutive pa_mixed_step
    calls (pa_mixed_step_split, each step's prefill pairs planned from its
    host lengths; the unpartitioned pa_mixed_step timed beside it); after
    every step a seeded 10 % finish and their blocks are reused by as many
    prompts U[16,512], prefilled in the next step.  The index trace
    (lengths, tables, slots) is the one the parity test checks; the rows are
    drawn on the device.  Each step timed with CUDA events; the pools (2.3 GB)
    exceed L2."""
    ch = wl.Churn(pool_device=dev, draw_values=False)
    shape = ch.shape
    steps = [ch.step() for _ in range(ch.steps)]
    kp, vp = ch.initial_pool()
    tod = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    Tmax = max(int(st.q_start_loc[-1]) for st in steps)
    g = torch.Generator(device=dev).manual_seed(55)
    rows = lambda h: torch.randn(Tmax, h, shape.head_dim, generator=g, device=dev).to(torch.bfloat16)
    qb, kb, vb = rows(shape.num_q_heads), rows(shape.num_kv_heads), rows(shape.num_kv_heads)
    outb = torch.empty_like(qb)
    ws = pa.workspace(shape, 512, 8192 + 80, dev)
    dev_steps = []
    bytes_dec, flops_pre, rows_pre = [], [], []
    for st in steps:
        T, nd = int(st.q_start_loc[-1]), st.num_decode
        rows_n = np.diff(st.q_start_loc)
        pairs = pa.mixed_prefill_pairs(shape, st.seq_lens[:nd], rows_n[nd:], st.seq_lens[nd:] - rows_n[nd:])
        dev_steps.append((T, nd, tod(st.q_start_loc), tod(st.seq_lens), tod(st.slot_mapping), tod(st.block_table),
                          int(st.seq_lens.max()), int(rows_n[nd:].max()) if len(rows_n) > nd else 1, pairs))
        bytes_dec.append(T * shape.num_kv_heads * shape.head_dim * 8 + 4 * T)  # + the decode's, below
        n = rows_n[nd:].tolist()
        flops_pre.append(causal_flops(n, [0] * len(n), shape.num_q_heads, shape.head_dim))
        rows_pre.append(int(sum(n)))

    def run(i, split=True):
        T, nd, qs, lens, slots, bt, ml, mq, pairs = dev_steps[i]
        pa.mixed_step(shape, qb[:T], kb[:T], vb[:T], qs, lens, slots, bt, nd, ml, mq, kp, vp, out=outb[:T], ws=ws,
                      prefill_pairs=pairs if split else None)

    def timed(split):
        for i in range(max(3, warmup)):
            run(i % len(dev_steps), split)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in dev_steps]
        for i in range(len(dev_steps)):
            ev[i][0].record()
            run(i, split)
            ev[i][1].record()
        torch.cuda.synchronize(dev)
        pa.check_device_error()
        return np.array([a.elapsed_time(b) for a, b in ev]) / 1e3

    # The rows each step appends are the same rows to the same slots every
    # pass, so the unpartitioned pass sees the same pools.
    t_shared = timed(False)
    t = timed(True)
    # Accounting pass (untimed): each step again, then the split its plan
    # launch took, for the decode's algorithmic bytes (the rows appended again
    # are the same rows to the same slots).
    for i, st in enumerate(steps):
        run(i)
        torch.cuda.synchronize(dev)
        nd = st.num_decode
        split = pa.planned_split(ws, shape, nd, dev_steps[i][6])
        bytes_dec[i] += decode_step_bytes(shape, st.seq_lens[:nd], split, shape.block_size)["decode"]
    pa.check_device_error()
    bound = np.maximum(np.array(bytes_dec) / (hbm_peak * 1e9), np.array(flops_pre) / (bf16_peak * 1e12))
    del kp, vp
    return {"workload": "512 seqs, log-uniform context [1,8192], Hq 32 / Hkv 8, d 128, B 32, 64 steps, 10 % "
                        "replaced per step by prompts U[16,512]",
            "steps": len(t), "step_ms_mean": round(float(t.mean()) * 1e3, 5),
            "step_ms_mean_unpartitioned": round(float(t_shared.mean()) * 1e3, 5),
            "prefill_pairs_mean": round(float(np.mean([s[8] for s in dev_steps])), 1),
            "step_ms_p10_p90": [round(float(np.percentile(t, 10)) * 1e3, 5), round(float(np.percentile(t, 90)) * 1e3, 5)],
            "decode_append_GB_per_step": round(float(np.mean(bytes_dec)) / 1e9, 4),
            "prefill_rows_per_step": round(float(np.mean(rows_pre)), 1),
            "prefill_GFLOP_per_step": round(float(np.mean(flops_pre)) / 1e9, 2),
            "kv_GBps": round(float(np.sum(bytes_dec) / t.sum()) / 1e9, 1),
            "prefill_tflops": round(float(np.sum(flops_pre) / t.sum()) / 1e12, 1),
            "step_bound_ms_mean": round(float(bound.mean()) * 1e3, 5),
            "frac": round(float(bound.sum() / t.sum()), 4),
            "l2": "inputs larger than L2 (pools 2.3 GB); no flush"}


def measure_chunked_prefill(pa, wl, dev, bf16_peak, iters):
    """Chunked prefill over a cached prefix: 4 sequences, each with 3072
    tokens in the pool and its next 1024-token chunk (bottom-right causal),
    Hq 32 / Hkv 8, d 128, B 16, through pa_prefill with prefix_lens.  FLOPs
    over the unmasked pairs (prefix keys and the chunk's causal triangle)."""
    shape, kp, vp, st, pre = wl.chunked_prefill(pool_device=dev)
    tod = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev) if isinstance(x, np.ndarray) else x.to(dev)
    q, kn, vn = tod(st.q), tod(st.k_new), tod(st.v_new)
    pa.kv_append(shape, kn, vn, tod(st.slot_mapping), kp, vp)
    cu, bt, pl = tod(st.q_start_loc), tod(st.block_table), tod(pre)
    out = torch.empty_like(q)
    flush = l2_flush_buffer(dev)
    t = time_each(dev, lambda: pa.prefill(shape, q, kp, vp, cu, st.max_q_len, prefix_lens=pl, block_table=bt,
                                          out=out), iters, flush)
    pa.check_device_error()
    n = np.diff(st.q_start_loc).tolist()
    fl = causal_flops(n, pre.tolist(), shape.num_q_heads, shape.head_dim)
    del kp, vp
    return {"workload": "4 x (3072 cached + 1024 new rows), Hq 32 / Hkv 8, d 128, B 16",
            "kernel": "prefill_pair_kernel", "ms": round(t * 1e3, 5), "flops": fl,
            "tflops": round(fl / t / 1e12, 1), "frac": round(fl / t / 1e12 / bf16_peak, 4),
            "l2": "flushed (256 MB write) before each launch"}


# ------------------------------------------------------------ CPU oracle --
def oracle_step(oracle, shape, kp_h, vp_h, st, seqs, threads):
    """The oracle's append + decode for the sequences `seqs` of the step."""
    rows = np.asarray(seqs)
    kn = st.k_new[rows].contiguous().view(torch.int16).numpy().view(np.uint16)
    vn = st.v_new[rows].contiguous().view(torch.int16).numpy().view(np.uint16)
    qb = st.q[rows].contiguous().view(torch.int16).numpy().view(np.uint16)
    oracle.kv_append(kn, vn, st.slot_mapping[rows], kp_h, vp_h, inplace=True)
    return oracle.decode(qb, kp_h, vp_h, st.block_table[rows], st.seq_lens[rows], threads=threads)


def cpu_sample(st, seconds_budget, per_token_s):
    """Leading sequences whose decode fits in the time budget (at least 4)."""
    lens = st.seq_lens.astype(np.int64)
    est = np.cumsum(lens) * per_token_s
    k = int(np.searchsorted(est, seconds_budget)) + 1
    return list(range(max(4, min(k, len(lens)))))


def cpu_baseline(shape, kp, vp, st, split, seconds):
    """The oracle on the host cores: whole steps (or a leading sample of the
    sequences when one step would exceed the budget), repeated until about
    `seconds` of CPU work have run."""
    import oracle
    threads = oracle.default_threads()
    kp_h = kp.cpu().view(torch.int16).numpy().view(np.uint16)
    vp_h = vp.cpu().view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    oracle_step(oracle, shape, kp_h, vp_h, st, [0, 1], threads)
    per_tok = (time.perf_counter() - t0) / max(1, int(st.seq_lens[:2].sum()))
    seqs = cpu_sample(st, seconds, per_tok)
    b = decode_step_bytes(shape, st.seq_lens[seqs], split, shape.block_size)["step"]
    reps, t = 0, 0.0
    t0 = time.perf_counter()
    while reps == 0 or t < seconds:
        oracle_step(oracle, shape, kp_h, vp_h, st, seqs, threads)
        reps += 1
        t = time.perf_counter() - t0
    res = {"value": round(b * reps / t / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"{reps} x (append + decode of the first {len(seqs)} of {st.num_seqs} sequences, "
                     f"{int(st.seq_lens[seqs].sum())} context tokens), fp64, {t:.1f} s"}
    # The same oracle on one thread, on a sample sized to about half the budget.
    seqs1 = cpu_sample(st, seconds / 2, per_tok * threads)
    b1 = decode_step_bytes(shape, st.seq_lens[seqs1], split, shape.block_size)["step"]
    reps1, t1 = 0, 0.0
    t0 = time.perf_counter()
    while reps1 == 0 or t1 < seconds / 2:
        oracle_step(oracle, shape, kp_h, vp_h, st, seqs1, 1)
        reps1 += 1
        t1 = time.perf_counter() - t0
    res["single_thread"] = {"value": round(b1 * reps1 / t1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                            "sample": f"{reps1} x (append + decode of the first {len(seqs1)} sequences, "
                                      f"{int(st.seq_lens[seqs1].sum())} context tokens), fp64, {t1:.1f} s"}
    return res


# --------------------------------------------------------- reference arm --
def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_continuous_gb300 import workload as wl
    oracle.build()
    shape, kp, vp, st = wl.llama7b_decode(pool_device="cpu")
    threads = oracle.default_threads()
    kp_h = kp.view(torch.int16).numpy().view(np.uint16)
    vp_h = vp.view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    oracle_step(oracle, shape, kp_h, vp_h, st, [0, 1], threads)
    per_tok = (time.perf_counter() - t0) / max(1, int(st.seq_lens[:2].sum()))
    budget = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    seqs = cpu_sample(st, budget, per_tok)
    for _ in range(args.warmup):
        oracle_step(oracle, shape, kp_h, vp_h, st, seqs, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(oracle, shape, kp_h, vp_h, st, seqs, threads)
    t = time.perf_counter() - t0
    # the bytes of the step without split partials (the oracle makes none; the
    # GPU arm counts the few its plan launch makes)
    b = decode_step_bytes(shape, st.seq_lens[seqs], 1 << 30, shape.block_size)["step"] * args.steps
    v = b / t / 1e9
    sample = (f"each step: append + decode of the first {len(seqs)} of {st.num_seqs} sequences "
              f"({int(st.seq_lens[seqs].sum())} context tokens), fp64 oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefill-iters", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["llama7b_decode", "long_context", "mixed", "churn", "chunked_prefill"],
                    default="llama7b_decode",
                    help="llama7b_decode prints the contract line; the others print secondary measurements")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        run_reference(args, world, rank)
        return
    if args.workload != "llama7b_decode":
        run_other_workload(args, local)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
