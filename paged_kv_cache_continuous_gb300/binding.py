"""Thin ctypes binding of libpagedattn (include/pa.h, include/pa_alloc.h).

Argument marshalling only: torch tensors become device pointers, the current
torch stream becomes the cudaStream_t, and every non-zero status raises
``PagedAttnError`` with the library's message.  All arithmetic runs in the
library's CUDA kernels; there is no fallback path.  If the shared library has
not been built, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

import numpy as np
import torch

from . import build as _build

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE = 3
ERR_CUDA = 4
ERR_BAD_INDEX = 5
ERR_NO_BLOCKS = 6
ERR_TIMEOUT = 7

# Every symbol the two headers declare (checked by the tests).
EXPORTS = [
    "pa_version", "pa_workspace_size", "pa_decode_plan", "pa_kv_append", "pa_decode", "pa_decode_append",
    "pa_decode_noalloc", "pa_prefill", "pa_mixed_step", "pa_mixed_step_split", "pa_mixed_prefill_pairs",
    "pa_copy_blocks", "pa_rope_append",
    "pa_kv_append_fp8", "pa_decode_fp8", "pa_set_validation", "pa_check_device_error", "pa_last_error",
    "pa_set_decode_split", "pa_set_prefill_pairs",
    "pa_alloc_create", "pa_alloc_destroy", "pa_alloc_ensure", "pa_alloc_release",
    "pa_alloc_num_free", "pa_alloc_num_blocks_of", "pa_alloc_block_table",
    "pa_sched_create", "pa_sched_destroy", "pa_sched_submit", "pa_sched_cancel", "pa_sched_plan",
    "pa_sched_commit", "pa_sched_stats",
    "pa_alloc_slot_mapping",
]


class PagedAttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"libpagedattn error {code}: {msg}")
        self.code = code


class PaShape(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("scale", ctypes.c_float)]


class SchedParams(ctypes.Structure):
    _fields_ = [("max_batch_prefill_tokens", ctypes.c_int), ("max_batch_total_tokens", ctypes.c_int),
                ("max_waiting_tokens", ctypes.c_int), ("waiting_served_ratio", ctypes.c_float),
                ("max_batch_size", ctypes.c_int), ("chunking", ctypes.c_int),
                ("max_input_tokens", ctypes.c_int), ("max_total_tokens", ctypes.c_int)]


_lib = None


def library_path() -> Path:
    return _build.LIB


def load():
    """Load the in-tree libpagedattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not path.exists():
        raise RuntimeError(f"{path} is missing: build it with paged_kv_cache_continuous_gb300.build.build()")
    lib = ctypes.CDLL(str(path))
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    SP = ctypes.POINTER(PaShape)
    sig = {
        "pa_version": ([], I),
        "pa_workspace_size": ([SP, I, I, ctypes.POINTER(S)], I),
        "pa_decode_plan": ([SP, I, I, ctypes.POINTER(I), ctypes.POINTER(I)], I),
        "pa_kv_append": ([SP, P, P, P, I, P, P, P], I),
        "pa_decode": ([SP, P, P, P, P, I, P, I, I, P, P, S, P], I),
        "pa_decode_noalloc": ([SP, P, P, P, P, I, P, I, I, P, P], I),
        "pa_decode_append": ([SP, P, P, P, P, P, P, P, I, P, I, I, P, P, S, P], I),
        "pa_prefill": ([SP, P, P, P, P, P, P, I, I, I, I, P, P], I),
        "pa_mixed_step": ([SP, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, P, S, P], I),
        "pa_mixed_step_split": ([SP, P, P, P, P, P, P, P, I, I, I, I, I, I, P, P, P, P, S, P, I], I),
        "pa_mixed_prefill_pairs": ([SP, P, I, P, P, I, I, ctypes.POINTER(I)], I),
        "pa_copy_blocks": ([SP, P, P, I, P, P, I, P, P, I, P], I),
        "pa_rope_append": ([SP, P, P, P, P, P, I, ctypes.c_float, P, P, P, P], I),
        "pa_kv_append_fp8": ([SP, P, P, P, I, P, P, P, P, P], I),
        "pa_decode_fp8": ([SP, P, P, P, P, P, P, I, P, I, I, P, P, S, P], I),
        "pa_set_validation": ([I], I),
        "pa_check_device_error": ([P], I),
        "pa_last_error": ([], ctypes.c_char_p),
        "pa_set_decode_split": ([I], I),
        "pa_set_prefill_pairs": ([I], I),
        "pa_alloc_create": ([I, I, P], P),
        "pa_alloc_destroy": ([P], None),
        "pa_alloc_ensure": ([P, ctypes.c_int64, I], I),
        "pa_alloc_release": ([P, ctypes.c_int64], I),
        "pa_alloc_num_free": ([P], I),
        "pa_alloc_num_blocks_of": ([P, ctypes.c_int64], I),
        "pa_alloc_block_table": ([P, P, I, I, ctypes.c_int32, P], I),
        "pa_alloc_slot_mapping": ([P, P, P, P, I, P], I),
        "pa_sched_create": ([ctypes.POINTER(SchedParams), I, I], P),
        "pa_sched_destroy": ([P], None),
        "pa_sched_submit": ([P, ctypes.c_int64, I, I], I),
        "pa_sched_cancel": ([P, ctypes.c_int64], I),
        "pa_sched_plan": ([P, I, I, I, P, P, P, P, P, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I)], I),
        "pa_sched_commit": ([P, P, I, ctypes.POINTER(I)], I),
        "pa_sched_stats": ([P, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I)], I),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def _check(rc: int):
    if rc != OK:
        raise PagedAttnError(rc, load().pa_last_error().decode())


def _shape(shape) -> PaShape:
    return PaShape(int(shape.num_q_heads), int(shape.num_kv_heads), int(shape.head_dim),
                   int(shape.block_size), int(shape.num_blocks), float(getattr(shape, "scale", 0.0)))


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to libpagedattn must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _i32(t: torch.Tensor, name: str):
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return _ptr(t)


def _bf16(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    return _ptr(t)


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def version() -> int:
    return load().pa_version()


def workspace_size(shape, max_seqs: int, max_seq_len: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().pa_workspace_size(ctypes.byref(_shape(shape)), int(max_seqs), int(max_seq_len),
                                    ctypes.byref(n)))
    return n.value


def decode_plan(shape, num_seqs: int, max_seq_len: int) -> tuple[int, int]:
    """(tokens per split, splits of the longest sequence) used by decode."""
    a, b = ctypes.c_int(0), ctypes.c_int(0)
    _check(load().pa_decode_plan(ctypes.byref(_shape(shape)), int(num_seqs), int(max_seq_len),
                                 ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def planned_split(ws: torch.Tensor, shape, num_seqs: int, max_seq_len: int) -> int:
    """Tokens per split that the last decode of (num_seqs, max_seq_len) with
    workspace `ws` used (its plan launch may take a multiple of decode_plan's
    split): the plan's second counter, after the partials and the items."""
    _, max_splits = decode_plan(shape, num_seqs, max_seq_len)
    n = num_seqs * shape.num_q_heads * max_splits
    partials = ((n * shape.head_dim * 4 + n * 2 * 4 + 15) & ~15) if max_splits > 1 else 0
    at = partials + num_seqs * max(max_splits, 1) * shape.num_kv_heads * 16
    return int(ws[at + 4:at + 8].cpu().view(torch.int32)[0])


def workspace(shape, max_seqs: int, max_seq_len: int, device="cuda") -> torch.Tensor:
    """A caller-owned workspace buffer of the size pa_workspace_size reports."""
    n = workspace_size(shape, max_seqs, max_seq_len)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def kv_append(shape, k_new, v_new, slot_mapping, k_pool, v_pool, stream=None):
    T = int(slot_mapping.shape[0])
    _check(load().pa_kv_append(ctypes.byref(_shape(shape)), _bf16(k_new, "k_new"), _bf16(v_new, "v_new"),
                               _i32(slot_mapping, "slot_mapping"), T, _bf16(k_pool, "k_pool"),
                               _bf16(v_pool, "v_pool"), _stream(stream)))


def copy_blocks(shape, src_k, src_v, dst_k, dst_v, src_ids, dst_ids, stream=None):
    """dst_k[dst_ids[i]] = src_k[src_ids[i]] (and V) for whole blocks.  Pools are
    [N, Hkv, B, d] bf16 tensors on the GPU or in pinned host memory; the id
    arrays are int32 on the GPU."""
    for t, name in ((src_k, "src_k"), (src_v, "src_v"), (dst_k, "dst_k"), (dst_v, "dst_v")):
        if not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    n = int(src_ids.shape[0])
    if int(dst_ids.shape[0]) != n:
        raise ValueError("src_ids and dst_ids differ in length")
    _check(load().pa_copy_blocks(ctypes.byref(_shape(shape)), _bf16(src_k, "src_k"), _bf16(src_v, "src_v"),
                                 int(src_k.shape[0]), _bf16(dst_k, "dst_k"), _bf16(dst_v, "dst_v"),
                                 int(dst_k.shape[0]), _i32(src_ids, "src_ids"), _i32(dst_ids, "dst_ids"), n,
                                 _stream(stream)))


def rope_append(shape, q, k_new, v_new, positions, slot_mapping, k_pool, v_pool, q_out=None,
                theta: float = 10000.0, stream=None) -> torch.Tensor:
    """pa_rope_append: rotate the new tokens' queries (into q_out, a new tensor
    unless given; pass q to rotate in place) and keys, and append the rotated
    keys and the values to the pools.  Returns q_out."""
    T = int(slot_mapping.shape[0])
    if q_out is None:
        q_out = torch.empty_like(q)
    _check(load().pa_rope_append(ctypes.byref(_shape(shape)), _bf16(q, "q"), _bf16(k_new, "k_new"),
                                 _bf16(v_new, "v_new"), _i32(positions, "positions"),
                                 _i32(slot_mapping, "slot_mapping"), T, float(theta), _bf16(q_out, "q_out"),
                                 _bf16(k_pool, "k_pool"), _bf16(v_pool, "v_pool"), _stream(stream)))
    return q_out


def _u8(t: torch.Tensor, name: str):
    if t.dtype != torch.uint8:
        raise TypeError(f"{name} must be uint8 (e4m3 codes)")
    return _ptr(t)


def _f32(t: torch.Tensor, name: str):
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    return _ptr(t)


def kv_append_fp8(shape, k_new, v_new, slot_mapping, k_scale, v_scale, k_pool, v_pool, stream=None):
    """pa_kv_append_fp8: quantising append into uint8 (e4m3 code) pools."""
    T = int(slot_mapping.shape[0])
    _check(load().pa_kv_append_fp8(ctypes.byref(_shape(shape)), _bf16(k_new, "k_new"), _bf16(v_new, "v_new"),
                                   _i32(slot_mapping, "slot_mapping"), T, _f32(k_scale, "k_scale"),
                                   _f32(v_scale, "v_scale"), _u8(k_pool, "k_pool"), _u8(v_pool, "v_pool"),
                                   _stream(stream)))


def decode_fp8(shape, q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, max_seq_len: int, out=None,
               ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """pa_decode_fp8: decode over uint8 (e4m3 code) pools with per-KV-head scales."""
    S = int(seq_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(shape, S, max_seq_len, q.device)
    _check(load().pa_decode_fp8(ctypes.byref(_shape(shape)), _bf16(q, "q"), _u8(k_pool, "k_pool"),
                                _u8(v_pool, "v_pool"), _f32(k_scale, "k_scale"), _f32(v_scale, "v_scale"),
                                _i32(block_table, "block_table"), int(block_table.shape[1]),
                                _i32(seq_lens, "seq_lens"), S, int(max_seq_len), _bf16(out, "out"), _ptr(ws),
                                ws.numel(), _stream(stream)))
    return out


def decode(shape, q, k_pool, v_pool, block_table, seq_lens, max_seq_len: int, out=None,
           ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    S = int(seq_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(shape, S, max_seq_len, q.device)
    _check(load().pa_decode(ctypes.byref(_shape(shape)), _bf16(q, "q"), _bf16(k_pool, "k_pool"),
                            _bf16(v_pool, "v_pool"), _i32(block_table, "block_table"),
                            int(block_table.shape[1]), _i32(seq_lens, "seq_lens"), S, int(max_seq_len),
                            _bf16(out, "out"), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def decode_append(shape, q, k_new, v_new, slot_mapping, k_pool, v_pool, block_table, seq_lens, max_seq_len: int,
                  out=None, ws: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """pa_decode_append: each sequence's new row appended at its slot, then
    decode, in one launch (plus the merge)."""
    S = int(seq_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(shape, S, max_seq_len, q.device)
    _check(load().pa_decode_append(ctypes.byref(_shape(shape)), _bf16(q, "q"), _bf16(k_new, "k_new"),
                                   _bf16(v_new, "v_new"), _i32(slot_mapping, "slot_mapping"),
                                   _bf16(k_pool, "k_pool"), _bf16(v_pool, "v_pool"),
                                   _i32(block_table, "block_table"), int(block_table.shape[1]),
                                   _i32(seq_lens, "seq_lens"), S, int(max_seq_len), _bf16(out, "out"), _ptr(ws),
                                   ws.numel(), _stream(stream)))
    return out


def decode_noalloc(shape, q, k_pool, v_pool, block_table, seq_lens, max_seq_len: int, out=None,
                   stream=None) -> torch.Tensor:
    """pa_decode_noalloc: decode with the library's built-in split-K scratch
    (for callers that cannot allocate a workspace); same result as decode()."""
    S = int(seq_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    _check(load().pa_decode_noalloc(ctypes.byref(_shape(shape)), _bf16(q, "q"), _bf16(k_pool, "k_pool"),
                                    _bf16(v_pool, "v_pool"), _i32(block_table, "block_table"),
                                    int(block_table.shape[1]), _i32(seq_lens, "seq_lens"), S,
                                    int(max_seq_len), _bf16(out, "out"), _stream(stream)))
    return out


def prefill(shape, q, k, v, cu_seqlens, max_q_len: int, prefix_lens=None, block_table=None,
            out=None, stream=None) -> torch.Tensor:
    S = int(cu_seqlens.shape[0]) - 1
    if out is None:
        out = torch.empty_like(q)
    mb = int(block_table.shape[1]) if block_table is not None else 0
    _check(load().pa_prefill(ctypes.byref(_shape(shape)), _bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"),
                             _i32(cu_seqlens, "cu_seqlens"),
                             None if prefix_lens is None else _i32(prefix_lens, "prefix_lens"),
                             None if block_table is None else _i32(block_table, "block_table"), mb, S,
                             int(q.shape[0]), int(max_q_len), _bf16(out, "out"), _stream(stream)))
    return out


def mixed_step(shape, q, k_new, v_new, q_start_loc, seq_lens, slot_mapping, block_table,
               num_decode: int, max_seq_len: int, max_q_len: int, k_pool, v_pool, out=None,
               ws: torch.Tensor | None = None, stream=None, prefill_pairs: int | None = None) -> torch.Tensor:
    """pa_mixed_step, or pa_mixed_step_split when prefill_pairs is given."""
    S = int(seq_lens.shape[0])
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(shape, max(num_decode, 1), max_seq_len, q.device)
    args = (ctypes.byref(_shape(shape)), _bf16(q, "q"), _bf16(k_new, "k_new"),
            _bf16(v_new, "v_new"), _i32(q_start_loc, "q_start_loc"),
            _i32(seq_lens, "seq_lens"), _i32(slot_mapping, "slot_mapping"),
            _i32(block_table, "block_table"), int(block_table.shape[1]), S,
            int(num_decode), int(q.shape[0]), int(max_seq_len), int(max_q_len),
            _bf16(k_pool, "k_pool"), _bf16(v_pool, "v_pool"), _bf16(out, "out"),
            _ptr(ws), ws.numel(), _stream(stream))
    if prefill_pairs is None:
        _check(load().pa_mixed_step(*args))
    else:
        _check(load().pa_mixed_step_split(*args, int(prefill_pairs)))
    return out


def mixed_prefill_pairs(shape, decode_lens, prompt_rows, prefix_lens=None, num_sms: int = 0) -> int:
    """Prefill CTA pairs for pa_mixed_step_split from host lengths (sequences of ints)."""
    d = np.ascontiguousarray(np.asarray(decode_lens, dtype=np.int32).reshape(-1))
    r = np.ascontiguousarray(np.asarray(prompt_rows, dtype=np.int32).reshape(-1))
    p = None if prefix_lens is None else np.ascontiguousarray(np.asarray(prefix_lens, dtype=np.int32).reshape(-1))
    if p is not None and p.shape[0] != r.shape[0]:
        raise ValueError("prefix_lens and prompt_rows differ in length")
    out = ctypes.c_int(0)
    _check(load().pa_mixed_prefill_pairs(ctypes.byref(_shape(shape)), d.ctypes.data if d.size else None,
                                         int(d.size), r.ctypes.data if r.size else None,
                                         None if p is None or not p.size else p.ctypes.data, int(r.size),
                                         int(num_sms), ctypes.byref(out)))
    return out.value


def set_validation(on: bool):
    _check(load().pa_set_validation(1 if on else 0))


def set_decode_split(tokens: int):
    _check(load().pa_set_decode_split(int(tokens)))


def set_prefill_pairs(pairs: int):
    _check(load().pa_set_prefill_pairs(int(pairs)))


def check_device_error(stream=None):
    """Synchronise the stream and raise if a kernel recorded an error."""
    _check(load().pa_check_device_error(_stream(stream)))


class BlockAllocator:
    """The library's host free-list allocator (include/pa_alloc.h)."""

    def __init__(self, num_blocks: int, block_size: int, initial_order=None):
        lib = load()
        self.block_size = int(block_size)
        order = None
        if initial_order is not None:
            self._order = np.ascontiguousarray(np.asarray(initial_order, dtype=np.int32))
            order = self._order.ctypes.data_as(ctypes.c_void_p)
        self._h = lib.pa_alloc_create(int(num_blocks), int(block_size), order)
        if not self._h:
            raise PagedAttnError(ERR_INVALID_ARG, "pa_alloc_create failed")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h and _lib is not None:
            _lib.pa_alloc_destroy(h)
            self._h = None

    def ensure(self, seq: int, num_tokens: int):
        rc = load().pa_alloc_ensure(self._h, int(seq), int(num_tokens))
        if rc != OK:
            raise PagedAttnError(rc, "no free blocks" if rc == ERR_NO_BLOCKS else "bad argument")

    def release(self, seq: int):
        rc = load().pa_alloc_release(self._h, int(seq))
        if rc != OK:
            raise PagedAttnError(rc, "unknown sequence")

    def num_free(self) -> int:
        return load().pa_alloc_num_free(self._h)

    def num_blocks_of(self, seq: int) -> int:
        return load().pa_alloc_num_blocks_of(self._h, int(seq))

    def block_table(self, seqs, width: int, fill: int = -1) -> np.ndarray:
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        out = np.empty((len(ids), int(width)), dtype=np.int32)
        rc = load().pa_alloc_block_table(self._h, ids.ctypes.data_as(ctypes.c_void_p), len(ids), int(width),
                                         int(fill), out.ctypes.data_as(ctypes.c_void_p))
        if rc != OK:
            raise PagedAttnError(rc, "block_table failed")
        return out

    def slot_mapping(self, seqs, n_new, total_after) -> np.ndarray:
        ids = np.ascontiguousarray(np.asarray(seqs, dtype=np.int64))
        nn = np.ascontiguousarray(np.asarray(n_new, dtype=np.int32))
        ta = np.ascontiguousarray(np.asarray(total_after, dtype=np.int32))
        out = np.empty(int(nn.sum()), dtype=np.int32)
        rc = load().pa_alloc_slot_mapping(self._h, ids.ctypes.data_as(ctypes.c_void_p),
                                          nn.ctypes.data_as(ctypes.c_void_p), ta.ctypes.data_as(ctypes.c_void_p),
                                          len(ids), out.ctypes.data_as(ctypes.c_void_p))
        if rc != OK:
            raise PagedAttnError(rc, "slot_mapping failed")
        return out


class Scheduler:
    """The host continuous-batching scheduler (include/pa_sched.h).  plan()
    returns the arrays of one pa_mixed_step (numpy, host), or None when
    nothing is to run; commit() advances the step and returns the finished
    request ids."""

    def __init__(self, num_blocks: int, block_size: int, max_batch_prefill_tokens: int = 4096,
                 max_batch_total_tokens: int = 0, max_waiting_tokens: int = 20, waiting_served_ratio: float = 1.2,
                 max_batch_size: int = 0, chunking: bool = False, max_input_tokens: int = 1024,
                 max_total_tokens: int = 2048, max_seqs: int = 4096, max_tokens: int = 65536, width: int = 1024):
        lib = load()
        self.params = SchedParams(max_batch_prefill_tokens, max_batch_total_tokens, max_waiting_tokens,
                                  waiting_served_ratio, max_batch_size, int(chunking), max_input_tokens,
                                  max_total_tokens)
        self._h = lib.pa_sched_create(ctypes.byref(self.params), int(num_blocks), int(block_size))
        if not self._h:
            raise ValueError("pa_sched_create: bad arguments")
        self.max_seqs, self.max_tokens, self.width = max_seqs, max_tokens, width
        self._ids = np.zeros(max_seqs, dtype=np.int64)
        self._qs = np.zeros(max_seqs + 1, dtype=np.int32)
        self._lens = np.zeros(max_seqs, dtype=np.int32)
        self._bt = np.zeros((max_seqs, width), dtype=np.int32)
        self._slots = np.zeros(max_tokens, dtype=np.int32)
        self._fin = np.zeros(max_seqs, dtype=np.int64)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            load().pa_sched_destroy(h)
            self._h = None

    def submit(self, request_id: int, input_tokens: int, max_new_tokens: int):
        _check(load().pa_sched_submit(self._h, int(request_id), int(input_tokens), int(max_new_tokens)))

    def cancel(self, request_id: int):
        _check(load().pa_sched_cancel(self._h, int(request_id)))

    def plan(self):
        S, D, T = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
        p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
        _check(load().pa_sched_plan(self._h, self.max_seqs, self.max_tokens, self.width, p(self._ids), p(self._qs),
                                    p(self._lens), p(self._bt), p(self._slots), ctypes.byref(S), ctypes.byref(D),
                                    ctypes.byref(T)))
        if S.value == 0:
            return None
        n = S.value
        return {"seq_ids": self._ids[:n].copy(), "q_start_loc": self._qs[:n + 1].copy(),
                "seq_lens": self._lens[:n].copy(), "block_table": self._bt[:n].copy(),
                "slot_mapping": self._slots[:T.value].copy(), "num_decode": D.value, "num_tokens": T.value}

    def commit(self):
        nf = ctypes.c_int(0)
        _check(load().pa_sched_commit(self._h, self._fin.ctypes.data_as(ctypes.c_void_p), self.max_seqs,
                                      ctypes.byref(nf)))
        return self._fin[:min(nf.value, self.max_seqs)].tolist()

    def stats(self):
        q, r, f, w = (ctypes.c_int(0) for _ in range(4))
        _check(load().pa_sched_stats(self._h, ctypes.byref(q), ctypes.byref(r), ctypes.byref(f), ctypes.byref(w)))
        return {"queued": q.value, "running": r.value, "free_blocks": f.value, "waiting_steps": w.value}

