"""fp64 CPU oracle for paged KV-cache attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never does, and the two
share no code: the arithmetic lives in ``oracle.c`` (plain C, double
precision), reached here through ``ctypes``.

Every function takes bf16 tensors as their raw 16-bit patterns (``numpy``
``uint16`` arrays) and returns float64 results.  What each one computes, and
the passage it follows, is written beside the C function it wraps:

* ``kv_append``      -- bit copy of new K/V rows into pool slots.
* ``expected_slots`` -- slot = block_table[s][p // B] * B + p % B.
* ``decode``         -- one query token per sequence over its cached context.
* ``prefill``        -- causal attention over packed (ragged) prompts, with an
  optional cached prefix read through the block table.
* ``mixed_step``     -- append, then decode for the first ``num_decode``
  sequences and prefill for the rest.
* ``rope``           -- rotary position embedding of head vectors.
* ``rope_append``    -- rotate the new tokens' queries and keys, then append
  the rotated keys (rounded to bf16) and the values to the pool.
* ``to_bf16``        -- round doubles to bf16 bit patterns.
* ``e4m3_from_float``, ``e4m3_to_double`` -- fp8 (e4m3) codes.
* ``kv_append_fp8``  -- append with quantisation to e4m3 (one scale per KV head).
* ``decode_fp8``     -- decode over e4m3 code pools (value = code * scale).

Parity pins: tests/test_oracle_pins.py checks these functions against a
library routine (torch's scaled-dot-product attention in float64 on dense
gathered inputs), closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "oracle.c"
_BUILD = _HERE / "_build"
_LIB_PATH = _BUILD / "liboracle.so"

OK = 0
ERR_SLOT_RANGE = -1
ERR_SLOT_DUP = -2
ERR_BLOCK_RANGE = -3
ERR_ARG = -4
ERR_NOMEM = -5


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> Path:
    """Compile oracle.c with gcc into oracle/_build/liboracle.so."""
    _BUILD.mkdir(exist_ok=True)
    if (not force and _LIB_PATH.exists()
            and _LIB_PATH.stat().st_mtime >= _SRC.stat().st_mtime):
        return _LIB_PATH
    tmp = _BUILD / f"liboracle.{os.getpid()}.so"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", str(_SRC), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(str(build()))
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.oracle_kv_append.argtypes = [I, I, I, I, I, P, P, P, P, P]
        lib.oracle_expected_slots.argtypes = [I, P, P, P, I, I, P]
        lib.oracle_decode.argtypes = [I, I, I, I, I, I, D, P, P, P, P, I, P, P, I, P, I]
        lib.oracle_prefill.argtypes = [I, I, I, I, I, I, D, P, P, P, P, P, P, I, P, I, P, I]
        lib.oracle_rope.argtypes = [I, I, I, P, P, D, P]
        lib.oracle_to_bf16.argtypes = [ctypes.c_longlong, P, P]
        lib.oracle_e4m3_from_float.argtypes = [ctypes.c_longlong, P, P]
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_longlong, P, P]
        lib.oracle_kv_append_fp8.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P]
        lib.oracle_decode_fp8.argtypes = [I, I, I, I, I, I, D, P, P, P, P, P, P, I, P, P, I, P, I]
        for f in (lib.oracle_kv_append, lib.oracle_expected_slots,
                  lib.oracle_decode, lib.oracle_prefill, lib.oracle_rope, lib.oracle_to_bf16,
                  lib.oracle_e4m3_from_float, lib.oracle_e4m3_to_double, lib.oracle_kv_append_fp8,
                  lib.oracle_decode_fp8):
            f.restype = I
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"expected bf16 bit patterns as uint16, got {a.dtype}")
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(status: int, what: str):
    if status != OK:
        names = {ERR_SLOT_RANGE: "slot out of range", ERR_SLOT_DUP: "duplicate slot",
                 ERR_BLOCK_RANGE: "block index out of range", ERR_ARG: "bad argument",
                 ERR_NOMEM: "out of memory"}
        raise OracleError(f"{what}: {names.get(status, status)}")


def kv_append(k_new, v_new, slot_mapping, k_pool, v_pool, inplace: bool = False):
    """Return (k_pool, v_pool) with the new rows written at their slots:
    copies, or the given arrays themselves with ``inplace`` (they must then be
    contiguous uint16 arrays).

    k_new/v_new: uint16 [T, Hkv, d]; pools: uint16 [N, Hkv, B, d].
    """
    k_new, v_new = _u16(k_new), _u16(v_new)
    if inplace:
        kp, vp = k_pool, v_pool
        assert kp.dtype == np.uint16 and vp.dtype == np.uint16
        assert kp.flags.c_contiguous and vp.flags.c_contiguous
    else:
        kp, vp = _u16(k_pool).copy(), _u16(v_pool).copy()
    sm = _i32(slot_mapping)
    N, Hkv, B, d = kp.shape
    T = sm.shape[0]
    assert k_new.shape == (T, Hkv, d) and v_new.shape == (T, Hkv, d)
    st = _load().oracle_kv_append(T, Hkv, d, B, N, _ptr(k_new), _ptr(v_new), _ptr(sm),
                                  _ptr(kp), _ptr(vp))
    _check(st, "kv_append")
    return kp, vp


def copy_blocks(src_k, src_v, dst_k, dst_v, src_ids, dst_ids):
    """Whole-block copies between pools (Blitzscale docs, sections
    "CacheManager" -- the cache's GPU and CPU regions -- and "migration_queue"):
    return copies of (dst_k, dst_v) with dst[dst_ids[i]] = src[src_ids[i]].
    Every copy reads the source as it was before the call.  Raises on an id
    outside a pool, and -- when src and dst are the same pool -- on a
    destination that is also a source.

    Pools: uint16 [N, Hkv, B, d]; ids: int32 [n].
    """
    sk, sv = _u16(src_k), _u16(src_v)
    dk, dv = _u16(dst_k).copy(), _u16(dst_v).copy()
    si, di = _i32(src_ids), _i32(dst_ids)
    if si.shape != di.shape:
        raise ValueError("src_ids and dst_ids differ in length")
    if sk.shape[1:] != dk.shape[1:]:
        raise ValueError("pools differ in block shape")
    if np.any((si < 0) | (si >= sk.shape[0])) or np.any((di < 0) | (di >= dk.shape[0])):
        raise ValueError("copy_blocks: block id out of range")
    if src_k is dst_k and np.intersect1d(si, di).size:
        raise ValueError("copy_blocks: a destination block is also a source")
    for s_, d_ in zip(si.tolist(), di.tolist()):
        dk[d_] = sk[s_]
        dv[d_] = sv[s_]
    return dk, dv


def expected_slots(q_start_loc, seq_lens, block_table, block_size) -> np.ndarray:
    qs, sl, bt = _i32(q_start_loc), _i32(seq_lens), _i32(block_table)
    S = sl.shape[0]
    out = np.full(int(qs[-1]), -1, dtype=np.int32)
    st = _load().oracle_expected_slots(S, _ptr(qs), _ptr(sl), _ptr(bt), bt.shape[1],
                                       block_size, _ptr(out))
    _check(st, "expected_slots")
    return out


def decode(q, k_pool, v_pool, block_table, seq_lens, scale: float = 0.0,
           pairs=None, threads: int | None = None) -> np.ndarray:
    """fp64 decode attention.  q: uint16 [S, Hq, d]; returns float64 [S, Hq, d],
    or [n, d] for an (s, h) sample list ``pairs`` of shape [n, 2]."""
    q, kp, vp = _u16(q), _u16(k_pool), _u16(v_pool)
    bt, sl = _i32(block_table), _i32(seq_lens)
    S, Hq, d = q.shape
    N, Hkv, B, d2 = kp.shape
    assert d2 == d and vp.shape == kp.shape and bt.shape[0] >= S and sl.shape[0] == S
    pr = None if pairs is None else _i32(pairs).reshape(-1, 2)
    n = S * Hq if pr is None else pr.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    st = _load().oracle_decode(S, Hq, Hkv, d, B, N, float(scale), _ptr(q), _ptr(kp), _ptr(vp),
                               _ptr(bt), bt.shape[1], _ptr(sl), _ptr(pr),
                               0 if pr is None else pr.shape[0], _ptr(out),
                               threads or default_threads())
    _check(st, "decode")
    return out.reshape(S, Hq, d) if pr is None else out


def prefill(q, k, v, cu_seqlens_q, prefix_lens=None, block_table=None,
            num_kv_heads: int | None = None, scale: float = 0.0, pairs=None,
            threads: int | None = None) -> np.ndarray:
    """fp64 causal prefill over packed prompts.

    Paged form (block_table given): k, v are pools uint16 [N, Hkv, B, d] that
    already hold every key of the sequence; prefix_lens[s] (default 0) is the
    number of cached tokens before the prompt rows.
    Dense form (block_table None): k, v are packed uint16 [T, Hkv, d].
    Returns float64 [T, Hq, d], or [n, d] for a (row, h) sample list."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    cu = _i32(cu_seqlens_q)
    S = cu.shape[0] - 1
    T, Hq, d = q.shape
    pre = None if prefix_lens is None else _i32(prefix_lens)
    if block_table is not None:
        bt = _i32(block_table)
        N, Hkv, B, d2 = k.shape
        maxb = bt.shape[1]
    else:
        bt = None
        _, Hkv, d2 = k.shape
        N, B, maxb = 1, 1, 0
    assert d2 == d
    pr = None if pairs is None else _i32(pairs).reshape(-1, 2)
    n = T * Hq if pr is None else pr.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    st = _load().oracle_prefill(S, Hq, Hkv, d, B, N, float(scale), _ptr(q), _ptr(k), _ptr(v),
                                _ptr(cu), _ptr(pre), _ptr(bt), maxb, _ptr(pr),
                                0 if pr is None else pr.shape[0], _ptr(out),
                                threads or default_threads())
    _check(st, "prefill")
    return out.reshape(T, Hq, d) if pr is None else out


def mixed_step(q, k_new, v_new, q_start_loc, seq_lens, slot_mapping, block_table,
               num_decode: int, k_pool, v_pool, scale: float = 0.0,
               threads: int | None = None):
    """One continuous-batching step: append every new token, then decode
    attention for sequences [0, num_decode) (one query row each) and causal
    prefill with prefix for the rest.  Returns (out float64 [T, Hq, d],
    k_pool, v_pool) with the pools after the append."""
    qs, sl, bt = _i32(q_start_loc), _i32(seq_lens), _i32(block_table)
    kp, vp = kv_append(k_new, v_new, slot_mapping, k_pool, v_pool)
    q = _u16(q)
    T, Hq, d = q.shape
    out = np.zeros((T, Hq, d), dtype=np.float64)
    nd = int(num_decode)
    if nd > 0:
        assert np.all(qs[1:nd + 1] - qs[:nd] == 1)
        rows = qs[:nd]
        out[rows] = decode(q[rows], kp, vp, bt[:nd], sl[:nd], scale=scale, threads=threads)
    S = sl.shape[0]
    if S > nd:
        r0, r1 = int(qs[nd]), int(qs[S])
        cu = qs[nd:] - r0
        n = cu[1:] - cu[:-1]
        pre = sl[nd:] - n
        out[r0:r1] = prefill(q[r0:r1], kp, vp, cu, prefix_lens=pre, block_table=bt[nd:],
                             scale=scale, threads=threads)
    return out, kp, vp


def rope(x, positions, theta: float = 10000.0) -> np.ndarray:
    """fp64 rotary embedding (oracle.c: ``oracle_rope``).  x: uint16 bits
    [T, H, d]; positions: int32 [T].  Returns float64 [T, H, d]."""
    xb = _u16(x)
    if xb.ndim != 3:
        raise ValueError("x must be [T, H, d]")
    T, H, d = xb.shape
    pos = _i32(positions)
    if pos.shape != (T,):
        raise ValueError("positions must be [T]")
    out = np.zeros((T, H, d), dtype=np.float64)
    _check(_load().oracle_rope(T, H, d, _ptr(xb), _ptr(pos), ctypes.c_double(float(theta)), _ptr(out)), "rope")
    return out


def to_bf16(x) -> np.ndarray:
    """Round float64 values to bf16 bit patterns (ties to even)."""
    xa = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.zeros(xa.shape, dtype=np.uint16)
    _check(_load().oracle_to_bf16(ctypes.c_longlong(xa.size), _ptr(xa), _ptr(out)), "to_bf16")
    return out


def rope_append(q, k_new, v_new, positions, slot_mapping, k_pool, v_pool, theta: float = 10000.0):
    """The new tokens' queries and keys rotated (``rope``), the rotated keys
    rounded to bf16 and appended with the values (``kv_append``).  Returns
    (q_rot float64, k_rot float64, k_pool, v_pool)."""
    q_rot = rope(q, positions, theta)
    k_rot = rope(k_new, positions, theta)
    k_pool2, v_pool2 = kv_append(to_bf16(k_rot), v_new, slot_mapping, k_pool, v_pool)
    return q_rot, k_rot, k_pool2, v_pool2


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.uint8))


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def e4m3_from_float(x) -> np.ndarray:
    """float32 values -> e4m3 codes (nearest, ties to even, saturating)."""
    xa = _f32(x)
    out = np.zeros(xa.shape, dtype=np.uint8)
    _check(_load().oracle_e4m3_from_float(ctypes.c_longlong(xa.size), _ptr(xa), _ptr(out)), "e4m3_from_float")
    return out


def e4m3_to_double(codes) -> np.ndarray:
    c = _u8(codes)
    out = np.zeros(c.shape, dtype=np.float64)
    _check(_load().oracle_e4m3_to_double(ctypes.c_longlong(c.size), _ptr(c), _ptr(out)), "e4m3_to_double")
    return out


def kv_append_fp8(k_new, v_new, slot_mapping, k_scale, v_scale, k_pool, v_pool):
    """Quantising append (oracle.c: ``oracle_kv_append_fp8``).  k_new, v_new:
    uint16 bf16 bits [T, Hkv, d]; scales float32 [Hkv]; pools uint8 codes
    [N, Hkv, B, d].  Returns new pools."""
    kn, vn = _u16(k_new), _u16(v_new)
    kp, vp = _u8(k_pool).copy(), _u8(v_pool).copy()
    sl = _i32(slot_mapping)
    N, H, B, d = kp.shape
    _check(_load().oracle_kv_append_fp8(sl.shape[0], H, d, B, N, _ptr(kn), _ptr(vn), _ptr(sl),
                                        _ptr(_f32(k_scale)), _ptr(_f32(v_scale)), _ptr(kp), _ptr(vp)),
           "kv_append_fp8")
    return kp, vp


def decode_fp8(q, k_pool, v_pool, k_scale, v_scale, block_table, seq_lens, scale: float = 0.0,
               pairs=None, threads: int | None = None) -> np.ndarray:
    """fp64 decode over e4m3 code pools (value = code * scale of the KV
    head).  q: uint16 [S, Hq, d]; returns float64 [S, Hq, d] or [n, d]."""
    qb, kp, vp = _u16(q), _u8(k_pool), _u8(v_pool)
    bt, sl = _i32(block_table), _i32(seq_lens)
    S, Hq, d = qb.shape
    N, H, B, _ = kp.shape
    pr = None if pairs is None else _i32(pairs)
    n = S * Hq if pr is None else pr.shape[0]
    out = np.zeros((n, d), dtype=np.float64)
    _check(_load().oracle_decode_fp8(S, Hq, H, d, B, N, ctypes.c_double(scale), _ptr(qb), _ptr(kp), _ptr(vp),
                                     _ptr(_f32(k_scale)), _ptr(_f32(v_scale)), _ptr(bt), bt.shape[1], _ptr(sl),
                                     _ptr(pr), 0 if pr is None else pr.shape[0], _ptr(out),
                                     threads or default_threads()), "decode_fp8")
    return out.reshape(S, Hq, d) if pr is None else out

