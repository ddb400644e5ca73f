"""The C-ABI library loads and exports every declared symbol; host-side
argument checks reject bad calls before anything reaches a GPU (CPU only)."""
import ctypes
import re
from pathlib import Path

import pytest

from paged_kv_cache_continuous_gb300 import binding, build

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    names = set()
    for h in (ROOT / "include").glob("*.h"):
        text = re.sub(r"/\*.*?\*/", "", h.read_text(), flags=re.S)
        names |= set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    declared = declared_functions()
    assert declared == set(binding.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_version(lib):
    assert lib.pa_version() >= 100


def _shape(**kw):
    d = dict(num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16, num_blocks=10, scale=0.0)
    d.update(kw)
    return binding.PaShape(**d)


DUMMY = ctypes.c_void_p(0x1000)  # never dereferenced: every case fails on the host first


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), binding.ERR_UNSUPPORTED),
    (dict(block_size=8), binding.ERR_UNSUPPORTED),
    (dict(num_q_heads=6, num_kv_heads=4), binding.ERR_UNSUPPORTED),
    (dict(num_q_heads=34, num_kv_heads=2), binding.ERR_UNSUPPORTED),
    (dict(num_blocks=0), binding.ERR_INVALID_ARG),
    (dict(scale=-1.0), binding.ERR_INVALID_ARG),
])
def test_bad_shapes_rejected(lib, kw, code):
    sh = _shape(**kw)
    rc = lib.pa_kv_append(ctypes.byref(sh), DUMMY, DUMMY, DUMMY, 4, DUMMY, DUMMY, None)
    assert rc == code
    assert lib.pa_last_error()


def test_null_and_misaligned_pointers(lib):
    sh = _shape()
    assert lib.pa_kv_append(ctypes.byref(sh), None, DUMMY, DUMMY, 4, DUMMY, DUMMY, None) == binding.ERR_INVALID_ARG
    odd = ctypes.c_void_p(0x1002)
    assert lib.pa_kv_append(ctypes.byref(sh), odd, DUMMY, DUMMY, 4, DUMMY, DUMMY, None) == binding.ERR_INVALID_ARG
    assert lib.pa_decode(ctypes.byref(sh), DUMMY, DUMMY, DUMMY, None, 4, DUMMY, 3, 64, DUMMY, None, 0,
                         None) == binding.ERR_INVALID_ARG
    # max_seq_len that cannot fit in the table width
    assert lib.pa_decode(ctypes.byref(sh), DUMMY, DUMMY, DUMMY, DUMMY, 4, DUMMY, 3, 65, DUMMY, None, 0,
                         None) == binding.ERR_INVALID_ARG
    # prefix lengths without a block table
    assert lib.pa_prefill(ctypes.byref(sh), DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, None, 0, 2, 10, 8, DUMMY,
                          None) == binding.ERR_INVALID_ARG
    # decode sequences must come first and be covered by the rows
    assert lib.pa_mixed_step(ctypes.byref(sh), DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, 4, 2, 3, 8,
                             64, 8, DUMMY, DUMMY, DUMMY, DUMMY, 0, None) == binding.ERR_INVALID_ARG


def test_copy_blocks_host_checks(lib):
    sh = _shape()
    odd = ctypes.c_void_p(0x1002)
    # negative sizes, NULL and misaligned pools fail before any launch
    assert lib.pa_copy_blocks(ctypes.byref(sh), DUMMY, DUMMY, 4, DUMMY, DUMMY, 4, DUMMY, DUMMY, -1,
                              None) == binding.ERR_INVALID_ARG
    assert lib.pa_copy_blocks(ctypes.byref(sh), DUMMY, DUMMY, -4, DUMMY, DUMMY, 4, DUMMY, DUMMY, 1,
                              None) == binding.ERR_INVALID_ARG
    assert lib.pa_copy_blocks(ctypes.byref(sh), DUMMY, None, 4, DUMMY, DUMMY, 4, DUMMY, DUMMY, 1,
                              None) == binding.ERR_INVALID_ARG
    assert lib.pa_copy_blocks(ctypes.byref(sh), DUMMY, DUMMY, 4, odd, DUMMY, 4, DUMMY, DUMMY, 1,
                              None) == binding.ERR_INVALID_ARG
    bad = _shape(head_dim=96)
    assert lib.pa_copy_blocks(ctypes.byref(bad), DUMMY, DUMMY, 4, DUMMY, DUMMY, 4, DUMMY, DUMMY, 1,
                              None) == binding.ERR_UNSUPPORTED
    # nothing to copy: a no-op even with NULL pointers
    assert lib.pa_copy_blocks(ctypes.byref(sh), None, None, 0, None, None, 0, None, None, 0, None) == binding.OK


def test_empty_calls_are_noops(lib):
    sh = _shape()
    assert lib.pa_kv_append(ctypes.byref(sh), None, None, None, 0, None, None, None) == binding.OK
    assert lib.pa_decode(ctypes.byref(sh), None, None, None, None, 0, None, 0, 0, None, None, 0, None) == binding.OK
    assert lib.pa_last_error() == b""


def _ws_bytes(S, Hq, Hkv, d, splits):
    """The documented workspace: split partials (fp32 acc and (max, sum) per
    sequence, query head and split, rounded up to 16 bytes; none for one
    split), then the plan's work items (16 bytes per sequence, split and KV
    head), its 16 bytes of counters, 8 bytes per sequence and, when anything
    can split, a merge count per sequence and KV head (4 bytes)."""
    partials = -(-(S * Hq * splits * (d + 2) * 4) // 16) * 16 if splits > 1 else 0
    return partials + S * splits * Hkv * 16 + 16 + S * 8 + (S * Hkv * 4 if splits > 1 else 0)


def test_workspace_size(lib):
    sh = binding.PaShape(32, 8, 128, 16, 100, 0.0)
    n = ctypes.c_size_t()
    assert lib.pa_workspace_size(ctypes.byref(sh), 128, 256, ctypes.byref(n)) == 0
    assert n.value == _ws_bytes(128, 32, 8, 128, 1)  # one split: the plan only
    assert lib.pa_workspace_size(ctypes.byref(sh), 128, 2049, ctypes.byref(n)) == 0
    splits = -(-2049 // 256)
    assert n.value == _ws_bytes(128, 32, 8, 128, splits)
    assert lib.pa_set_decode_split(64) == 0
    assert lib.pa_workspace_size(ctypes.byref(sh), 2, 2049, ctypes.byref(n)) == 0
    assert n.value == _ws_bytes(2, 32, 8, 128, -(-2049 // 64))
    assert lib.pa_set_decode_split(0) == 0
    assert lib.pa_set_decode_split(-1) == binding.ERR_INVALID_ARG
    assert lib.pa_set_prefill_pairs(3) == 0
    assert lib.pa_set_prefill_pairs(0) == 0
    assert lib.pa_set_prefill_pairs(-1) == binding.ERR_INVALID_ARG


def _pairs(lib, sh, dec, rows, prefix=None, sms=152):
    arr = lambda xs: (ctypes.c_int32 * max(1, len(xs)))(*xs)
    out = ctypes.c_int(-7)
    rc = lib.pa_mixed_prefill_pairs(ctypes.byref(sh), arr(dec), len(dec), arr(rows),
                                    None if prefix is None else arr(prefix), len(rows), sms, ctypes.byref(out))
    return rc, out.value


def test_mixed_prefill_pairs_planner(lib):
    """The SM partition of a mixed step: 0 when a half is empty or head_dim is
    64, else the balance point of the cost model, inside [1, S/2 - 1]."""
    sh = binding.PaShape(32, 8, 128, 16, 100, 0.0)
    assert _pairs(lib, sh, [], [512]) == (0, 0)
    assert _pairs(lib, sh, [1000], []) == (0, 0)
    assert _pairs(lib, binding.PaShape(32, 8, 64, 16, 100, 0.0), [1000], [512]) == (0, 0)
    # One 128-row prompt: 8 head groups of 4 (Hq 32 / Hkv 8), one tile each:
    # A = 8 * 1 + 8 * 2 pair-us.  One decode of L tokens moves
    # L * 8 * 128 * 4 bytes at 50 GB/s per SM.
    for L in (2000, 20000, 200000):
        a = 8 * 1.0 + 8 * 2.0
        b = L * 8 * 128 * 4 / 50e3
        want = max(1, min(round(152 * a / (b + 2 * a)), 75))
        assert _pairs(lib, sh, [L], [128]) == (0, want)
    # more decode work -> fewer pairs; more prefill work (rows, prefix) -> more
    base = _pairs(lib, sh, [1500] * 64, [256, 512])[1]
    assert 1 <= base <= 75
    assert _pairs(lib, sh, [1500] * 128, [256, 512])[1] < base
    assert _pairs(lib, sh, [1500] * 64, [256, 512, 1024])[1] > base
    assert _pairs(lib, sh, [1500] * 64, [256, 512], [4096, 4096])[1] > base
    # clamps: a tiny decode leaves the prefill all but one pair, and a huge
    # one still gives the prefill a pair
    assert _pairs(lib, sh, [1], [4096] * 8)[1] == 75
    assert _pairs(lib, sh, [10 ** 6] * 64, [16])[1] == 1
    assert _pairs(lib, sh, [1], [4096] * 8, sms=100)[1] == 49
    # group 2 (two row tiles a unit) and group 1 (four)
    for hq, hkv in ((16, 8), (8, 8)):
        assert 1 <= _pairs(lib, binding.PaShape(hq, hkv, 128, 16, 100, 0.0), [3000] * 32, [700, 300])[1] <= 75
    bad = ctypes.c_int()
    assert lib.pa_mixed_prefill_pairs(ctypes.byref(sh), None, 1, None, None, 0, 152,
                                      ctypes.byref(bad)) == binding.ERR_INVALID_ARG
    assert lib.pa_mixed_prefill_pairs(ctypes.byref(sh), None, 0, None, None, 0, 152, None) == binding.ERR_INVALID_ARG
    # the split step rejects a negative count before anything else
    assert lib.pa_mixed_step_split(ctypes.byref(sh), DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, DUMMY, 4, 2, 1, 8,
                                   64, 8, DUMMY, DUMMY, DUMMY, DUMMY, 0, None, -1) == binding.ERR_INVALID_ARG


def test_mixed_prefill_pairs_binding(lib):
    shape = binding.PaShape(32, 8, 128, 16, 100, 0.0)
    n = binding.mixed_prefill_pairs(shape, [1500] * 64, [256, 512], num_sms=152)
    assert n == _pairs(lib, shape, [1500] * 64, [256, 512])[1]
    assert binding.mixed_prefill_pairs(shape, [], [256], num_sms=152) == 0
