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
    head), its 16 bytes of counters and 8 bytes per sequence."""
    partials = -(-(S * Hq * splits * (d + 2) * 4) // 16) * 16 if splits > 1 else 0
    return partials + S * splits * Hkv * 16 + 16 + S * 8


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
