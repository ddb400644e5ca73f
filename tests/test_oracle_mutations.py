"""Each plausible mistake planted in a copy of the oracle (on the CPU) must be
caught by at least one pin; the pins are only worth what they catch."""
import os
import subprocess
import tempfile
from pathlib import Path

import numpy as np
import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = Path(oracle.__file__).resolve().parent / "oracle.c"

# (name, original text, replacement, expected count of occurrences)
MUTATIONS = [
    ("drop_scale", "x[j] = scale * dot;", "x[j] = dot;", 2),
    ("gqa_head_mod", "int g = (int)(h / dc->G);", "int g = (int)(h % (dc->Hq / dc->G));", 1),
    ("prefill_gqa_head_mod", "int g = (int)(h / pc->G);", "int g = (int)(h % (pc->Hq / pc->G));", 1),
    ("causal_off_by_one", "int L = (int)(p0 + i + 1);", "int L = (int)(p0 + i);", 1),
    ("no_normalise", "for (int e = 0; e < d; ++e) out[e] /= Z;", "", 2),
    ("append_swaps_kv", "k_pool[dst + e] = k_new[src + e];", "k_pool[dst + e] = v_new[src + e];", 1),
    ("v_read_from_k_pool", "(which ? pv->v_pool : pv->k_pool)[at]", "(which ? pv->k_pool : pv->k_pool)[at]", 1),
    ("pool_layout_nhd", "size_t dst = (size_t)(((blk * num_kv_heads + h) * block_size + off) * head_dim);",
     "size_t dst = (size_t)(((blk * block_size + off) * num_kv_heads + h) * head_dim);", 2),
    ("block_offset_wrong", "const size_t krow = (size_t)(((long long)blk * H + g) * B + j % B);",
     "const size_t krow = (size_t)(((long long)blk * H + g) * B + (B - 1 - j % B));", 1),
    ("prefix_ignored", "int p0 = pc->prefix ? pc->prefix[s] : 0;", "int p0 = 0;", 1),
    ("default_scale_wrong", "1.0 / sqrt((double)head_dim)", "1.0 / (double)head_dim", 1),
    ("slot_formula_wrong", "slots_out[q_start[s] + i] = blk * block_size + p % block_size;",
     "slots_out[q_start[s] + i] = blk * block_size + p / block_size;", 1),
    ("dup_check_dropped", "if (seen[slot]) { free(seen); return OR_ERR_SLOT_DUP; }", "", 2),
    ("rope_sign", "out[base + i] = x0 * c - x1 * s;", "out[base + i] = x0 * c + x1 * s;", 1),
    ("rope_interleaved_pairs", "x1 = bf16_to_double(x[base + i + half]);", "x1 = bf16_to_double(x[base + (i ^ 1)]);", 1),
    ("rope_frequency", "pow(theta, -2.0 * (double)i / (double)head_dim)", "pow(theta, -1.0 * (double)i / (double)head_dim)", 1),
    ("bf16_truncates", "nearbyint(ldexp(a, -qexp))", "floor(ldexp(a, -qexp))", 1),
    ("e4m3_bias", "ldexp(8.0 + m, e - 10)", "ldexp(8.0 + m, e - 9)", 1),
    ("e4m3_rounds_down", "double q = nearbyint(ldexp(a, 3 - e));", "double q = floor(ldexp(a, 3 - e));", 1),
    ("fp8_scale_multiplied", "(float)bf16_to_double(k_new[src + e]) / k_scale[h];", "(float)bf16_to_double(k_new[src + e]) * k_scale[h];", 1),
    ("fp8_read_scale_dropped", "return e4m3_to_double(p8[at]) * (double)sc[g];", "return e4m3_to_double(p8[at]);", 1),
]


def _build_mutant(tmp: Path, orig: str, repl: str, count: int) -> Path:
    text = SRC.read_text()
    assert text.count(orig) == count, (orig, text.count(orig))
    src = tmp / "oracle_mut.c"
    src.write_text(text.replace(orig, repl))
    lib = tmp / "liboracle_mut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    str(src), "-o", str(lib), "-lm"], check=True)
    return lib


@pytest.mark.parametrize("name,orig,repl,count", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(name, orig, repl, count, monkeypatch):
    with tempfile.TemporaryDirectory() as d:
        lib = _build_mutant(Path(d), orig, repl, count)
        monkeypatch.setattr(oracle, "_lib", None)
        monkeypatch.setattr(oracle, "build", lambda force=False: lib)
        caught = []
        for pin in ALL_PINS:
            try:
                pin()
            except (AssertionError, oracle.OracleError):
                caught.append(pin.__name__)
        assert caught, f"mutation {name} passed every pin"


# Python-level mistakes in the block copy (it is plain numpy, not C).
_copy = oracle.copy_blocks


def _copy_k_only(sk, sv, dk, dv, si, di):
    dk2, _ = _copy(sk, sv, dk, dv, si, di)
    return dk2, np.array(dv, dtype=np.uint16, copy=True)


def _ids_swapped(sk, sv, dk, dv, si, di):
    if sk is dk:
        dk, dv = np.array(dk, copy=True), np.array(dv, copy=True)
    return _copy(sk, sv, dk, dv, di, si)


def _next_block(sk, sv, dk, dv, si, di):
    n = np.asarray(dk).shape[0]
    return _copy(sk, sv, dk, dv, si, ((np.asarray(di, dtype=np.int64) + 1) % n).astype(np.int32))


def _no_checks(sk, sv, dk, dv, si, di):
    sk, sv = np.asarray(sk), np.asarray(sv)
    dk2, dv2 = np.array(dk, copy=True), np.array(dv, copy=True)
    for s_, d_ in zip(np.asarray(si).tolist(), np.asarray(di).tolist()):
        dk2[d_ % dk2.shape[0]] = sk[s_ % sk.shape[0]]
        dv2[d_ % dv2.shape[0]] = sv[s_ % sv.shape[0]]
    return dk2, dv2


COPY_MUTANTS = [("copy_k_only", _copy_k_only), ("ids_swapped", _ids_swapped),
                ("next_block", _next_block), ("no_checks", _no_checks)]


@pytest.mark.parametrize("name,fn", COPY_MUTANTS, ids=[m[0] for m in COPY_MUTANTS])
def test_copy_mutant_is_caught(name, fn, monkeypatch):
    monkeypatch.setattr(oracle, "copy_blocks", fn)
    caught = []
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, oracle.OracleError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"mutation {name} passed every pin"
