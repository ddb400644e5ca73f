"""bench.py's reference arm (the fp64 oracle on the host cores) prints one
JSON line with the contract's keys, on the CPU."""
import json
import subprocess
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.strip().startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["dtype"] == "f64" and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_decode_step_bytes_split_rule():
    """The decode's algorithmic bytes count split partials by the documented
    split rule: ceil(L / split) splits, one fewer when the last would hold at
    most split / 8 tokens; partials only for sequences with two or more."""
    import numpy as np
    sys.path.insert(0, str(ROOT))
    import bench

    class Sh:
        num_q_heads, num_kv_heads, head_dim = 8, 2, 64

    lens = np.array([256, 257, 256 + 32, 256 + 33, 512 + 32, 512 + 33, 1], dtype=np.int32)
    nsplit = np.array([1, 1, 1, 2, 2, 3, 1])
    got = bench.decode_step_bytes(Sh, lens, 256, 16)
    L = lens.astype(np.int64)
    kv = int(L.sum()) * 2 * 64 * 2 * 2
    qo = 2 * 7 * 8 * 64 * 2
    tables = int(np.ceil(L / 16).sum()) * 4 + 7 * 4
    partials = int(nsplit[nsplit > 1].sum()) * 8 * (64 + 2) * 4 * 2
    assert got["decode"] == kv + qo + tables + partials
