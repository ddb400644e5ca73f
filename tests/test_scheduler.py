"""The host continuous-batching scheduler (include/pa_sched.h) against the
reference scheduler of the oracle package: the reference pinned on
hand-worked schedules, then the library's plans compared with it step by
step on random arrival traces (bit-exact: every decision is integer), and
the library's block tables and slots checked for validity."""
import numpy as np
import pytest

from oracle.scheduler import RefScheduler
from paged_kv_cache_continuous_gb300 import binding as pa


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_continuous_gb300 import build
    build.build()
    return pa.load()


def _run(ref, n_steps):
    out = []
    for _ in range(n_steps):
        steps, nd = ref.plan()
        out.append(([(i, r, L) for i, r, L, _ in steps], nd, ref.commit()))
    return out


# ----------------------------------------------------------------- pins --
def test_ref_plain_two_requests():
    """Both prompts are prefilled in step 1 (their first tokens); B leaves
    after its 2nd token (step 2), A after its 3rd (step 3)."""
    ref = RefScheduler(100, 16)
    ref.submit("A", 100, 3)
    ref.submit("B", 50, 2)
    got = _run(ref, 4)
    assert got[0] == ([("A", 100, 100), ("B", 50, 50)], 0, [])
    assert got[1] == ([("A", 1, 101), ("B", 1, 51)], 2, ["B"])
    assert got[2] == ([("A", 1, 102)], 1, ["A"])
    assert got[3] == ([], 0, [])


def test_ref_backpressure_and_forced_admission():
    """5 running, 5 waiting: 5 < floor(5 x 1.2) = 6, so nobody is admitted
    until max_waiting_tokens (3) steps have passed without an admission."""
    ref = RefScheduler(1000, 16, max_waiting_tokens=3, waiting_served_ratio=1.2)
    for i in range(5):
        ref.submit(f"r{i}", 10, 100)
    _run(ref, 1)  # all five admitted (nothing was running)
    for i in range(5):
        ref.submit(f"w{i}", 10, 100)
    hist = _run(ref, 4)
    admitted = [any(x[0].startswith("w") for x in step) for step, _, _ in hist]
    assert admitted == [False, False, False, True]  # waiting = 0, 1, 2, then 3 >= 3
    assert [len(s) for s, _, _ in hist] == [5, 5, 5, 10]


def test_ref_prefill_budget_fifo():
    """Prompts of 3000 and 2000 under a 4096-row prefill budget: the first
    alone; the second is not skipped over to admit the third (1000)."""
    ref = RefScheduler(2000, 16, max_input_tokens=4000, max_total_tokens=8000)
    for rid, n in (("x", 3000), ("y", 2000), ("z", 1000)):
        ref.submit(rid, n, 5)
    steps, _ = ref.plan()
    assert [s[0] for s in steps] == ["x"]


def test_ref_token_budget():
    """Pool of 10 blocks x 16 tokens: reservations (block-aligned prompt +
    max_new) of 48 and 64 fit, a further 64 does not (48 + 64 + 64 > 160)."""
    ref = RefScheduler(10, 16)
    ref.submit("a", 30, 10)   # 40 -> 48
    ref.submit("b", 50, 10)   # 60 -> 64
    ref.submit("c", 50, 10)
    steps, _ = ref.plan()
    assert [s[0] for s in steps] == ["a", "b"]


def test_ref_chunking():
    """Chunked prefill, 100 rows per step: 10 decoding requests leave 90
    rows for a 250-row prompt: chunks 90, 90, 70; its first token comes with
    the last chunk."""
    ref = RefScheduler(10000, 16, max_batch_prefill_tokens=100, chunking=True)
    for i in range(10):
        ref.submit(i, 5, 50)
    ref.plan(); ref.commit()  # 50 rows: all ten prompts
    ref.submit("big", 250, 3)
    chunks = []
    for _ in range(4):
        steps, nd = ref.plan()
        chunks.append([(r, L) for i, r, L, _ in steps if i == "big"])
        ref.commit()
    assert chunks == [[(90, 90)], [(90, 180)], [(70, 250)], [(1, 251)]]


# ---------------------------------------------------- library vs reference --
def _trace(seed, steps, chunking, max_batch_size):
    rng = np.random.default_rng(seed)
    kw = dict(max_batch_prefill_tokens=int(rng.choice([256, 1024, 4096])), max_waiting_tokens=int(rng.integers(0, 6)),
              waiting_served_ratio=float(rng.choice([0.0, 1.2, 2.0])), max_batch_size=max_batch_size,
              chunking=chunking)
    nb, B = int(rng.choice([64, 400])), int(rng.choice([16, 32]))
    lib_s = pa.Scheduler(nb, B, **kw)
    ref = RefScheduler(nb, B, **kw)
    nid = 0
    for step in range(steps):
        for _ in range(int(rng.poisson(1.5))):
            n, m = int(rng.integers(1, 700)), int(rng.integers(1, 300))
            ok_ref = True
            try:
                ref.submit(nid, n, m)
            except ValueError:
                ok_ref = False
            if ok_ref:
                lib_s.submit(nid, n, m)
            else:
                with pytest.raises(pa.PagedAttnError):
                    lib_s.submit(nid, n, m)
            nid += 1
        if rng.random() < 0.05 and (ref.queue or ref.running):
            pool = ref.queue + ref.running
            victim = pool[int(rng.integers(0, len(pool)))]["id"]
            ref.cancel(victim)
            lib_s.cancel(victim)
        rsteps, rnd = ref.plan()
        got = lib_s.plan()
        if not rsteps:
            assert got is None
        else:
            S = len(rsteps)
            assert got["seq_ids"].tolist() == [s[0] for s in rsteps]
            assert np.diff(got["q_start_loc"]).tolist() == [s[1] for s in rsteps]
            assert got["seq_lens"].tolist() == [s[2] for s in rsteps]
            assert got["num_decode"] == rnd
            # blocks: enough for each sequence, none shared; slots follow the tables
            owned = {}
            for r in range(S):
                nbk = -(-rsteps[r][2] // B)
                row = got["block_table"][r]
                assert (row[:nbk] >= 0).all() and (row[nbk:] == -1).all()
                for b in row[:nbk].tolist():
                    assert owned.setdefault(b, got["seq_ids"][r]) == got["seq_ids"][r], "block shared"
                t0, n_new = got["q_start_loc"][r], rsteps[r][1]
                for j in range(n_new):
                    pos = rsteps[r][2] - n_new + j
                    assert got["slot_mapping"][t0 + j] == row[pos // B] * B + pos % B
        assert lib_s.commit() == ref.commit()
        st = lib_s.stats()
        assert (st["queued"], st["running"], st["free_blocks"]) == (len(ref.queue), len(ref.running), ref.free_blocks)
        assert st["waiting_steps"] == ref.waiting


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("chunking", [False, True])
def test_library_matches_reference(lib, seed, chunking):
    _trace(seed, 120, chunking, max_batch_size=[0, 24][seed % 2])


def test_submit_rejections(lib):
    s = pa.Scheduler(100, 16)
    s.submit(1, 10, 10)
    for args in ((1, 10, 10), (2, 0, 5), (3, 5, 0), (4, 1025, 1), (5, 1000, 1049)):
        with pytest.raises(pa.PagedAttnError):
            s.submit(*args)
