"""The schedule fuzzer and comparator on the CPU, against the paged stand-in
engine (tests/standin.py): random arrivals, chunked prefill co-scheduled with
decodes, preemption and evict/readmit (pages freed, context recomputed by
prefill) must leave every produced row equal to the request's solo run when
the engine is batch-invariant, and the comparator must see a difference when
it is not (the harness has teeth)."""
import numpy as np

from invariant_fixed_order_gb300 import sched
from tests.standin import StandInEngine, V


def make_requests(n, seed):
    rng = np.random.default_rng(seed)
    return [sched.Request(i, rng.integers(0, V, int(rng.integers(5, 90))).astype(np.int32)) for i in range(n)]


def solo_rows(prompts, n_decode, batch_dependent=False):
    out = {}
    for rid, p in prompts.items():
        runner = sched.Runner(StandInEngine(batch_dependent=batch_dependent))
        r = sched.Request(rid, p)
        out[rid] = sched.run_solo(runner, r, n_decode)
    return out


def compare(fuzzed, solo):
    diffs = checked = 0
    for rid, rows in fuzzed.items():
        for pos, row in rows.items():
            checked += 1
            if not sched.bitwise_equal(row, solo[rid][pos]):
                diffs += 1
    return diffs, checked


def test_fuzzed_schedules_reproduce_solo_rows():
    reqs = make_requests(12, 3)
    solo = solo_rows({r.rid: r.prompt for r in reqs}, 10)
    total = 0
    for k in range(6):
        rng = np.random.default_rng(1000 + k)
        runner = sched.Runner(StandInEngine())
        fresh = [sched.Request(r.rid, r.prompt) for r in reqs]
        cfg = sched.FuzzConfig(token_budget=64, chunk_min=3, chunk_max=40, p_evict=0.15, readmit_delay=(1, 3),
                               arrival_span=5)
        fuzzed = sched.fuzz_continuous(runner, fresh, 10, rng, cfg)
        diffs, checked = compare(fuzzed, solo)
        assert diffs == 0, (k, diffs, checked)
        assert runner.eng.pool.n_free == runner.eng.pool.num_pages   # every page returned
        total += checked
    assert total > 500


def test_fuzzer_catches_a_batch_dependent_engine():
    reqs = make_requests(8, 4)
    solo = solo_rows({r.rid: r.prompt for r in reqs}, 6, batch_dependent=True)
    rng = np.random.default_rng(7)
    runner = sched.Runner(StandInEngine(batch_dependent=True))
    fresh = [sched.Request(r.rid, r.prompt) for r in reqs]
    fuzzed = sched.fuzz_continuous(runner, fresh, 6, rng, sched.FuzzConfig(token_budget=64, chunk_min=3,
                                                                          chunk_max=40, p_evict=0.1))
    diffs, checked = compare(fuzzed, solo)
    assert diffs > 0 and checked > 0
