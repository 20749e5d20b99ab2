"""Decode-verify-rollback host logic on the CPU, against a stand-in engine.

The stand-in keeps a paged token cache exactly as the real KV cache is kept
(pages from the pool, slot = position % 16) and predicts each row's next token
from the tokens cached at positions 0..p of its request: an "invariant" rule,
and a "variant" rule that differs from it at a seeded tenth of the histories
(the fast path's occasional flips).  dvr_generate and the Runner run
unchanged on top of it, so the test checks the loop itself: the windows, the
verify groups, the rollback and cache truncation, and the per-request opt-in.
"""
import numpy as np
import pytest

from invariant_fixed_order_gb300 import dvr, sched
from tests.standin import INVARIANT, VARIANT, V, StandInEngine as FakeEngine, rule


def greedy(prompt, n_new, mode):
    seq = list(int(x) for x in prompt)
    gen = []
    for _ in range(n_new):
        gen.append(rule(seq, mode))
        seq.append(gen[-1])
    return gen


@pytest.mark.parametrize("window,verify_batch", [(4, 2), (8, 3), (16, 8)])
def test_dvr_commits_invariant_tokens_and_opt_in_is_per_request(window, verify_batch):
    rng = np.random.default_rng(window)
    prompts = [rng.integers(0, V, int(rng.integers(3, 40))).astype(np.int32) for _ in range(10)]
    n_new = 37
    runner = sched.Runner(FakeEngine(), mode=INVARIANT)
    det = {0, 2, 3, 7, 9}
    reqs = [sched.Request(i, p, is_deterministic=i in det) for i, p in enumerate(prompts)]
    st = dvr.dvr_generate(runner, reqs, n_new, window=window, verify_batch=verify_batch, fast_mode=VARIANT)
    for r in reqs:
        want = greedy(r.prompt, n_new, INVARIANT if r.is_deterministic else VARIANT)
        assert r.generated == want, r.rid
    assert st.verified == det
    assert st.committed == len(reqs) * n_new
    assert st.mismatched_windows > 0 and st.discarded > 0   # the fast path's flips were caught
    # every verify step (window-long replays from inside the sequence; prefills start at position 0) held at
    # most verify_batch requests, all deterministic
    verify_steps = [{rid for rid, p, n in step if n == window and p > 0} for step in runner.log]
    verify_steps = [s_ for s_ in verify_steps if s_]
    assert verify_steps
    for rids in verify_steps:
        assert rids <= det and len(rids) <= verify_batch


def test_dvr_forced_divergence_is_rolled_back():
    rng = np.random.default_rng(1)
    prompts = [rng.integers(0, V, 20).astype(np.int32) for _ in range(4)]
    runner = sched.Runner(FakeEngine(), mode=INVARIANT)
    reqs = [sched.Request(i, p) for i, p in enumerate(prompts)]
    bad = {(i, 20 + 3 + 5 * i) for i in range(4)}
    st = dvr.dvr_generate(runner, reqs, 30, window=8, verify_batch=2, fast_mode=INVARIANT,
                          corrupt=lambda rid, pos: (rid, pos) in bad)
    for r in reqs:
        assert r.generated == greedy(r.prompt, 30, INVARIANT), r.rid
    assert st.mismatched_windows == len(bad)


def test_dvr_window_statistics():
    """Forced divergences at known offsets inside the windows: each rolled-back window's first-mismatch index
    is recorded, and each verified window commits its matching prefix plus the verifier's token."""
    rng = np.random.default_rng(2)
    prompts = [rng.integers(0, V, 20).astype(np.int32) for _ in range(4)]
    runner = sched.Runner(FakeEngine(), mode=INVARIANT)
    reqs = [sched.Request(i, p) for i, p in enumerate(prompts)]
    # the first window of request i covers positions 21 .. 28 (prompt 20, first token from the prefill)
    bad = {(i, 21 + 2 * i) for i in range(4)}
    st = dvr.dvr_generate(runner, reqs, 30, window=8, verify_batch=2, fast_mode=INVARIANT,
                          corrupt=lambda rid, pos: (rid, pos) in bad)
    assert sorted(st.first_mismatch) == [0, 2, 4, 6]
    d = st.as_dict(window=8)
    assert d["first_mismatch_mean"] == 3.0 and d["first_mismatch_median"] == 4
    assert d["first_mismatch_hist"]["0-0"] == 1 and d["first_mismatch_hist"]["1-3"] == 1
    assert d["first_mismatch_hist"]["4-15"] == 2
    # windows without a mismatch commit all 8; the four rolled-back ones commit k + 1
    assert sorted(k for k in st.window_committed if k < 8) == [1, 3, 5, 7]
    assert len(st.window_committed) == st.windows
    assert 0 < d["committed_fraction_mean"] <= 1


def test_results_record_is_atomic_and_complete(tmp_path, monkeypatch):
    from invariant_fixed_order_gb300 import results
    monkeypatch.setenv("BI_GIT_SHA", "0123abc")
    assert results.record("x", {"a": 1}, directory=None) is None or "BI_RESULTS_DIR" in __import__("os").environ
    path = results.record("unique", {"max_completions": 1, "bound": 0.0009}, directory=str(tmp_path))
    import json
    import os
    j = json.load(open(path))
    assert j["name"] == "unique" and j["result"]["max_completions"] == 1
    assert j["environment"]["git_sha"] == "0123abc" and "time_utc" in j["environment"]
    assert [f for f in os.listdir(tmp_path)] == ["unique.json"]  # no temporary left behind
