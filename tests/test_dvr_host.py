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
import torch

from invariant_fixed_order_gb300 import dvr, sched
from invariant_fixed_order_gb300.engine import PagePool

INVARIANT, VARIANT = 0, 1
V = 997
PAGE = 16


def rule(history, mode):
    h = 7
    for t in history:
        h = (h * 1000003 + int(t) + 1) % 2147483647
    tok = h % V
    if mode == VARIANT and (h >> 7) % 10 == 0:
        tok = (tok + 1) % V
    return tok


class FakeEngine:
    class cfg:
        V = V

    def __init__(self, num_pages=4096, max_pages=64):
        self.max_pages = max_pages
        self.pool = PagePool(num_pages, seed=0)
        self.cache = {}

    def step(self, q_len, pos0, ids, table, rows, mode=INVARIANT):
        out, t = [], 0
        for i, (n, p0) in enumerate(zip(q_len, pos0)):
            for j in range(n):
                p = p0 + j
                self.cache[(int(table[i][p // PAGE]), p % PAGE)] = int(ids[t + j])
            for j in range(n):
                p = p0 + j
                hist = [self.cache[(int(table[i][q // PAGE]), q % PAGE)] for q in range(p + 1)]
                out.append(rule(hist, mode))
            t += n
        tokens = torch.tensor([out[r] for r in rows], dtype=torch.int32)
        return None, tokens, None


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
