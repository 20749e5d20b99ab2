"""Decode-verify-rollback over the batch-variant fast path.

"LLM-42: How Microsoft Made LLM Inference Reproducible Without Killing
Throughput", "The Decode-Verify-Rollback Protocol": a window of candidate
tokens is decoded with dynamic batching on the fast path (here: BI_VARIANT
mode, whose reductions follow the batch), then replayed under a fixed-shape
schedule (here: BI_INVARIANT mode, teacher-forced prefill of the window) in
groups of requests; tokens that match are committed, the first mismatching
one is replaced and the rest are discarded.

"Per-Request Opt-In and Mixed Workloads": only requests marked
is_deterministic are verified (their prompts are prefilled in invariant
mode); the others share the fast path's batches and commit its tokens as they
come, so the verifier's work follows the deterministic share of the traffic.

Reading of the rollback step (the page says only that the system rolls back
to the last verified consistent position): at the first mismatch the
verifier's own token at that position is committed too, as in speculative
decoding.  The committed sequence then equals pure invariant greedy decoding:
the invariant prefill logits at a position equal the invariant decode logits
there (same per-chunk arithmetic), and every verified input token is itself a
committed one.  After verification the KV cache holds invariant K/V for every
committed position (the replay overwrote the window's slots), so rolling back
is only a matter of truncating the request's length.
"""
from __future__ import annotations

import time
from dataclasses import dataclass, field

import torch

from . import bi
from .sched import Request, Runner, StepItem


@dataclass
class DvrStats:
    windows: int = 0            # request-windows verified
    mismatched_windows: int = 0
    committed: int = 0          # generated tokens committed (capped at n_new per request)
    discarded: int = 0          # candidate tokens thrown away
    t_prefill: float = 0.0
    t_decode: float = 0.0
    t_verify: float = 0.0
    verified: set = field(default_factory=set)  # request ids whose windows were verified
    first_mismatch: list = field(default_factory=list)    # per rolled-back window: index of its first mismatch
    window_committed: list = field(default_factory=list)  # per verified window: tokens it committed

    @property
    def rollback_rate(self) -> float:
        return self.mismatched_windows / self.windows if self.windows else 0.0

    @property
    def verify_overhead(self) -> float:
        tot = self.t_decode + self.t_verify
        return self.t_verify / tot if tot else 0.0

    def as_dict(self, window: int | None = None) -> dict:
        """Counts, times and where windows break: the first-mismatch position of each rolled-back window (its
        mean, median and a histogram) and the tokens each verified window committed (the verifier's token
        included).  A window that commits c of its W candidates (plus the verifier's) pays for W fast-path
        steps and one replay, which is why DVR only pays when mismatches are rare and late."""
        tot = self.t_prefill + self.t_decode + self.t_verify
        fm = sorted(self.first_mismatch)
        edges = [0, 1, 4, 16, 64, 1 << 30]
        hist = {f"{a}-{b - 1}" if b - 1 < (1 << 29) else f"{a}+": sum(1 for k in fm if a <= k < b)
                for a, b in zip(edges[:-1], edges[1:])}
        wc = self.window_committed
        d = {"windows": self.windows, "mismatched_windows": self.mismatched_windows,
             "rollback_rate": self.rollback_rate, "committed": self.committed, "discarded": self.discarded,
             "committed_tok_s": self.committed / tot if tot else 0.0, "verify_overhead": self.verify_overhead,
             "t_prefill_s": self.t_prefill, "t_decode_s": self.t_decode, "t_verify_s": self.t_verify,
             "first_mismatch_mean": sum(fm) / len(fm) if fm else None,
             "first_mismatch_median": fm[len(fm) // 2] if fm else None,
             "first_mismatch_hist": hist,
             "committed_per_window_mean": sum(wc) / len(wc) if wc else None}
        if window:
            d["committed_fraction_mean"] = (sum(wc) / len(wc)) / window if wc else None
        return d


def _groups(seq, n):
    return [seq[i:i + n] for i in range(0, len(seq), n)]


def _now():
    if torch.cuda.is_available():
        torch.cuda.synchronize()  # device work counts towards the phase it was issued in
    return time.perf_counter()


def dvr_generate(runner: Runner, reqs: list, n_new: int, window: int = 64, verify_batch: int = 8,
                 fast_mode: int = bi.VARIANT, corrupt=None) -> DvrStats:
    """Generates n_new greedy tokens per request with decode-verify-rollback.

    corrupt(rid, position) -> bool, if given, replaces the fast path's
    candidate at that position by another token (a forced divergence that the
    verifier must catch).  On return each request's ``generated`` holds exactly
    its n_new committed tokens."""
    st = DvrStats()
    V = runner.eng.cfg.V
    t0 = _now()
    # prompts, in groups; the first token comes from the prefill: invariant for
    # deterministic requests, the fast path for the others
    det = [r for r in reqs if r.is_deterministic]
    free = [r for r in reqs if not r.is_deterministic]
    for group, mode in [(g, bi.INVARIANT) for g in _groups(det, verify_batch)] + \
                       [(g, fast_mode) for g in _groups(free, verify_batch)]:
        items = [StepItem(r, len(r.prompt), "last") for r in group]
        logits, tokens, sl = runner.step(items, mode=mode)
        toks = tokens.cpu().tolist()
        for it, s in zip(items, sl):
            it.req.generated.append(int(toks[s][-1] if isinstance(toks[s], list) else toks[s.stop - 1]))
    t1 = _now()
    st.t_prefill += t1 - t0
    active = [r for r in reqs if len(r.generated) < n_new]
    while active:
        # ---- decode a window on the fast path, all active requests batched ----
        W = window
        start = {r.rid: len(r.tokens) for r in active}   # L: committed length
        t0 = _now()
        for _ in range(W):
            items = [StepItem(r, 1, "last") for r in active]
            logits, tokens, sl = runner.step(items, mode=fast_mode)
            toks = tokens.cpu().tolist()
            for it, s in zip(items, sl):
                t = int(toks[s.start])
                pos = len(it.req.tokens)
                if corrupt is not None and corrupt(it.req.rid, pos):
                    t = (t + 1) % V
                it.req.generated.append(t)
        t1 = _now()
        st.t_decode += t1 - t0
        # ---- verify: invariant teacher-forced prefill of the window, in groups ----
        for group in _groups([r for r in active if r.is_deterministic], verify_batch):
            items = []
            for r in group:
                L = start[r.rid]
                r.n_cached = L - 1                       # replay positions L-1 .. L+W-2
                items.append(StepItem(r, W, "all"))
            logits, tokens, sl = runner.step(items, mode=bi.INVARIANT)
            toks = tokens.cpu().tolist()
            for it, s in zip(items, sl):
                r = it.req
                L = start[r.rid]
                verified = toks[s.start:s.stop]          # predictions for positions L .. L+W-1
                cand = r.tokens[L:L + W].tolist()
                k = next((j for j in range(W) if verified[j] != cand[j]), None)
                st.windows += 1
                st.verified.add(r.rid)
                n_prompt = len(r.prompt)
                if k is None:
                    r.n_cached = L + W - 1
                    st.window_committed.append(W)
                else:
                    st.mismatched_windows += 1
                    st.discarded += W - k
                    st.first_mismatch.append(k)
                    st.window_committed.append(k + 1)
                    r.generated = r.generated[:L + k - n_prompt] + [int(verified[k])]
                    r.n_cached = L + k
        st.t_verify += _now() - t1
        for r in active:
            if not r.is_deterministic:
                r.n_cached = len(r.tokens) - 1   # fast-path tokens are committed as decoded
        active = [r for r in active if len(r.generated) < n_new]
    for r in reqs:
        del r.generated[n_new:]
        st.committed += len(r.generated)
    return st
