"""Host-side continuous-batching harness around the forward step.

"Lockstep", "Proving it": the harness enumerates and randomises what a
scheduler may vary — which requests share a batch, in what order they arrive,
where preemption lands, how continuous batching evicts and readmits — and
compares every request's logits bit for bit with its single-request run.

Pieces:
  * ``Request`` / ``Runner``: per-request paged KV bookkeeping (pages from a
    shuffled pool, freed on evict, recomputed by prefill on readmit) and the
    ragged step builder;
  * ``set_partitions_with_sizes``: every split of n requests into batches of
    allowed sizes;
  * ``fuzz_continuous``: a randomised continuous-batching schedule with
    arrivals, chunked prefill, preemption and evict/readmit;
  * ``bitwise_equal`` / ``diff_report``: the pure comparator (no tolerance);
  * ``rule_of_three``: the 95% upper bound on a divergence rate after zero
    divergences in n trials (llamacpp-batch-invariance README, "Rule of three").
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Iterator

import numpy as np
import torch

from . import bi


# ---------------------------------------------------------------------------
# pure helpers
# ---------------------------------------------------------------------------

def set_partitions_with_sizes(items: list, sizes: set) -> Iterator[list]:
    """Yields every partition of `items` into blocks whose sizes are in `sizes`
    (blocks are lists; the first item of each block is its smallest index)."""
    items = list(items)
    if not items:
        yield []
        return
    first, rest = items[0], items[1:]
    n = len(rest)
    for size in sorted(sizes):
        if size - 1 > n:
            continue
        for combo in _combinations(rest, size - 1):
            block = [first] + list(combo)
            remaining = [x for x in rest if x not in combo]
            for tail in set_partitions_with_sizes(remaining, sizes):
                yield [block] + tail


def _combinations(seq, k):
    seq = list(seq)
    if k == 0:
        yield ()
        return
    for i in range(len(seq) - k + 1):
        for tail in _combinations(seq[i + 1:], k - 1):
            yield (seq[i],) + tail


def rule_of_three(n_trials: int) -> float:
    """95% upper bound on the true divergence rate after 0 divergences in n trials."""
    return 3.0 / n_trials if n_trials > 0 else 1.0


def bitwise_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Exact equality of the bit patterns (NaN payloads and signed zeros included)."""
    if a.shape != b.shape or a.dtype != b.dtype:
        return False
    if a.dtype == torch.float32:
        return bool(torch.equal(a.view(torch.int32), b.view(torch.int32)))
    if a.dtype == torch.bfloat16:
        return bool(torch.equal(a.view(torch.int16), b.view(torch.int16)))
    return bool(torch.equal(a, b))


def diff_report(a: torch.Tensor, b: torch.Tensor) -> dict:
    """Number of differing elements and the largest absolute difference."""
    if a.shape != b.shape:
        return {"shape_mismatch": (tuple(a.shape), tuple(b.shape))}
    ai = a.view(torch.int32) if a.dtype == torch.float32 else a
    bi_ = b.view(torch.int32) if b.dtype == torch.float32 else b
    ne = (ai != bi_)
    n = int(ne.sum().item())
    mx = float((a.float() - b.float()).abs().max().item()) if n else 0.0
    return {"n_diff": n, "max_abs": mx, "numel": a.numel()}


# ---------------------------------------------------------------------------
# requests and the step builder
# ---------------------------------------------------------------------------

@dataclass
class Request:
    rid: int
    prompt: np.ndarray
    generated: list = field(default_factory=list)
    pages: list = field(default_factory=list)
    n_cached: int = 0
    # "Per-Request Opt-In and Mixed Workloads": a deterministic request's
    # committed tokens must not depend on the batch; the others may take the
    # batch-variant fast path unverified
    is_deterministic: bool = True

    @property
    def tokens(self) -> np.ndarray:
        return np.concatenate([self.prompt, np.asarray(self.generated, np.int32)]).astype(np.int32)


@dataclass
class StepItem:
    req: Request
    n_new: int             # tokens appended this step (from req.tokens[n_cached:])
    logits: str = "last"   # "last" | "all" | "none"


class Runner:
    """Builds ragged steps for an Engine and keeps per-request page tables."""

    def __init__(self, engine, mode: int = bi.INVARIANT):
        self.eng = engine
        self.mode = mode
        self.log = []  # per step: list of (rid, pos0, n_new)

    def ensure_pages(self, req: Request, n_pos: int) -> None:
        need = (n_pos + bi.PAGE - 1) // bi.PAGE
        if need > self.eng.max_pages:
            raise ValueError(f"request {req.rid}: {n_pos} positions exceed max_pages")
        if need > len(req.pages):
            req.pages.extend(self.eng.pool.alloc(need - len(req.pages)))

    def evict(self, req: Request) -> None:
        """Frees the request's KV pages; a later step must recompute them by prefill."""
        self.eng.pool.free(req.pages)
        req.pages = []
        req.n_cached = 0

    def step(self, items: list, mode: int | None = None):
        """Runs one forward step.  Returns (logits, tokens, slices) where
        slices[i] is the range of logits rows that belong to items[i]."""
        mode = self.mode if mode is None else mode
        q_len, pos0, ids, rows, slices = [], [], [], [], []
        table = np.zeros((len(items), self.eng.max_pages), np.int32)
        t = 0
        for i, it in enumerate(items):
            req = it.req
            toks = req.tokens[req.n_cached:req.n_cached + it.n_new]
            assert len(toks) == it.n_new and it.n_new >= 1, (req.rid, it.n_new, len(toks))
            self.ensure_pages(req, req.n_cached + it.n_new)
            table[i, :len(req.pages)] = req.pages
            q_len.append(it.n_new)
            pos0.append(req.n_cached)
            ids.append(toks)
            r0 = len(rows)
            if it.logits == "all":
                rows.extend(range(t, t + it.n_new))
            elif it.logits == "last":
                rows.append(t + it.n_new - 1)
            slices.append(slice(r0, len(rows)))
            t += it.n_new
        self.log.append([(it.req.rid, p, n) for it, p, n in zip(items, pos0, q_len)])
        logits, tokens, _ = self.eng.step(q_len, pos0, np.concatenate(ids), table, rows, mode=mode)
        for it in items:
            it.req.n_cached += it.n_new
        return logits, tokens, slices


# ---------------------------------------------------------------------------
# solo baselines and schedules
# ---------------------------------------------------------------------------

def run_solo(runner: Runner, req: Request, n_decode: int, prefill_chunks=None):
    """Prefill the prompt alone (all-position logits) then decode greedily alone.
    Returns logits [len(prompt) + n_decode - 1 ... ] as a list of per-position
    device tensors keyed by position, and the generated tokens."""
    out = {}
    chunks = prefill_chunks or [len(req.prompt)]
    for n in chunks:
        logits, tokens, sl = runner.step([StepItem(req, n, "all")])
        base = req.n_cached - n
        for j in range(n):
            out[base + j] = logits[sl[0]][j].clone()
        last_tok = int(tokens[sl[0]][-1].item())
    for _ in range(n_decode):
        req.generated.append(last_tok)
        logits, tokens, sl = runner.step([StepItem(req, 1, "last")])
        out[req.n_cached - 1] = logits[sl[0]][0].clone()
        last_tok = int(tokens[sl[0]][0].item())
    return out


@dataclass
class FuzzConfig:
    token_budget: int = 4096        # tokens per step
    chunk_min: int = 256
    chunk_max: int = 2048
    p_evict: float = 0.05           # chance per step that a running request is evicted
    readmit_delay: tuple = (1, 4)   # steps before an evicted request is readmitted
    arrival_span: int = 6           # arrivals spread over this many steps


def fuzz_continuous(runner: Runner, requests: list, n_decode: int, rng: np.random.Generator,
                    cfg: FuzzConfig, teacher: dict | None = None, all_prompt_logits: bool = True,
                    stats: dict | None = None):
    """A randomised continuous-batching run.  Requests arrive at random steps,
    prefill in random chunks (within the token budget, co-scheduled with the
    decodes of running requests), may be evicted (pages freed) and readmitted
    (context recomputed by prefill in random chunks).  Each request decodes
    n_decode tokens; when `teacher` maps rid -> token list, those tokens are
    appended instead of the argmax (so logits stay comparable after a
    divergence).  Returns {rid: {position: logits row}} for every position
    whose logits were produced (prompt positions during the first prefill and
    each decode position).  stats (optional) receives the counts of steps, evictions and readmissions."""
    if stats is not None:
        for k in ("steps", "evictions", "readmissions", "prefill_tokens"):
            stats.setdefault(k, 0)
    arrival = {r.rid: int(rng.integers(0, cfg.arrival_span)) for r in requests}
    order = list(requests)
    rng.shuffle(order)
    waiting = []                         # admitted, context not fully cached
    running = []                         # fully cached, decoding
    out = {r.rid: {} for r in requests}
    done = set()
    evicted_until = {}
    step_no = 0
    produced_prompt = {r.rid: False for r in requests}
    while len(done) < len(requests):
        for r in order:
            if arrival[r.rid] == step_no and r not in waiting:
                waiting.append(r)
        for rid, until in list(evicted_until.items()):
            if until <= step_no:
                r = next(x for x in requests if x.rid == rid)
                waiting.append(r)
                del evicted_until[rid]
                if stats is not None:
                    stats["readmissions"] += 1
        items = []
        budget = cfg.token_budget
        rng.shuffle(running)
        for r in running:
            if budget <= 0:
                break
            items.append(StepItem(r, 1, "last"))
            budget -= 1
        rng.shuffle(waiting)
        for r in list(waiting):
            if budget <= 0:
                break
            remaining = len(r.tokens) - r.n_cached
            chunk = int(rng.integers(cfg.chunk_min, cfg.chunk_max + 1))
            n = min(remaining, chunk, budget)
            if n <= 0:
                continue
            first_prefill = (all_prompt_logits and not produced_prompt[r.rid] and r.n_cached == 0
                             and not r.generated)
            items.append(StepItem(r, n, "all" if first_prefill else "last"))
            budget -= n
        if not items:
            step_no += 1
            continue
        order_idx = rng.permutation(len(items))
        items = [items[i] for i in order_idx]
        logits, tokens, slices = runner.step(items)
        if stats is not None:
            stats["steps"] += 1
            stats["prefill_tokens"] += sum(it.n_new for it in items if it.n_new > 1)
        for it, sl in zip(items, slices):
            r = it.req
            rows = logits[sl]
            if it.logits == "all":
                base = r.n_cached - it.n_new
                for j in range(it.n_new):
                    out[r.rid][base + j] = rows[j].clone()
            complete = r.n_cached == len(r.tokens)
            if it.logits == "all" and complete:
                produced_prompt[r.rid] = True
            if it.logits == "last" and complete:
                out[r.rid][r.n_cached - 1] = rows[0].clone()
            if complete:
                if r in waiting:
                    waiting.remove(r)
                    if r not in running:
                        running.append(r)
                if len(r.generated) >= n_decode:
                    if r in running:
                        running.remove(r)
                    if r.rid not in done:
                        done.add(r.rid)
                        runner.evict(r)
                    continue
                # choose the next token
                if teacher is not None:
                    nxt = int(teacher[r.rid][len(r.generated)])
                else:
                    nxt = int(tokens[sl][-1].item())
                r.generated.append(nxt)
        # preemption: evict a running request, readmit later (recompute by prefill)
        for r in list(running):
            if rng.random() < cfg.p_evict and r.rid not in done:
                running.remove(r)
                runner.evict(r)
                evicted_until[r.rid] = step_no + int(rng.integers(*cfg.readmit_delay))
                if stats is not None:
                    stats["evictions"] += 1
        step_no += 1
    return out
