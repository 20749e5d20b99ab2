"""A CPU stand-in for the engine, for host-logic tests of the step builder,
the schedule fuzzer and decode-verify-rollback.

It keeps tokens in a paged cache exactly as the KV cache is kept (pages from
the pool, slot = position % 16) and computes each row's output from the
tokens cached at positions 0..p of its request alone: a next-token rule
(INVARIANT, or VARIANT which differs at a seeded tenth of the histories) and
a small "logits" row.  With batch_dependent=True the logits also depend on
the number of rows in the step, as a batch-variant kernel's would: the
comparators must catch it.
"""
import torch

from invariant_fixed_order_gb300.engine import PagePool

INVARIANT, VARIANT = 0, 1
V = 997
PAGE = 16


def history_hash(history) -> int:
    h = 7
    for t in history:
        h = (h * 1000003 + int(t) + 1) % 2147483647
    return h


def rule(history, mode) -> int:
    h = history_hash(history)
    tok = h % V
    if mode == VARIANT and (h >> 7) % 10 == 0:
        tok = (tok + 1) % V
    return tok


class StandInEngine:
    class cfg:
        V = V

    def __init__(self, num_pages=4096, max_pages=64, batch_dependent=False):
        self.max_pages = max_pages
        self.pool = PagePool(num_pages, seed=0)
        self.cache = {}
        self.batch_dependent = batch_dependent

    def step(self, q_len, pos0, ids, table, rows, mode=INVARIANT):
        toks, logit_rows, t = [], [], 0
        n_rows = len(rows)
        for i, (n, p0) in enumerate(zip(q_len, pos0)):
            for j in range(n):
                p = p0 + j
                self.cache[(int(table[i][p // PAGE]), p % PAGE)] = int(ids[t + j])
            for j in range(n):
                p = p0 + j
                hist = [self.cache[(int(table[i][q // PAGE]), q % PAGE)] for q in range(p + 1)]
                toks.append(rule(hist, mode))
                h = history_hash(hist) + (n_rows if self.batch_dependent else 0)
                logit_rows.append([float((h >> (3 * k)) % 1024) for k in range(8)])
            t += n
        tokens = torch.tensor([toks[r] for r in rows], dtype=torch.int32)
        logits = torch.tensor([logit_rows[r] for r in rows], dtype=torch.float32).reshape(len(rows), 8)
        return logits, tokens, None
