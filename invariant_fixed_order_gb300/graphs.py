"""CUDA graphs of the decode step on a bucket ladder.

"Batch invariance and reproducible inference", "3 · Kernel selection changing
with shape" and "The regression that only reproduces at one batch size": a
graph is captured per bucket of a ladder, and a batch replays the smallest
bucket that holds it, padded with rows that do no harm.  Padding changes the
launch geometry (M of every GEMM, the attention grid) but, with every
reduction fixed per request, never a real row's bits; the tests use the
ladder as a fuzz axis (eager step, smallest bucket, a larger bucket: the same
logits bit for bit).

The step is captured through ``bi_batch.meta``: its per-token metadata lives
on the device, so replay needs only new contents of the bucket's buffers
(token ids, page-table rows, positions).  Padding rows decode token 0 at
position 0 of a reserved scratch page, which no request ever owns.
"""
from __future__ import annotations

import numpy as np
import torch

from . import bi

LADDER = (1, 2, 4, 8, 16, 24, 32, 48, 64)


class DecodeGraphs:
    def __init__(self, eng, max_ctx: int, ladder=LADDER, mode: int = bi.INVARIANT):
        """eng: an Engine; max_ctx: the largest context (positions + 1) any replayed request may reach."""
        if max_ctx > eng.max_seq:
            raise ValueError("max_ctx beyond the engine's max_seq")
        self.eng, self.mode, self.max_ctx = eng, mode, max_ctx
        self.scratch = eng.pool.alloc(1)[0]
        self.stream = torch.cuda.Stream(device=eng.device)
        self.buckets = {}
        cfg, dev = eng.cfg, eng.device
        self.stream.wait_stream(torch.cuda.current_stream(dev))
        for Bk in sorted(ladder):
            if Bk > eng.max_B or Bk > eng.max_R or Bk > eng.max_T:
                break
            bufs = {
                "ids": torch.zeros(Bk, dtype=torch.int32, device=dev),
                "table": torch.full((Bk, eng.max_pages), self.scratch, dtype=torch.int32, device=dev),
                "meta": torch.from_numpy(self._meta(np.zeros(Bk, np.int32), Bk)).to(dev),
                "logits": torch.empty(Bk, cfg.V, dtype=torch.float32, device=dev),
                "tokens": torch.empty(Bk, dtype=torch.int32, device=dev),
            }
            with torch.cuda.stream(self.stream):
                self._run(bufs, Bk)  # once outside the capture: one-time setup of every kernel
            self.stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self._run(bufs, Bk)
            self.buckets[Bk] = (g, bufs)
        torch.cuda.current_stream(dev).wait_stream(self.stream)

    @staticmethod
    def _meta(positions: np.ndarray, Bk: int) -> np.ndarray:
        """[request of token t][position of token t][decode tokens][prefill tokens: none][logit rows]."""
        ar = np.arange(Bk, dtype=np.int32)
        return np.concatenate([ar, positions.astype(np.int32), ar, ar])

    def _run(self, bufs: dict, Bk: int) -> None:
        # the captured shapes: Bk decode rows whose contexts may reach max_ctx
        self.eng.model.forward_step([1] * Bk, [self.max_ctx - 1] * Bk, bufs["ids"], bufs["table"], self.eng.k,
                                    self.eng.v, list(range(Bk)), self.eng.ws, self.eng.status,
                                    logits_out=bufs["logits"], tokens_out=bufs["tokens"], mode=self.mode,
                                    stream=self.stream, meta=bufs["meta"])

    def bucket_for(self, B: int) -> int:
        for Bk in sorted(self.buckets):
            if Bk >= B:
                return Bk
        raise ValueError(f"no captured bucket holds {B} rows")

    def step(self, token_ids, positions, page_rows, bucket: int | None = None):
        """One decode step of B requests by graph replay: token_ids, positions (host int sequences, the new
        token's position) and page_rows (host [B, max_pages]).  Returns (logits [B, V], greedy tokens [B]),
        views of the bucket's buffers valid until its next replay."""
        B = len(token_ids)
        Bk = self.bucket_for(B) if bucket is None else bucket
        if Bk not in self.buckets or Bk < B:
            raise ValueError(f"bucket {Bk} cannot hold {B} rows")
        pos = np.zeros(Bk, np.int32)
        pos[:B] = np.asarray(positions, np.int32)
        if B and (pos[:B].min() < 0 or pos[:B].max() >= self.max_ctx):
            raise ValueError("position outside the captured range")
        ids = np.zeros(Bk, np.int32)
        ids[:B] = np.asarray(token_ids, np.int32)
        table = np.full((Bk, self.eng.max_pages), self.scratch, np.int32)
        table[:B] = np.asarray(page_rows, np.int32).reshape(B, -1)[:, : self.eng.max_pages]
        g, bufs = self.buckets[Bk]
        cur = torch.cuda.current_stream(self.eng.device)
        self.stream.wait_stream(cur)
        with torch.cuda.stream(self.stream):
            bufs["ids"].copy_(torch.from_numpy(ids))
            bufs["table"].copy_(torch.from_numpy(table))
            bufs["meta"].copy_(torch.from_numpy(self._meta(pos, Bk)))
            g.replay()
        cur.wait_stream(self.stream)
        return bufs["logits"][:B], bufs["tokens"][:B]

    def close(self) -> None:
        self.buckets.clear()
        self.eng.pool.free([self.scratch])
