"""Engine: a model's weights, its paged KV pools and a forward-step workspace on
one GPU, around the C ABI's bi_forward_step.

Weights are random (seeded), drawn on the device by ``synth``; gate and up are
packed into the interleaved layout the SwiGLU epilogue reads.  All compute
runs in libbi; this class only owns memory and marshals arguments.
"""
from __future__ import annotations

import numpy as np
import torch

from . import bi, synth
from .config import ModelConfig


class PagePool:
    """Free list of physical KV pages, handed out in a seeded shuffled order."""

    def __init__(self, num_pages: int, seed: int = 0):
        self.num_pages = num_pages
        rng = np.random.default_rng(seed)
        self._free = [int(p) for p in rng.permutation(num_pages)]

    def alloc(self, n: int) -> list:
        if n > len(self._free):
            raise MemoryError(f"KV pool exhausted: need {n} pages, {len(self._free)} free")
        out, self._free = self._free[:n], self._free[n:]
        return out

    def free(self, pages) -> None:
        self._free.extend(int(p) for p in pages)

    @property
    def n_free(self) -> int:
        return len(self._free)


class Engine:
    def __init__(self, cfg: ModelConfig, *, seed: int = 1234, num_pages: int, max_pages: int, max_T: int,
                 max_B: int, max_R: int, max_seq: int | None = None, device: str = "cuda",
                 keep_logical: bool = False, weights: dict | None = None):
        self.cfg = cfg
        self.device = device
        self.max_pages = max_pages
        self.max_seq = max_seq or max_pages * bi.PAGE
        max_pos = self.max_seq + 1
        self.logical = [] if keep_logical else None
        layers = []
        for l in range(cfg.n_layers):
            w = weights["layers"][l] if weights else synth.layer_weights(cfg, seed, device, l)
            if keep_logical:
                self.logical.append(w)
            layers.append({
                "gamma_attn": w["gamma_attn"], "w_qkv": w["w_qkv"], "w_o": w["w_o"],
                "gamma_ffn": w["gamma_ffn"], "w_gu": bi.pack_gate_up(w["w_gate"], w["w_up"]),
                "w_down": w["w_down"],
            })
            if not keep_logical:
                del w
        self.head = weights["head"] if weights else synth.head_weights(cfg, seed, device)
        self.layers = layers
        self.model = bi.Model(cfg, layers, self.head, max_pos)
        shape = (num_pages, cfg.Hkv, bi.PAGE, cfg.Dh)
        self.k = [torch.zeros(shape, dtype=torch.bfloat16, device=device) for _ in range(cfg.n_layers)]
        self.v = [torch.zeros(shape, dtype=torch.bfloat16, device=device) for _ in range(cfg.n_layers)]
        self.pool = PagePool(num_pages, seed)
        self.ws = torch.empty(self.model.workspace_size(max_T, max_B, max_R, self.max_seq), dtype=torch.uint8,
                              device=device)
        self.status = bi.new_status(device)
        self.max_T, self.max_B, self.max_R = max_T, max_B, max_R

    def step(self, q_len, pos0, token_ids, page_table, logit_rows, mode: int = bi.INVARIANT,
             want_logits: bool = True, want_hidden: bool = False, stream=None, logits_out=None, tokens_out=None):
        """One forward step.  token_ids / page_table: device int32 tensors (or
        host arrays, copied here); q_len, pos0, logit_rows: host sequences."""
        if not isinstance(token_ids, torch.Tensor) or token_ids.device.type != "cuda":
            token_ids = torch.as_tensor(np.asarray(token_ids, np.int32)).to(self.device)
        if not isinstance(page_table, torch.Tensor) or page_table.device.type != "cuda":
            page_table = torch.as_tensor(np.ascontiguousarray(page_table, np.int32)).to(self.device)
        R = len(logit_rows)
        T = int(sum(int(q) for q in q_len))
        if logits_out is None and want_logits:
            logits_out = torch.empty(R, self.cfg.V, dtype=torch.float32, device=self.device)
        if tokens_out is None:
            tokens_out = torch.empty(max(R, 1), dtype=torch.int32, device=self.device)
        hidden = torch.empty(T, self.cfg.d, dtype=torch.bfloat16, device=self.device) if want_hidden else None
        self.model.forward_step(q_len, pos0, token_ids, page_table, self.k, self.v, logit_rows, self.ws,
                                self.status, logits_out=logits_out, tokens_out=tokens_out, hidden_out=hidden,
                                mode=mode, stream=stream)
        return logits_out, tokens_out[:R], hidden

    def check(self, stream=None) -> None:
        bi.check_status(self.status, stream)

    def close(self) -> None:
        self.model.close()
