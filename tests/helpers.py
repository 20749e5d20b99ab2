"""Shared helpers for the tests: paged-cache construction, metrics, tolerances."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances stated for this path: attention outputs max-abs <= 1e-3 (fp32
# kernel outputs from bf16-exact inputs); logits max-abs <= 2e-2 * max|ref| and
# relative Frobenius <= 5e-3.
ATTN_MAX_ABS = 1e-3
LOGIT_MAX_ABS_REL = 2e-2
LOGIT_REL_FRO = 5e-3


def rel_fro(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def assert_logits_close(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    assert err <= LOGIT_MAX_ABS_REL * scale, f"max-abs {err} > {LOGIT_MAX_ABS_REL} * {scale}"
    rf = rel_fro(got, ref)
    assert rf <= LOGIT_REL_FRO, f"relative Frobenius {rf} > {LOGIT_REL_FRO}"


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy()


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a tensor, for bitwise comparisons."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy()
    return t.numpy()


class PagedKV:
    """A paged KV pool [num_pages, Hkv, 16, Dh] (bf16) plus page tables.

    Pages are handed out in a shuffled order so that a request's logical pages
    are scattered over the pool."""

    def __init__(self, num_pages: int, Hkv: int, Dh: int, max_pages: int, n_req: int, seed: int = 0,
                 device="cuda", n_layers: int = 1):
        self.num_pages, self.Hkv, self.Dh, self.max_pages = num_pages, Hkv, Dh, max_pages
        self.k = [torch.zeros(num_pages, Hkv, 16, Dh, dtype=torch.bfloat16, device=device) for _ in range(n_layers)]
        self.v = [torch.zeros(num_pages, Hkv, 16, Dh, dtype=torch.bfloat16, device=device) for _ in range(n_layers)]
        rng = np.random.default_rng(seed)
        self.free = list(rng.permutation(num_pages))
        self.table = np.full((n_req, max_pages), -1, np.int32)
        self.n_alloc = np.zeros(n_req, np.int64)
        self.device = device

    def ensure(self, req: int, n_pos: int):
        need = (n_pos + 15) // 16
        while self.n_alloc[req] < need:
            self.table[req, self.n_alloc[req]] = self.free.pop()
            self.n_alloc[req] += 1

    def table_tensor(self, rows=None) -> torch.Tensor:
        t = self.table if rows is None else self.table[rows]
        return torch.from_numpy(np.ascontiguousarray(np.where(t < 0, 0, t))).to(self.device)

    def write(self, req: int, k: torch.Tensor, v: torch.Tensor, layer: int = 0, start: int = 0):
        """Scatter history k, v [n, Hkv, Dh] (bf16) of request req to positions start.."""
        n = k.shape[0]
        self.ensure(req, start + n)
        pos = np.arange(start, start + n)
        pages = torch.from_numpy(self.table[req, pos // 16].astype(np.int64)).to(self.device)
        slots = torch.from_numpy((pos % 16).astype(np.int64)).to(self.device)
        self.k[layer][pages, :, slots, :] = k.to(self.device)
        self.v[layer][pages, :, slots, :] = v.to(self.device)

    def read(self, req: int, n: int, layer: int = 0):
        pos = np.arange(n)
        pages = torch.from_numpy(self.table[req, pos // 16].astype(np.int64)).to(self.device)
        slots = torch.from_numpy((pos % 16).astype(np.int64)).to(self.device)
        return self.k[layer][pages, :, slots, :], self.v[layer][pages, :, slots, :]
