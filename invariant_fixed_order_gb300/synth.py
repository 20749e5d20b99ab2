"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module only draws random numbers; it holds none of the forward step's
arithmetic.  Weights and activations are drawn in fp32 by torch's seeded
generator and rounded to bf16 by torch's own conversion (round to nearest
even); both the CUDA path and the oracle receive the same tensors.

Recipe (weights seed 1234, data seed 42+cfg, schedules 1000+k by convention):
  * linear weights N(0, 0.02) bf16;
  * RMSNorm gains 1 + N(0, 0.02) bf16 (a gain near zero would flatten the
    attention scores and the tests would lose their teeth);
  * embedding rows N(0, 1) bf16 so the first layer sees unit-scale activations;
  * KV history N(0, 1) bf16; hidden states N(0, 1) bf16;
  * token ids uniform over the vocabulary; context lengths uniform in a range.
"""
from __future__ import annotations

import numpy as np
import torch

from .config import ModelConfig


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu", mean: float = 0.0) -> torch.Tensor:
    g = generator(seed, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def layer_weights(cfg: ModelConfig, seed: int, device="cpu", layer: int = 0) -> dict:
    """Logical weights of one decoder layer (gate and up kept separate)."""
    s = int(seed) * 1000 + layer * 16
    return {
        "gamma_attn": normal_bf16((cfg.d,), 0.02, s + 1, device, mean=1.0),
        "w_qkv": normal_bf16((cfg.qkv_dim, cfg.d), 0.02, s + 2, device),
        "w_o": normal_bf16((cfg.d, cfg.H * cfg.Dh), 0.02, s + 3, device),
        "gamma_ffn": normal_bf16((cfg.d,), 0.02, s + 4, device, mean=1.0),
        "w_gate": normal_bf16((cfg.F, cfg.d), 0.02, s + 5, device),
        "w_up": normal_bf16((cfg.F, cfg.d), 0.02, s + 6, device),
        "w_down": normal_bf16((cfg.d, cfg.F), 0.02, s + 7, device),
    }


def head_weights(cfg: ModelConfig, seed: int, device="cpu") -> dict:
    s = int(seed) * 1000 + 999 * 16
    return {
        "embed": normal_bf16((cfg.V, cfg.d), 1.0, s + 1, device),
        "gamma_final": normal_bf16((cfg.d,), 0.02, s + 2, device, mean=1.0),
        "w_lm": normal_bf16((cfg.V, cfg.d), 0.02, s + 3, device),
    }


def hidden(T: int, d: int, seed: int, device="cpu") -> torch.Tensor:
    return normal_bf16((T, d), 1.0, seed, device)


def kv_history(n: int, Hkv: int, Dh: int, seed: int, device="cpu"):
    """K and V history of one request: two bf16 tensors [n, Hkv, Dh] ~ N(0, 1)."""
    k = normal_bf16((n, Hkv, Dh), 1.0, seed * 2 + 1, device)
    v = normal_bf16((n, Hkv, Dh), 1.0, seed * 2 + 2, device)
    return k, v


def token_ids(n: int, V: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(0, V, size=n, dtype=np.int64).astype(np.int32)


def uniform_ints(n: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """n integers uniform on [lo, hi] inclusive."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=n, dtype=np.int64).astype(np.int32)


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


def to_f32_numpy(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> float32 numpy array (exact)."""
    return t.detach().to("cpu", torch.float32).contiguous().numpy()
