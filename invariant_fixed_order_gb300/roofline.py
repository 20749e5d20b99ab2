"""Algorithmic bytes and FLOPs of the forward step (what a step must move).

These counts are the roofline numerators: weights read once per step, the KV of
each request's own context, activations in and out, and 2*T*params FLOPs.  They
are not the padded tile FLOPs: a 128-row MMA tile over one real row does 128x
the arithmetic but moves the same bytes ("Batch invariance and reproducible
inference", "Fixed GEMM tiles: also cheap at batch 1").
"""
from __future__ import annotations

from .config import ModelConfig

BF16 = 2
F32 = 4


def layer_weight_bytes(cfg: ModelConfig) -> int:
    """Bytes of one decoder layer's weights (four GEMMs plus two RMSNorm gains)."""
    d, F = cfg.d, cfg.F
    gemm = cfg.qkv_dim * d + d * cfg.H * cfg.Dh + 2 * F * d + d * F
    return (gemm + 2 * d) * BF16


def qkv_weight_bytes(cfg: ModelConfig) -> int:
    return cfg.qkv_dim * cfg.d * BF16


def lm_head_bytes(cfg: ModelConfig) -> int:
    return (cfg.V * cfg.d + cfg.d) * BF16


def step_weight_bytes(cfg: ModelConfig, with_lm_head: bool = True) -> int:
    """Weights one decode step reads: every layer plus the LM head (the embedding
    table is only gathered, T rows)."""
    return cfg.n_layers * layer_weight_bytes(cfg) + (lm_head_bytes(cfg) if with_lm_head else 0)


def kv_bytes_per_layer(cfg: ModelConfig, seq_len: int) -> int:
    """K and V of one request's context in one layer: 2 * s * Hkv * Dh * 2 bytes."""
    return 2 * seq_len * cfg.Hkv * cfg.Dh * BF16


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def gemm_weight_intensity(M: int, N: int, K: int) -> float:
    """FLOP per weight byte of an [M,K]x[K,N] GEMM whose bytes are the weights: M."""
    return gemm_flops(M, N, K) / (K * N * BF16)


def layer_flops(cfg: ModelConfig, T: int) -> int:
    """GEMM FLOPs of one layer over T tokens: 2 * T * (weight elements)."""
    d, F = cfg.d, cfg.F
    params = cfg.qkv_dim * d + d * cfg.H * cfg.Dh + 2 * F * d + d * F
    return 2 * T * params


def attention_flops(cfg: ModelConfig, q_positions) -> int:
    """Score and value FLOPs of causal attention: 4 * H * Dh per (query, key)."""
    keys = sum(int(p) + 1 for p in q_positions)
    return 4 * cfg.H * cfg.Dh * keys


def decode_layer_bytes(cfg: ModelConfig, seq_lens) -> int:
    """Algorithmic HBM bytes of one layer of one decode step over a batch whose
    requests have the given context lengths (the current token included):
    weights once, each request's KV once, and per token the activations the
    step stores and reads back: the residual stream and the two norm outputs
    (six d-vectors), the rotated q and the appended k and v (written once by
    the QKV GEMM's epilogue; the fp32 projection is never stored), q read by
    attention, the attention output written and read, the SwiGLU output
    written and read."""
    B = len(seq_lens)
    kv = sum(kv_bytes_per_layer(cfg, int(s)) for s in seq_lens)
    act = B * (cfg.d * BF16 * 6 + cfg.qkv_dim * BF16 + cfg.H * cfg.Dh * BF16 * 3
               + cfg.F * BF16 * 2)
    return layer_weight_bytes(cfg) + kv + act


def decode_step_bytes(cfg: ModelConfig, seq_lens, with_lm_head: bool = True) -> int:
    B = len(seq_lens)
    lm = (lm_head_bytes(cfg) + B * (cfg.V * F32 + cfg.d * BF16 * 2)) if with_lm_head else 0
    return cfg.n_layers * decode_layer_bytes(cfg, seq_lens) + lm
