"""Model shapes and the method's fixed constants.

The constants below never depend on a batch: they are the fixed split points
("Lockstep", "The fix": every reduction has a fixed order with fixed split
points chosen independently of batch shape).
"""
from __future__ import annotations

from dataclasses import dataclass

# Attention key chunk: split count = ceil(seq_len / KV_CHUNK), a function of the
# request alone ("Batch invariance and reproducible inference", "1 · Split-K and
# segmented attention reductions": the Triton split tile defaults to 256).
KV_CHUNK = 256
# KV cache page size in tokens.
PAGE = 16
# GEMM tiling: one MMA instruction shape and one K tile for every M.
GEMM_BLOCK_M = 128
GEMM_BLOCK_K = 64


@dataclass(frozen=True)
class ModelConfig:
    name: str
    d: int          # hidden size
    H: int          # query heads
    Hkv: int        # key/value heads
    Dh: int         # head dim
    F: int          # SwiGLU ffn width
    V: int          # vocabulary
    n_layers: int
    eps: float = 1e-5
    rope_theta: float = 500000.0

    @property
    def qkv_dim(self) -> int:
        return (self.H + 2 * self.Hkv) * self.Dh

    @property
    def group(self) -> int:
        return self.H // self.Hkv

    def with_layers(self, n: int) -> "ModelConfig":
        return ModelConfig(self.name, self.d, self.H, self.Hkv, self.Dh, self.F, self.V, n,
                           self.eps, self.rope_theta)


# Tiny single decoder layer + LM head.
TINY = ModelConfig("tiny-1L", d=256, H=4, Hkv=2, Dh=64, F=1024, V=2048, n_layers=1)
# Llama-3-8B shapes (random init).
LLAMA3_8B = ModelConfig("llama3-8b-shape", d=4096, H=32, Hkv=8, Dh=128, F=14336, V=128256,
                        n_layers=32)
LLAMA3_8B_1L = LLAMA3_8B.with_layers(1)
