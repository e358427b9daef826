"""Decode workloads: the layer shapes and cache lengths the library is measured on.

Each workload is one batch-B decode step of a GQA decoder stack with 4-bit
(or bf16) weights ("把基础打牢" primer §1.2 decode_step; Unsloth/Qwen-27B
article §三 for the 27B-class shape).  Weights are random (N(0, 0.02)),
RMSNorm weights 1 + N(0, 0.1), eps 1e-6, KV history N(0, 1) bf16, the new
token at position = cache length, input x N(0, 1) bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    D: int
    H_q: int
    H_kv: int
    head_dim: int
    d_ff: int
    rope_base: float
    kv_len: int          # history length S; the new token sits at position S
    layers: int
    batch: int = 1
    eps: float = 1e-6
    seed: int = 0
    weights: str = "int4"  # "int4" (symmetric, group 64, bf16 scales) or "bf16"

    @property
    def group(self) -> int:
        return self.H_q // self.H_kv

    @property
    def Nq(self) -> int:
        return self.H_q * self.head_dim

    @property
    def Nkv(self) -> int:
        return self.H_kv * self.head_dim

    @property
    def pos(self) -> int:
        return self.kv_len

    def with_(self, **kw) -> "DecodeConfig":
        return replace(self, **kw)


# One small decode layer: D=512, 8 query heads over 2 KV heads, hd 64, cache 128.
SMALL_LAYER = DecodeConfig("small-layer-d512-kv128", D=512, H_q=8, H_kv=2, head_dim=64,
                           d_ff=1408, rope_base=1e4, kv_len=128, layers=1, seed=0)

# One Qwen2.5-7B-shaped layer with a 4096-token cache.
QWEN7B_LAYER = DecodeConfig("qwen2.5-7b-layer-kv4096", D=3584, H_q=28, H_kv=4, head_dim=128,
                            d_ff=18944, rope_base=1e6, kv_len=4096, layers=1, seed=1)

# The 27B-class 64-layer stack at batch 1 with an 8192-token cache (the headline).
STACK27B = DecodeConfig("27b-class-64L-int4-kv8192-b1", D=5120, H_q=64, H_kv=8, head_dim=128,
                        d_ff=25600, rope_base=1e6, kv_len=8192, layers=64, seed=2)

# The same 27B-class stack, batch sweep with a 4096-token cache per sequence.
STACK27B_SWEEP = DecodeConfig("27b-class-64L-kv4096-sweep", D=5120, H_q=64, H_kv=8,
                              head_dim=128, d_ff=25600, rope_base=1e6, kv_len=4096, layers=64,
                              seed=3)
SWEEP_BATCHES = (1, 4, 16, 64)

# Llama-3-70B-shaped 80-layer stack with a 32768-token cache.
LLAMA70B_STACK = DecodeConfig("llama3-70b-80L-int4-kv32768-b1", D=8192, H_q=64, H_kv=8,
                              head_dim=128, d_ff=28672, rope_base=5e5, kv_len=32768, layers=80,
                              seed=4)

# Vocabulary of the LM head: the Qwen-class vocabulary of about 152 thousand
# entries (Unsloth/Qwen-27B article §三), 152064 = 16 x 9504.
VOCAB = 152064

ALL = (SMALL_LAYER, QWEN7B_LAYER, STACK27B, STACK27B_SWEEP, LLAMA70B_STACK)
BY_NAME = {c.name: c for c in ALL}
