"""Algorithmic bytes and FLOPs of a decode step, and the roofline arithmetic.

Decode at small batch is bound by HBM bandwidth: every step reads every
weight once plus each sequence's KV history ("把基础打牢" primer §1.2: decode
latency is about the time to read the weights once; §1.3 roofline with
intensity I = FLOPs / bytes; roofline reply §一-§二: ridge point and the
batch-1 intensity of about 1 op/byte).

Bytes counted per step (activations, < 0.1 MB per layer, are excluded):
  weights   INT4: N*K/2 packed codes + 2*N*K/64 bf16 scales per matrix
            bf16: 2*N*K per matrix
  norms     2 bf16 vectors of D per layer
  KV        per sequence, per layer: read S history rows and write 1 new row
            of K and V: 2 * H_kv * hd * 2 bytes * (S + 1)
FLOPs: 2 per multiply-add of every matrix row and sequence, plus
4 * H_q * hd * (S + 1) per sequence and layer for q.K and p.V.
"""
from __future__ import annotations

GROUP = 64


def matrix_dims(cfg) -> list[tuple[int, int]]:
    """[N, K] of the seven matrices of one layer."""
    D, F, Nq, Nkv = cfg.D, cfg.d_ff, cfg.Nq, cfg.Nkv
    return [(Nq, D), (Nkv, D), (Nkv, D), (D, Nq), (F, D), (F, D), (D, F)]


def weight_bytes_per_layer(cfg, weights: str | None = None) -> int:
    w = weights or cfg.weights
    tot = 0
    for N, K in matrix_dims(cfg):
        tot += (N * K // 2 + 2 * N * (K // GROUP)) if w == "int4" else 2 * N * K
    return tot + 2 * 2 * cfg.D


def kv_bytes_per_layer(cfg, batch: int | None = None) -> int:
    B = cfg.batch if batch is None else batch
    return B * 2 * cfg.H_kv * cfg.head_dim * 2 * (cfg.kv_len + 1)


def step_bytes(cfg, batch: int | None = None, weights: str | None = None,
               layers: int | None = None) -> int:
    L = cfg.layers if layers is None else layers
    return L * (weight_bytes_per_layer(cfg, weights) + kv_bytes_per_layer(cfg, batch))


def step_flops(cfg, batch: int | None = None, layers: int | None = None) -> int:
    B = cfg.batch if batch is None else batch
    L = cfg.layers if layers is None else layers
    mac = sum(N * K for N, K in matrix_dims(cfg))
    att = 4 * cfg.H_q * cfg.head_dim * (cfg.kv_len + 1)
    return L * B * (2 * mac + att)


def intensity(flops: float, nbytes: float) -> float:
    """Operational intensity I = FLOPs / bytes (primer §1.3)."""
    return flops / nbytes


def roofline_seconds(nbytes: float, bandwidth_bytes_per_s: float) -> float:
    """Lower bound on a memory-bound step: bytes / bandwidth (primer §1.2)."""
    return nbytes / bandwidth_bytes_per_s


def estimate_mem(params_billion: float, L: int, D: int, H_q: int, H_kv: int, d_h: int,
                 S: int, B: int, bytes_per: int = 2) -> dict:
    """Memory bill of a dense LLM in bytes (primer §1.4): weights, KV cache,
    Adam state (fp32 m, v + 16-bit master) and training activations."""
    p = params_billion * 1e9
    return {
        "weights": p * bytes_per,
        "kv": 2 * H_kv * d_h * bytes_per * L * B * S,
        "adam": p * (4 + 4 + 2),
        "act_train": B * S * L * D * 2 * bytes_per,
    }
