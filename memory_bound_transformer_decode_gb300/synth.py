"""Seeded synthetic inputs for the decode step.

This module only draws random numbers: it holds none of the decode step's
arithmetic and serves both the CUDA path and the oracle (the only module they
share).  Every tensor has its own sub-seed

    seed * 2**32 + (layer + 1) * 64 + tensor_id

with tensor ids norm1 0, wq 1, wk 2, wv 3, wo 4, norm2 5, wg 6, wu 7, wd 8,
K cache 9, V cache 10; the input x (id 0), the embedding table (id 11) and
the final norm weight (id 12) use layer = -1.  Values are drawn as fp32
normals (mean + std * N(0, 1)) and rounded to bf16 by PyTorch's
round-to-nearest-even conversion.

Two generators: on a CUDA device, torch's Philox generator (fast enough for
the 16-35 GB stacks); on the host, numpy's PCG64 (platform independent, used
for the small CPU-side cases).  A test that compares the two sides draws once
and hands the same tensors to both.
"""
from __future__ import annotations

import numpy as np
import torch

TENSOR_IDS = {"norm1": 0, "wq": 1, "wk": 2, "wv": 3, "wo": 4, "norm2": 5, "wg": 6,
              "wu": 7, "wd": 8, "kcache": 9, "vcache": 10, "embed": 11, "norm_f": 12}
WEIGHT_STD = 0.02
NORM_STD = 0.1


def subseed(seed: int, layer: int, tid: int) -> int:
    return (int(seed) << 32) + (int(layer) + 1) * 64 + int(tid)


def normal_bf16(shape, *, seed: int, mean: float = 0.0, std: float = 1.0,
                device="cpu") -> torch.Tensor:
    """bf16 tensor of mean + std * N(0, 1), drawn in fp32 then rounded RNE."""
    device = torch.device(device)
    shape = tuple(int(s) for s in shape)
    if device.type == "cuda":
        g = torch.Generator(device=device)
        g.manual_seed(int(seed))
        z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    else:
        rng = np.random.Generator(np.random.PCG64(int(seed)))
        z = torch.from_numpy(rng.standard_normal(shape, dtype=np.float32))
    if std != 1.0:
        z.mul_(std)
    if mean != 0.0:
        z.add_(mean)
    return z.to(torch.bfloat16)


def matrix_shapes(cfg) -> dict:
    """[N, K] of each weight matrix (y = W x, W row-major [out, in])."""
    return {"wq": (cfg.Nq, cfg.D), "wk": (cfg.Nkv, cfg.D), "wv": (cfg.Nkv, cfg.D),
            "wo": (cfg.D, cfg.Nq), "wg": (cfg.d_ff, cfg.D), "wu": (cfg.d_ff, cfg.D),
            "wd": (cfg.D, cfg.d_ff)}


def layer_weights(cfg, layer: int, device="cpu", names=None) -> dict:
    """bf16 master weights of one layer: matrices N(0, 0.02), norms 1 + N(0, 0.1)."""
    out = {}
    shapes = matrix_shapes(cfg)
    for name in names or ("norm1", "wq", "wk", "wv", "wo", "norm2", "wg", "wu", "wd"):
        sd = subseed(cfg.seed, layer, TENSOR_IDS[name])
        if name.startswith("norm"):
            out[name] = normal_bf16((cfg.D,), seed=sd, mean=1.0, std=NORM_STD, device=device)
        else:
            out[name] = normal_bf16(shapes[name], seed=sd, std=WEIGHT_STD, device=device)
    return out


def kv_cache(cfg, layer: int, s_max: int, device="cpu", batch=None):
    """K and V caches [B, H_kv, s_max, hd] bf16: slots 0..kv_len-1 N(0, 1), rest 0."""
    B = cfg.batch if batch is None else batch
    out = []
    for name in ("kcache", "vcache"):
        hist = normal_bf16((B, cfg.H_kv, cfg.kv_len, cfg.head_dim),
                           seed=subseed(cfg.seed, layer, TENSOR_IDS[name]), device=device)
        full = torch.zeros((B, cfg.H_kv, s_max, cfg.head_dim), dtype=torch.bfloat16,
                           device=device)
        full[:, :, :cfg.kv_len] = hist
        out.append(full)
    return out[0], out[1]


def input_x(cfg, device="cpu", batch=None) -> torch.Tensor:
    """Layer-0 input x [B, D] bf16, N(0, 1)."""
    B = cfg.batch if batch is None else batch
    return normal_bf16((B, cfg.D), seed=subseed(cfg.seed, -1, 0), device=device)


def head_weights(cfg, vocab: int, device="cpu") -> dict:
    """The embedding table [vocab, D] (N(0, 0.02), also the output matrix) and
    the final norm weight [D] (1 + N(0, 0.1)), bf16."""
    return {"embed": normal_bf16((vocab, cfg.D), seed=subseed(cfg.seed, -1, TENSOR_IDS["embed"]),
                                 std=WEIGHT_STD, device=device),
            "norm_f": normal_bf16((cfg.D,), seed=subseed(cfg.seed, -1, TENSOR_IDS["norm_f"]),
                                  mean=1.0, std=NORM_STD, device=device)}


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16 tensor, on the host."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
