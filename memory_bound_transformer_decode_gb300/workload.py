"""Device-resident decode workloads built through the C ABI.

build_stack() draws each layer's bf16 master weights with the seeded
generator, quantizes them with ddl_quantize_int4 (or keeps bf16), packs them
with ddl_pack_layer, frees the masters, and draws the KV history.  The result
holds exactly what a decode step reads: packed weights, norm weights, caches.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import ddl, synth

MATS = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


@dataclass
class Stack:
    cfg: object
    wtype: int
    batch: int
    s_max: int
    shape: ddl.Shape
    layers: list = field(default_factory=list)   # dicts: packed, norm1, norm2
    kvs: list = field(default_factory=list)      # (K, V) [B, H_kv, s_max, hd] bf16
    x: torch.Tensor | None = None                 # [B, D] bf16
    workspace: torch.Tensor | None = None

    @property
    def pos(self) -> int:
        return self.cfg.kv_len

    def decode(self, out_bf16=None, resid_out=None, x=None, stream=None):
        ddl.ddl_stack_decode(self.shape, self.wtype, self.layers, self.kvs, self.pos,
                             x_bf16=self.x if x is None else x, resid_out=resid_out,
                             out_bf16=out_bf16, workspace=self.workspace, stream=stream)


def pack_layer_from_master(shape, wtype: int, w: dict) -> torch.Tensor:
    """Quantize (INT4) or pass through (bf16) one layer's masters and pack them."""
    if wtype == ddl.INT4:
        mats = {n: ddl.ddl_quantize_int4(w[n]) for n in MATS}
    else:
        mats = {n: w[n] for n in MATS}
    return ddl.ddl_pack_layer(shape, wtype, mats)


def build_stack(cfg, *, batch: int | None = None, wtype: int | None = None, layers: int | None = None,
                s_max: int | None = None, device="cuda") -> Stack:
    B = cfg.batch if batch is None else batch
    if wtype is None:
        wtype = ddl.INT4 if cfg.weights == "int4" else ddl.BF16
    L = cfg.layers if layers is None else layers
    s_max = cfg.kv_len + 1 if s_max is None else s_max
    shape = ddl.make_shape(cfg)
    st = Stack(cfg=cfg, wtype=wtype, batch=B, s_max=s_max, shape=shape)
    for layer in range(L):
        w = synth.layer_weights(cfg, layer, device=device)
        packed = pack_layer_from_master(shape, wtype, w)
        st.layers.append({"packed": packed, "norm1": w["norm1"], "norm2": w["norm2"]})
        del w
        st.kvs.append(synth.kv_cache(cfg, layer, s_max, device=device, batch=B))
    st.x = synth.input_x(cfg, device=device, batch=B)
    n = ddl.ddl_workspace_bytes(shape, B, s_max)
    st.workspace = torch.zeros(n, dtype=torch.uint8, device=device)
    torch.cuda.synchronize()
    return st
