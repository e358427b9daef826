"""Shared helpers of the GPU parity tests: run the oracle on the same seeded
inputs a device stack was built from, and compare with the stated tolerances.

Tolerances (the decode step's floating-point bar, read per layer output):
  * relative L2 error of the bf16 output vs the oracle's fp64 z <= 2e-3
  * max-abs error of the fp32 residual output vs the oracle's z <= 2e-2
  * each stage (q after RoPE, attn, y, a) relative L2 <= 2e-3 vs the oracle
  * the appended K/V rows within one bf16 ulp plus 1e-4 of the rows' RMS
    (k, v are rounded to bf16 on both sides from values that differ by the
    fp32 error of the projection)
  * the quantizer, the packer and the KV append bit-exact
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from memory_bound_transformer_decode_gb300 import ddl, synth

REL_L2 = 2e-3
MAX_ABS = 2e-2


def tensor_core_path(st) -> bool:
    """The batched path on the tcgen05 tensor cores: INT4 from 16 sequences,
    bf16 weights from 5."""
    return (st.wtype == ddl.INT4 and st.batch >= 16) or (st.wtype == ddl.BF16 and st.batch > 4)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def bf16_bits_close(a: np.ndarray, b: np.ndarray, ulps: int = 1) -> bool:
    """Stored bf16 rows agree: |a - b| <= `ulps` bf16 ulps of the value plus an
    absolute 1e-4 of the rows' RMS.  The two sides round k, v to bf16 from
    values that differ by the fp32 error of the projection, whose size follows
    the row's scale, not each element's; near zero that is many ulps of the
    element, hence the absolute term."""
    av = oracle.bf16_to_f64(a)
    bv = oracle.bf16_to_f64(b)
    mag = np.maximum(np.abs(av), np.abs(bv))
    ulp = np.exp2(np.floor(np.log2(np.maximum(mag, 1e-38))) - 7)
    rms = float(np.sqrt(np.mean(bv * bv))) if bv.size else 0.0
    return bool(np.all(np.abs(av - bv) <= ulps * ulp + 1e-4 * rms))


def host_layer(cfg, layer: int, wtype: int):
    """The oracle's layer dict from the same seeded masters the device used."""
    w = synth.layer_weights(cfg, layer, device="cuda")
    wb = {k: synth.bits(v) for k, v in w.items()}
    del w
    return oracle.quantized_layer(wb) if wtype == ddl.INT4 else oracle.bf16_layer(wb)


def oracle_stack(st, kv_host=None, stages_last: bool = False, collect=()):
    """Run the oracle over every layer of device stack `st` (untethered: the
    oracle's own residual is carried from layer to layer).  kv_host: list of
    (K, V) uint16 host copies of the caches taken before the device step
    (slots < pos are identical after it anyway).  Returns (z, stages of the
    last layer or None, {layer: z} for layers in `collect`, caches)."""
    cfg = st.cfg
    x = oracle.bf16_to_f64(synth.bits(st.x))
    L = len(st.layers)
    zs = {}
    caches = []
    stages = None
    for l in range(L):
        lw = host_layer(cfg, l, st.wtype)
        if kv_host is not None:
            kc, vc = kv_host[l]
        else:
            kc, vc = (synth.bits(t) for t in st.kvs[l])
        kc, vc = kc.copy(), vc.copy()
        want_st = stages_last and l == L - 1
        r = oracle.layer_decode(cfg, lw, kc, vc, st.pos, x, stages=want_st)
        if want_st:
            x, stages = r
        else:
            x = r
        if l in collect:
            zs[l] = x.copy()
        caches.append((kc, vc))
    return x, stages, zs, caches


def device_outputs(st, mode: int | None = None):
    """Run one device decode step; returns (out_bf16 bits, resid fp32, stages)."""
    if mode is not None:
        ddl.ddl_set_launch_mode(mode)
    try:
        B, D = st.batch, st.cfg.D
        out = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
        res = torch.empty((B, D), dtype=torch.float32, device="cuda")
        st.decode(out_bf16=out, resid_out=res)
        torch.cuda.synchronize()
        status = ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max)
        assert status == 0, f"device status {status}"
        v = ddl.ddl_workspace_view(st.shape, B, st.s_max)
        cfg = st.cfg
        stages = {
            "q": ddl.ws_tensor(st.workspace, v.q, B * cfg.Nq).view(B, -1).cpu().numpy().copy(),
            "attn": ddl.ws_tensor(st.workspace, v.attn, B * cfg.Nq).view(B, -1).cpu().numpy().copy(),
            "y": ddl.ws_tensor(st.workspace, v.y, B * cfg.D).view(B, -1).cpu().numpy().copy(),
            "a": ddl.ws_tensor(st.workspace, v.a, B * cfg.d_ff).view(B, -1).cpu().numpy().copy(),
        }
        return synth.bits(out), res.cpu().numpy().astype(np.float64), stages
    finally:
        if mode is not None:
            ddl.ddl_set_launch_mode(0)
