"""The batched decode step on the tcgen05 tensor cores, against the oracle.

INT4 weights from 16 sequences on, bf16 weights from 5: the weight stages run
as tensor-core GEMMs (weights expanded to fp16 code * scale into tensor
memory, activations as three fp16 limbs, fp32 accumulators), the attention
stage as in the smaller batches.  Checked like the other batches: the bf16
output and every stage against the oracle's fp64 values at the step's
tolerance, the appended K/V rows within one bf16 ulp, the history and the
slots after pos bit-exact; runs are deterministic.  Shapes cover ragged row
tiles (a matrix height that is not a multiple of 128), head_dim 64 and 128,
query groups of 1-8 heads, several layers, and caches with spare slots.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_transformer_decode_gb300 import configs, ddl, synth, workload
from tests.gpu_helpers import (MAX_ABS, REL_L2, bf16_bits_close, device_outputs, host_layer,
                               oracle_stack, rel_l2)

pytestmark = pytest.mark.gpu

SMALL = configs.DecodeConfig("tc-small", D=256, H_q=8, H_kv=2, head_dim=128, d_ff=320, rope_base=1e4,
                             kv_len=45, layers=2, seed=51)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddl.load(build_if_missing=True)
    yield
    ddl.ddl_set_launch_mode(0)
    torch.cuda.empty_cache()


def _check(st, kv0, stages=True):
    out, res, dst = device_outputs(st)
    z, ost, _, caches = oracle_stack(st, kv0, stages_last=stages)
    e_out = rel_l2(oracle.bf16_to_f64(out), z)
    e_res = float(np.max(np.abs(res - z)))
    assert e_out <= REL_L2, f"bf16 output rel-L2 {e_out:.3e}"
    assert e_res <= MAX_ABS, f"fp32 residual max-abs {e_res:.3e}"
    p = st.pos
    for l, (kc_o, vc_o) in enumerate(caches):
        kd, vd = synth.bits(st.kvs[l][0]), synth.bits(st.kvs[l][1])
        assert bf16_bits_close(kd[:, :, p], kc_o[:, :, p]), f"appended K, layer {l}"
        assert bf16_bits_close(vd[:, :, p], vc_o[:, :, p]), f"appended V, layer {l}"
        np.testing.assert_array_equal(kd[:, :, :p], kv0[l][0][:, :, :p])
        np.testing.assert_array_equal(kd[:, :, p + 1:], kv0[l][0][:, :, p + 1:])
        np.testing.assert_array_equal(vd[:, :, p + 1:], kv0[l][1][:, :, p + 1:])
    if stages:
        for name in ("q", "attn", "y", "a"):
            e = rel_l2(dst[name], ost[name])
            assert e <= REL_L2, f"stage {name} rel-L2 {e:.3e}"
    return out, res


def _stack(cfg, B, wtype=ddl.INT4, s_max=None):
    st = workload.build_stack(cfg, batch=B, wtype=wtype, s_max=s_max)
    kv0 = [(synth.bits(k).copy(), synth.bits(v).copy()) for k, v in st.kvs]
    return st, kv0


@pytest.mark.parametrize("B", [16, 20, 33, 64])
def test_int4_batches(B):
    st, kv0 = _stack(SMALL, B)
    _check(st, kv0)


@pytest.mark.parametrize("B", [5, 16, 64])
def test_bf16_weight_batches(B):
    st, kv0 = _stack(SMALL.with_(seed=52), B, wtype=ddl.BF16)
    _check(st, kv0)


@pytest.mark.parametrize("cfg", [
    SMALL.with_(D=2112, d_ff=4160, H_q=6, H_kv=2, kv_len=70, layers=1, name="ragged-rows"),
    SMALL.with_(H_q=8, H_kv=1, head_dim=128, D=192, d_ff=192, kv_len=5, layers=1, name="g8"),
    SMALL.with_(H_q=4, H_kv=2, head_dim=64, D=128, d_ff=192, kv_len=20, layers=3, name="hd64-3L"),
    SMALL.with_(H_q=2, H_kv=2, head_dim=64, D=64, d_ff=64, kv_len=0, layers=1, name="mha-empty-history"),
])
def test_shapes(cfg):
    st, kv0 = _stack(cfg, 16)
    _check(st, kv0)


def test_spare_slots_and_determinism():
    st, kv0 = _stack(SMALL.with_(seed=53), 24, s_max=SMALL.kv_len + 30)
    # slots after pos hold a planted pattern that must neither be read nor written
    for (kc, vc), (k0, v0) in zip(st.kvs, kv0):
        kc.view(torch.int16)[:, :, st.pos + 1:] = 0x4800
        vc.view(torch.int16)[:, :, st.pos + 1:] = 0x4800
        k0[:, :, st.pos + 1:] = 0x4800
        v0[:, :, st.pos + 1:] = 0x4800
    torch.cuda.synchronize()
    out1, res1 = _check(st, kv0)
    out2, res2, _ = device_outputs(st)
    np.testing.assert_array_equal(out1, out2)
    np.testing.assert_array_equal(res1, res2)
    ddl.ddl_set_launch_mode(1)  # the tensor-core path launches per stage either way
    try:
        out3, res3, _ = device_outputs(st)
    finally:
        ddl.ddl_set_launch_mode(0)
    np.testing.assert_array_equal(out1, out3)
    np.testing.assert_array_equal(res1, res3)


def test_layer_decode_with_residual_input():
    st, kv0 = _stack(SMALL.with_(layers=1, seed=54), 32)
    B, D = st.batch, SMALL.D
    resid = synth.normal_bf16((B, D), seed=55, std=3.0, device="cuda").float()
    out = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
    res = torch.empty((B, D), dtype=torch.float32, device="cuda")
    ddl.ddl_layer_decode(st.shape, st.wtype, st.layers[0], st.kvs[0], st.pos, resid_in=resid,
                         resid_out=res, out_bf16=out, workspace=st.workspace)
    torch.cuda.synchronize()
    assert ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max) == 0
    kc, vc = kv0[0][0].copy(), kv0[0][1].copy()
    z = oracle.layer_decode(SMALL, host_layer(SMALL.with_(seed=54), 0, st.wtype), kc, vc, st.pos,
                            resid.cpu().numpy().astype(np.float64))
    assert rel_l2(oracle.bf16_to_f64(synth.bits(out)), z) <= REL_L2
    assert float(np.max(np.abs(res.cpu().numpy().astype(np.float64) - z))) <= MAX_ABS
