"""Prefill (ddl_stack_prefill: S prompt tokens of one sequence as one batched
step) on the GPU vs the fp64 oracle's prefill (the rows in order on the
sequence's cache), through the C ABI: the bf16 outputs and fp32 residuals of
every row at the step's bars, the K/V rows appended at p0 .. p0 + S - 1, and
every other slot bit-unchanged.  Covers the batch <= 4 kernel (both launch
modes), the wide-batch kernel, the tcgen05 path (INT4 and bf16 weights, up to
64 rows), an empty history, a prompt in two chunks, and a 27B-class layer.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_transformer_decode_gb300 import configs, ddl, synth, workload
from tests.gpu_helpers import MAX_ABS, REL_L2, bf16_bits_close, host_layer, rel_l2

pytestmark = pytest.mark.gpu

SMALL = configs.SMALL_LAYER


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddl.load(build_if_missing=True)
    yield
    ddl.ddl_set_launch_mode(0)
    torch.cuda.empty_cache()


def _seq(cfg, p0, S_total, layers=1, wtype=ddl.INT4, spare=19):
    """One sequence: a history of p0 tokens, room for S_total prompt tokens;
    slots from p0 on hold a fixed pattern."""
    c = cfg.with_(kv_len=p0, layers=layers)
    st = workload.build_stack(c, batch=1, wtype=wtype, s_max=p0 + S_total + spare)
    for k, v in st.kvs:
        k[:, :, p0:] = 0.75
        v[:, :, p0:] = -0.5
    torch.cuda.synchronize()
    kv0 = [(synth.bits(k).copy(), synth.bits(v).copy()) for k, v in st.kvs]
    return st, kv0


def _prompt(cfg, S, seed):
    return synth.normal_bf16((S, cfg.D), seed=seed, device="cuda")


def _device(st, p0, x, mode=0):
    S, D = x.shape
    ws = torch.zeros(ddl.ddl_workspace_bytes(st.shape, S, st.s_max), dtype=torch.uint8, device="cuda")
    out = torch.empty((S, D), dtype=torch.bfloat16, device="cuda")
    res = torch.empty((S, D), dtype=torch.float32, device="cuda")
    ddl.ddl_set_launch_mode(mode)
    try:
        ddl.ddl_stack_prefill(st.shape, st.wtype, st.layers, st.kvs, p0, x_bf16=x, resid_out=res, out_bf16=out,
                              workspace=ws)
        torch.cuda.synchronize()
        assert ddl.ddl_read_device_status(ws, st.shape, S, st.s_max) == 0
    finally:
        ddl.ddl_set_launch_mode(0)
    return synth.bits(out), res.cpu().numpy().astype(np.float64)


def _oracle(st, kv, p0, x64):
    """The oracle's prefill over every layer; kv: host caches, updated in place."""
    for l in range(len(st.layers)):
        x64 = oracle.layer_prefill(st.cfg, host_layer(st.cfg, l, st.wtype), kv[l][0], kv[l][1], p0, x64)
    return x64


def _check(st, kv0, kv_ref, p0, S, out, res, z, kv_ulp=True):
    assert rel_l2(oracle.bf16_to_f64(out), z) <= REL_L2
    assert float(np.max(np.abs(res - z))) <= MAX_ABS
    for l in range(len(st.layers)):
        kd, vd = synth.bits(st.kvs[l][0]), synth.bits(st.kvs[l][1])
        for dev, ref, before in ((kd, kv_ref[l][0], kv0[l][0]), (vd, kv_ref[l][1], kv0[l][1])):
            for p in range(p0, p0 + S):
                if kv_ulp:
                    assert bf16_bits_close(dev[0, :, p], ref[0, :, p]), f"layer {l}, slot {p}"
                else:
                    assert rel_l2(oracle.bf16_to_f64(dev[0, :, p]), oracle.bf16_to_f64(ref[0, :, p])) <= REL_L2
            np.testing.assert_array_equal(dev[:, :, :p0], before[:, :, :p0])
            np.testing.assert_array_equal(dev[:, :, p0 + S:], before[:, :, p0 + S:])


@pytest.mark.parametrize("p0,S,mode", [(100, 1, 0), (100, 3, 0), (0, 3, 1), (45, 4, 1)])
def test_narrow_rows_two_layers(p0, S, mode):
    st, kv0 = _seq(SMALL, p0, S, layers=2)
    x = _prompt(SMALL, S, seed=p0 + S)
    out, res = _device(st, p0, x, mode)
    kv = [(k.copy(), v.copy()) for k, v in kv0]
    z = _oracle(st, kv, p0, oracle.bf16_to_f64(synth.bits(x)))
    _check(st, kv0, kv, p0, S, out, res, z)


def test_wide_rows():
    p0, S = 60, 9
    st, kv0 = _seq(SMALL, p0, S)
    x = _prompt(SMALL, S, seed=5)
    out, res = _device(st, p0, x)
    kv = [(k.copy(), v.copy()) for k, v in kv0]
    z = _oracle(st, kv, p0, oracle.bf16_to_f64(synth.bits(x)))
    _check(st, kv0, kv, p0, S, out, res, z, kv_ulp=False)  # the wide-batch kernel: K/V at the stage bar


@pytest.mark.parametrize("wtype,p0,S", [(ddl.INT4, 0, 16), (ddl.INT4, 33, 37), (ddl.INT4, 100, 64),
                                        (ddl.BF16, 17, 7)])
def test_tensor_core_rows(wtype, p0, S):
    st, kv0 = _seq(SMALL, p0, S, wtype=wtype)
    x = _prompt(SMALL, S, seed=S)
    out, res = _device(st, p0, x)
    kv = [(k.copy(), v.copy()) for k, v in kv0]
    z = _oracle(st, kv, p0, oracle.bf16_to_f64(synth.bits(x)))
    _check(st, kv0, kv, p0, S, out, res, z)


def test_prompt_in_two_chunks():
    p0, S = 20, 16
    st, kv0 = _seq(SMALL, p0, 2 * S, layers=2)
    x = _prompt(SMALL, 2 * S, seed=7)
    out1, res1 = _device(st, p0, x[:S])
    out2, res2 = _device(st, p0 + S, x[S:])
    kv = [(k.copy(), v.copy()) for k, v in kv0]
    z = _oracle(st, kv, p0, oracle.bf16_to_f64(synth.bits(x)))
    _check(st, kv0, kv, p0, 2 * S, np.concatenate([out1, out2]), np.concatenate([res1, res2]), z)


def test_27b_layer_prompt_after_long_history():
    cfg = configs.STACK27B.with_(layers=1)
    p0, S = 4000, 16
    st, kv0 = _seq(cfg, p0, S, spare=16)
    x = _prompt(cfg, S, seed=3)
    out, res = _device(st, p0, x)
    kv = [(k.copy(), v.copy()) for k, v in kv0]
    z = _oracle(st, kv, p0, oracle.bf16_to_f64(synth.bits(x)))
    _check(st, kv0, kv, p0, S, out, res, z)


def test_prompt_past_the_cache_is_refused():
    st, _ = _seq(SMALL, 10, 4, spare=0)
    x = _prompt(SMALL, 5, seed=1)
    ws = torch.zeros(ddl.ddl_workspace_bytes(st.shape, 5, st.s_max), dtype=torch.uint8, device="cuda")
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_stack_prefill(st.shape, st.wtype, st.layers, st.kvs, 10, x_bf16=x, workspace=ws)
    assert e.value.status == 2
