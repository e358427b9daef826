"""Sequences at their own positions (ddl_stack_decode_ragged) on the GPU vs the
fp64 oracle run sequence by sequence, through the C ABI: the bf16 output and
the fp32 residual at the step's bars, the last layer's stages, the appended
K/V rows at each sequence's own slot, and every other slot of every cache
bit-unchanged (the history beyond a sequence's position holds junk that must
not reach its result).  Covers the batch <= 4 kernel, the wide-batch kernel,
the tcgen05 path (INT4 and bf16 weights), both launch modes, positions 0 and
at tile edges, and a 27B-class layer with an 8192-token history.
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


def _stack(cfg, B, pos, layers=1, wtype=ddl.INT4, spare=23):
    """History drawn up to max(pos); slots from there on hold a fixed pattern."""
    S = max(pos)
    c = cfg.with_(kv_len=S, layers=layers)
    st = workload.build_stack(c, batch=B, wtype=wtype, s_max=S + 1 + spare)
    for k, v in st.kvs:
        k[:, :, S:] = 0.75
        v[:, :, S:] = -0.5
    torch.cuda.synchronize()
    kv0 = [(synth.bits(k).copy(), synth.bits(v).copy()) for k, v in st.kvs]
    return st, kv0


def _run(st, pos, mode=0):
    ddl.ddl_set_launch_mode(mode)
    try:
        B, D = st.batch, st.cfg.D
        out = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
        res = torch.empty((B, D), dtype=torch.float32, device="cuda")
        ddl.ddl_stack_decode_ragged(st.shape, st.wtype, st.layers, st.kvs, pos, x_bf16=st.x, resid_out=res,
                                    out_bf16=out, workspace=st.workspace)
        torch.cuda.synchronize()
        assert ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max) == 0
        v = ddl.ddl_workspace_view(st.shape, B, st.s_max)
        cfg = st.cfg
        stages = {n: ddl.ws_tensor(st.workspace, off, B * k).view(B, -1).cpu().numpy().copy()
                  for n, off, k in (("q", v.q, cfg.Nq), ("attn", v.attn, cfg.Nq), ("y", v.y, cfg.D),
                                    ("a", v.a, cfg.d_ff))}
        return synth.bits(out), res.cpu().numpy().astype(np.float64), stages
    finally:
        ddl.ddl_set_launch_mode(0)


def _check(st, kv0, pos, mode=0, kv_ulp=True):
    out, res, dst = _run(st, pos, mode)
    cfg = st.cfg
    x = oracle.bf16_to_f64(synth.bits(st.x))
    L = len(st.layers)
    for l in range(L):
        kc, vc = kv0[l][0].copy(), kv0[l][1].copy()
        r = oracle.layer_decode_ragged(cfg, host_layer(cfg, l, st.wtype), kc, vc, pos, x, stages=l == L - 1)
        x, ost = r if l == L - 1 else (r, None)
        kd, vd = synth.bits(st.kvs[l][0]), synth.bits(st.kvs[l][1])
        for b, p in enumerate(pos):
            if kv_ulp:
                assert bf16_bits_close(kd[b, :, p], kc[b, :, p]), f"appended K, layer {l}, sequence {b}"
                assert bf16_bits_close(vd[b, :, p], vc[b, :, p]), f"appended V, layer {l}, sequence {b}"
            else:
                assert rel_l2(oracle.bf16_to_f64(kd[b, :, p]), oracle.bf16_to_f64(kc[b, :, p])) <= REL_L2
                assert rel_l2(oracle.bf16_to_f64(vd[b, :, p]), oracle.bf16_to_f64(vc[b, :, p])) <= REL_L2
            for t0, t1 in ((kd, kv0[l][0]), (vd, kv0[l][1])):
                np.testing.assert_array_equal(t0[b, :, :p], t1[b, :, :p])
                np.testing.assert_array_equal(t0[b, :, p + 1:], t1[b, :, p + 1:])
    e_out = rel_l2(oracle.bf16_to_f64(out), x)
    e_res = float(np.max(np.abs(res - x)))
    assert e_out <= REL_L2, f"bf16 output rel-L2 {e_out:.3e}"
    assert e_res <= MAX_ABS, f"fp32 residual max-abs {e_res:.3e}"
    for name in ("q", "attn", "y", "a"):
        e = rel_l2(dst[name], ost[name])
        assert e <= REL_L2, f"stage {name} rel-L2 {e:.3e}"
    return out, res


@pytest.mark.parametrize("mode", [0, 1])
def test_narrow_batch_two_layers(mode):
    pos = [0, 17, 100]
    st, kv0 = _stack(SMALL, 3, pos, layers=2)
    _check(st, kv0, pos, mode)


@pytest.mark.parametrize("pos", [[37], [15, 16, 31, 32]])
def test_narrow_tile_edges(pos):
    st, kv0 = _stack(SMALL, len(pos), pos)
    _check(st, kv0, pos)


def test_wide_batch():
    pos = [5, 90, 0, 64, 127, 33, 16, 100]
    st, kv0 = _stack(SMALL, 8, pos)
    _check(st, kv0, pos, kv_ulp=False)  # the wide-batch kernel carries 11-bit activations: K/V at the stage bar


@pytest.mark.parametrize("wtype,B", [(ddl.INT4, 16), (ddl.BF16, 5)])
def test_tensor_core_path(wtype, B):
    pos = [(37 * b) % 130 for b in range(B)]
    st, kv0 = _stack(SMALL, B, pos, wtype=wtype)
    _check(st, kv0, pos)


def test_equal_positions_match_the_shared_position_call():
    """The ragged call with every sequence at one position agrees with the
    plain call (same kernels; the RoPE table comes from the device)."""
    pos = [64, 64, 64]
    st, kv0 = _stack(SMALL, 3, pos)
    out_r, res_r = _check(st, kv0, pos)
    for l, (k, v) in enumerate(st.kvs):  # restore the caches
        k.copy_(torch.from_numpy(kv0[l][0].view(np.int16)).view(torch.bfloat16))
        v.copy_(torch.from_numpy(kv0[l][1].view(np.int16)).view(torch.bfloat16))
    out = torch.empty((3, SMALL.D), dtype=torch.bfloat16, device="cuda")
    res = torch.empty((3, SMALL.D), dtype=torch.float32, device="cuda")
    ddl.ddl_stack_decode(st.shape, st.wtype, st.layers, st.kvs, 64, x_bf16=st.x, resid_out=res, out_bf16=out,
                         workspace=st.workspace)
    torch.cuda.synchronize()
    assert rel_l2(res.cpu().numpy().astype(np.float64), res_r) <= 1e-6


def test_qwen7b_layer_and_27b_layer_with_long_history():
    for cfg, pos in ((configs.QWEN7B_LAYER, [4095, 1000]), (configs.STACK27B.with_(layers=1), [8192, 10, 4000, 0])):
        st, kv0 = _stack(cfg, len(pos), pos, spare=16)
        _check(st, kv0, pos)
        del st
        torch.cuda.empty_cache()


def test_positions_out_of_range_are_refused():
    pos = [3, 4]
    st, _ = _stack(SMALL, 2, pos)
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_stack_decode_ragged(st.shape, st.wtype, st.layers, st.kvs, [3, st.s_max], x_bf16=st.x,
                                    workspace=st.workspace)
    assert e.value.status == 2
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_stack_decode_ragged(st.shape, st.wtype, st.layers, st.kvs, [-1, 2], x_bf16=st.x,
                                    workspace=st.workspace)
    assert e.value.status == 2
