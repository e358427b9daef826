"""The C-ABI boundary as a caller uses it, against the fp64 oracle.

* KV caches sized for a longer context than the step needs (s_max well above
  pos + 1, the normal production layout): the fused append writes slot pos of
  the [B][H_kv][s_max][hd] layout and nothing else; the slots before pos keep
  their history bit for bit and the slots after pos keep a planted pattern
  bit for bit (attention must never read them: the pattern is a large finite
  value that would swamp the softmax), in both launch modes.
* ddl_layer_decode, the one-layer entry point, on the small D=512 layer and on
  the Qwen2.5-7B-shaped layer, with the bf16 input x and with an fp32
  residual input.
* One 27B-class layer whose caches hold 16384 slots for an 8192-token history.

Tolerances are those of the decode step (tests/gpu_helpers.py).
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_transformer_decode_gb300 import configs, ddl, synth, workload
from tests.gpu_helpers import MAX_ABS, REL_L2, bf16_bits_close, host_layer, rel_l2

pytestmark = pytest.mark.gpu

POISON = 0x4800  # bf16 131072.0: any read of a slot after pos would dominate its softmax


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddl.load(build_if_missing=True)
    yield
    ddl.ddl_set_launch_mode(0)
    torch.cuda.empty_cache()


def _poison_after(st, first: int):
    for kc, vc in st.kvs:
        kc.view(torch.int16)[:, :, first:] = POISON
        vc.view(torch.int16)[:, :, first:] = POISON
    torch.cuda.synchronize()


def _run(st, mode: int):
    ddl.ddl_set_launch_mode(mode)
    try:
        B, D = st.batch, st.cfg.D
        out = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
        res = torch.empty((B, D), dtype=torch.float32, device="cuda")
        st.decode(out_bf16=out, resid_out=res)
        torch.cuda.synchronize()
        assert ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max) == 0
        return synth.bits(out), res.cpu().numpy().astype(np.float64)
    finally:
        ddl.ddl_set_launch_mode(0)


SPARE = [
    # (batch, H_q, H_kv, head_dim, history length)
    (1, 8, 1, 128, 45),
    (3, 8, 2, 64, 45),
    (3, 16, 8, 128, 31),
    (16, 8, 2, 128, 45),
    (16, 8, 8, 64, 17),
]


@pytest.mark.parametrize("mode", [0, 1])
@pytest.mark.parametrize("B,H_q,H_kv,hd,S", SPARE)
def test_cache_with_spare_slots(B, H_q, H_kv, hd, S, mode):
    cfg = configs.DecodeConfig("spare", D=256, H_q=H_q, H_kv=H_kv, head_dim=hd, d_ff=320,
                               rope_base=1e4, kv_len=S, layers=2, seed=31 + B + H_kv)
    s_max = S + 37
    st = workload.build_stack(cfg, batch=B, s_max=s_max)
    p = st.pos
    _poison_after(st, p)  # slot p too: the step must overwrite it
    before = [(synth.bits(k).copy(), synth.bits(v).copy()) for k, v in st.kvs]
    out, res = _run(st, mode)
    # the oracle on the same caches (it reads slots 0..p and writes slot p)
    x = oracle.bf16_to_f64(synth.bits(st.x))
    for l in range(cfg.layers):
        kc, vc = before[l][0].copy(), before[l][1].copy()
        x = oracle.layer_decode(cfg, host_layer(cfg, l, st.wtype), kc, vc, p, x)
        kd, vd = synth.bits(st.kvs[l][0]), synth.bits(st.kvs[l][1])
        for name, dev, pre, orc in (("K", kd, before[l][0], kc), ("V", vd, before[l][1], vc)):
            np.testing.assert_array_equal(dev[:, :, :p], pre[:, :, :p], err_msg=f"{name} history, layer {l}")
            np.testing.assert_array_equal(dev[:, :, p + 1:], pre[:, :, p + 1:],
                                          err_msg=f"{name} slots after pos, layer {l}")
            assert np.all(pre[:, :, p + 1:] == POISON)
            if B <= 4:  # x carried to ~22 bits: one bf16 ulp
                assert bf16_bits_close(dev[:, :, p], orc[:, :, p]), f"appended {name}, layer {l}"
            else:  # wide batches carry x in fp16: the stage tolerance
                e = rel_l2(oracle.bf16_to_f64(dev[:, :, p]), oracle.bf16_to_f64(orc[:, :, p]))
                assert e <= REL_L2, f"appended {name} rel-L2 {e:.3e}, layer {l}"
    e_out = rel_l2(oracle.bf16_to_f64(out), x)
    e_res = float(np.max(np.abs(res - x)))
    assert e_out <= REL_L2, f"bf16 output rel-L2 {e_out:.3e}"
    assert e_res <= MAX_ABS, f"fp32 residual max-abs {e_res:.3e}"


@pytest.mark.parametrize("cfg", [configs.SMALL_LAYER, configs.QWEN7B_LAYER])
@pytest.mark.parametrize("use_resid", [False, True])
def test_layer_decode_entry_point(cfg, use_resid):
    """ddl_layer_decode through the C ABI: one layer, bf16 x or fp32 residual in."""
    st = workload.build_stack(cfg, s_max=cfg.kv_len + 9)
    B, D = st.batch, cfg.D
    kc0, vc0 = (synth.bits(t).copy() for t in st.kvs[0])
    if use_resid:
        resid = synth.normal_bf16((B, D), seed=77, std=3.0, device="cuda").float()
        resid.add_(synth.normal_bf16((B, D), seed=78, std=1e-3, device="cuda").float())
        x64 = resid.cpu().numpy().astype(np.float64)
    else:
        resid = None
        x64 = oracle.bf16_to_f64(synth.bits(st.x))
    out = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
    res = torch.empty((B, D), dtype=torch.float32, device="cuda")
    ddl.ddl_layer_decode(st.shape, st.wtype, st.layers[0], st.kvs[0], st.pos,
                         x_bf16=None if use_resid else st.x, resid_in=resid, resid_out=res,
                         out_bf16=out, workspace=st.workspace)
    torch.cuda.synchronize()
    assert ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max) == 0
    kc, vc = kc0.copy(), vc0.copy()
    z = oracle.layer_decode(cfg, host_layer(cfg, 0, st.wtype), kc, vc, st.pos, x64)
    e_out = rel_l2(oracle.bf16_to_f64(synth.bits(out)), z)
    e_res = float(np.max(np.abs(res.cpu().numpy().astype(np.float64) - z)))
    assert e_out <= REL_L2, f"bf16 output rel-L2 {e_out:.3e}"
    assert e_res <= MAX_ABS, f"fp32 residual max-abs {e_res:.3e}"
    kd, vd = (synth.bits(t) for t in st.kvs[0])
    p = st.pos
    np.testing.assert_array_equal(kd[:, :, :p], kc0[:, :, :p])
    np.testing.assert_array_equal(kd[:, :, p + 1:], kc0[:, :, p + 1:])
    np.testing.assert_array_equal(vd[:, :, p + 1:], vc0[:, :, p + 1:])
    assert bf16_bits_close(kd[:, :, p], kc[:, :, p])
    assert bf16_bits_close(vd[:, :, p], vc[:, :, p])


def test_27b_layer_with_16384_slot_cache():
    cfg = configs.STACK27B.with_(layers=1)
    st = workload.build_stack(cfg, s_max=16384)
    p = st.pos
    _poison_after(st, p + 1)
    kc0, vc0 = (synth.bits(t).copy() for t in st.kvs[0])
    out, res = _run(st, 0)
    kc, vc = kc0.copy(), vc0.copy()
    z = oracle.layer_decode(cfg, host_layer(cfg, 0, st.wtype), kc, vc, p,
                            oracle.bf16_to_f64(synth.bits(st.x)))
    assert rel_l2(oracle.bf16_to_f64(out), z) <= REL_L2
    assert float(np.max(np.abs(res - z))) <= MAX_ABS
    kd, vd = (synth.bits(t) for t in st.kvs[0])
    np.testing.assert_array_equal(kd[:, :, p + 1:], kc0[:, :, p + 1:])
    np.testing.assert_array_equal(vd[:, :, p + 1:], vc0[:, :, p + 1:])
    assert bf16_bits_close(kd[:, :, p], kc[:, :, p])
    assert bf16_bits_close(vd[:, :, p], vc[:, :, p])
