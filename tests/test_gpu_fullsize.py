"""Parity at the full sizes of the stack workloads, through the C ABI, in the
launch configuration the benchmark times (one persistent launch of the whole
stack per step).

* 27B-class stack, 64 layers, INT4, batch 1, KV 8192: teacher-forced checks
  of layers {0, 1, 32, 63} plus four seeded others (the device's own fp32
  input to the layer, from a device step over the layers before it, goes
  through the device layer and the oracle's), and the device step against the
  oracle run untethered over all 64 layers (each layer takes the oracle's own
  residual; rel-L2 of the output held to the step's bar, the residual's drift
  reported).
* the same stack with a 4096-token cache per sequence, INT4 at batches 4, 16
  and 64 and bf16 weights at batches 1, 16 and 64: the full step,
  teacher-forced layers {0, 63} plus two seeded others, and 120 repeats each
  of the full step and of layer 16 alone, bit-identical to the first run.
* Llama-3-70B-shaped stack, 80 layers, KV 32768: the device step against the
  oracle run untethered over all 80 layers, and teacher-forced layers
  {0, 1, 40, 79} plus two seeded others.

Tolerances are those of the decode step (gpu_helpers): rel-L2 of the bf16
output vs the oracle's fp64 z <= 2e-3 and max-abs of the fp32 residual <= 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_transformer_decode_gb300 import configs, ddl, synth, workload
from tests.gpu_helpers import MAX_ABS, REL_L2, host_layer, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddl.load(build_if_missing=True)
    ddl.ddl_set_launch_mode(0)
    yield
    torch.cuda.empty_cache()


def _device_run(st, lo: int, hi: int, resid_in=None):
    """Device step over layers [lo, hi); layer 0 takes the bf16 input x."""
    B, D = st.batch, st.cfg.D
    out = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
    res = torch.empty((B, D), dtype=torch.float32, device="cuda")
    ddl.ddl_stack_decode(st.shape, st.wtype, st.layers[lo:hi], st.kvs[lo:hi], st.pos,
                         x_bf16=st.x if resid_in is None else None, resid_in=resid_in,
                         resid_out=res, out_bf16=out, workspace=st.workspace)
    torch.cuda.synchronize()
    status = ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max)
    assert status == 0, f"device status {status}"
    return out, res


def _host_cache(st, layer: int):
    k, v = st.kvs[layer]
    return synth.bits(k).copy(), synth.bits(v).copy()


def _sampled(L: int, fixed, extra: int, seed: int):
    rng = np.random.default_rng(seed)
    rest = [l for l in range(L) if l not in fixed]
    return sorted(set(fixed) | set(int(x) for x in rng.choice(rest, size=extra, replace=False)))


def _teacher_forced(st, layer: int, lw: dict):
    """Device layer `layer` on the device's own input vs the oracle on it."""
    if layer == 0:
        x_in = None
        x64 = oracle.bf16_to_f64(synth.bits(st.x))
    else:
        _, x_in = _device_run(st, 0, layer)
        x64 = x_in.cpu().numpy().astype(np.float64)
    out, res = _device_run(st, layer, layer + 1, resid_in=x_in)
    kc, vc = _host_cache(st, layer)
    z = oracle.layer_decode(st.cfg, lw, kc, vc, st.pos, x64)
    e_out = rel_l2(oracle.bf16_to_f64(synth.bits(out)), z)
    e_res = float(np.max(np.abs(res.cpu().numpy().astype(np.float64) - z)))
    return e_out, e_res


def _repeats_differing(st, reps: int, mid: int = 16):
    """Steps repeated on the same inputs (each rewrites the same K/V slots with
    the same values): the full step, and layer `mid` alone on the device's own
    input after a step over the layers before it.  Partial sums are added in a
    fixed order, so every repeat must give the first one's bits; returns the
    repeats that did not."""
    L = st.cfg.layers
    _, ref = _device_run(st, 0, L)
    _, x_mid = _device_run(st, 0, mid)
    _, ref1 = _device_run(st, mid, mid + 1, resid_in=x_mid)
    bad = []
    for r in range(reps):
        _, res = _device_run(st, 0, L)
        if not torch.equal(res.view(torch.int32), ref.view(torch.int32)):
            bad.append(("full", r))
        _device_run(st, 0, mid)
        _, res1 = _device_run(st, mid, mid + 1, resid_in=x_mid)
        if not torch.equal(res1.view(torch.int32), ref1.view(torch.int32)):
            bad.append((f"layer {mid}", r))
    return bad


def _check(errs: dict):
    print({k: (f"{a:.2e}", f"{b:.2e}") for k, (a, b) in errs.items()})
    for k, (e_out, e_res) in errs.items():
        assert e_out <= REL_L2, f"{k}: rel-L2 {e_out:.3e}"
        assert e_res <= MAX_ABS, f"{k}: max-abs {e_res:.3e}"


def test_27b_stack_64_layers_full_and_teacher_forced():
    cfg = configs.STACK27B
    st = workload.build_stack(cfg)
    out, res = _device_run(st, 0, cfg.layers)
    out = oracle.bf16_to_f64(synth.bits(out))
    res = res.cpu().numpy().astype(np.float64)
    sampled = _sampled(cfg.layers, (0, 1, cfg.layers // 2, cfg.layers - 1), 4, seed=11)
    errs = {}
    x = oracle.bf16_to_f64(synth.bits(st.x))
    for l in range(cfg.layers):
        lw = host_layer(cfg, l, st.wtype)
        kc, vc = _host_cache(st, l)
        x = oracle.layer_decode(cfg, lw, kc, vc, st.pos, x)  # untethered
        if l in sampled:
            errs[f"layer {l}"] = _teacher_forced(st, l, lw)
        del lw
    del st
    torch.cuda.empty_cache()
    _check(errs)
    # Untethered over 64 layers the two residual streams drift apart (each
    # layer feeds the next its own fp32 rounding): the bf16 output is held to
    # the step's rel-L2 bar; the fp32 residual's max-abs error is reported and
    # held only to 1e-3 of the largest |z| (the per-layer 2e-2 bar is for a
    # layer fed the device's own input, checked above).
    e_out, e_res = rel_l2(out, x), float(np.max(np.abs(res - x)))
    print(f"untethered 64-layer stack: rel-L2 {e_out:.3e}, max-abs {e_res:.3e} (max |z| {np.max(np.abs(x)):.1f})")
    assert e_out <= REL_L2
    assert e_res <= 1e-3 * float(np.max(np.abs(x)))


@pytest.mark.parametrize("wtype,B", [(ddl.INT4, 4), (ddl.INT4, 16), (ddl.INT4, 64), (ddl.BF16, 1),
                                     (ddl.BF16, 16), (ddl.BF16, 64)])
def test_27b_stack_batch_teacher_forced(wtype, B):
    """The 64-layer batch/weight sweep shape (4096-token caches): batches on the
    warp-level path (4 INT4, 1 bf16) and on the tcgen05 path (16 and 64, INT4
    and bf16 weights), the full step's status and teacher-forced layers."""
    cfg = configs.STACK27B_SWEEP
    st = workload.build_stack(cfg, batch=B, wtype=wtype)
    _device_run(st, 0, cfg.layers)  # the full step runs clean (status checked)
    errs = {}
    for l in _sampled(cfg.layers, (0, cfg.layers - 1), 2, seed=12):
        errs[f"layer {l}"] = _teacher_forced(st, l, host_layer(cfg, l, st.wtype))
    # (a tensor-core GEMM whose ring stage could be refilled before one of
    # its readers had waited for it gave one such repeat in about 60 a wrong
    # 128-row tile at 64 sequences with bf16 weights)
    bad = _repeats_differing(st, 120)
    del st
    torch.cuda.empty_cache()
    _check(errs)
    assert not bad, f"repeats differing from the first run: {bad[:8]} ({len(bad)} of 240)"


def test_70b_stack_80_layers_full_and_teacher_forced():
    """The full 80-layer step against the oracle run untethered over all 80
    layers (output rel-L2 at the step's bar, the fp32 residual within 1e-3 of
    the largest |z|, as for the 64-layer stack), and teacher-forced layers."""
    cfg = configs.LLAMA70B_STACK
    st = workload.build_stack(cfg)
    out, res = _device_run(st, 0, cfg.layers)
    out = oracle.bf16_to_f64(synth.bits(out))
    res = res.cpu().numpy().astype(np.float64)
    sampled = _sampled(cfg.layers, (0, 1, cfg.layers // 2, cfg.layers - 1), 2, seed=13)
    errs = {}
    x = oracle.bf16_to_f64(synth.bits(st.x))
    for l in range(cfg.layers):
        lw = host_layer(cfg, l, st.wtype)
        kc, vc = _host_cache(st, l)
        x = oracle.layer_decode(cfg, lw, kc, vc, st.pos, x)  # untethered
        if l in sampled:
            errs[f"layer {l}"] = _teacher_forced(st, l, lw)
        del lw
    del st
    torch.cuda.empty_cache()
    _check(errs)
    e_out, e_res = rel_l2(out, x), float(np.max(np.abs(res - x)))
    print(f"untethered 80-layer stack: rel-L2 {e_out:.3e}, max-abs {e_res:.3e} (max |z| {np.max(np.abs(x)):.1f})")
    assert e_out <= REL_L2
    assert e_res <= 1e-3 * float(np.max(np.abs(x)))
