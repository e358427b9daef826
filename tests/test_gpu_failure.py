"""Failure detection without a GPU fault: a bounded device wait that gives up.

The test hook ddl_test_hold_barrier makes one grid barrier of a cooperative
decode call wait for one arrival more than the grid makes (a count that
nothing reaches).  With the wait limit lowered to a few milliseconds, every
CTA's bounded wait gives up, the kernel records DDL_ERR_TIMEOUT in the device
status word, waits for its copies in flight and returns; nothing faults or
traps.  The call must end within a bounded time, report the timeout through
ddl_read_device_status, and leave the context usable: the next normal call on
the same workspace agrees with the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from memory_bound_transformer_decode_gb300 import configs, ddl, synth, workload
from tests.gpu_helpers import MAX_ABS, REL_L2, oracle_stack, rel_l2

pytestmark = pytest.mark.gpu

CFG = configs.DecodeConfig("timeout-3L", D=256, H_q=8, H_kv=2, head_dim=128, d_ff=320, rope_base=1e4,
                           kv_len=45, layers=3, seed=41)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddl.load(build_if_missing=True)
    ddl.ddl_set_launch_mode(0)
    yield
    ddl.ddl_test_hold_barrier(-1)
    ddl.ddl_set_wait_limit_ns(0)


@pytest.mark.parametrize("held", [3, 7, 14])  # in front of layer 0's Wo, layer 1's attention, layer 2's down
def test_held_barrier_times_out_and_the_context_recovers(held):
    st = workload.build_stack(CFG, batch=1)
    kv0 = [(synth.bits(k).copy(), synth.bits(v).copy()) for k, v in st.kvs]
    out = torch.empty((1, CFG.D), dtype=torch.bfloat16, device="cuda")
    res = torch.empty((1, CFG.D), dtype=torch.float32, device="cuda")
    ddl.ddl_set_wait_limit_ns(2_000_000)  # 2 ms
    ddl.ddl_test_hold_barrier(held)
    try:
        t0 = time.perf_counter()
        st.decode(out_bf16=out, resid_out=res)
        status = ddl.ddl_read_device_status(st.workspace, st.shape, 1, st.s_max)
        dt = time.perf_counter() - t0
    finally:
        ddl.ddl_test_hold_barrier(-1)
        ddl.ddl_set_wait_limit_ns(0)
    assert status == 7, f"status {status}"  # DDL_ERR_TIMEOUT
    assert dt < 5.0, f"the timed-out call took {dt:.2f} s"
    # the same workspace, a normal call: the step agrees with the oracle
    st.decode(out_bf16=out, resid_out=res)
    assert ddl.ddl_read_device_status(st.workspace, st.shape, 1, st.s_max) == 0
    z, _, _, _ = oracle_stack(st, kv0)
    assert rel_l2(oracle.bf16_to_f64(synth.bits(out)), z) <= REL_L2
    assert float(np.max(np.abs(res.cpu().numpy().astype(np.float64) - z))) <= MAX_ABS


def test_hold_hook_off_by_default_and_stage_zero_has_no_barrier():
    st = workload.build_stack(CFG, batch=1)
    ddl.ddl_set_wait_limit_ns(2_000_000)
    ddl.ddl_test_hold_barrier(0)  # nothing waits in front of the first stage
    try:
        st.decode()
        status = ddl.ddl_read_device_status(st.workspace, st.shape, 1, st.s_max)
    finally:
        ddl.ddl_test_hold_barrier(-1)
        ddl.ddl_set_wait_limit_ns(0)
    assert status == 0
