"""ddl_stack_decode_noalloc against ddl_stack_decode.

The allocation-free entry point serves callers that cannot allocate device
memory (a plugin that is handed only its inputs and outputs, or a loop that
must not pay cudaMalloc's implicit device synchronization); it takes its
scratch from the library's static device array.  The decode path is
deterministic (partial sums are added in a fixed order), so two calls in a
row must give the workspace entry point's outputs bit for bit (the second
call runs on whatever the first left in the shared array), and the status
word of each call, read back from the static array, must be DDL_OK.  A
problem larger than the array must be rejected before anything is launched.
This file is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from memory_bound_transformer_decode_gb300 import configs, ddl, synth, workload

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice():
    ddl.load(build_if_missing=True)
    cfg = configs.DecodeConfig("noalloc-3L", D=256, H_q=8, H_kv=2, head_dim=128, d_ff=320,
                               rope_base=1e4, kv_len=37, layers=3, seed=21)
    st = workload.build_stack(cfg, batch=2)
    B, D = st.batch, cfg.D
    out_ref = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
    res_ref = torch.empty((B, D), dtype=torch.float32, device="cuda")
    st.decode(out_bf16=out_ref, resid_out=res_ref)
    torch.cuda.synchronize()
    assert ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max) == 0
    ref_o = synth.bits(out_ref)
    ref_r = res_ref.cpu().numpy()
    for _ in range(2):
        out = torch.full((B, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        res = torch.full((B, D), float("nan"), dtype=torch.float32, device="cuda")
        ddl.ddl_stack_decode_noalloc(st.shape, st.wtype, st.layers, st.kvs, st.pos, x_bf16=st.x,
                                     resid_out=res, out_bf16=out)
        torch.cuda.synchronize()
        assert ddl.ddl_read_device_status(None, st.shape, B, st.s_max) == 0
        np.testing.assert_array_equal(synth.bits(out), ref_o)
        np.testing.assert_array_equal(res.cpu().numpy(), ref_r)


def test_noalloc_rejects_problems_larger_than_its_scratch():
    lib = ddl.load(build_if_missing=True)
    # the first supported shape that needs more scratch than the static array
    cands = [ddl.Shape(32768, 64, 8, 128, 65536, 1e-6, 5e5), ddl.Shape(16384, 64, 64, 128, 65536, 1e-6, 5e5),
             ddl.Shape(32768, 128, 16, 128, 65536, 1e-6, 5e5)]
    big = next((c for c in cands if lib.ddl_workspace_bytes(ctypes.byref(c), 4, 1024) > (32 << 20)), None)
    assert big is not None
    # NULL device pointers: should the size check ever come after the
    # argument checks, the call still returns an error without a launch
    lw = (ddl.LayerW * 1)(ddl.LayerW(None, None, None))
    kv = (ddl.KV * 1)(ddl.KV(None, None, 1024))
    st = lib.ddl_stack_decode_noalloc(ctypes.byref(big), ddl.INT4, lw, kv, 1, 4, 0, None,
                                      None, None, None, None)
    assert st == 4  # DDL_ERR_WORKSPACE, before any launch
