"""Paged KV caches (ddl_stack_decode_paged, ddl_stack_prefill_paged) on the GPU
vs the fp64 oracle's paged step, through the C ABI: the bf16 output and fp32
residual at the step's bars, the last layer's stages, each new K/V row in the
page and row its page table names, and every other byte of every pool
bit-unchanged (pages nobody owns and slots past each position hold junk).
The same step on the same data laid out contiguously (ddl_stack_decode_ragged)
gives bit-identical results: paging moves where a tile comes from, not the
arithmetic.  Covers the batch <= 4 kernel (both launch modes), the wide-batch
kernel, the tcgen05 path, page sizes 16 to 256, shared read-only prefix pages,
a 27B-class layer with an 8192-token history, and prefill into pages.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_transformer_decode_gb300 import configs, ddl, synth, workload
from tests.gpu_helpers import MAX_ABS, REL_L2, bf16_bits_close, host_layer, rel_l2

pytestmark = pytest.mark.gpu

SMALL = configs.SMALL_LAYER
JUNK_K, JUNK_V = 0.75, -0.5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddl.load(build_if_missing=True)
    yield
    ddl.ddl_set_launch_mode(0)
    torch.cuda.empty_cache()


def _paged_stack(cfg, B, pos, ps, layers=1, wtype=ddl.INT4, extra=5, seed=0, share=0):
    """A stack whose caches are cut into pages of ps slots and scattered over a
    pool with `extra` unowned junk pages; slots past each position hold junk.
    share: sequence 1 reads sequence 0's first `share` pages instead of its own."""
    S = max(pos)
    s_max = -(-(S + 1 + 7) // ps) * ps
    st = workload.build_stack(cfg.with_(kv_len=S, layers=layers), batch=B, wtype=wtype, s_max=s_max)
    npg = s_max // ps
    rng = np.random.default_rng(seed)
    n_phys = B * npg + extra
    perm = rng.permutation(n_phys)[: B * npg]
    table = perm.reshape(B, npg).astype(np.int32)
    if share:
        table[1, :share] = table[0, :share]
    pools = []
    for k, v in st.kvs:
        for b, p in enumerate(pos):
            k[b, :, p:] = JUNK_K
            v[b, :, p:] = JUNK_V
        H, hd = k.shape[1], k.shape[3]
        kp = torch.full((n_phys, H, ps, hd), -JUNK_K, dtype=torch.bfloat16, device="cuda")
        vp = torch.full((n_phys, H, ps, hd), -JUNK_V, dtype=torch.bfloat16, device="cuda")
        idx = torch.from_numpy(perm).cuda()
        kp[idx] = k.reshape(B, H, npg, ps, hd).permute(0, 2, 1, 3, 4).reshape(-1, H, ps, hd)
        vp[idx] = v.reshape(B, H, npg, ps, hd).permute(0, 2, 1, 3, 4).reshape(-1, H, ps, hd)
        if share:  # the contiguous copy sees what the shared pages hold
            k[1, :, : share * ps] = k[0, :, : share * ps]
            v[1, :, : share * ps] = v[0, :, : share * ps]
        pools.append((kp, vp))
    torch.cuda.synchronize()
    return st, pools, table


def _run_paged(st, pools, table, pos, ps, mode=0):
    B, D = st.batch, st.cfg.D
    out = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
    res = torch.empty((B, D), dtype=torch.float32, device="cuda")
    ddl.ddl_set_launch_mode(mode)
    try:
        ddl.ddl_stack_decode_paged(st.shape, st.wtype, st.layers, pools, pos, table, ps, x_bf16=st.x,
                                   resid_out=res, out_bf16=out, workspace=st.workspace)
        torch.cuda.synchronize()
    finally:
        ddl.ddl_set_launch_mode(0)
    assert ddl.ddl_read_device_status(st.workspace, st.shape, B, st.s_max) == 0
    v = ddl.ddl_workspace_view(st.shape, B, st.s_max)
    cfg = st.cfg
    stages = {n: ddl.ws_tensor(st.workspace, off, B * k).view(B, -1).cpu().numpy().copy()
              for n, off, k in (("q", v.q, cfg.Nq), ("attn", v.attn, cfg.Nq), ("y", v.y, cfg.D),
                                ("a", v.a, cfg.d_ff))}
    return synth.bits(out), res.cpu().numpy().astype(np.float64), stages


def _check(st, pools, table, pos, ps, mode=0, kv_ulp=True, against_ragged=True):
    before = [(synth.bits(k).copy(), synth.bits(v).copy()) for k, v in pools]
    out, res, dst = _run_paged(st, pools, table, pos, ps, mode)
    cfg, L = st.cfg, len(st.layers)
    x = oracle.bf16_to_f64(synth.bits(st.x))
    for l in range(L):
        kp, vp = before[l][0].copy(), before[l][1].copy()
        r = oracle.layer_decode_paged(cfg, host_layer(cfg, l, st.wtype), kp, vp, table, ps, pos, x,
                                      stages=l == L - 1)
        x, ost = r if l == L - 1 else (r, None)
        kd, vd = synth.bits(pools[l][0]), synth.bits(pools[l][1])
        written = {(int(table[b][p // ps]), p % ps) for b, p in enumerate(pos)}
        for dev, ref, old in ((kd, kp, before[l][0]), (vd, vp, before[l][1])):
            for pg, row in written:
                if kv_ulp:
                    assert bf16_bits_close(dev[pg, :, row], ref[pg, :, row]), f"layer {l}, page {pg} row {row}"
                else:
                    assert rel_l2(oracle.bf16_to_f64(dev[pg, :, row]), oracle.bf16_to_f64(ref[pg, :, row])) <= REL_L2
            mask = np.ones(dev.shape[:1] + dev.shape[2:3], bool)  # [page, row]
            for pg, row in written:
                mask[pg, row] = False
            np.testing.assert_array_equal(dev.transpose(0, 2, 1, 3)[mask], old.transpose(0, 2, 1, 3)[mask])
    assert rel_l2(oracle.bf16_to_f64(out), x) <= REL_L2
    assert float(np.max(np.abs(res - x))) <= MAX_ABS
    for name in ("q", "attn", "y", "a"):
        e = rel_l2(dst[name], ost[name])
        assert e <= REL_L2, f"stage {name} rel-L2 {e:.3e}"
    if against_ragged:  # the contiguous layout of the same data: the same bits
        B, D = st.batch, cfg.D
        out2 = torch.empty((B, D), dtype=torch.bfloat16, device="cuda")
        res2 = torch.empty((B, D), dtype=torch.float32, device="cuda")
        ddl.ddl_set_launch_mode(mode)
        try:
            ddl.ddl_stack_decode_ragged(st.shape, st.wtype, st.layers, st.kvs, pos, x_bf16=st.x, resid_out=res2,
                                        out_bf16=out2, workspace=st.workspace)
            torch.cuda.synchronize()
        finally:
            ddl.ddl_set_launch_mode(0)
        np.testing.assert_array_equal(synth.bits(out2), out)
        np.testing.assert_array_equal(res2.cpu().numpy().astype(np.float64), res)


@pytest.mark.parametrize("ps,mode", [(16, 0), (64, 0), (16, 1)])
def test_narrow_batch_two_layers(ps, mode):
    pos = [0, 17, 100]
    st, pools, table = _paged_stack(SMALL, 3, pos, ps, layers=2)
    _check(st, pools, table, pos, ps, mode)


def test_shared_prefix_pages():
    pos, ps = [40, 50], 16
    st, pools, table = _paged_stack(SMALL, 2, pos, ps, share=2)
    _check(st, pools, table, pos, ps)


def test_wide_batch():
    pos = [5, 90, 0, 64, 127, 33, 16, 100]
    st, pools, table = _paged_stack(SMALL, 8, pos, 32)
    _check(st, pools, table, pos, 32, kv_ulp=False)  # the wide-batch kernel: K/V at the stage bar


@pytest.mark.parametrize("wtype,B,ps", [(ddl.INT4, 16, 16), (ddl.BF16, 5, 64)])
def test_tensor_core_path(wtype, B, ps):
    pos = [(37 * b) % 130 for b in range(B)]
    st, pools, table = _paged_stack(SMALL, B, pos, ps, wtype=wtype)
    _check(st, pools, table, pos, ps)


def test_27b_layer_with_long_history():
    pos, ps = [8192, 10, 4000, 0], 256
    st, pools, table = _paged_stack(configs.STACK27B.with_(layers=1), 4, pos, ps)
    _check(st, pools, table, pos, ps)


def test_prefill_into_pages():
    """S prompt rows of one sequence through its page-table row vs the oracle's
    prefill on the gathered slots, and the rows written to their pages."""
    cfg, ps, p0, S = SMALL, 32, 45, 16
    st = workload.build_stack(cfg.with_(kv_len=p0, layers=2), batch=1, s_max=4 * ps)
    rng = np.random.default_rng(3)
    row = rng.permutation(9)[:4].astype(np.int32)
    pools = []
    for k, v in st.kvs:
        H, hd = k.shape[1], k.shape[3]
        kp = torch.full((9, H, ps, hd), JUNK_K, dtype=torch.bfloat16, device="cuda")
        vp = torch.full((9, H, ps, hd), JUNK_V, dtype=torch.bfloat16, device="cuda")
        idx = torch.from_numpy(row).cuda()
        kp[idx] = k.reshape(1, H, 4, ps, hd).permute(0, 2, 1, 3, 4).reshape(-1, H, ps, hd)
        vp[idx] = v.reshape(1, H, 4, ps, hd).permute(0, 2, 1, 3, 4).reshape(-1, H, ps, hd)
        pools.append((kp, vp))
    torch.cuda.synchronize()
    before = [(synth.bits(k).copy(), synth.bits(v).copy()) for k, v in pools]
    x = synth.normal_bf16((S, cfg.D), seed=11, device="cuda")
    ws = torch.zeros(ddl.ddl_workspace_bytes(st.shape, S, st.s_max), dtype=torch.uint8, device="cuda")
    out = torch.empty((S, cfg.D), dtype=torch.bfloat16, device="cuda")
    res = torch.empty((S, cfg.D), dtype=torch.float32, device="cuda")
    ddl.ddl_stack_prefill_paged(st.shape, st.wtype, st.layers, pools, p0, row, ps, x_bf16=x, resid_out=res,
                                out_bf16=out, workspace=ws)
    torch.cuda.synchronize()
    assert ddl.ddl_read_device_status(ws, st.shape, S, st.s_max) == 0
    z = oracle.bf16_to_f64(synth.bits(x))
    table = row.reshape(1, -1)
    for l in range(2):
        kc = oracle.paged_gather(before[l][0], table, ps, 0, 4 * ps)
        vc = oracle.paged_gather(before[l][1], table, ps, 0, 4 * ps)
        z = oracle.layer_prefill(cfg, host_layer(cfg, l, st.wtype), kc, vc, p0, z)
        kd, vd = synth.bits(pools[l][0]), synth.bits(pools[l][1])
        for t in range(4 * ps):
            pg, r = int(row[t // ps]), t % ps
            for dev, ref, old in ((kd, kc, before[l][0]), (vd, vc, before[l][1])):
                if p0 <= t < p0 + S:
                    assert bf16_bits_close(dev[pg, :, r], ref[0, :, t]), f"layer {l}, slot {t}"
                else:
                    np.testing.assert_array_equal(dev[pg, :, r], old[pg, :, r])
        for dev, old in ((kd, before[l][0]), (vd, before[l][1])):
            others = np.setdiff1d(np.arange(9), row)
            np.testing.assert_array_equal(dev[others], old[others])
    assert rel_l2(oracle.bf16_to_f64(synth.bits(out)), z) <= REL_L2
    assert float(np.max(np.abs(res.cpu().numpy().astype(np.float64) - z))) <= MAX_ABS


def test_bad_page_tables_are_refused():
    pos, ps = [3, 20], 16
    st, pools, table = _paged_stack(SMALL, 2, pos, ps)
    bad = table.copy()
    bad[1, 1] = len(pools[0][0])  # past the pool
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_stack_decode_paged(st.shape, st.wtype, st.layers, pools, pos, bad, ps, x_bf16=st.x,
                                   workspace=st.workspace)
    assert e.value.status == 8
    bad = table.copy()
    bad[1, 1] = bad[0, 0]  # sequence 1 writes a page sequence 0 reads
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_stack_decode_paged(st.shape, st.wtype, st.layers, pools, pos, bad, ps, x_bf16=st.x,
                                   workspace=st.workspace)
    assert e.value.status == 8
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_stack_decode_paged(st.shape, st.wtype, st.layers, pools, [3, table.shape[1] * ps], table, ps,
                                   x_bf16=st.x, workspace=st.workspace)
    assert e.value.status == 2
