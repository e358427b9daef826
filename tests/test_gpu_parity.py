"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Bit-exact for the quantizer, the packer and the KV append; the decode step
within the tolerances stated in gpu_helpers.  Sizes span several tiles,
k-chunks and 16-key tiles with ragged tails; edge cases cover an empty KV
history, single-key attention, ragged last tiles, batches 1-4, head_dim 64
and 128, query groups of 1-8 heads and k-chunked inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_transformer_decode_gb300 import configs, ddl, synth, workload
from tests.gpu_helpers import (MAX_ABS, REL_L2, bf16_bits_close, device_outputs, oracle_stack,
                               rel_l2, tensor_core_path)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddl.load(build_if_missing=True)
    torch.manual_seed(0)
    yield


# ------------------------------------------------------------------ quantizer


@pytest.mark.parametrize("N,K", [(1, 64), (37, 128), (300, 5120), (64, 2112)])
def test_quantize_bit_exact(N, K):
    w = synth.normal_bf16((N, K), seed=N * 7 + K, std=0.02, device="cuda")
    if N > 10:  # special groups: zero, one value, exact multiples, huge/tiny values
        w[1, :64] = 0
        w[2, :64] = 0
        w[2, 5] = -0.0371
        w[3, :64] = (torch.arange(64, device="cuda") % 15 - 7).to(torch.bfloat16) * 2.0 ** -5
        w[4, :64] *= 1e30
        w[5, :64] *= 1e-30
    q, s = ddl.ddl_quantize_int4(w)
    qo, so = oracle.quantize_int4(synth.bits(w))
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    np.testing.assert_array_equal(synth.bits(s), so)


def test_kv_append_bit_exact():
    B, Hkv, s_max, hd, pos = 3, 2, 37, 128, 29
    kc = synth.normal_bf16((B, Hkv, s_max, hd), seed=1, device="cuda")
    vc = synth.normal_bf16((B, Hkv, s_max, hd), seed=2, device="cuda")
    kn = synth.normal_bf16((B, Hkv, hd), seed=3, device="cuda")
    vn = synth.normal_bf16((B, Hkv, hd), seed=4, device="cuda")
    k0, v0 = kc.clone(), vc.clone()
    ddl.ddl_kv_append(kc, vc, pos, kn, vn)
    torch.cuda.synchronize()
    k0[:, :, pos] = kn
    v0[:, :, pos] = vn
    assert torch.equal(kc.view(torch.int16), k0.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), v0.view(torch.int16))


# ------------------------------------------------------------------ packer


def _geoms(cfg, wtype):
    """Packed-layer geometry recomputed from the documented layout."""
    Nq, Nkv = cfg.Nq, cfg.Nkv
    dims = [(Nq + 2 * Nkv, cfg.D), (cfg.D, Nq), (2 * cfg.d_ff, cfg.D), (cfg.D, cfg.d_ff)]
    out, off = [], 0
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    for N, K in dims:
        G = K // 64
        Gc = min(G, 32)
        g = dict(N=N, K=K, NT=N // 16, G=G, Gc=Gc, Sk=-(-G // Gc), T=(N // 16) * G, woff=off)
        off = al(off + g["T"] * (544 if wtype == ddl.INT4 else 2048))  # INT4: 512 B codes + 32 B scales
        out.append(g)
    return out, off


def _tile_rows(kind, T, hd):
    r = np.arange(16)
    if kind == 0:
        tph = hd // 16
        head, mm = T // tph, T % tph
        return head * hd + np.where(r < 8, 8 * mm + r, 8 * mm + r - 8 + hd // 2)
    if kind == 2:
        return np.where(r < 8, 8 * T + r, 8 * T + r - 8)  # gate rows, then up rows
    return 16 * T + r


def _block_coords(g):
    b = np.arange(g["T"])
    per = g["NT"] * g["Gc"]
    kc = np.minimum(b // per, g["Sk"] - 1)
    rem = b - kc * per
    gk = np.where(kc == g["Sk"] - 1, g["G"] - (g["Sk"] - 1) * g["Gc"], g["Gc"])
    return kc, rem // gk, rem % gk


@pytest.mark.parametrize("cfg", [configs.SMALL_LAYER,
                                 configs.SMALL_LAYER.with_(D=2112, d_ff=4160, name="chunked")])
def test_pack_layer_is_the_documented_permutation(cfg):
    shape = ddl.make_shape(cfg)
    w = synth.layer_weights(cfg, 0, device="cuda")
    mats = {n: ddl.ddl_quantize_int4(w[n]) for n in workload.MATS}
    blob = ddl.ddl_pack_layer(shape, ddl.INT4, mats).cpu().numpy()
    geoms, total = _geoms(cfg, ddl.INT4)
    assert blob.size == total == ddl.ddl_packed_layer_bytes(shape, ddl.INT4)
    codes = {n: oracle.unpack_int4(mats[n][0].cpu().numpy()) for n in workload.MATS}
    scales = {n: synth.bits(mats[n][1]) for n in workload.MATS}
    combos = [np.concatenate([codes["wq"], codes["wk"], codes["wv"]]), codes["wo"],
              None, codes["wd"]]
    scombos = [np.concatenate([scales["wq"], scales["wk"], scales["wv"]]), scales["wo"],
               None, scales["wd"]]
    lanes = np.arange(32)
    gg, tt = lanes // 4, lanes % 4
    for kind, g in enumerate(geoms):
        kc, T, gi = _block_coords(g)
        blocks = blob[g["woff"]: g["woff"] + g["T"] * 544].view(np.uint32).reshape(-1, 136)
        words = blocks[:, :128].reshape(-1, 32, 4)
        sw = blocks[:, 128:]
        for b in range(0, g["T"], max(1, g["T"] // 97)):  # a spread sample of blocks
            rows = _tile_rows(kind, T[b], cfg.head_dim)
            if kind == 2:
                src = np.concatenate([codes["wg"][rows[:8]], codes["wu"][rows[8:]]])
                ssrc = np.concatenate([scales["wg"][rows[:8]], scales["wu"][rows[8:]]])
            else:
                src, ssrc = combos[kind][rows], scombos[kind][rows]
            grp = kc[b] * g["Gc"] + gi[b]
            for j in range(4):
                k0 = grp * 64 + 16 * j + 2 * tt
                wd = words[b, :, j].astype(np.int64)
                nib = [(wd >> (4 * s)) & 0xF for s in range(8)]
                want = [src[gg, k0], src[gg + 8, k0], src[gg, k0 + 8], src[gg + 8, k0 + 8],
                        src[gg, k0 + 1], src[gg + 8, k0 + 1], src[gg, k0 + 9], src[gg + 8, k0 + 9]]
                for s in range(8):
                    np.testing.assert_array_equal(nib[s], want[s].astype(np.int64) & 0xF)
            np.testing.assert_array_equal(sw[b] & 0xFFFF, ssrc[:8, grp])
            np.testing.assert_array_equal(sw[b] >> 16, ssrc[8:, grp])


# ------------------------------------------------------------------ decode step


def _check_layer(st, mode=None, stages=True):
    out, res, dst = device_outputs(st, mode)
    kv_host = None
    z, ost, _, caches = oracle_stack(st, kv_host, stages_last=stages)
    e_out = rel_l2(oracle.bf16_to_f64(out), z)
    e_res = float(np.max(np.abs(res - z)))
    assert e_out <= REL_L2, f"bf16 output rel-L2 {e_out:.3e}"
    assert e_res <= MAX_ABS, f"fp32 residual max-abs {e_res:.3e}"
    # the appended K/V rows (last layer's cache)
    kc_dev, vc_dev = (synth.bits(t) for t in st.kvs[-1])
    kc_o, vc_o = caches[-1]
    p = st.pos
    if st.batch <= 4 or tensor_core_path(st):  # x carried to >= 22 bits: k, v within a bf16 ulp
        assert bf16_bits_close(kc_dev[:, :, p], kc_o[:, :, p]), "appended K"
        assert bf16_bits_close(vc_dev[:, :, p], vc_o[:, :, p]), "appended V"
    else:  # the warp-level wide path (5-15 sequences) carries x in fp16 (11 bits): the stage tolerance
        for name, d, o in (("K", kc_dev, kc_o), ("V", vc_dev, vc_o)):
            e = rel_l2(oracle.bf16_to_f64(d[:, :, p]), oracle.bf16_to_f64(o[:, :, p]))
            assert e <= REL_L2, f"appended {name} rel-L2 {e:.3e}"
    np.testing.assert_array_equal(kc_dev[:, :, :p], kc_o[:, :, :p])
    errs = {"out": e_out, "res_maxabs": e_res}
    if stages:
        for name in ("q", "attn", "y", "a"):
            e = rel_l2(dst[name], ost[name])
            errs[name] = e
            assert e <= REL_L2, f"stage {name} rel-L2 {e:.3e}"
    return errs, out, res


@pytest.mark.parametrize("cfg", [configs.SMALL_LAYER, configs.QWEN7B_LAYER])
def test_layer_parity_named_configs(cfg):
    st = workload.build_stack(cfg)
    errs, _, _ = _check_layer(st)
    print(cfg.name, {k: f"{v:.2e}" for k, v in errs.items()})


EDGE = configs.DecodeConfig("edge", D=128, H_q=4, H_kv=2, head_dim=64, d_ff=192, rope_base=1e4,
                            kv_len=20, layers=1, seed=9)


@pytest.mark.parametrize("kv_len", [0, 1, 15, 16, 17, 100])
def test_layer_parity_cache_lengths(kv_len):
    errs, _, _ = _check_layer(workload.build_stack(EDGE.with_(kv_len=kv_len)))
    print(kv_len, errs)


@pytest.mark.parametrize("B", [2, 3, 4, 5, 8, 9, 16])
def test_layer_parity_batches(B):
    """Batches 2-4 carry x as fp16 hi/lo columns; 5-16 as fp16 columns in one
    or two n-tiles of 8 (the wide-batch stage)."""
    _check_layer(workload.build_stack(EDGE.with_(kv_len=33), batch=B))


@pytest.mark.parametrize("B", [6, 16])
def test_wide_batch_shapes(B):
    cfg = EDGE.with_(D=2112, d_ff=4160, H_q=8, H_kv=2, head_dim=128, kv_len=70, name="chunked-wide")
    _check_layer(workload.build_stack(cfg, batch=B))


def test_wide_batch_stack_launch_modes_agree():
    cfg = EDGE.with_(layers=3, kv_len=45, D=256, H_q=8, H_kv=2, head_dim=128, d_ff=320, name="s3w")
    st = workload.build_stack(cfg, batch=12)
    kv0 = [(synth.bits(k).copy(), synth.bits(v).copy()) for k, v in st.kvs]
    out_c, res_c, _ = device_outputs(st, mode=0)
    out_s, res_s, _ = device_outputs(st, mode=1)
    np.testing.assert_array_equal(out_c, out_s)
    np.testing.assert_array_equal(res_c, res_s)
    z, _, _, _ = oracle_stack(st, kv0)
    assert rel_l2(oracle.bf16_to_f64(out_c), z) <= REL_L2
    assert np.max(np.abs(res_c - z)) <= MAX_ABS


@pytest.mark.parametrize("B", [5, 8, 16])
def test_wide_batch_bf16_weights(B):
    """bf16 weights beyond 4 sequences run on the tcgen05 tensor cores."""
    _check_layer(workload.build_stack(EDGE.with_(kv_len=24, D=256, d_ff=320), wtype=ddl.BF16, batch=B))


@pytest.mark.parametrize("cfg", [
    EDGE.with_(H_q=7, H_kv=1, head_dim=128, D=256, kv_len=40, name="g7"),
    EDGE.with_(H_q=8, H_kv=1, head_dim=128, D=192, kv_len=5, name="g8"),
    EDGE.with_(H_q=2, H_kv=2, head_dim=64, D=64, d_ff=64, kv_len=3, name="mha-tiny"),
    EDGE.with_(D=2112, d_ff=4160, H_q=6, H_kv=2, head_dim=128, kv_len=70, name="chunked"),
])
def test_layer_parity_shapes(cfg):
    _check_layer(workload.build_stack(cfg))


def test_stack_parity_small_and_launch_modes_agree():
    cfg = EDGE.with_(layers=5, kv_len=45, D=256, H_q=8, H_kv=2, head_dim=128, d_ff=320, name="s5")
    st = workload.build_stack(cfg, batch=2)
    kv0 = [(synth.bits(k).copy(), synth.bits(v).copy()) for k, v in st.kvs]
    out_c, res_c, _ = device_outputs(st, mode=0)
    out_s, res_s, _ = device_outputs(st, mode=1)
    np.testing.assert_array_equal(out_c, out_s)
    np.testing.assert_array_equal(res_c, res_s)
    out_r, res_r, _ = device_outputs(st, mode=0)  # deterministic re-run
    np.testing.assert_array_equal(res_r, res_c)
    z, _, _, _ = oracle_stack(st, kv0)
    assert rel_l2(oracle.bf16_to_f64(out_c), z) <= REL_L2
    assert np.max(np.abs(res_c - z)) <= MAX_ABS


def test_stack_longer_than_one_launch():
    """100 layers: two cooperative launches of at most 96 layers, the second
    starting with its own maxima, counters and empty partial slots; bit-equal
    to one launch per stage, and to the oracle run untethered over all 100
    layers (output rel-L2 at the step's bar; the fp32 residual held to 1e-3 of
    the largest |z|, as for the 64-layer stack)."""
    cfg = EDGE.with_(layers=100, kv_len=45, D=256, H_q=8, H_kv=2, head_dim=128, d_ff=320, name="s100")
    st = workload.build_stack(cfg, batch=1)
    kv0 = [(synth.bits(k).copy(), synth.bits(v).copy()) for k, v in st.kvs]
    out_c, res_c, _ = device_outputs(st, mode=0)
    out_s, res_s, _ = device_outputs(st, mode=1)
    np.testing.assert_array_equal(out_c, out_s)
    np.testing.assert_array_equal(res_c, res_s)
    z, _, _, _ = oracle_stack(st, kv0)
    assert rel_l2(oracle.bf16_to_f64(out_c), z) <= REL_L2
    assert np.max(np.abs(res_c - z)) <= 1e-3 * np.max(np.abs(z))


def test_bf16_weight_layer_parity():
    st = workload.build_stack(EDGE.with_(kv_len=24, D=256, d_ff=320), wtype=ddl.BF16, batch=2)
    _check_layer(st)


# ------------------------------------------------------------------ argument errors


def test_argument_errors_are_reported():
    st = workload.build_stack(EDGE.with_(kv_len=4))
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_stack_decode(st.shape, st.wtype, st.layers, st.kvs, st.s_max, x_bf16=st.x,
                             workspace=st.workspace)
    assert e.value.status == 2
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_stack_decode(st.shape, st.wtype, st.layers, st.kvs, st.pos, x_bf16=st.x,
                             workspace=st.workspace[:64])
    assert e.value.status == 4
    with pytest.raises(ddl.DDLError) as e:
        ws = st.workspace.view(torch.uint8)[8:]
        ddl.ddl_stack_decode(st.shape, st.wtype, st.layers, st.kvs, st.pos, x_bf16=st.x,
                             workspace=ws)
    assert e.value.status in (3, 4)
    bad = ddl.Shape(128, 4, 2, 96, 192, 1e-6, 1e4)
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_workspace_bytes(bad, 1, 16)
    x65 = synth.normal_bf16((65, st.cfg.D), seed=1, device="cuda")  # beyond DDL_MAX_BATCH
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_stack_decode(st.shape, st.wtype, st.layers, st.kvs, st.pos, x_bf16=x65,
                             workspace=st.workspace)
    assert e.value.status == 5
