"""Host-side checks of the C-ABI library that need no GPU: it builds for
sm_103a, loads, exports every entry point include/ddl.h declares, and its
host-only calls (status strings, packed-layer sizes, argument checks) behave.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from memory_bound_transformer_decode_gb300 import build, configs, ddl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "ddl.h")).read()
    return sorted(set(re.findall(r"^(?:int|size_t|const char\*)\s+(ddl_\w+)\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ddl.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(ddl.EXPORTED)


def test_status_strings(lib):
    for code in range(9):
        assert lib.ddl_status_string(code)
    assert lib.ddl_status_string(99) == b"unknown status"


def _geom_bytes(cfg, int4: bool) -> int:
    al = lambda x: (x + 255) // 256 * 256  # noqa: E731
    dims = [(cfg.Nq + 2 * cfg.Nkv, cfg.D), (cfg.D, cfg.Nq), (2 * cfg.d_ff, cfg.D), (cfg.D, cfg.d_ff)]
    off = 0
    for N, K in dims:
        T = (N // 16) * (K // 64)
        off = al(off + T * (544 if int4 else 2048))  # INT4 block: 512 B of codes, then its 32 B of scales
    return off


@pytest.mark.parametrize("cfg", configs.ALL)
def test_packed_layer_bytes(lib, cfg):
    shape = ddl.make_shape(cfg)
    n4 = ddl.ddl_packed_layer_bytes(shape, ddl.INT4)
    nb = ddl.ddl_packed_layer_bytes(shape, ddl.BF16)
    assert n4 == _geom_bytes(cfg, True)
    assert nb == _geom_bytes(cfg, False)
    # exactly the codes and scales (or bf16 values), up to 256-byte alignment
    mac = sum(n * k for n, k in [(cfg.Nq + 2 * cfg.Nkv, cfg.D), (cfg.D, cfg.Nq),
                                 (2 * cfg.d_ff, cfg.D), (cfg.D, cfg.d_ff)])
    assert 0 <= n4 - (mac // 2 + mac // 32) < 8 * 256
    assert 0 <= nb - 2 * mac < 4 * 256


def test_shape_rules(lib):
    bad = [ddl.Shape(128, 4, 2, 96, 192, 1e-6, 1e4),   # head_dim
           ddl.Shape(100, 4, 2, 64, 192, 1e-6, 1e4),   # D % 64
           ddl.Shape(128, 4, 3, 64, 192, 1e-6, 1e4),   # H_q % H_kv
           ddl.Shape(128, 16, 1, 64, 192, 1e-6, 1e4),  # group > 8
           ddl.Shape(128, 4, 2, 64, 100, 1e-6, 1e4)]   # d_ff % 64
    for s in bad:
        assert ddl.ddl_packed_layer_bytes(s, ddl.INT4) == 0


def test_host_argument_checks(lib):
    assert lib.ddl_set_launch_mode(7) == 8
    assert lib.ddl_set_launch_mode(0) == 0
    assert lib.ddl_test_hold_barrier(-2) == 8
    assert lib.ddl_test_hold_barrier(-1) == 0
    assert lib.ddl_set_wait_limit_ns(5_000_000) == 0
    assert lib.ddl_set_wait_limit_ns(0) == 0
    assert lib.ddl_quantize_int4(None, 4, 64, None, None, None) == 8
    kv = ddl.KV(16, 16, 10)
    assert lib.ddl_kv_append(ctypes.byref(kv), 1, 1, 64, 10, ctypes.c_void_p(16),
                             ctypes.c_void_p(16), None) == 2


def test_token_step_host_checks(lib):
    # sizes: INT4 blocks of 544 bytes, bf16 of 2048, over ceil(V / 16) tiles x D / 64 groups
    assert lib.ddl_packed_head_bytes(512, 1000, ddl.INT4) == 63 * 8 * 544
    assert lib.ddl_packed_head_bytes(512, 1008, ddl.BF16) == 63 * 8 * 2048
    assert lib.ddl_packed_head_bytes(500, 1000, ddl.INT4) == 0
    assert lib.ddl_packed_head_bytes(512, 0, ddl.INT4) == 0
    m = ddl.Mat(None, None, None)
    assert lib.ddl_pack_head(ctypes.byref(m), 512, 1000, ddl.INT4, ctypes.c_void_p(256), None) == 8
    assert lib.ddl_pack_head(ctypes.byref(m), 500, 1000, ddl.INT4, ctypes.c_void_p(256), None) == 1
    p = ctypes.c_void_p(256)
    assert lib.ddl_embed(None, 10, 64, p, 1, p, None, None) == 8
    assert lib.ddl_embed(p, 10, 100, p, 1, p, None, None) == 1
    assert lib.ddl_embed(p, 10, 64, p, 65, p, None, None) == 5
    assert lib.ddl_embed(ctypes.c_void_p(258), 10, 64, p, 1, p, None, None) == 3
    head = lambda **kw: lib.ddl_lm_head(  # noqa: E731
        kw.get("D", 512), kw.get("V", 1000), ddl.INT4, p, None, 1e-6, kw.get("B", 1), p, kw.get("k", 1),
        ctypes.c_float(kw.get("T", 1.0)), kw.get("u", None), p, None, None, kw.get("ws", p), 1 << 30, None)
    assert head(D=500) == 1
    assert head(B=65) == 5
    assert head(k=1025, u=p) == 5
    assert head(k=-1) == 8
    assert head(k=4) == 8             # sampling without uniforms
    assert head(k=4, u=p, T=0.0) == 8
    assert head(ws=None) == 8


def test_ragged_decode_host_checks(lib):
    s = ddl.Shape(512, 8, 2, 64, 1408, 1e-6, 1e4)
    p = ctypes.c_void_p(256)
    pos = (ctypes.c_int64 * 2)(3, 4)
    assert lib.ddl_stack_decode_ragged(ctypes.byref(s), ddl.INT4, None, None, 1, 2, None, None, p, None, p,
                                       p, 1 << 20, None) == 8  # no positions
    assert lib.ddl_stack_decode_ragged(ctypes.byref(s), ddl.INT4, None, None, 1, 65, pos, None, p, None, p,
                                       p, 1 << 20, None) == 5  # batch past the limit


def test_paged_decode_host_checks(lib):
    """The page-table rules are checked on the host before any device work: a
    call that passes them goes on to the device query (no GPU here: a CUDA
    error), one that breaks them returns DDL_ERR_ARG / DDL_ERR_POS."""
    if torch.cuda.is_available():  # fake device pointers must never reach a GPU
        pytest.skip("host checks with fake pointers run without a GPU; tests/test_gpu_paged.py has real buffers")
    s = ddl.Shape(512, 8, 2, 64, 1408, 1e-6, 1e4)
    p = ctypes.c_void_p(256)
    lw = (ddl.LayerW * 2)(ddl.LayerW(256, 256, 256), ddl.LayerW(256, 256, 256))

    def call(table, pos, ps=16, pages=(10, 10), per=None):
        kv = (ddl.KVPages * 2)(*[ddl.KVPages(256, 256, n) for n in pages])
        t = np.asarray(table, np.int32)
        per = t.shape[1] if per is None else per
        pt = (ctypes.c_int32 * t.size)(*t.ravel().tolist())
        pv = (ctypes.c_int64 * len(pos))(*pos)
        return lib.ddl_stack_decode_paged(ctypes.byref(s), ddl.INT4, lw, kv, 2, len(pos), pv, pt, per, ps, None,
                                          p, None, None, p, 1 << 30, None)

    good = [[0, 1, 2], [3, 4, 9]]
    assert call(good, [40, 33]) == 6                  # past the host checks: no device here
    assert call(good, [40, 33], ps=24) == 8           # page size not a power of two
    assert call(good, [40, 33], ps=8) == 8            # below one 16-key tile
    assert call(good, [40, 48]) == 2                  # slot 48 past 3 pages of 16
    assert call([[0, 1, 2], [3, 4, 10]], [40, 33]) == 8   # page 10 of a 10-page pool
    assert call([[0, 1, -1], [3, 4, 9]], [40, 33]) == 8   # negative page id
    assert call([[0, 1, 2], [3, 4, 77]], [40, 15]) == 6   # dead entries are not read
    assert call([[0, 1, 2], [0, 1, 9]], [40, 33]) == 6    # a shared read-only prefix
    assert call([[0, 1, 2], [0, 2, 9]], [40, 33]) == 8    # page 2 receives a row that another sequence reads
    assert call([[0, 1, 1], [3, 4, 9]], [40, 33]) == 8    # a sequence mapping its written page twice
    assert call(good, [40, 33], pages=(10, 11)) == 8      # pools of different sizes
    # prefill through one page-table row: the pages written must be its own
    kv = (ddl.KVPages * 2)(*[ddl.KVPages(256, 256, 10) for _ in range(2)])

    def pre(row, p0, S):
        pt = (ctypes.c_int32 * len(row))(*row)
        return lib.ddl_stack_prefill_paged(ctypes.byref(s), ddl.INT4, lw, kv, 2, S, p0, pt, len(row), 16, None, p,
                                           None, None, p, 1 << 30, None)

    assert pre([5, 6, 7], 10, 20) == 6
    assert pre([5, 6, 6], 10, 30) == 8                # page 6 mapped twice and written
    assert pre([5, 6, 7], 40, 9) == 2                 # past 48 slots
