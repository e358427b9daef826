"""ctypes binding of the C ABI in include/ddl.h (argument marshalling only).

Every function here has the name of the C entry point it wraps, takes torch
tensors (device memory owned by the caller) and passes their data pointers,
sizes and the current CUDA stream.  Every step of the decode runs in the
library's CUDA kernels; nothing falls back to the CPU.  The library must have
been built (``build.build()``); loading fails loudly otherwise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import build as _build

INT4, BF16 = 0, 1
STATUS = {0: "DDL_OK", 1: "DDL_ERR_SHAPE", 2: "DDL_ERR_POS", 3: "DDL_ERR_ALIGN",
          4: "DDL_ERR_WORKSPACE", 5: "DDL_ERR_UNSUPPORTED", 6: "DDL_ERR_CUDA",
          7: "DDL_ERR_TIMEOUT", 8: "DDL_ERR_ARG"}
EXPORTED = ("ddl_quantize_int4", "ddl_packed_layer_bytes", "ddl_pack_layer", "ddl_kv_append",
            "ddl_workspace_bytes", "ddl_workspace_view", "ddl_layer_decode", "ddl_stack_decode",
            "ddl_stack_decode_noalloc", "ddl_set_launch_mode", "ddl_set_wait_limit_ns",
            "ddl_test_hold_barrier", "ddl_set_trace", "ddl_read_device_status", "ddl_status_string",
            "ddl_last_cuda_error", "ddl_embed", "ddl_packed_head_bytes", "ddl_pack_head",
            "ddl_head_workspace_bytes", "ddl_lm_head", "ddl_stack_decode_ragged",
            "ddl_stack_prefill", "ddl_stack_decode_paged", "ddl_stack_prefill_paged")


class DDLError(RuntimeError):
    def __init__(self, func: str, status: int, lib=None):
        msg = f"{func} failed: {STATUS.get(status, status)}"
        if lib is not None:
            msg += f" ({lib.ddl_status_string(status).decode()})"
            if status == 6:
                msg += f": {lib.ddl_last_cuda_error().decode()}"
        super().__init__(msg)
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int32), ("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("eps", ctypes.c_float),
                ("rope_base", ctypes.c_double)]


class Mat(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("w", ctypes.c_void_p)]


class LayerSrc(ctypes.Structure):
    _fields_ = [(n, Mat) for n in ("wq", "wk", "wv", "wo", "wg", "wu", "wd")]


class LayerW(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("norm1", ctypes.c_void_p), ("norm2", ctypes.c_void_p)]


class KV(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("s_max", ctypes.c_int64)]


class KVPages(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("pages", ctypes.c_int64)]


class WsView(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("q", "attn", "y", "a", "status")]


_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libddl.so (building it first only when asked)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA decode library not built ({path} missing); "
                               "run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        P = ctypes.POINTER
        lib.ddl_quantize_int4.argtypes = [vp, i64, i64, vp, vp, vp]
        lib.ddl_packed_layer_bytes.argtypes = [P(Shape), ctypes.c_int]
        lib.ddl_packed_layer_bytes.restype = sz
        lib.ddl_pack_layer.argtypes = [P(Shape), ctypes.c_int, P(LayerSrc), vp, vp]
        lib.ddl_kv_append.argtypes = [P(KV), i32, i32, i32, i64, vp, vp, vp]
        lib.ddl_workspace_bytes.argtypes = [P(Shape), i32, i64]
        lib.ddl_workspace_bytes.restype = sz
        lib.ddl_workspace_view.argtypes = [P(Shape), i32, i64, P(WsView)]
        lib.ddl_layer_decode.argtypes = [P(Shape), ctypes.c_int, P(LayerW), P(KV), i32, i64, vp, vp,
                                         vp, vp, vp, sz, vp]
        lib.ddl_stack_decode.argtypes = [P(Shape), ctypes.c_int, P(LayerW), P(KV), i32, i32, i64,
                                         vp, vp, vp, vp, vp, sz, vp]
        lib.ddl_stack_decode_ragged.argtypes = [P(Shape), ctypes.c_int, P(LayerW), P(KV), i32, i32, P(i64),
                                                vp, vp, vp, vp, vp, sz, vp]
        lib.ddl_stack_prefill.argtypes = [P(Shape), ctypes.c_int, P(LayerW), P(KV), i32, i32, i64, vp, vp, vp, vp,
                                          vp, sz, vp]
        lib.ddl_stack_decode_paged.argtypes = [P(Shape), ctypes.c_int, P(LayerW), P(KVPages), i32, i32, P(i64),
                                               P(i32), i32, i32, vp, vp, vp, vp, vp, sz, vp]
        lib.ddl_stack_prefill_paged.argtypes = [P(Shape), ctypes.c_int, P(LayerW), P(KVPages), i32, i32, i64,
                                                P(i32), i32, i32, vp, vp, vp, vp, vp, sz, vp]
        lib.ddl_stack_decode_noalloc.argtypes = [P(Shape), ctypes.c_int, P(LayerW), P(KV), i32, i32,
                                                 i64, vp, vp, vp, vp, vp]
        lib.ddl_set_launch_mode.argtypes = [i32]
        lib.ddl_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.ddl_test_hold_barrier.argtypes = [i32]
        lib.ddl_set_trace.argtypes = [vp, sz]
        lib.ddl_read_device_status.argtypes = [vp, P(Shape), i32, i64, P(i32), vp]
        lib.ddl_status_string.argtypes = [ctypes.c_int]
        lib.ddl_status_string.restype = ctypes.c_char_p
        lib.ddl_last_cuda_error.restype = ctypes.c_char_p
        lib.ddl_embed.argtypes = [vp, i64, i32, vp, i32, vp, vp, vp]
        lib.ddl_packed_head_bytes.argtypes = [i32, i64, ctypes.c_int]
        lib.ddl_packed_head_bytes.restype = sz
        lib.ddl_pack_head.argtypes = [P(Mat), i32, i64, ctypes.c_int, vp, vp]
        lib.ddl_head_workspace_bytes.argtypes = [i32, i64, i32]
        lib.ddl_head_workspace_bytes.restype = sz
        lib.ddl_lm_head.argtypes = [i32, i64, ctypes.c_int, vp, vp, ctypes.c_float, i32, vp, i32,
                                    ctypes.c_float, vp, vp, vp, vp, vp, sz, vp]
        for name in EXPORTED:
            if not hasattr(lib, name):
                raise RuntimeError(f"{path} does not export {name}")
        _lib = lib
        return lib


def _check(func: str, status: int):
    if status != 0:
        raise DDLError(func, status, _lib)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_shape(cfg) -> Shape:
    return Shape(cfg.D, cfg.H_q, cfg.H_kv, cfg.head_dim, cfg.d_ff, float(cfg.eps),
                 float(cfg.rope_base))


def _u16(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


# ------------------------------------------------------------------ weights

def ddl_quantize_int4(w_bf16: torch.Tensor, stream=None):
    """Symmetric INT4 (group 64, bf16 scales) of a bf16 [N, K] device tensor.
    Returns (q uint8 [N, K/2], scale bf16 [N, K/64])."""
    lib = load()
    assert w_bf16.is_cuda and w_bf16.dtype == torch.bfloat16 and w_bf16.is_contiguous()
    N, K = w_bf16.shape
    q = torch.empty((N, K // 2), dtype=torch.uint8, device=w_bf16.device)
    s = torch.empty((N, K // 64), dtype=torch.bfloat16, device=w_bf16.device)
    _check("ddl_quantize_int4", lib.ddl_quantize_int4(_ptr(w_bf16), N, K, _ptr(q), _ptr(s),
                                                      _stream(stream)))
    return q, s


def ddl_packed_layer_bytes(shape: Shape, wtype: int) -> int:
    return int(load().ddl_packed_layer_bytes(ctypes.byref(shape), wtype))


def ddl_pack_layer(shape: Shape, wtype: int, mats: dict, out: torch.Tensor | None = None,
                   stream=None) -> torch.Tensor:
    """Pack one layer's canonical matrices (dict name -> (q, scale) for INT4 or
    bf16 tensor for BF16) into the kernel-native blob (uint8 device tensor)."""
    lib = load()
    n = ddl_packed_layer_bytes(shape, wtype)
    if n == 0:
        raise DDLError("ddl_packed_layer_bytes", 1, lib)
    dev = next(iter(mats.values()))
    dev = (dev[0] if isinstance(dev, tuple) else dev).device
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=dev)
    src = LayerSrc()
    keep = []
    for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
        m = mats[name]
        if wtype == INT4:
            q, s = m
            keep += [q, s]
            setattr(src, name, Mat(q.data_ptr(), s.data_ptr(), None))
        else:
            keep.append(m)
            setattr(src, name, Mat(None, None, m.data_ptr()))
    _check("ddl_pack_layer", lib.ddl_pack_layer(ctypes.byref(shape), wtype, ctypes.byref(src),
                                                _ptr(out), _stream(stream)))
    return out


# ------------------------------------------------------------------ KV cache

def ddl_kv_append(kc: torch.Tensor, vc: torch.Tensor, pos: int, k_new: torch.Tensor,
                  v_new: torch.Tensor, stream=None):
    """Write k_new, v_new [B, H_kv, hd] bf16 into slot pos of kc, vc [B, H_kv, s_max, hd]."""
    lib = load()
    B, Hkv, s_max, hd = kc.shape
    kv = KV(kc.data_ptr(), vc.data_ptr(), s_max)
    _check("ddl_kv_append", lib.ddl_kv_append(ctypes.byref(kv), B, Hkv, hd, int(pos),
                                              _ptr(k_new), _ptr(v_new), _stream(stream)))


# ------------------------------------------------------------------ decode

def ddl_workspace_bytes(shape: Shape, B: int, s_max: int) -> int:
    n = int(load().ddl_workspace_bytes(ctypes.byref(shape), B, s_max))
    if n == 0:
        raise DDLError("ddl_workspace_bytes", 1, _lib)
    return n


def ddl_workspace_view(shape: Shape, B: int, s_max: int) -> WsView:
    v = WsView()
    _check("ddl_workspace_view", load().ddl_workspace_view(ctypes.byref(shape), B, s_max,
                                                           ctypes.byref(v)))
    return v


def _layers_and_kv(layers, kvs):
    L = len(layers)
    lw = (LayerW * L)()
    kv = (KV * L)()
    for i, (layer, (kc, vc)) in enumerate(zip(layers, kvs)):
        lw[i] = LayerW(layer["packed"].data_ptr(), layer["norm1"].data_ptr(),
                       layer["norm2"].data_ptr())
        kv[i] = KV(kc.data_ptr(), vc.data_ptr(), kc.shape[2])
    return lw, kv


def ddl_stack_decode(shape: Shape, wtype: int, layers: list, kvs: list, pos: int, *,
                     x_bf16: torch.Tensor | None = None, resid_in: torch.Tensor | None = None,
                     resid_out: torch.Tensor | None = None, out_bf16: torch.Tensor | None = None,
                     workspace: torch.Tensor, stream=None):
    """One decode step of len(layers) layers.  layers: dicts with 'packed',
    'norm1', 'norm2' device tensors; kvs: (K, V) caches [B, H_kv, s_max, hd]."""
    lib = load()
    B = (x_bf16 if x_bf16 is not None else resid_in).shape[0]
    lw, kv = _layers_and_kv(layers, kvs)
    st = lib.ddl_stack_decode(ctypes.byref(shape), wtype, lw, kv, len(layers), B, int(pos),
                              _ptr(resid_in), _ptr(x_bf16), _ptr(resid_out), _ptr(out_bf16),
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream(stream))
    _check("ddl_stack_decode", st)


def ddl_stack_decode_ragged(shape: Shape, wtype: int, layers: list, kvs: list, pos, *,
                            x_bf16: torch.Tensor | None = None, resid_in: torch.Tensor | None = None,
                            resid_out: torch.Tensor | None = None, out_bf16: torch.Tensor | None = None,
                            workspace: torch.Tensor, stream=None):
    """ddl_stack_decode with sequence b at its own position pos[b]."""
    lib = load()
    B = (x_bf16 if x_bf16 is not None else resid_in).shape[0]
    lw, kv = _layers_and_kv(layers, kvs)
    pv = (ctypes.c_int64 * B)(*[int(p) for p in pos])
    st = lib.ddl_stack_decode_ragged(ctypes.byref(shape), wtype, lw, kv, len(layers), B, pv,
                                     _ptr(resid_in), _ptr(x_bf16), _ptr(resid_out), _ptr(out_bf16),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream))
    _check("ddl_stack_decode_ragged", st)


def _layers_and_pages(layers, pools):
    L = len(layers)
    lw = (LayerW * L)()
    kv = (KVPages * L)()
    for i, (layer, (kp, vp_)) in enumerate(zip(layers, pools)):
        lw[i] = LayerW(layer["packed"].data_ptr(), layer["norm1"].data_ptr(),
                       layer["norm2"].data_ptr())
        kv[i] = KVPages(kp.data_ptr(), vp_.data_ptr(), kp.shape[0])
    return lw, kv


def _page_table(table):
    """(ctypes int32 array, rows, entries per row) of a 2-D page table."""
    t = np.ascontiguousarray(np.asarray(table, dtype=np.int32))
    if t.ndim != 2:
        raise ValueError("page table: [rows][pages_per_seq]")
    return (ctypes.c_int32 * t.size)(*t.ravel().tolist()), t.shape[0], t.shape[1]


def ddl_stack_decode_paged(shape: Shape, wtype: int, layers: list, pools: list, pos, page_table, page_size: int,
                           *, x_bf16: torch.Tensor | None = None, resid_in: torch.Tensor | None = None,
                           resid_out: torch.Tensor | None = None, out_bf16: torch.Tensor | None = None,
                           workspace: torch.Tensor, stream=None):
    """ddl_stack_decode_ragged on paged caches.  pools: (K, V) per layer, each
    [pages, H_kv, page_size, hd]; page_table: [B][pages_per_seq] page ids."""
    lib = load()
    B = (x_bf16 if x_bf16 is not None else resid_in).shape[0]
    lw, kv = _layers_and_pages(layers, pools)
    pv = (ctypes.c_int64 * B)(*[int(p) for p in pos])
    pt, _, per = _page_table(page_table)
    st = lib.ddl_stack_decode_paged(ctypes.byref(shape), wtype, lw, kv, len(layers), B, pv, pt, per,
                                    int(page_size), _ptr(resid_in), _ptr(x_bf16), _ptr(resid_out),
                                    _ptr(out_bf16), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream))
    _check("ddl_stack_decode_paged", st)


def ddl_stack_prefill_paged(shape: Shape, wtype: int, layers: list, pools: list, p0: int, page_row, page_size: int,
                            *, x_bf16: torch.Tensor | None = None, resid_in: torch.Tensor | None = None,
                            resid_out: torch.Tensor | None = None, out_bf16: torch.Tensor | None = None,
                            workspace: torch.Tensor, stream=None):
    """ddl_stack_prefill into paged caches through one page-table row."""
    lib = load()
    S = (x_bf16 if x_bf16 is not None else resid_in).shape[0]
    lw, kv = _layers_and_pages(layers, pools)
    pt, _, per = _page_table(np.asarray(page_row).reshape(1, -1))
    st = lib.ddl_stack_prefill_paged(ctypes.byref(shape), wtype, lw, kv, len(layers), S, int(p0), pt, per,
                                     int(page_size), _ptr(resid_in), _ptr(x_bf16), _ptr(resid_out),
                                     _ptr(out_bf16), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream))
    _check("ddl_stack_prefill_paged", st)


def ddl_stack_prefill(shape: Shape, wtype: int, layers: list, kvs: list, p0: int, *,
                      x_bf16: torch.Tensor | None = None, resid_in: torch.Tensor | None = None,
                      resid_out: torch.Tensor | None = None, out_bf16: torch.Tensor | None = None,
                      workspace: torch.Tensor, stream=None):
    """S prompt tokens (rows of x) of one sequence at positions p0 .. p0 + S - 1;
    kvs: that sequence's (K, V) caches [1, H_kv, s_max, hd]."""
    lib = load()
    S = (x_bf16 if x_bf16 is not None else resid_in).shape[0]
    lw, kv = _layers_and_kv(layers, kvs)
    st = lib.ddl_stack_prefill(ctypes.byref(shape), wtype, lw, kv, len(layers), S, int(p0), _ptr(resid_in),
                               _ptr(x_bf16), _ptr(resid_out), _ptr(out_bf16), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check("ddl_stack_prefill", st)


def ddl_stack_decode_noalloc(shape: Shape, wtype: int, layers: list, kvs: list, pos: int, *,
                             x_bf16: torch.Tensor | None = None,
                             resid_in: torch.Tensor | None = None,
                             resid_out: torch.Tensor | None = None,
                             out_bf16: torch.Tensor | None = None, stream=None):
    """ddl_stack_decode with the library's static scratch instead of a
    workspace, for callers that cannot allocate device memory."""
    lib = load()
    B = (x_bf16 if x_bf16 is not None else resid_in).shape[0]
    lw, kv = _layers_and_kv(layers, kvs)
    st = lib.ddl_stack_decode_noalloc(ctypes.byref(shape), wtype, lw, kv, len(layers), B, int(pos),
                                      _ptr(resid_in), _ptr(x_bf16), _ptr(resid_out),
                                      _ptr(out_bf16), _stream(stream))
    _check("ddl_stack_decode_noalloc", st)


def ddl_layer_decode(shape: Shape, wtype: int, layer: dict, kv: tuple, pos: int, *,
                     x_bf16=None, resid_in=None, resid_out=None, out_bf16=None, workspace,
                     stream=None):
    lib = load()
    B = (x_bf16 if x_bf16 is not None else resid_in).shape[0]
    lw, kvs = _layers_and_kv([layer], [kv])
    st = lib.ddl_layer_decode(ctypes.byref(shape), wtype, lw, kvs, B, int(pos), _ptr(resid_in),
                              _ptr(x_bf16), _ptr(resid_out), _ptr(out_bf16), _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check("ddl_layer_decode", st)


def ddl_set_launch_mode(mode: int):
    _check("ddl_set_launch_mode", load().ddl_set_launch_mode(mode))


def ddl_set_wait_limit_ns(ns: int):
    """Limit of every bounded device wait (0: the default of 2 s)."""
    _check("ddl_set_wait_limit_ns", load().ddl_set_wait_limit_ns(int(ns)))


def ddl_test_hold_barrier(stage: int):
    """Test hook: hold the grid barrier in front of flattened stage `stage`
    (-1: off), so that the bounded waits give up and report a timeout."""
    _check("ddl_test_hold_barrier", load().ddl_test_hold_barrier(int(stage)))


def ddl_set_trace(buf: torch.Tensor | None):
    """Turn the per-(stage, CTA) timing trace on (a device tensor) or off."""
    lib = load()
    if buf is None:
        _check("ddl_set_trace", lib.ddl_set_trace(None, 0))
    else:
        _check("ddl_set_trace", lib.ddl_set_trace(_ptr(buf), buf.numel() * buf.element_size()))


def ddl_read_device_status(workspace: torch.Tensor | None, shape: Shape, B: int, s_max: int,
                           stream=None) -> int:
    """Status word of the last decode call on `workspace` (None: the static
    scratch of ddl_stack_decode_noalloc)."""
    out = ctypes.c_int32(0)
    _check("ddl_read_device_status",
           load().ddl_read_device_status(_ptr(workspace), ctypes.byref(shape), B, s_max,
                                         ctypes.byref(out), _stream(stream)))
    return int(out.value)


def ws_tensor(workspace: torch.Tensor, offset: int, n: int) -> torch.Tensor:
    """fp32 view of n floats at byte offset `offset` of a workspace tensor."""
    assert offset % 4 == 0
    return workspace.view(torch.uint8)[offset: offset + 4 * n].view(torch.float32)


# ------------------------------------------------------------------ token step

def ddl_embed(table: torch.Tensor, tokens: torch.Tensor, out: torch.Tensor | None = None,
              bad: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Rows tokens (int32 [B], device) of the bf16 table [V, D] -> bf16 [B, D].
    bad: optional int32 [1] device flag set to 1 by an id outside [0, V)."""
    lib = load()
    V, D = table.shape
    B = tokens.numel()
    if out is None:
        out = torch.empty((B, D), dtype=torch.bfloat16, device=table.device)
    _check("ddl_embed", lib.ddl_embed(_ptr(table), V, D, _ptr(tokens), B, _ptr(out), _ptr(bad),
                                      _stream(stream)))
    return out


def ddl_packed_head_bytes(D: int, V: int, wtype: int) -> int:
    return int(load().ddl_packed_head_bytes(D, V, wtype))


def ddl_pack_head(w, D: int, V: int, wtype: int, out: torch.Tensor | None = None,
                  stream=None) -> torch.Tensor:
    """Pack the output matrix [V, D]: (q, scale) for INT4 or a bf16 tensor."""
    lib = load()
    n = ddl_packed_head_bytes(D, V, wtype)
    if n == 0:
        raise DDLError("ddl_packed_head_bytes", 1, lib)
    if wtype == INT4:
        q, s = w
        m, dev = Mat(q.data_ptr(), s.data_ptr(), None), q.device
    else:
        m, dev = Mat(None, None, w.data_ptr()), w.device
    if out is None:
        out = torch.empty(n, dtype=torch.uint8, device=dev)
    _check("ddl_pack_head", lib.ddl_pack_head(ctypes.byref(m), D, V, wtype, _ptr(out), _stream(stream)))
    return out


def ddl_head_workspace_bytes(D: int, V: int, B: int) -> int:
    n = int(load().ddl_head_workspace_bytes(D, V, B))
    if n == 0:
        raise DDLError("ddl_head_workspace_bytes", 1, _lib)
    return n


def ddl_lm_head(D: int, V: int, wtype: int, head_packed: torch.Tensor, x: torch.Tensor,
                norm_f: torch.Tensor | None = None, eps: float = 0.0, top_k: int = 1,
                temperature: float = 1.0, u: torch.Tensor | None = None,
                tokens: torch.Tensor | None = None, logits: torch.Tensor | None = None,
                lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """Next-token ids (int32 [B]) from the fp32 hidden states x [B, D]: greedy
    for top_k <= 1, else top-k sampling with the uniforms u (fp32 [B])."""
    lib = load()
    B = x.shape[0]
    if tokens is None:
        tokens = torch.empty(B, dtype=torch.int32, device=x.device)
    if workspace is None:
        workspace = torch.empty(ddl_head_workspace_bytes(D, V, B), dtype=torch.uint8, device=x.device)
    _check("ddl_lm_head", lib.ddl_lm_head(D, V, wtype, _ptr(head_packed), _ptr(norm_f), float(eps), B,
                                          _ptr(x), int(top_k), float(temperature), _ptr(u),
                                          _ptr(tokens), _ptr(logits), _ptr(lse), _ptr(workspace),
                                          workspace.numel(), _stream(stream)))
    return tokens
