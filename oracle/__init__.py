"""fp64 CPU oracle of the batch-B INT4 GQA decode step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It never
imports the CUDA library package and shares no code with it; the only thing
both sides share is the seeded input generator (``synth``), which holds none
of the method's arithmetic.

The arithmetic lives in ``ddl_oracle.c`` (plain C, fp64, OpenMP over
independent outputs), compiled here with gcc at first use.  Each function
states the passage it follows; see the C file's header for the readings of
the pages taken where they are silent.

Pinning: every function below is pinned by ``tests/test_oracle_pins.py``
against closed forms, invariants, library routines and brute force; the
composed layer is additionally pinned against a composition of PyTorch
library routines (F.rms_norm, scaled_dot_product_attention, F.silu) and
against residual-identity special cases.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ddl_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ddl_oracle.c to a shared library (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Shape(ctypes.Structure):
    _fields_ = [("D", ctypes.c_int64), ("H_q", ctypes.c_int64), ("H_kv", ctypes.c_int64),
                ("head_dim", ctypes.c_int64), ("d_ff", ctypes.c_int64),
                ("rope_base", ctypes.c_double), ("eps", ctypes.c_double)]


class _Mat(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("w", ctypes.c_void_p)]


class _Layer(ctypes.Structure):
    _fields_ = [("norm1", ctypes.c_void_p), ("wq", _Mat), ("wk", _Mat), ("wv", _Mat),
                ("wo", _Mat), ("norm2", ctypes.c_void_p), ("wg", _Mat), ("wu", _Mat),
                ("wd", _Mat)]


class _Stages(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("h", "q", "k", "v", "attn", "y", "a")]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dbl, vp = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.orc_bf16_to_f64.restype = dbl
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_from_f64.restype = ctypes.c_uint16
            lib.orc_bf16_from_f64.argtypes = [dbl]
            lib.orc_bf16_from_f64_array.argtypes = [vp, i64, vp]
            lib.orc_quantize_int4.argtypes = [vp, i64, i64, vp, vp]
            lib.orc_unpack_int4.argtypes = [vp, i64, i64, vp]
            lib.orc_gemv_int4.argtypes = [vp, vp, i64, i64, vp, vp]
            lib.orc_gemv_bf16.argtypes = [vp, i64, i64, vp, vp]
            lib.orc_rmsnorm.argtypes = [vp, vp, i64, dbl, vp]
            lib.orc_rope.argtypes = [vp, i64, i64, dbl]
            lib.orc_attention.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, vp, vp]
            lib.orc_layer_decode.restype = ctypes.c_int
            lib.orc_layer_decode.argtypes = [ctypes.POINTER(_Shape), ctypes.POINTER(_Layer),
                                             vp, vp, i64, i64, i64, vp, vp,
                                             ctypes.POINTER(_Stages)]
            lib.orc_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_load().orc_num_threads())


# ---------------------------------------------------------------- bf16

def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    b = _c(bits, np.uint16)
    with np.errstate(invalid="ignore"):
        return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_from_f64(x) -> np.ndarray:
    """Round fp64 values to bf16 bit patterns, nearest-even, one rounding."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().orc_bf16_from_f64_array(_p(x), x.size, _p(out))
    return out


# ---------------------------------------------------------------- INT4

def quantize_int4(w_bf16) -> tuple[np.ndarray, np.ndarray]:
    """Symmetric INT4, group 64 along K (Unsloth article §二.3 4-bit weights).

    w_bf16: uint16 [N, K] bf16 bits.  Returns (q uint8 [N, K/2] with even k in
    the low nibble, s uint16 [N, K/64] bf16 scales)."""
    w = _c(w_bf16, np.uint16)
    N, K = w.shape
    if K % 64:
        raise ValueError("K must be a multiple of 64")
    q = np.zeros((N, K // 2), np.uint8)
    s = np.zeros((N, K // 64), np.uint16)
    _load().orc_quantize_int4(_p(w), N, K, _p(q), _p(s))
    return q, s


def unpack_int4(q) -> np.ndarray:
    """Codes int8 [N, K] of a packed [N, K/2] matrix."""
    q = _c(q, np.uint8)
    N, Kh = q.shape
    out = np.empty((N, 2 * Kh), np.int8)
    _load().orc_unpack_int4(_p(q), N, 2 * Kh, _p(out))
    return out


# ---------------------------------------------------------------- primitives

def gemv_int4(q, s, x) -> np.ndarray:
    """y = (q*s) x in fp64 (primer §1.1 projections with dequantized weights)."""
    q = _c(q, np.uint8)
    s = _c(s, np.uint16)
    x = _c(x, np.float64)
    N, Kh = q.shape
    y = np.empty(N, np.float64)
    _load().orc_gemv_int4(_p(q), _p(s), N, 2 * Kh, _p(x), _p(y))
    return y


def gemv_bf16(w, x) -> np.ndarray:
    w = _c(w, np.uint16)
    x = _c(x, np.float64)
    N, K = w.shape
    y = np.empty(N, np.float64)
    _load().orc_gemv_bf16(_p(w), N, K, _p(x), _p(y))
    return y


def rmsnorm(x, w_bf16, eps: float) -> np.ndarray:
    """x * w / sqrt(mean(x^2) + eps) (primer §1.1 rmsnorm)."""
    x = _c(x, np.float64)
    w = _c(w_bf16, np.uint16)
    out = np.empty_like(x)
    _load().orc_rmsnorm(_p(x), _p(w), x.size, float(eps), _p(out))
    return out


def rope(v, pos: int, base: float) -> np.ndarray:
    """Half-split RoPE of one head vector (roofline reply §五)."""
    v = np.array(v, np.float64, copy=True, order="C")
    _load().orc_rope(_p(v), v.size, int(pos), float(base))
    return v


def attention(q, kc, vc, n_keys: int, return_probs: bool = False):
    """Softmax attention of one query token per head over keys 0..n_keys-1.

    q: [H_q, hd] fp64; kc, vc: [H_kv, s_max, hd] bf16 bits (one sequence).
    Returns o [H_q, hd] (and the weights [H_q, n_keys] when asked)."""
    q = _c(q, np.float64)
    kc = _c(kc, np.uint16)
    vc = _c(vc, np.uint16)
    Hq, hd = q.shape
    Hkv, s_max, _ = kc.shape
    out = np.empty((Hq, hd), np.float64)
    probs = np.empty((Hq, n_keys), np.float64) if return_probs else None
    _load().orc_attention(_p(q), _p(kc), _p(vc), Hq, Hkv, hd, s_max, int(n_keys),
                          _p(out), _p(probs))
    return (out, probs) if return_probs else out


# ---------------------------------------------------------------- layer

@dataclass
class OracleMat:
    """A weight matrix [N, K]: INT4 (q, s) or bf16 (w)."""
    q: np.ndarray | None = None
    s: np.ndarray | None = None
    w: np.ndarray | None = None


def quantized_layer(weights: dict) -> dict:
    """Quantize every matrix of a bf16 layer dict with the oracle's quantizer."""
    out = {"norm1": weights["norm1"], "norm2": weights["norm2"]}
    for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
        q, s = quantize_int4(weights[name])
        out[name] = OracleMat(q=q, s=s)
    return out


def bf16_layer(weights: dict) -> dict:
    out = {"norm1": weights["norm1"], "norm2": weights["norm2"]}
    for name in ("wq", "wk", "wv", "wo", "wg", "wu", "wd"):
        out[name] = OracleMat(w=_c(weights[name], np.uint16))
    return out


def layer_decode(shape, layer: dict, kc, vc, pos: int, x, stages: bool = False):
    """One decode step of one layer for B sequences (primer §1.2 decode_step).

    shape: object with D, H_q, H_kv, head_dim, d_ff, rope_base, eps.
    layer: dict from quantized_layer() / bf16_layer().
    kc, vc: uint16 [B, H_kv, s_max, hd], modified in place (slot pos written).
    x: fp64 [B, D].  Returns z [B, D] (and a dict of stage outputs)."""
    lib = _load()
    x = _c(x, np.float64)
    B, D = x.shape
    assert kc.dtype == np.uint16 and kc.flags.c_contiguous
    assert vc.dtype == np.uint16 and vc.flags.c_contiguous
    s_max = kc.shape[2]
    sh = _Shape(shape.D, shape.H_q, shape.H_kv, shape.head_dim, shape.d_ff,
                float(shape.rope_base), float(shape.eps))
    keep = []

    def mat(m: OracleMat) -> _Mat:
        arrs = [None if a is None else np.ascontiguousarray(a) for a in (m.q, m.s, m.w)]
        keep.extend(a for a in arrs if a is not None)
        return _Mat(*[_p(a) for a in arrs])

    n1 = _c(layer["norm1"], np.uint16)
    n2 = _c(layer["norm2"], np.uint16)
    L = _Layer(_p(n1), mat(layer["wq"]), mat(layer["wk"]), mat(layer["wv"]), mat(layer["wo"]),
               _p(n2), mat(layer["wg"]), mat(layer["wu"]), mat(layer["wd"]))
    z = np.empty((B, D), np.float64)
    st = None
    st_arrays = {}
    if stages:
        Nq = shape.H_q * shape.head_dim
        Nkv = shape.H_kv * shape.head_dim
        sizes = {"h": D, "q": Nq, "k": Nkv, "v": Nkv, "attn": Nq, "y": D, "a": shape.d_ff}
        st_arrays = {k: np.empty((B, n), np.float64) for k, n in sizes.items()}
        st = _Stages(*[_p(st_arrays[k]) for k in ("h", "q", "k", "v", "attn", "y", "a")])
    rc = lib.orc_layer_decode(ctypes.byref(sh), ctypes.byref(L), _p(kc), _p(vc), s_max, B,
                              int(pos), _p(x), _p(z), ctypes.byref(st) if st else None)
    if rc != 0:
        raise ValueError(f"oracle rejected the shape/position (rc={rc})")
    return (z, st_arrays) if stages else z


# ---------------------------------------------------------------- token step
# The steps on either side of the layer stack in the primer's §1.2
# decode step: the last token's embedding row before the layers, and after
# them a token drawn from the logits of the last hidden state against the
# embedding table, with the Unsloth/Qwen-27B article's §三 vocabulary of about
# 152 thousand entries.  Readings where the pages are silent: the output
# matrix is the (tied) embedding table, in the same weight format as the
# layers (INT4 quantized from the bf16 table, or the bf16 table itself); an
# optional final RMSNorm weight (the pages show none; the Qwen/Llama models of
# the workload shapes apply one before the output matrix); greedy decoding
# takes the lowest id among equal maxima; top-k sampling is inverse-CDF
# sampling over the k largest logits (equal logits at the boundary: lower ids
# first) with weights exp((l - l_max) / T) and a caller-drawn uniform u.

def embed(table_bf16, tokens) -> np.ndarray:
    """Rows `tokens` of the embedding table (primer §1.2 `embed`).

    table_bf16: uint16 [V, D] bf16 bits.  tokens: int [B].  Returns a uint16
    [B, D] copy.  Ids outside [0, V) raise ValueError."""
    table = np.asarray(table_bf16, np.uint16)
    ids = np.asarray(tokens, np.int64).reshape(-1)
    if np.any((ids < 0) | (ids >= table.shape[0])):
        raise ValueError("token id outside the vocabulary")
    out = np.empty((ids.size, table.shape[1]), np.uint16)
    for b, t in enumerate(ids):
        out[b] = table[t]
    return out


def lm_head_logits(x, head: OracleMat, norm_w=None, eps: float = 0.0) -> np.ndarray:
    """Logits over the vocabulary of B hidden states (primer §1.2
    decode step: the last hidden state times the transposed embedding table): l = W h with h = rmsnorm(x, norm_w) when a final
    norm weight is given, else h = x.

    x: fp64 [B, D].  head: OracleMat [V, D], INT4 (q, s) or bf16 (w).
    Returns fp64 [B, V]."""
    x = np.atleast_2d(np.asarray(x, np.float64))
    rows = []
    for b in range(x.shape[0]):
        h = rmsnorm(x[b], norm_w, eps) if norm_w is not None else x[b]
        rows.append(gemv_int4(head.q, head.s, h) if head.w is None else gemv_bf16(head.w, h))
    return np.stack(rows)


def greedy_token(logits) -> np.ndarray:
    """Greedy decoding: the id of the largest logit, the lowest id among
    equal maxima.  logits: [B, V] (or [V]).  Returns int64 [B]."""
    l = np.atleast_2d(np.asarray(logits, np.float64))
    return np.argmax(l, axis=1).astype(np.int64)  # first occurrence of the maximum


def logsumexp(logits) -> np.ndarray:
    """log sum_v exp(l_v) per row, with the maximum taken out first."""
    l = np.atleast_2d(np.asarray(logits, np.float64))
    m = l.max(axis=1, keepdims=True)
    return (m + np.log(np.exp(l - m).sum(axis=1, keepdims=True)))[:, 0]


def top_k_cdf(logits_row, k: int, temperature: float):
    """The k candidates of top-k sampling in draw order (logit descending, id
    ascending among equal logits) and their cumulative weights divided by the
    total: candidate j is drawn for u in [cdf[j-1], cdf[j])."""
    l = np.asarray(logits_row, np.float64).reshape(-1)
    if temperature <= 0:
        raise ValueError("temperature must be positive")
    k = max(1, min(int(k), l.size))
    order = np.lexsort((np.arange(l.size), -l))[:k]  # sort by -l, then by id
    w = np.exp((l[order] - l[order[0]]) / temperature)
    c = np.cumsum(w)
    return order.astype(np.int64), c / c[-1]


def sample_top_k(logits, k: int, temperature: float, u) -> np.ndarray:
    """Top-k sampling (primer §1.2 `sample`) by inverse CDF with one uniform
    u in [0, 1) per sequence; k <= 1 is greedy decoding.  logits: [B, V].
    Returns int64 [B]."""
    l = np.atleast_2d(np.asarray(logits, np.float64))
    u = np.asarray(u, np.float64).reshape(-1)
    if k <= 1:
        return greedy_token(l)
    out = np.empty(l.shape[0], np.int64)
    for b in range(l.shape[0]):
        ids, cdf = top_k_cdf(l[b], k, temperature)
        j = int(np.searchsorted(cdf, u[b], side="right"))  # first j with cdf[j] > u
        out[b] = ids[min(j, ids.size - 1)]
    return out


def layer_decode_ragged(shape, layer: dict, kc, vc, pos, x, stages: bool = False):
    """One decode step of one layer for B sequences each at its own position
    pos[b] (the primer's §1.2 decode_step per sequence; §1.3 batching of
    sequences of different lengths): sequence b is the plain step on its own
    cache, its own input row and its position, independently of the others.

    kc, vc: uint16 [B, H_kv, s_max, hd], slot pos[b] of sequence b written in
    place.  x: fp64 [B, D].  Returns z [B, D] (and the per-sequence stage
    outputs stacked, as layer_decode)."""
    x = np.atleast_2d(np.asarray(x, np.float64))
    B = x.shape[0]
    pos = [int(p) for p in pos]
    zs, sts = [], []
    for b in range(B):
        kb = np.ascontiguousarray(kc[b:b + 1])
        vb = np.ascontiguousarray(vc[b:b + 1])
        r = layer_decode(shape, layer, kb, vb, pos[b], x[b:b + 1], stages=stages)
        kc[b:b + 1] = kb
        vc[b:b + 1] = vb
        if stages:
            zs.append(r[0])
            sts.append(r[1])
        else:
            zs.append(r)
    z = np.concatenate(zs)
    if not stages:
        return z
    return z, {k: np.concatenate([s[k] for s in sts]) for k in sts[0]}


def paged_gather(pool, table, page_size: int, b: int, n: int):
    """The first n logical slots of sequence b from a paged cache: slot t sits
    in physical page table[b][t // page_size] at row t % page_size.
    pool: [pages, H_kv, page_size, hd]; returns [1, H_kv, n, hd] (a copy)."""
    H, hd = pool.shape[1], pool.shape[3]
    out = np.empty((1, H, n, hd), pool.dtype)
    for t in range(n):
        out[0, :, t] = pool[int(table[b][t // page_size]), :, t % page_size]
    return out


def layer_decode_paged(shape, layer: dict, kpool, vpool, table, page_size: int, pos, x, stages: bool = False):
    """One decode step of one layer for B sequences at their own positions
    whose caches are paged (the primer's §1.3 continuous batching with the
    cache kept in fixed-size pages): sequence b's logical slots 0 .. pos[b]
    are gathered through its page-table row, the plain step runs on them,
    and its new K/V row goes back to logical slot pos[b], i.e. physical page
    table[b][pos[b] // page_size], row pos[b] % page_size.

    kpool, vpool: uint16 [pages, H_kv, page_size, hd], written in place at
    the new slots only.  table: [B][>= pos[b] // page_size + 1] page ids.
    x: fp64 [B, D].  Returns z [B, D] (and the stacked stages)."""
    x = np.atleast_2d(np.asarray(x, np.float64))
    pos = [int(p) for p in pos]
    zs, sts = [], []
    for b in range(x.shape[0]):
        n = pos[b] + 1
        kb = paged_gather(kpool, table, page_size, b, n)
        vb = paged_gather(vpool, table, page_size, b, n)
        r = layer_decode(shape, layer, kb, vb, pos[b], x[b:b + 1], stages=stages)
        pg, row = int(table[b][pos[b] // page_size]), pos[b] % page_size
        kpool[pg, :, row] = kb[0, :, pos[b]]
        vpool[pg, :, row] = vb[0, :, pos[b]]
        if stages:
            zs.append(r[0])
            sts.append(r[1])
        else:
            zs.append(r)
    z = np.concatenate(zs)
    if not stages:
        return z
    return z, {k: np.concatenate([s[k] for s in sts]) for k in sts[0]}


def layer_prefill(shape, layer: dict, kc, vc, p0: int, x, stages: bool = False):
    """S prompt tokens of one sequence through one layer (the primer's §1.2
    prefill, its K/V kept in the cache): row i is the token at position
    p0 + i and sees the history and the rows before it.  Causality makes it
    the plain decode step row after row on the one cache: row i appends slot
    p0 + i before row i + 1 attends.

    kc, vc: uint16 [1, H_kv, s_max, hd], slots p0 .. p0 + S - 1 written in
    place.  x: fp64 [S, D].  Returns z [S, D] (and the rows' stages)."""
    x = np.atleast_2d(np.asarray(x, np.float64))
    zs, sts = [], []
    for i in range(x.shape[0]):
        r = layer_decode(shape, layer, kc, vc, int(p0) + i, x[i:i + 1], stages=stages)
        if stages:
            zs.append(r[0])
            sts.append(r[1])
        else:
            zs.append(r)
    z = np.concatenate(zs)
    if not stages:
        return z
    return z, {k: np.concatenate([s[k] for s in sts]) for k in sts[0]}
