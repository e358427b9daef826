"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a library
routine (PyTorch's bf16 conversion, rms_norm, scaled_dot_product_attention,
numpy matmul, complex multiplication), a closed form, an invariant, a
hand-derived example, or brute force.  A plausible slip anywhere in the
oracle (a dropped term, a wrong sign or index, a transposed operand, a wrong
nibble order or rounding rule) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from memory_bound_transformer_decode_gb300 import configs, synth

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------ bf16


def _torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_bf16_matches_torch_on_fp32_values():
    # fp32 inputs: one rounding of the exact value == PyTorch's RNE conversion.
    x = np.concatenate([
        RNG.standard_normal(20000).astype(np.float32),
        (RNG.standard_normal(2000) * 1e-39).astype(np.float32),  # subnormals
        (RNG.standard_normal(2000) * 1e38).astype(np.float32),
        # exact ties: bf16 value + half an ulp
        (np.arange(1, 300, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        (np.arange(1, 300, dtype=np.uint32) << 16 | 0x18000).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 3.39e38, 3.40e38, -1.0e-45], np.float32),
    ])
    got = oracle.bf16_from_f64(x.astype(np.float64))
    want = _torch_bf16_bits(x)
    np.testing.assert_array_equal(got, want)
    assert oracle.bf16_from_f64(np.array([np.nan]))[0] & 0x7FFF > 0x7F80


def test_bf16_is_nearest_even_on_fp64_values():
    # brute force against the two bf16 neighbours of each fp64 value
    x = RNG.standard_normal(5000) * np.exp(RNG.uniform(-20, 20, 5000))
    b = oracle.bf16_from_f64(x).astype(np.int64)
    for xi, bi in zip(x[:2000], b[:2000]):
        mag = bi & 0x7FFF
        cands = [c for c in (mag - 1, mag, mag + 1) if 0 <= c < 0x7F80]
        vals = [abs(abs(xi) - oracle.bf16_to_f64(np.array([c], np.uint16))[0]) for c in cands]
        best = min(vals)
        ties = [c for c, v in zip(cands, vals) if v == best]
        assert mag in ties
        if len(ties) > 1:
            assert mag % 2 == 0
        assert (bi >> 15) == (1 if xi < 0 else 0)


def test_bf16_widening_exact():
    bits = np.arange(0, 65536, 97, dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_to_f64(bits)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])


# ------------------------------------------------------------------ INT4


def _bits_of(vals) -> np.ndarray:
    return _torch_bf16_bits(np.asarray(vals, np.float32))


def _numpy_codes(q: np.ndarray) -> np.ndarray:
    lo = (q & 0xF).astype(np.int16)
    hi = (q >> 4).astype(np.int16)
    codes = np.stack([lo, hi], axis=-1).reshape(q.shape[0], -1)
    return np.where(codes >= 8, codes - 16, codes).astype(np.int8)


def test_quantize_hand_example():
    # absmax 1.75 -> s = 1.75 / 7 = 0.25 exactly; codes by round-half-even.
    w = np.zeros((1, 64), np.float32)
    vals = {0: 0.125, 1: 0.375, 2: 0.625, 3: -0.625, 4: 1.75, 5: -1.75, 6: 0.3, 7: -0.0}
    for k, v in vals.items():
        w[0, k] = v
    q, s = oracle.quantize_int4(_bits_of(w))
    assert oracle.bf16_to_f64(s)[0, 0] == 0.25
    # 0.5 -> 0 (tie to even), 1.5 -> 2, 2.5 -> 2, -2.5 -> -2, 7, -7, 1.2 -> 1
    want_codes = [0, 2, 2, -2, 7, -7, 1, 0]
    assert list(_numpy_codes(q)[0, :8]) == want_codes
    # low nibble first: byte0 = codes (0, 2) -> 0x20; byte1 = (2, -2) -> 0xE2;
    # byte2 = (7, -7) -> 0x97; byte3 = (1, 0) -> 0x01
    assert list(q[0, :4]) == [0x20, 0xE2, 0x97, 0x01]


def test_quantize_zero_group_and_single_value():
    w = np.zeros((2, 128), np.float32)
    w[1, 70] = -0.0371
    q, s = oracle.quantize_int4(_bits_of(w))
    assert s[0, 0] == 0 and s[0, 1] == 0 and s[1, 0] == 0 and np.all(q[0] == 0)
    codes = _numpy_codes(q)
    assert codes[1, 70] == -7 and np.count_nonzero(codes[1]) == 1
    wb = oracle.bf16_to_f64(_bits_of([-0.0371]))[0]
    want_s = oracle.bf16_to_f64(_bits_of([abs(wb) / 7]))[0]
    assert oracle.bf16_to_f64(s)[1, 1] == want_s


def test_quantize_reproduces_integer_multiples():
    c = RNG.integers(-7, 8, size=(5, 256))
    c[:, ::64] = 7  # each group reaches the clamp value, so s = 2^-5 exactly
    w = c.astype(np.float32) * 2.0 ** -5
    q, s = oracle.quantize_int4(_bits_of(w))
    np.testing.assert_array_equal(oracle.bf16_to_f64(s), 2.0 ** -5)
    np.testing.assert_array_equal(_numpy_codes(q), c)


def test_quantize_error_bound_and_range():
    w_bits = synth.bits(synth.normal_bf16((64, 512), seed=7, std=0.02))
    q, s = oracle.quantize_int4(w_bits)
    codes = _numpy_codes(q).astype(np.float64)
    assert codes.min() >= -7 and codes.max() <= 7
    sd = np.repeat(oracle.bf16_to_f64(s), 64, axis=1)
    w = oracle.bf16_to_f64(w_bits)
    err = np.abs(w - codes * sd)
    inside = np.abs(w) <= 7 * sd
    assert np.all(err[inside] <= sd[inside] / 2 * (1 + 1e-12))
    # outside (scale rounded down): only the clamp error, at most one step
    assert np.all(err[~inside] <= sd[~inside] * 1.01)
    np.testing.assert_array_equal(oracle.unpack_int4(q), _numpy_codes(q))


def test_quantize_brute_force_tiny():
    w_bits = synth.bits(synth.normal_bf16((2, 64), seed=11, std=0.02))
    q, s = oracle.quantize_int4(w_bits)
    w = oracle.bf16_to_f64(w_bits)
    codes = _numpy_codes(q)
    for n in range(2):
        sv = oracle.bf16_to_f64(s[n:n + 1])[0]
        # brute force: the code minimising |w - c s| over c in [-7, 7], ties to even
        for k in range(64):
            errs = [abs(w[n, k] - c * sv) for c in range(-7, 8)]
            best = min(errs)
            allowed = [c for c, e in zip(range(-7, 8), errs) if e == best]
            if len(allowed) > 1:
                allowed = [c for c in allowed if c % 2 == 0]
            assert codes[n, k] in allowed


# ------------------------------------------------------------------ GEMV


@pytest.mark.parametrize("N,K", [(1, 64), (3, 128), (7, 192), (5, 64)])
def test_gemv_int4_vs_numpy_matmul(N, K):
    w_bits = synth.bits(synth.normal_bf16((N, K), seed=N * 100 + K, std=0.02))
    q, s = oracle.quantize_int4(w_bits)
    x = RNG.standard_normal(K)
    W = _numpy_codes(q).astype(np.float64) * np.repeat(oracle.bf16_to_f64(s), 64, axis=1)
    np.testing.assert_allclose(oracle.gemv_int4(q, s, x), W @ x, rtol=1e-12, atol=1e-14)
    Wb = oracle.bf16_to_f64(w_bits)
    np.testing.assert_allclose(oracle.gemv_bf16(w_bits, x), Wb @ x, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ RMSNorm


def test_rmsnorm_unit_weight_and_scale_invariance():
    x = RNG.standard_normal(512) * 3.0
    one = _bits_of(np.ones(512))
    h = oracle.rmsnorm(x, one, 0.0)
    assert abs(math.sqrt(np.mean(h * h)) - 1.0) < 1e-14
    np.testing.assert_allclose(oracle.rmsnorm(17.5 * x, one, 0.0), h, rtol=1e-13)
    eps = 0.25
    ms = np.mean(x * x)
    assert abs(math.sqrt(np.mean(oracle.rmsnorm(x, one, eps) ** 2)) - math.sqrt(ms / (ms + eps))) < 1e-13


def test_rmsnorm_vs_torch():
    x = RNG.standard_normal(640)
    w_bits = synth.bits(synth.normal_bf16((640,), seed=3, mean=1.0, std=0.1))
    w = torch.from_numpy(oracle.bf16_to_f64(w_bits))
    want = F.rms_norm(torch.from_numpy(x), (640,), weight=w, eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rmsnorm(x, w_bits, 1e-6), want, rtol=1e-13)


# ------------------------------------------------------------------ RoPE


def test_rope_invariants():
    hd, base = 128, 1e6
    q, k = RNG.standard_normal(hd), RNG.standard_normal(hd)
    np.testing.assert_array_equal(oracle.rope(q, 0, base), q)
    for p in (1, 77, 8192, 32768):
        assert abs(np.linalg.norm(oracle.rope(q, p, base)) - np.linalg.norm(q)) < 1e-12
    # <R(m) q, R(n) k> depends only on m - n
    d0 = oracle.rope(q, 100, base) @ oracle.rope(k, 37, base)
    d1 = oracle.rope(q, 5063, base) @ oracle.rope(k, 5000, base)
    assert abs(d0 - d1) < 1e-9


def test_rope_vs_complex_rotation():
    # pair (i, i + hd/2) as a complex number times exp(i * p * theta_i)
    hd, p, base = 64, 128, 1e4
    v = RNG.standard_normal(hd)
    z = v[: hd // 2] + 1j * v[hd // 2:]
    theta = np.power(base, -np.arange(0, hd, 2, dtype=np.float64) / hd)
    zr = z * np.exp(1j * p * theta)
    got = oracle.rope(v, p, base)
    np.testing.assert_allclose(got[: hd // 2], zr.real, atol=1e-12)
    np.testing.assert_allclose(got[hd // 2:], zr.imag, atol=1e-12)
    # hd = 2: a single pair rotated by exactly p radians
    np.testing.assert_allclose(oracle.rope([1.0, 0.0], 1, base), [math.cos(1), math.sin(1)],
                               atol=1e-15)


# ------------------------------------------------------------------ attention


def _cache(Hkv, s_max, hd, seed):
    return synth.bits(synth.normal_bf16((Hkv, s_max, hd), seed=seed))


def test_attention_single_key_returns_v():
    q = RNG.standard_normal((4, 64))
    kc, vc = _cache(2, 10, 64, 1), _cache(2, 10, 64, 2)
    o = oracle.attention(q, kc, vc, 1)
    v0 = oracle.bf16_to_f64(vc[:, 0])
    np.testing.assert_array_equal(o, np.repeat(v0, 2, axis=0))


def test_attention_equal_keys_give_mean_of_v_and_probs_sum_to_one():
    q = RNG.standard_normal((8, 64))
    kc = np.repeat(_cache(2, 1, 64, 3), 33, axis=1)
    vc = _cache(2, 33, 64, 4)
    o, p = oracle.attention(q, kc, vc, 33, return_probs=True)
    np.testing.assert_allclose(p, 1.0 / 33, rtol=1e-13)
    mean_v = oracle.bf16_to_f64(vc).mean(axis=1)
    np.testing.assert_allclose(o, np.repeat(mean_v, 4, axis=0), rtol=1e-12, atol=1e-15)
    q2 = RNG.standard_normal((8, 64)) * 4
    _, p2 = oracle.attention(q2, _cache(2, 50, 64, 5), vc.repeat(2, axis=1)[:, :50], 50,
                             return_probs=True)
    np.testing.assert_allclose(p2.sum(axis=1), 1.0, rtol=1e-13)


def test_attention_gqa_equals_mha_with_repeated_heads():
    Hq, Hkv, hd, n = 8, 2, 64, 40
    q = RNG.standard_normal((Hq, hd))
    kc, vc = _cache(Hkv, n, hd, 6), _cache(Hkv, n, hd, 7)
    gqa = oracle.attention(q, kc, vc, n)
    mha = oracle.attention(q, np.repeat(kc, Hq // Hkv, axis=0), np.repeat(vc, Hq // Hkv, axis=0), n)
    np.testing.assert_array_equal(gqa, mha)


def test_attention_vs_torch_sdpa():
    Hq, Hkv, hd, s_max, n = 7, 1, 128, 300, 257
    q = RNG.standard_normal((Hq, hd)) * 2
    kc, vc = _cache(Hkv, s_max, hd, 8), _cache(Hkv, s_max, hd, 9)
    K = torch.from_numpy(oracle.bf16_to_f64(kc[:, :n]))
    V = torch.from_numpy(oracle.bf16_to_f64(vc[:, :n]))
    want = F.scaled_dot_product_attention(
        torch.from_numpy(q)[:, None, :], K.repeat_interleave(Hq // Hkv, 0),
        V.repeat_interleave(Hq // Hkv, 0))[:, 0].numpy()
    np.testing.assert_allclose(oracle.attention(q, kc, vc, n), want, rtol=1e-11, atol=1e-13)


# ------------------------------------------------------------------ layer

TINY = configs.DecodeConfig("tiny", D=128, H_q=4, H_kv=2, head_dim=32, d_ff=192,
                            rope_base=1e4, kv_len=20, layers=1, batch=2, seed=5)


def _torch_layer(cfg, w, kc_bits, vc_bits, pos, x):
    """The decode layer composed from PyTorch library routines in fp64."""
    def dq(m):
        codes = torch.from_numpy(_numpy_codes(m.q).astype(np.float64))
        sc = torch.from_numpy(np.repeat(oracle.bf16_to_f64(m.s), 64, axis=1))
        return codes * sc

    def rope(t, hd):  # t [..., hd]: complex rotation of pairs (i, i + hd/2)
        theta = torch.pow(torch.tensor(cfg.rope_base, dtype=torch.float64),
                          -torch.arange(0, hd, 2, dtype=torch.float64) / hd)
        z = torch.complex(t[..., : hd // 2], t[..., hd // 2:]) * torch.polar(
            torch.ones_like(theta), pos * theta)
        return torch.cat([z.real, z.imag], dim=-1)

    n1 = torch.from_numpy(oracle.bf16_to_f64(w["norm1"]))
    n2 = torch.from_numpy(oracle.bf16_to_f64(w["norm2"]))
    hd, B = cfg.head_dim, x.shape[0]
    xt = torch.from_numpy(x)
    h = F.rms_norm(xt, (cfg.D,), weight=n1, eps=cfg.eps)
    q = (h @ dq(w["wq"]).T).view(B, cfg.H_q, hd)
    k = (h @ dq(w["wk"]).T).view(B, cfg.H_kv, hd)
    v = (h @ dq(w["wv"]).T).view(B, cfg.H_kv, hd)
    q, k = rope(q, hd), rope(k, hd)
    kb = torch.from_numpy(oracle.bf16_to_f64(kc_bits)).clone()
    vb = torch.from_numpy(oracle.bf16_to_f64(vc_bits)).clone()
    kb[:, :, pos] = k.to(torch.bfloat16).to(torch.float64)
    vb[:, :, pos] = v.to(torch.bfloat16).to(torch.float64)
    att = F.scaled_dot_product_attention(q[:, :, None, :], kb[:, :, : pos + 1],
                                         vb[:, :, : pos + 1], enable_gqa=True)
    att = att[:, :, 0, :].reshape(B, -1)
    y = xt + att @ dq(w["wo"]).T
    h2 = F.rms_norm(y, (cfg.D,), weight=n2, eps=cfg.eps)
    a = F.silu(h2 @ dq(w["wg"]).T) * (h2 @ dq(w["wu"]).T)
    return (y + a @ dq(w["wd"]).T).numpy(), att.numpy()


def _tiny_inputs(cfg, s_max):
    wb = {k: synth.bits(v) for k, v in synth.layer_weights(cfg, 0).items()}
    kc, vc = synth.kv_cache(cfg, 0, s_max)
    x = synth.bits(synth.input_x(cfg))
    return wb, synth.bits(kc), synth.bits(vc), oracle.bf16_to_f64(x)


@pytest.mark.parametrize("cfg", [TINY, configs.SMALL_LAYER])
def test_layer_vs_torch_composition(cfg):
    s_max = cfg.kv_len + 3
    wb, kc, vc, x = _tiny_inputs(cfg, s_max)
    lw = oracle.quantized_layer(wb)
    want, want_att = _torch_layer(cfg, lw, kc, vc, cfg.pos, x)
    kc2, vc2 = kc.copy(), vc.copy()
    z, st = oracle.layer_decode(cfg, lw, kc2, vc2, cfg.pos, x, stages=True)
    np.testing.assert_allclose(z, want, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(st["attn"], want_att, rtol=1e-10, atol=1e-12)
    # only slot pos changed in the cache, and it holds bf16(k), bf16(v)
    changed = np.argwhere(kc2 != kc)
    assert set(changed[:, 2]) <= {cfg.pos}
    np.testing.assert_array_equal(kc2[:, :, cfg.pos].reshape(cfg.batch, -1),
                                  oracle.bf16_from_f64(st["k"]))
    np.testing.assert_array_equal(vc2[:, :, cfg.pos].reshape(cfg.batch, -1),
                                  oracle.bf16_from_f64(st["v"]))


def test_layer_bf16_weights_vs_int4_path_structure():
    cfg = TINY
    wb, kc, vc, x = _tiny_inputs(cfg, cfg.kv_len + 1)
    z_b = oracle.layer_decode(cfg, oracle.bf16_layer(wb), kc.copy(), vc.copy(), cfg.pos, x)
    z_q = oracle.layer_decode(cfg, oracle.quantized_layer(wb), kc.copy(), vc.copy(), cfg.pos, x)
    # INT4 quantization noise is small but not zero on this random layer
    rel = np.linalg.norm(z_q - z_b) / np.linalg.norm(z_b)
    assert 1e-5 < rel < 5e-2


def test_layer_residual_identity():
    # Wo = 0 and Wd = 0 (all-zero groups quantize to s = 0): z == x exactly
    cfg = TINY
    wb, kc, vc, x = _tiny_inputs(cfg, cfg.kv_len + 1)
    wb["wo"] = np.zeros_like(wb["wo"])
    wb["wd"] = np.zeros_like(wb["wd"])
    z = oracle.layer_decode(cfg, oracle.quantized_layer(wb), kc, vc, cfg.pos, x)
    np.testing.assert_array_equal(z, x)


def test_layer_zero_norm_gives_uniform_attention():
    # norm1 = 0 -> h = 0 -> q = k = v = 0: every score is 0, so attention is the
    # mean of V over slots 0..pos with the new (zero) row included
    cfg = TINY
    wb, kc, vc, x = _tiny_inputs(cfg, cfg.kv_len + 1)
    wb["norm1"] = np.zeros_like(wb["norm1"])
    _, st = oracle.layer_decode(cfg, oracle.quantized_layer(wb), kc, vc, cfg.pos, x, stages=True)
    vhist = oracle.bf16_to_f64(vc[:, :, : cfg.pos])
    mean = vhist.sum(axis=2) / (cfg.pos + 1)  # [B, H_kv, hd]
    want = np.repeat(mean, cfg.group, axis=1).reshape(cfg.batch, -1)
    np.testing.assert_allclose(st["attn"], want, rtol=1e-12, atol=1e-15)
    assert np.all(st["q"] == 0) and np.all(st["k"] == 0)


def test_layer_rejects_bad_position():
    cfg = TINY
    wb, kc, vc, x = _tiny_inputs(cfg, cfg.kv_len)
    with pytest.raises(ValueError):
        oracle.layer_decode(cfg, oracle.quantized_layer(wb), kc, vc, cfg.kv_len, x)


# ------------------------------------------------------------------ token step


def test_embed_is_the_table_rows():
    # hand example: row v of the table holds the bf16 value v + 1 everywhere
    V, D = 5, 64
    table = np.stack([_bits_of(np.full(D, v + 1.0)) for v in range(V)])
    got = oracle.embed(table, [4, 0, 4, 2])
    np.testing.assert_array_equal(oracle.bf16_to_f64(got)[:, 0], [5.0, 1.0, 5.0, 3.0])
    np.testing.assert_array_equal(got[1], table[0])
    for bad in ([-1], [V]):
        with pytest.raises(ValueError):
            oracle.embed(table, bad)


@pytest.mark.parametrize("V,D", [(300, 128), (17, 64)])
@pytest.mark.parametrize("with_norm", [False, True])
def test_lm_head_logits_vs_library_routines(V, D, with_norm):
    # W from the independently unpacked codes times the scales, the norm from
    # torch's rms_norm, the product from numpy's matmul
    w_bits = synth.bits(synth.normal_bf16((V, D), seed=V + D, std=0.02))
    q, s = oracle.quantize_int4(w_bits)
    x = RNG.standard_normal((3, D)) * 7.0
    nw = synth.bits(synth.normal_bf16((D,), seed=5, mean=1.0, std=0.1)) if with_norm else None
    eps = 1e-6
    if with_norm:
        h = F.rms_norm(torch.from_numpy(x), (D,), torch.from_numpy(oracle.bf16_to_f64(nw)), eps).numpy()
    else:
        h = x
    W4 = _numpy_codes(q).astype(np.float64) * np.repeat(oracle.bf16_to_f64(s), 64, axis=1)
    got = oracle.lm_head_logits(x, oracle.OracleMat(q=q, s=s), nw, eps)
    np.testing.assert_allclose(got, h @ W4.T, rtol=1e-10, atol=1e-12)
    gotb = oracle.lm_head_logits(x, oracle.OracleMat(w=w_bits), nw, eps)
    np.testing.assert_allclose(gotb, h @ oracle.bf16_to_f64(w_bits).T, rtol=1e-10, atol=1e-12)


def test_greedy_token_ties_and_brute_force():
    assert oracle.greedy_token([[1.0, 3.0, 3.0, 2.0]])[0] == 1  # lowest id among equal maxima
    assert oracle.greedy_token([[-5.0, -2.0, -9.0]])[0] == 1
    l = RNG.standard_normal((4, 1000))
    for b in range(4):
        best = 0
        for i in range(1000):
            if l[b, i] > l[b, best]:
                best = i
        assert oracle.greedy_token(l)[b] == best


def test_logsumexp_closed_forms_and_scipy():
    scipy_special = pytest.importorskip("scipy.special")
    l = RNG.standard_normal((3, 5000)) * 4.0
    np.testing.assert_allclose(oracle.logsumexp(l), scipy_special.logsumexp(l, axis=1), rtol=1e-14)
    # all equal: c + log V; shift: lse(l + c) = lse(l) + c (no overflow at 1e3)
    np.testing.assert_allclose(oracle.logsumexp(np.full((1, 152064), 2.5)), 2.5 + math.log(152064), rtol=1e-14)
    np.testing.assert_allclose(oracle.logsumexp(l + 1000.0), oracle.logsumexp(l) + 1000.0, rtol=1e-14)
    assert oracle.logsumexp([[7.25]])[0] == 7.25


def test_top_k_candidates_and_order():
    l = np.array([5.0, 2.0, 2.0, 2.0, 1.0, 6.0])
    ids, cdf = oracle.top_k_cdf(l, 3, 1.0)
    np.testing.assert_array_equal(ids, [5, 0, 1])  # descending; the tie at the boundary takes the lower id
    w = np.exp(np.array([6.0, 5.0, 2.0]) - 6.0)
    np.testing.assert_allclose(cdf, np.cumsum(w) / w.sum(), rtol=1e-15)
    ids, _ = oracle.top_k_cdf(l, 100, 1.0)  # k beyond V: every id
    np.testing.assert_array_equal(ids, [5, 0, 1, 2, 3, 4])
    r = RNG.standard_normal(2000)
    ids, _ = oracle.top_k_cdf(r, 50, 0.7)
    np.testing.assert_array_equal(np.sort(ids), np.sort(np.argsort(-r)[:50]))


def test_sample_top_k_special_cases():
    l = RNG.standard_normal((2, 3000)) * 2.0
    g = oracle.greedy_token(l)
    for u in (0.0, 0.3, 0.999):
        np.testing.assert_array_equal(oracle.sample_top_k(l, 1, 1.0, [u, u]), g)  # k = 1: greedy
    np.testing.assert_array_equal(oracle.sample_top_k(l, 40, 1.0, [0.0, 0.0]), g)  # u = 0: the largest
    last = [oracle.top_k_cdf(l[b], 40, 1.0)[0][-1] for b in range(2)]
    np.testing.assert_array_equal(oracle.sample_top_k(l, 40, 1.0, [1 - 1e-15] * 2), last)
    # a tiny temperature is greedy; a huge one is uniform over the k candidates
    np.testing.assert_array_equal(oracle.sample_top_k(l, 40, 1e-6, [0.9, 0.9]), g)
    ids, cdf = oracle.top_k_cdf(l[0], 8, 1e9)
    np.testing.assert_allclose(cdf, np.arange(1, 9) / 8.0, rtol=1e-8)
    # candidate j is drawn for u in [cdf[j-1], cdf[j]): at u = 1/2 exactly, two
    # equal logits give the second candidate
    two = np.array([[0.0, 0.0, -50.0]])
    assert oracle.sample_top_k(two, 2, 1.0, [0.5])[0] == 1
    assert oracle.sample_top_k(two, 2, 1.0, [0.5 - 2 ** -53])[0] == 0


def test_sample_top_k_frequencies_match_softmax():
    # draws at the midpoints of a fine grid of u land on each candidate in
    # proportion to its softmax weight over the top k (scipy's softmax)
    scipy_special = pytest.importorskip("scipy.special")
    l = RNG.standard_normal(500) * 1.5
    k, T, n = 12, 0.8, 20000
    u = (np.arange(n) + 0.5) / n
    toks = np.array([oracle.sample_top_k(l[None, :], k, T, [ui])[0] for ui in u])
    top = np.argsort(-l)[:k]
    p = scipy_special.softmax(l[top] / T)
    for j, v in enumerate(top):
        assert abs(np.count_nonzero(toks == v) / n - p[j]) <= 1.0 / n + 1e-12
    assert set(np.unique(toks)) <= set(top.tolist())


# ------------------------------------------------------------------ sequences at their own positions


def _small_batch(B, S):
    cfg = configs.SMALL_LAYER.with_(kv_len=S)
    w = {k: synth.bits(v) for k, v in synth.layer_weights(cfg, 0).items()}
    lw = oracle.quantized_layer(w)
    kc, vc = (synth.bits(t).copy() for t in synth.kv_cache(cfg, 0, S + 1, batch=B))
    x = oracle.bf16_to_f64(synth.bits(synth.input_x(cfg, batch=B)))
    return cfg, lw, kc, vc, x


def test_ragged_equal_positions_is_the_batched_step():
    cfg, lw, kc, vc, x = _small_batch(3, 40)
    k1, v1, k2, v2 = kc.copy(), vc.copy(), kc.copy(), vc.copy()
    z1, s1 = oracle.layer_decode(cfg, lw, k1, v1, 40, x, stages=True)
    z2, s2 = oracle.layer_decode_ragged(cfg, lw, k2, v2, [40, 40, 40], x, stages=True)
    np.testing.assert_array_equal(z1, z2)
    for k in s1:
        np.testing.assert_array_equal(s1[k], s2[k])
    np.testing.assert_array_equal(k1, k2)
    np.testing.assert_array_equal(v1, v2)


def test_ragged_sequences_are_independent_and_ignore_slots_past_their_position():
    cfg, lw, kc, vc, x = _small_batch(3, 40)
    pos = [0, 17, 40]
    z = oracle.layer_decode_ragged(cfg, lw, kc.copy(), vc.copy(), pos, x)
    # junk in the slots past each position changes nothing
    kj, vj = kc.copy(), vc.copy()
    for b, p in enumerate(pos):
        kj[b, :, p + 1:] = 0x7F7F  # a large bf16 value
        vj[b, :, p + 1:] = 0xFF7F
    zj = oracle.layer_decode_ragged(cfg, lw, kj, vj, pos, x)
    np.testing.assert_array_equal(z, zj)
    # moving sequence 1 changes only sequence 1
    z2 = oracle.layer_decode_ragged(cfg, lw, kc.copy(), vc.copy(), [0, 30, 40], x)
    np.testing.assert_array_equal(z[[0, 2]], z2[[0, 2]])
    assert not np.array_equal(z[1], z2[1])


# ------------------------------------------------------------------ paged KV cache


def _pages_of(cache, ps):
    """A contiguous cache [B, H, s_max, hd] as pages [B * s_max / ps, H, ps, hd],
    sequence b's logical page j at physical page b * (s_max / ps) + j (a
    reshape and a transpose, no loop)."""
    B, H, S, hd = cache.shape
    return np.ascontiguousarray(cache.reshape(B, H, S // ps, ps, hd).transpose(0, 2, 1, 3, 4)).reshape(-1, H, ps, hd)


def _paged_case(B=3, s_max=64):
    cfg = configs.SMALL_LAYER.with_(kv_len=s_max - 1)
    w = {k: synth.bits(v) for k, v in synth.layer_weights(cfg, 0).items()}
    lw = oracle.quantized_layer(w)
    kc, vc = (synth.bits(t).copy() for t in synth.kv_cache(cfg, 0, s_max, batch=B))
    x = oracle.bf16_to_f64(synth.bits(synth.input_x(cfg, batch=B)))
    return cfg, lw, kc, vc, x


@pytest.mark.parametrize("ps", [16, 32])
def test_paged_identity_layout_is_the_ragged_step(ps):
    cfg, lw, kc, vc, x = _paged_case()
    pos = [0, 33, 63]
    npg = kc.shape[2] // ps
    table = np.arange(3 * npg).reshape(3, npg)
    kp, vp = _pages_of(kc, ps), _pages_of(vc, ps)
    z, st = oracle.layer_decode_paged(cfg, lw, kp, vp, table, ps, pos, x, stages=True)
    z2, st2 = oracle.layer_decode_ragged(cfg, lw, kc, vc, pos, x, stages=True)
    np.testing.assert_array_equal(z, z2)
    for k in st:
        np.testing.assert_array_equal(st[k], st2[k])
    # the new rows landed where the contiguous step put them, nothing else moved
    np.testing.assert_array_equal(kp, _pages_of(kc, ps))
    np.testing.assert_array_equal(vp, _pages_of(vc, ps))


def test_paged_permuted_pages_with_junk_pages():
    cfg, lw, kc, vc, x = _paged_case()
    ps, pos = 16, [5, 47, 16]
    npg = kc.shape[2] // ps
    kp0, vp0 = _pages_of(kc, ps), _pages_of(vc, ps)
    rng = np.random.default_rng(5)
    n_phys = 3 * npg + 7  # 7 pages nobody owns, full of junk
    perm = rng.permutation(n_phys)[: 3 * npg]  # logical page (b, j) -> physical page
    kp = np.full((n_phys,) + kp0.shape[1:], 0x7F7F, np.uint16)
    vp = np.full((n_phys,) + vp0.shape[1:], 0xFF7F, np.uint16)
    kp[perm], vp[perm] = kp0, vp0
    table = perm.reshape(3, npg)
    kpb, vpb = kp.copy(), vp.copy()
    z = oracle.layer_decode_paged(cfg, lw, kp, vp, table, ps, pos, x)
    z2 = oracle.layer_decode_ragged(cfg, lw, kc, vc, pos, x)
    np.testing.assert_array_equal(z, z2)
    np.testing.assert_array_equal(kp[perm], _pages_of(kc, ps))
    np.testing.assert_array_equal(vp[perm], _pages_of(vc, ps))
    junk = np.setdiff1d(np.arange(n_phys), perm)
    np.testing.assert_array_equal(kp[junk], kpb[junk])
    np.testing.assert_array_equal(vp[junk], vpb[junk])
    # exactly one row of one page per sequence changed
    diff = np.argwhere((kp != kpb).any(axis=(1, 3)))
    assert sorted(map(tuple, diff)) == sorted((int(table[b][p // ps]), p % ps) for b, p in enumerate(pos))


def test_paged_shared_prefix_pages():
    """Two sequences whose first two pages are one physical copy read the same
    history as two sequences holding it twice."""
    cfg, lw, kc, vc, x = _paged_case(B=2)
    ps, pos = 16, [40, 50]
    kc[1, :, : 2 * ps] = kc[0, :, : 2 * ps]  # the contiguous reference: prefix duplicated
    vc[1, :, : 2 * ps] = vc[0, :, : 2 * ps]
    kp0, vp0 = _pages_of(kc, ps), _pages_of(vc, ps)  # 4 pages per sequence
    keep = [0, 1, 2, 3, 6, 7]  # sequence 1's first two pages dropped: it reads sequence 0's
    kp, vp = kp0[keep].copy(), vp0[keep].copy()
    table = np.array([[0, 1, 2, 3], [0, 1, 4, 5]])
    z = oracle.layer_decode_paged(cfg, lw, kp, vp, table, ps, pos, x)
    z2 = oracle.layer_decode_ragged(cfg, lw, kc, vc, pos, x)
    np.testing.assert_array_equal(z, z2)


# ------------------------------------------------------------------ prefill


def _torch_prefill(cfg, w, kc_bits, vc_bits, p0, x):
    """A prefill layer from PyTorch routines in fp64: all rows at once, RoPE at
    positions p0 + i, the new K/V rows rounded to bf16, one attention call
    with a causal mask over the history and the prompt."""
    def dq(m):
        codes = torch.from_numpy(_numpy_codes(m.q).astype(np.float64))
        sc = torch.from_numpy(np.repeat(oracle.bf16_to_f64(m.s), 64, axis=1))
        return codes * sc

    S, hd = x.shape[0], cfg.head_dim
    posn = torch.arange(p0, p0 + S, dtype=torch.float64)

    def rope(t):  # t [S, H, hd]
        theta = torch.pow(torch.tensor(cfg.rope_base, dtype=torch.float64),
                          -torch.arange(0, hd, 2, dtype=torch.float64) / hd)
        ang = posn[:, None, None] * theta[None, None, :]
        z = torch.complex(t[..., : hd // 2], t[..., hd // 2:]) * torch.polar(torch.ones_like(ang), ang)
        return torch.cat([z.real, z.imag], dim=-1)

    xt = torch.from_numpy(x)
    h = F.rms_norm(xt, (cfg.D,), weight=torch.from_numpy(oracle.bf16_to_f64(w["norm1"])), eps=cfg.eps)
    q = rope((h @ dq(w["wq"]).T).view(S, cfg.H_q, hd))
    k = rope((h @ dq(w["wk"]).T).view(S, cfg.H_kv, hd))
    v = (h @ dq(w["wv"]).T).view(S, cfg.H_kv, hd)
    kb = torch.from_numpy(oracle.bf16_to_f64(kc_bits))[0, :, :p0].clone()  # [H_kv, p0, hd]
    vb = torch.from_numpy(oracle.bf16_to_f64(vc_bits))[0, :, :p0].clone()
    kk = torch.cat([kb, k.to(torch.bfloat16).to(torch.float64).transpose(0, 1)], dim=1)
    vv = torch.cat([vb, v.to(torch.bfloat16).to(torch.float64).transpose(0, 1)], dim=1)
    mask = torch.arange(p0 + S)[None, :] <= (p0 + torch.arange(S))[:, None]  # row i sees keys <= p0 + i
    att = F.scaled_dot_product_attention(q.transpose(0, 1)[None], kk[None], vv[None], attn_mask=mask,
                                         enable_gqa=True)
    att = att[0].transpose(0, 1).reshape(S, -1)
    y = xt + att @ dq(w["wo"]).T
    h2 = F.rms_norm(y, (cfg.D,), weight=torch.from_numpy(oracle.bf16_to_f64(w["norm2"])), eps=cfg.eps)
    a = F.silu(h2 @ dq(w["wg"]).T) * (h2 @ dq(w["wu"]).T)
    return (y + a @ dq(w["wd"]).T).numpy()


@pytest.mark.parametrize("p0,S", [(0, 5), (37, 9)])
def test_prefill_vs_causal_torch_composition(p0, S):
    cfg = configs.SMALL_LAYER.with_(kv_len=p0)
    wb = {k: synth.bits(v) for k, v in synth.layer_weights(cfg, 0).items()}
    lw = oracle.quantized_layer(wb)
    kc, vc = (synth.bits(t).copy() for t in synth.kv_cache(cfg, 0, p0 + S + 3, batch=1))
    x = oracle.bf16_to_f64(synth.bits(synth.normal_bf16((S, cfg.D), seed=99)))
    want = _torch_prefill(cfg, lw, kc, vc, p0, x)
    k2, v2 = kc.copy(), vc.copy()
    z = oracle.layer_prefill(cfg, lw, k2, v2, p0, x)
    np.testing.assert_allclose(z, want, rtol=1e-10, atol=1e-10)
    # slots p0 .. p0 + S - 1 written, nothing else
    changed = set(np.argwhere(k2 != kc)[:, 2]) | set(np.argwhere(v2 != vc)[:, 2])
    assert changed <= set(range(p0, p0 + S))
    # causal: a later row's input changes nothing before it
    x2 = x.copy()
    x2[-1] += 1.0
    z2 = oracle.layer_prefill(cfg, lw, kc.copy(), vc.copy(), p0, x2)
    np.testing.assert_array_equal(z2[:-1], z[:-1])
