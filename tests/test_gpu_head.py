"""The token step around the stack on the GPU vs the fp64 oracle, through the
C ABI: embedding rows bit-exact; LM-head logits (INT4 and bf16 output
matrices, with and without the final RMSNorm, ragged vocabularies, batches
1-64) element by element at the step's rel-L2 bar; log-sum-exp; greedy ids
equal wherever the oracle's top-2 gap exceeds the logits' error, else a
near-maximal id; top-k sampling equal to the oracle's draw for uniforms at
the middle of a candidate's CDF interval and valid (within the error margin
of the drawn candidate's interval) for random uniforms; ties at the maximum
and at the top-k boundary resolved to the lower id.
"""
import numpy as np
import pytest
import torch

import oracle
from memory_bound_transformer_decode_gb300 import configs, ddl, synth
from tests.gpu_helpers import REL_L2, rel_l2

pytestmark = pytest.mark.gpu

EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ddl.load(build_if_missing=True)
    yield
    torch.cuda.empty_cache()


class Head:
    """A seeded output matrix on the device (packed) and on the host (oracle)."""

    def __init__(self, D, V, wtype, seed, with_norm=True, table=None):
        cfg = configs.SMALL_LAYER.with_(D=D, seed=seed)
        hw = synth.head_weights(cfg, V, device="cuda")
        self.table = hw["embed"] if table is None else table
        self.norm = hw["norm_f"] if with_norm else None
        self.D, self.V, self.wtype = D, V, wtype
        tb = synth.bits(self.table)
        if wtype == ddl.INT4:
            q, s = ddl.ddl_quantize_int4(self.table)
            self.packed = ddl.ddl_pack_head((q, s), D, V, wtype)
            qo, so = oracle.quantize_int4(tb)
            self.omat = oracle.OracleMat(q=qo, s=so)
            del q, s
        else:
            self.packed = ddl.ddl_pack_head(self.table, D, V, wtype)
            self.omat = oracle.OracleMat(w=tb)
        self.norm_bits = synth.bits(self.norm) if self.norm is not None else None

    def run(self, x, top_k=1, temperature=1.0, u=None):
        B = x.shape[0]
        logits = torch.empty((B, self.V), dtype=torch.float32, device="cuda")
        lse = torch.empty(B, dtype=torch.float32, device="cuda")
        tok = ddl.ddl_lm_head(self.D, self.V, self.wtype, self.packed, x, norm_f=self.norm, eps=EPS,
                              top_k=top_k, temperature=temperature, u=u, logits=logits, lse=lse)
        torch.cuda.synchronize()
        return tok.cpu().numpy(), logits.cpu().numpy().astype(np.float64), lse.cpu().numpy()

    def oracle_logits(self, x):
        return oracle.lm_head_logits(x.cpu().numpy().astype(np.float64), self.omat, self.norm_bits, EPS)


def _x(B, D, seed, std=3.0):
    return synth.normal_bf16((B, D), seed=seed, std=std, device="cuda").float()


def _check_logits_and_greedy(tok, lg, lse, ref):
    assert rel_l2(lg, ref) <= REL_L2 * 1e-2, rel_l2(lg, ref)  # the bar is 2e-3; fp32 reaches ~1e-6
    err = float(np.max(np.abs(lg - ref)))
    np.testing.assert_allclose(lse, oracle.logsumexp(ref), rtol=1e-5, atol=1e-5)
    want = oracle.greedy_token(ref)
    for b in range(ref.shape[0]):
        top2 = np.sort(ref[b])[-2:]
        if top2[1] - top2[0] > 4 * err + 1e-9:
            assert tok[b] == want[b], (b, tok[b], want[b])
        else:  # a near tie: the device's id must be one of the near-maximal ones
            assert ref[b, tok[b]] >= top2[1] - 4 * err - 1e-9
    return err


def test_embed_rows_bit_exact_and_bad_ids():
    D, V = 512, 1000
    table = synth.normal_bf16((V, D), seed=77, std=0.02, device="cuda")
    toks = torch.tensor([3, 999, 0, 3], dtype=torch.int32, device="cuda")
    out = ddl.ddl_embed(table, toks)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(synth.bits(out), oracle.embed(synth.bits(table), [3, 999, 0, 3]))
    bad = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ddl.ddl_embed(table, torch.tensor([-1, V, 5], dtype=torch.int32, device="cuda"), bad=bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == 1
    got = synth.bits(out)
    assert not got[:2].any()
    np.testing.assert_array_equal(got[2], synth.bits(table)[5])
    bad.zero_()
    ddl.ddl_embed(table, toks, bad=bad)
    torch.cuda.synchronize()
    assert int(bad.item()) == 0


@pytest.mark.parametrize("D,V,B,wtype,with_norm", [
    (512, configs.VOCAB, 1, ddl.INT4, True),
    (512, 1000, 3, ddl.INT4, True),        # ragged: 62 tiles + 8 rows
    (512, 4099, 5, ddl.INT4, False),       # ragged, two n-tiles, no final norm
    (512, 20000, 16, ddl.INT4, True),
    (512, 20000, 64, ddl.INT4, True),
    (576, 3001, 2, ddl.BF16, True),        # D not a power of two
    (512, 20000, 33, ddl.BF16, False),
])
def test_head_logits_lse_and_greedy(D, V, B, wtype, with_norm):
    h = Head(D, V, wtype, seed=D + V + B, with_norm=with_norm)
    x = _x(B, D, seed=V + B)
    tok, lg, lse = h.run(x)
    _check_logits_and_greedy(tok, lg, lse, h.oracle_logits(x))


@pytest.mark.parametrize("wtype,B", [(ddl.INT4, 1), (ddl.BF16, 4)])
def test_head_27b_shape_full_vocabulary(wtype, B):
    """D = 5120 (the 27B-class model width) over the 152064-entry vocabulary."""
    h = Head(5120, configs.VOCAB, wtype, seed=2)
    x = _x(B, 5120, seed=21, std=20.0)
    tok, lg, lse = h.run(x)
    err = _check_logits_and_greedy(tok, lg, lse, h.oracle_logits(x))
    print(f"27B-shape head: max |logit error| {err:.2e}")


def test_head_without_logits_output_matches():
    """Greedy ids and log-sum-exp do not depend on asking for the logits."""
    h = Head(512, 20000, ddl.INT4, seed=9)
    x = _x(4, 512, seed=10)
    tok, _, lse = h.run(x)
    lse2 = torch.empty(4, dtype=torch.float32, device="cuda")
    tok2 = ddl.ddl_lm_head(512, 20000, ddl.INT4, h.packed, x, norm_f=h.norm, eps=EPS, lse=lse2)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(tok2.cpu().numpy(), tok)
    np.testing.assert_array_equal(lse2.cpu().numpy(), lse)  # deterministic: same reduction order


def _tied_table(D, V, seed):
    """Rows 40 and 7000 equal and largest for x = 1; rows 100, 200, 300 equal
    and next (x = 1, no final norm: logit = sum of the row)."""
    t = synth.normal_bf16((V, D), seed=seed, std=0.02, device="cuda")
    t[40] = 0.05
    t[7000] = 0.05
    for r in (100, 200, 300):
        t[r] = 0.025
    return t


@pytest.mark.parametrize("wtype", [ddl.INT4, ddl.BF16])
def test_ties_take_the_lower_id(wtype):
    D, V = 512, 9000
    h = Head(D, V, wtype, seed=5, with_norm=False, table=_tied_table(D, V, 55))
    x = torch.ones((3, D), dtype=torch.float32, device="cuda")
    tok, lg, _ = h.run(x)
    assert lg[0, 40] == lg[0, 7000] and lg[0, 100] == lg[0, 200] == lg[0, 300]
    assert (tok == 40).all()
    # k = 2: the two tied maxima in id order with equal weights: u < 1/2 -> 40
    u = torch.tensor([0.25, 0.75, 0.5], dtype=torch.float32, device="cuda")
    tok, _, _ = h.run(x, top_k=2, temperature=1.0, u=u)
    np.testing.assert_array_equal(tok, [40, 7000, 7000])
    # k = 3: the boundary tie among 100, 200, 300 takes 100
    u = torch.tensor([0.1, 0.6, 0.95], dtype=torch.float32, device="cuda")
    tok, _, _ = h.run(x, top_k=3, temperature=100.0, u=u)
    ids, cdf = oracle.top_k_cdf(h.oracle_logits(x)[0], 3, 100.0)
    np.testing.assert_array_equal(ids, [40, 7000, 100])
    want = [ids[int(np.searchsorted(cdf, v, side="right"))] for v in (0.1, 0.6, 0.95)]
    np.testing.assert_array_equal(tok, want)


@pytest.mark.parametrize("k,T", [(2, 0.8), (40, 1.0), (1024, 1.5)])
def test_top_k_sampling_matches_the_oracle_draw(k, T):
    D, V, B = 512, configs.VOCAB, 4
    h = Head(D, V, ddl.INT4, seed=13)
    x = _x(B, D, seed=14)
    _, lg, _ = h.run(x)
    ref = h.oracle_logits(x)
    rng = np.random.default_rng(k)
    # u at the middle of a wide candidate interval: the draw is decided far
    # from any boundary, so both sides must pick that candidate
    u_mid, want = [], []
    for b in range(B):
        ids, cdf = oracle.top_k_cdf(ref[b], k, T)
        lo = np.concatenate([[0.0], cdf[:-1]])
        widths = cdf - lo
        cands = np.flatnonzero(widths > 5e-4)  # the fp32 weights and sums move a boundary by < 1e-4
        j = int(rng.choice(cands)) if cands.size else int(np.argmax(widths))
        u_mid.append((lo[j] + cdf[j]) / 2)
        want.append(ids[j])
    u = torch.tensor(u_mid, dtype=torch.float32, device="cuda")
    tok, _, _ = h.run(x, top_k=k, temperature=T, u=u)
    np.testing.assert_array_equal(tok, want)
    # random uniforms: the drawn id is a candidate whose interval holds u
    # within the margin of the logits' and the fp32 sums' error
    for trial in range(5):
        uu = rng.random(B).astype(np.float32)
        tok, _, _ = h.run(x, top_k=k, temperature=T, u=torch.from_numpy(uu).cuda())
        for b in range(B):
            ids, cdf = oracle.top_k_cdf(ref[b], k, T)
            pos = np.flatnonzero(ids == tok[b])
            assert pos.size == 1, (b, tok[b])
            j = int(pos[0])
            lo = cdf[j - 1] if j else 0.0
            assert lo - 1e-3 <= uu[b] <= cdf[j] + 1e-3, (b, j, lo, cdf[j], uu[b])


def test_top_k_larger_than_vocabulary_and_u_zero():
    D, V, B = 512, 1000, 2
    h = Head(D, V, ddl.INT4, seed=31)
    x = _x(B, D, seed=32)
    ref = h.oracle_logits(x)
    u = torch.zeros(B, dtype=torch.float32, device="cuda")
    tok, _, _ = h.run(x, top_k=1024, temperature=1.0, u=u)  # k clipped to V
    np.testing.assert_array_equal(tok, oracle.greedy_token(ref))
    ids, cdf = oracle.top_k_cdf(ref[1], 1024, 2.0)
    assert ids.size == V
    lo = np.concatenate([[0.0], cdf[:-1]])
    j = int(np.flatnonzero(cdf - lo > 5e-4)[-1])  # the last candidate with a wide interval
    u = torch.tensor([0.0, (lo[j] + cdf[j]) / 2], dtype=torch.float32, device="cuda")
    tok, _, _ = h.run(x, top_k=1024, temperature=2.0, u=u)
    assert tok[1] == ids[j]


def test_head_argument_errors():
    D, V = 512, 1000
    h = Head(D, V, ddl.INT4, seed=1)
    x = _x(2, D, seed=2)
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_lm_head(D, V, ddl.INT4, h.packed, x, top_k=5, temperature=1.0, u=None)
    assert e.value.status == 8  # sampling without uniforms
    u = torch.zeros(2, dtype=torch.float32, device="cuda")
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_lm_head(D, V, ddl.INT4, h.packed, x, top_k=5, temperature=0.0, u=u)
    assert e.value.status == 8
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_lm_head(D, V, ddl.INT4, h.packed, x, top_k=2000, temperature=1.0, u=u)
    assert e.value.status == 5
    with pytest.raises(ddl.DDLError) as e:
        ddl.ddl_lm_head(D, V, ddl.INT4, h.packed, x, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 4
