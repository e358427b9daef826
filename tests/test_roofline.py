"""The bytes/FLOPs model against the pages' worked numbers (tests/golden)."""
import json
import os

import pytest

from memory_bound_transformer_decode_gb300 import configs, roofline

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                   "pages_worked_numbers.json")))


def test_intensity_27b_fp16():
    g = GOLD["intensity_27b_fp16"]
    flops = 2 * g["params"]
    nbytes = g["params"] * g["bytes_per_param"]
    assert flops == g["flops_per_token"] and nbytes == g["bytes_per_token"]
    assert roofline.intensity(flops, nbytes) == g["ops_per_byte"]
    util = 100 * roofline.intensity(flops, nbytes) / g["ridge_ops_per_byte"]
    assert round(util, 1) == g["utilisation_printed_percent"]


def test_int4_and_fusion_fraction():
    g = GOLD["int4_and_fusion"]
    assert 100 * (1 - g["int4_bytes_per_param"] / 2) == g["int4_saving_percent"]
    # 4-bit (x1/4) together with fusion (x1/4) -> 1/16 of the bytes, 16 op/byte
    frac = (g["int4_bytes_per_param"] / 2) * 0.25
    assert frac == g["combined_byte_fraction"]
    assert roofline.intensity(1.0, frac) == g["combined_ops_per_byte"]


def test_decode_floor_7b():
    g = GOLD["decode_floor_7b_h100"]
    t = roofline.roofline_seconds(g["weight_bytes"], g["bandwidth_bytes_per_s"])
    assert round(t * 1e3, 1) == g["printed_ms_per_token"]
    assert abs(1 / t - g["printed_tokens_per_s"]) / g["printed_tokens_per_s"] < 0.03


def test_estimate_mem_against_page_and_its_formula():
    g = GOLD["estimate_mem_llama3_70b"]
    m = roofline.estimate_mem(**g["args"])
    for k, v in g["formula_gb"].items():
        assert m[k] / 1e9 == pytest.approx(v, rel=1e-9)
    assert m["weights"] / 1e9 == g["printed_gb"]["weights"]
    assert m["adam"] / 1e9 == g["printed_gb"]["adam"]
    assert int(m["act_train"] / 1e9) == g["printed_gb"]["act_train"]
    # the printed KV figure disagrees with the page's own formula
    assert abs(m["kv"] / 1e9 - g["printed_gb"]["kv"]) > 1.0


def test_flops_per_token_llama3_70b():
    g = GOLD["flops_per_token_llama3_70b"]
    c = configs.LLAMA70B_STACK
    printed_formula = g["L"] * (4 * c.D ** 2 + 2 * c.D * c.d_ff)
    assert printed_formula / 1e9 == pytest.approx(59.06, abs=0.01)
    exact_mac = sum(n * k for n, k in roofline.matrix_dims(c)) * c.layers
    assert exact_mac / 1e9 == pytest.approx(68.45, abs=0.01)


def test_step_bytes_of_the_workloads():
    # the 27B-class stack: 18.727 GB per token; the 70B stack 47.105 GB
    assert roofline.step_bytes(configs.STACK27B) / 1e9 == pytest.approx(18.727, abs=0.001)
    assert roofline.step_bytes(configs.LLAMA70B_STACK) / 1e9 == pytest.approx(47.105, abs=0.001)
    sw = configs.STACK27B_SWEEP
    got = [roofline.step_bytes(sw, batch=b) / 1e9 for b in configs.SWEEP_BATCHES]
    assert got == pytest.approx([17.65, 20.88, 33.76, 85.32], abs=0.01)
    got = [roofline.step_bytes(sw, batch=b, weights="bf16") / 1e9 for b in configs.SWEEP_BATCHES]
    assert got == pytest.approx([63.49, 66.71, 79.60, 131.15], abs=0.01)
    # KV term is the page's per-sequence formula with S + 1 rows (read S, write 1)
    c = configs.STACK27B
    mem = roofline.estimate_mem(1, c.layers, c.D, c.H_q, c.H_kv, c.head_dim, c.kv_len + 1, 1)
    assert roofline.kv_bytes_per_layer(c) * c.layers == mem["kv"]
    assert roofline.step_flops(c) / 1e9 == pytest.approx(79.6, abs=0.1)
