"""The seeded input generators: shapes, determinism and the workload recipe."""
import math

import torch

import moe_inputs as mi


def test_mixtral_expert_parameter_count():
    # Mixture of Experts (waylandz.com, ch. 30) §30.3.2: each matrix 4096 x 14336
    # = 58.7M, about 176M per expert, about 1.408B for the 8 experts of a layer.
    w = mi.workload("mixtral")
    per_matrix = w.d_model * w.d_ff
    assert round(per_matrix / 1e5) == 587
    per_expert = 3 * per_matrix
    assert round(per_expert / 1e6) == 176
    assert abs(w.n_experts * per_expert / 1e9 - 1.408) < 0.002
    assert abs(w.n_experts * per_expert * 2 / 1e9 - 2.82) < 0.01   # bf16 bytes


def test_shapes_and_dtypes_small():
    w = mi.workload("deepseek").with_sizes(d_model=32, n_experts=8, d_ff=16, d_ff_shared=24)
    inp = mi.generate(w, 5)
    assert inp["x"].shape == (5, 32) and inp["x"].dtype == torch.bfloat16
    assert inp["w_r"].shape == (8, 32) and inp["w_r"].dtype == torch.float32
    assert inp["w1"].shape == (8, 16, 32) and inp["w3"].shape == (8, 16, 32)
    assert inp["w2"].shape == (8, 32, 16)
    assert inp["ws1"].shape == (24, 32) and inp["ws2"].shape == (32, 24)
    sb = inp["select_bias"]
    assert sb.shape == (8,) and float(sb.abs().max()) <= 0.05


def test_deterministic_and_T_independent_weights():
    w = mi.workload("switch").with_sizes(d_model=16, d_ff=32)
    a = mi.generate(w, 7)
    b = mi.generate(w, 9)
    for k in ("w_r", "w1", "w2", "logit_bias"):
        assert torch.equal(a[k], b[k])
    c = mi.generate(w, 7)
    assert torch.equal(a["x"], c["x"])
    assert a["w3"] is None                                   # ReLU experts
    assert abs(float(a["logit_bias"][0]) - mi.EXPERT0_LOGIT_OFFSET) < 1e-6


def test_zipf_offsets_and_scale():
    w = mi.workload("e896").with_sizes(d_model=64)
    inp = mi.generate(w, 3, with_experts=False)
    lb = inp["logit_bias"]
    assert lb.shape == (896,)
    assert abs(float(lb[0])) < 1e-7 and abs(float(lb[9]) + 1.1 * math.log(10)) < 1e-5
    wr = mi.generate(mi.workload("tiny"), 64)["w_r"]
    assert abs(float(wr.std()) - 1 / 8) < 0.03
