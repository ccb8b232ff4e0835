"""Precision of the router logits on the GPU at full sizes, against the fp64
oracle: the tensor-core router (E > 32, bf16: a two-part bf16 split of W_r
with the fp32 accumulation cut into chains) and the fp32 CUDA-core routers.

The logits stay on the device; the router hands out probs = softmax(logits),
so the test compares log probs on a seeded sample of tokens.  If logit e of
a token is off by D_e, log p_e is off by D_e - sum_j p_j D_j to first order,
so |D_e| <= B_e gives |d log p_e| <= B_e + sum_j p_j B_j, plus the fp32
rounding of the softmax itself.  The centred difference
d log p_e - mean_e d log p_e = D_e - mean_e D_e is reported as the logit
error.

Bounds, per token and expert, in units of S_e = sum_i |x_i| |W_r[e, i]|:

* fp32 CUDA-core router: d products and at most d additions, each rounded
  to nearest in fp32: (d + 2) 2^-24 S (the classical bound of recursive
  summation, whatever the order).
* tensor-core router: the split leaves |w - hi - lo| <= 2^-18 |w|, and the
  bf16 x bf16 products are exact in fp32.  A chain is at most 16 K blocks of
  64, i.e. 64 MMA steps of K = 16; each step is taken to add at most 2^-22
  (two fp32 units, truncation allowed) of the magnitudes it sums.  Chains
  and group planes are added in fp32: at most 2 d / 1024 + 4 roundings of
  2^-24.  Bound: (2^-18 + 64 2^-22 + (2 d / 1024 + 4) 2^-24) S.
* softmax in fp32: the logit and its difference to the row maximum rounded
  (2^-23 (|l_e| + |max l|)), exp, the sum of E terms and the division
  ((E + 8) 2^-24).

The tensor-core router is also held to the fp32 CUDA-core router on the same
tokens: its RMS logit error at most 4 times that router's."""
import dataclasses

import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle.moe_oracle as om
import sparse_mixture_experts_47_b300 as moe
from tests.parity import sample_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -24


def _gpu_probs(cfg, x, inp):
    r = moe.router_topk(cfg, x, inp["w_r"], inp.get("logit_bias"), None, want_probs=True,
                        want_p=False)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    return r["probs"]


def _oracle(inp, tokens):
    x = inp["x"][tokens].float().cpu().numpy().astype(np.float64)
    wr = inp["w_r"].cpu().numpy().astype(np.float64)
    lb = inp.get("logit_bias")
    lb = None if lb is None else lb.cpu().numpy()
    lg = om.router_logits(x, wr, lb)
    S = np.abs(x) @ np.abs(wr).T                          # sum_i |x_i| |W_r[e, i]|
    return lg, om.softmax(lg), S


def _errors(p_gpu, lg, p_orc, S, B_rel, E):
    """Check |d log p| against the bound; return (max, rms) of the centred
    logit error."""
    lp = np.log(p_gpu.astype(np.float64))
    d = lp - np.log(p_orc)
    B = B_rel * S
    soft = 2 * U * (np.abs(lg) + np.max(np.abs(lg), axis=1, keepdims=True)) + (E + 8) * U
    bound = B + np.sum(p_orc * B, axis=1, keepdims=True) + soft
    worst = np.max(d / bound)
    assert np.all(np.abs(d) <= bound), worst
    c = d - d.mean(axis=1, keepdims=True)
    return float(np.max(np.abs(c))), float(np.sqrt(np.mean(c ** 2))), float(worst)


CASES = [("e896", 16384, True), ("deepseek", 8192, True), ("deepseek", 128, True),
         ("mixtral", 16384, False), ("switch", 8192, False)]


@pytest.mark.parametrize("name,T,tensor_core", CASES, ids=[f"{n}-T{T}" for n, T, _ in CASES])
def test_router_logit_error(name, T, tensor_core):
    w = mi.workload(name)
    inp = mi.generate(w, T, DEV, with_experts=False)
    d, E = w.d_model, w.n_experts
    tokens = sample_tokens(T, min(T, 1024))
    lg, p_orc, S = _oracle(inp, tokens)
    cfg = dataclasses.replace(moe.config_for(w, T), quantile_balance=0)
    b_fp32 = (d + 2) * U
    b_tc = 2.0 ** -18 + 64 * 2.0 ** -22 + (2 * d / 1024 + 4) * U
    p = _gpu_probs(cfg, inp["x"], inp)[tokens].cpu().numpy()
    mx, rms, worst = _errors(p, lg, p_orc, S, b_tc if tensor_core else b_fp32, E)
    print(f"{name} T={T} {'tensor-core' if tensor_core else 'fp32'} router: logit error "
          f"max {mx:.2e} rms {rms:.2e}; worst |d log p| / bound {worst:.3f}")
    if not tensor_core:
        return
    # the same tokens through the fp32 CUDA-core router
    cfg32 = dataclasses.replace(cfg, dtype=moe.DTYPE_FP32)
    x32 = inp["x"].float()
    p32 = _gpu_probs(cfg32, x32, inp)[tokens].cpu().numpy()
    mx32, rms32, worst32 = _errors(p32, lg, p_orc, S, b_fp32, E)
    print(f"{name} T={T} fp32 router: logit error max {mx32:.2e} rms {rms32:.2e}; "
          f"worst |d log p| / bound {worst32:.3f}")
    assert rms <= 4 * rms32, (rms, rms32)
    del inp, x32
    torch.cuda.empty_cache()
