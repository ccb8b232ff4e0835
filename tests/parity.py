"""Parity helpers: run the layer through the C ABI and compare with the oracle.

Comparison rules (tolerances written here, used by every GPU test):
  * expert indices: for every token that is not a tie, the selected set is
    bit-exact, and the order is bit-exact when no two of its top-(k+1)
    selection scores are within the tie band; a tie is a token whose k-th and
    (k+1)-th oracle scores differ by less than 1e-6 relative (relative to the
    largest magnitude summed into the score: the score, the probability and
    the selection bias), widened by the largest bias difference when the bias
    is computed per batch;
  * gate weights: 1e-5 absolute;
  * counts, offsets, perm, inv, n_dropped: bit-exact (given the same indices);
  * y: max |y - y_oracle| <= tol * RMS(y_oracle), tol = 1e-4 (fp32 layer) or
    1e-2 (bf16 layer), over the compared tokens;
  * f, p: 1e-6 absolute; aux: 1e-5 relative.
"""
from __future__ import annotations

import numpy as np
import torch

import moe_inputs as mi
import oracle.moe_oracle as om
import sparse_mixture_experts_47_b300 as moe

W_ATOL = 1e-5
FP_ATOL = 1e-6
AUX_RTOL = 1e-5
TIE_REL = 1e-6


def y_tol(workload) -> float:
    return 1e-4 if workload.dtype == "fp32" else 1e-2


# Both sides round each expert output to the layer's storage type (reading
# R8); where the GPU's fp32 sum and the exact value straddle a rounding
# boundary the two roundings differ by one unit in the last place: for v in
# [2^e, 2^(e+1)) that is 2^(e-7) in bf16 (8 significant bits), at most 2^-7
# of |v|, and at most 2^-23 of |v| in fp32.  Each term |w o| of y may carry
# one such difference on top of the RMS-relative tolerance.
ROUND_FLIP = {"bf16": 2.0 ** -7, "fp32": 2.0 ** -23, "fp64": 0.0}


def y_allow(workload, rms, y_abs):
    """Elementwise bound on |y_gpu - y_oracle|."""
    return y_tol(workload) * rms + ROUND_FLIP[act_dtype(workload)] * y_abs


def weights_dict(inp):
    return {k: inp.get(k) for k in moe._WEIGHT_KEYS}


def gpu_layer(workload, T, inp, out_dtype=moe.DTYPE_FP32, want_unbiased=False, ws=None,
              want_slots=False):
    cfg = moe.config_for(workload, T, out_dtype)
    out = moe.layer_forward(cfg, inp["x"], weights_dict(inp), workspace=ws,
                            want_unbiased_counts=want_unbiased, want_slots=want_slots)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    return {k: (v.float().cpu().numpy() if v.dtype == torch.bfloat16 else v.cpu().numpy())
            for k, v in out.items() if isinstance(v, torch.Tensor)}


def act_dtype(workload) -> str:
    """Storage type of the experts' intermediate activation: the layer dtype."""
    return workload.dtype


def oracle_layer(workload, inp, tokens=None):
    return om.moe_forward(inp, workload.top_k, workload.act, workload.capacity_factor,
                          "probs", workload.quantile_balance, tokens, act_dtype(workload),
                          reroute_rounds=workload.reroute_rounds)


def tie_mask(r: "om.RouterOut", k: int, extra_abs: float = 0.0):
    """Tokens whose k-th and (k+1)-th selection scores are within the band,
    and tokens with any near-equal adjacent pair among their top k+1."""
    T, E = r.scores.shape
    order = np.argsort(-r.scores, axis=1, kind="stable")
    s = np.take_along_axis(r.scores, order, axis=1)
    pr = np.take_along_axis(r.probs, order, axis=1)
    bias = np.zeros(E) if r.select_bias is None else r.select_bias
    b = bias[order]
    mag = np.maximum(np.maximum(np.abs(s), np.abs(pr)), np.abs(b))
    if k >= E:
        kk = np.zeros(T, dtype=bool)
        adj = np.zeros(T, dtype=bool)
    else:
        gap = s[:, :k] - s[:, 1:k + 1]
        band = TIE_REL * mag[:, :k] + extra_abs
        kk = gap[:, k - 1] <= band[:, k - 1]
        adj = np.any(gap <= band, axis=1)
    if k > 1 and k >= E:
        gap = s[:, :k - 1] - s[:, 1:k]
        adj = np.any(gap <= TIE_REL * mag[:, :k - 1] + extra_abs, axis=1)
    return kk, adj


def compare_routing(workload, gpu, orc, extra_abs=0.0):
    r = orc["router"]
    k = workload.top_k
    ties, near = tie_mask(r, k, extra_abs)
    gi = gpu["idx"].astype(np.int64)
    ok = ~ties
    gs = np.sort(gi, axis=1)
    osr = np.sort(r.idx, axis=1)
    bad_set = np.nonzero(ok & np.any(gs != osr, axis=1))[0]
    assert bad_set.size == 0, f"expert sets differ on non-tie tokens {bad_set[:10]}"
    strict = ~near
    bad_ord = np.nonzero(strict & np.any(gi != r.idx, axis=1))[0]
    assert bad_ord.size == 0, f"expert order differs on tokens {bad_ord[:10]}"
    # weights: match by (token, expert) on non-tie tokens
    wo = np.take_along_axis(r.w, np.argsort(r.idx, axis=1), axis=1)
    wg = np.take_along_axis(gpu["w"].astype(np.float64), np.argsort(gi, axis=1), axis=1)
    err = np.abs(wo - wg)[ok]
    assert err.size == 0 or err.max() <= W_ATOL, f"gate weight error {err.max()}"
    return {"ties": int(ties.sum()), "near": int(near.sum()), "w_err": float(err.max()) if err.size else 0.0}


def compare_stats(workload, gpu, orc, n_ties):
    st = orc["stats"]
    E = workload.n_experts
    if n_ties == 0:
        assert np.array_equal(gpu["counts"].astype(np.int64), st["counts"])
        assert int(gpu["n_dropped"][0]) == orc["dispatch"].n_dropped
        assert np.max(np.abs(gpu["f"] - st["f"])) <= FP_ATOL
    else:
        diff = np.abs(gpu["counts"].astype(np.int64) - st["counts"]).sum()
        assert diff <= 2 * n_ties
    perr = float(np.max(np.abs(gpu["p"] - st["p"])))
    assert perr <= FP_ATOL, f"p error {perr}"
    if n_ties == 0:
        rel = abs(float(gpu["aux"][0]) - st["aux"]) / abs(st["aux"])
        assert rel <= AUX_RTOL, f"aux rel error {rel}"
        lr = abs(float(gpu["load_max_over_mean"][0]) - st["load_max_over_mean"])
        assert lr <= 1e-5 * st["load_max_over_mean"]
    return {"p_err": perr}


def compare_y(workload, gpu_y, orc, rows_mask=None):
    rows = orc["rows"]
    yo, ya = orc["y"], orc["y_abs"]
    yg = gpu_y[rows].astype(np.float64)
    if rows_mask is not None:
        yo, ya, yg = yo[rows_mask], ya[rows_mask], yg[rows_mask]
    rms = float(np.sqrt(np.mean(orc["y"] ** 2)))
    d = np.abs(yg - yo)
    err = float(np.max(d)) if yo.size else 0.0
    if yo.size:
        allow = y_allow(workload, rms, ya)
        i = np.unravel_index(np.argmax(d - allow), d.shape)
        assert np.all(d <= allow), (f"y error {d[i]:.3e} > {allow[i]:.3e} at {i} "
                                    f"({y_tol(workload)} x RMS {rms:.3e} + rounding)")
    return {"y_err_over_rms": err / rms if rms > 0 else 0.0}


def full_check(workload, T, inp, tokens=None, out_dtype=moe.DTYPE_FP32, ws=None):
    """Layer through the ABI vs the oracle on the same inputs; returns a report."""
    gpu = gpu_layer(workload, T, inp, out_dtype, ws=ws)
    orc = oracle_layer(workload, inp, tokens)
    extra = 0.0
    if workload.quantile_balance:
        db = np.abs(gpu["select_bias"].astype(np.float64) - orc["router"].select_bias)
        extra = float(db.max())
        assert extra <= 1e-6, f"quantile bias differs by {extra}"
    rep = compare_routing(workload, gpu, orc, extra)
    rep.update(compare_stats(workload, gpu, orc, rep["ties"]))
    # tokens affected by a tie (and, with capacity, everything after the first
    # tie in the same expert) are excluded from the y comparison
    ties, _ = tie_mask(orc["router"], workload.top_k, extra)
    mask = ~ties[orc["rows"]]
    if workload.capacity_factor > 0 and ties.any():
        first = int(np.nonzero(ties)[0].min())
        mask &= orc["rows"] < first
    rep.update(compare_y(workload, gpu["y"], orc, mask))
    return rep, gpu, orc


def sample_tokens(T, n, seed=7):
    g = np.random.default_rng(seed)
    if T <= n:
        return np.arange(T)
    s = set(g.choice(T, size=n, replace=False).tolist())
    s.update([0, T - 1])
    return np.array(sorted(s))
