"""Parity helpers: run the layer through the C ABI and compare with the oracle.

Comparison rules (tolerances written here, used by every GPU test):
  * expert indices: bit-exact on every token, with one freedom.  Where a
    token's selection scores tie within rounding, either order is a correct
    top-k, and the GPU (fp32 scores) may take the other one.  Such a pick is
    accepted only if it is a valid top-k of the oracle's fp64 scores under
    the tie band:
      - each selected expert scores no lower than the next selected one,
        minus the band;
      - no unselected expert scores above the lowest selected one by more
        than the band.
    With redirection the same holds for the GPU's candidates ranked after
    the top k.  The band is 1e-6 relative to the largest magnitude summed
    into the scores involved (the score, the probability and the selection bias).  It
    is widened by twice the largest GPU-oracle difference of a bias computed
    per batch, since one such difference can enter each of the two scores
    that are compared.  The oracle is then re-run with the accepted orders
    (``oracle.with_ranking``), so that everything after the selection is
    compared on every token: weights, counts, drops, statistics and y;
  * gate weights: 1e-5 absolute;
  * counts, offsets, perm, inv, n_dropped: bit-exact;
  * y: max |y - y_oracle| <= tol * RMS(y_oracle) over the compared tokens,
    tol = 1e-4 (fp32 layer) or 1e-2 (bf16 layer), with no other allowance;
  * f, p: 1e-6 absolute; aux and load max/mean: 1e-5 relative.
"""
from __future__ import annotations

from typing import Dict, Optional

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


def weights_dict(inp):
    return {k: inp.get(k) for k in moe._WEIGHT_KEYS}


def gpu_layer(workload, T, inp, out_dtype=moe.DTYPE_FP32, want_unbiased=False, ws=None,
              want_slots=False, want_layout=False):
    cfg = moe.config_for(workload, T, out_dtype)
    out = moe.layer_forward(cfg, inp["x"], weights_dict(inp), workspace=ws,
                            want_unbiased_counts=want_unbiased, want_slots=want_slots,
                            want_layout=want_layout)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    return {k: (v.float().cpu().numpy() if v.dtype == torch.bfloat16 else v.cpu().numpy())
            for k, v in out.items() if isinstance(v, torch.Tensor)}


def act_dtype(workload) -> str:
    """Storage type of the experts' intermediate activation: the layer dtype."""
    return workload.dtype


def oracle_route(workload, inp) -> "om.RouterOut":
    return om.route(inp["x"], inp["w_r"], workload.top_k, inp.get("logit_bias"),
                    inp.get("select_bias"), workload.select_space, workload.quantile_balance)


def oracle_layer(workload, inp, tokens=None, ranking=None, router=None):
    return om.moe_forward(inp, workload.top_k, workload.act, workload.capacity_factor,
                          workload.select_space, workload.quantile_balance, tokens, act_dtype(workload),
                          reroute_rounds=workload.reroute_rounds, ranking=ranking,
                          router=router)


def _magnitude(r: "om.RouterOut", t: int, experts) -> float:
    e = np.asarray(list(experts), dtype=np.int64)
    b = np.zeros(e.shape[0]) if r.select_bias is None else np.abs(r.select_bias[e])
    return float(max(np.max(np.abs(r.scores[t, e])), np.max(np.abs(r.probs[t, e])), np.max(b)))


def tie_band(r: "om.RouterOut", t: int, experts, bias_diff: float = 0.0) -> float:
    """Scores of token t closer than this may be ordered either way."""
    return TIE_REL * _magnitude(r, t, experts) + 2.0 * bias_diff


def tie_mask(r: "om.RouterOut", k: int, bias_diff: float = 0.0, depth: Optional[int] = None):
    """Tokens whose selection scores tie within the band: (a) the k-th and
    (k+1)-th, and (b) any adjacent pair among the top ``depth`` (default
    k + 1) ranked scores."""
    T, E = r.scores.shape
    depth = min(E, k + 1 if depth is None else depth)
    order = np.argsort(-r.scores, axis=1, kind="stable")[:, :depth]
    s = np.take_along_axis(r.scores, order, axis=1)
    pr = np.take_along_axis(r.probs, order, axis=1)
    b = (np.zeros_like(s) if r.select_bias is None else np.abs(r.select_bias[order]))
    mag = np.maximum(np.maximum(np.abs(s), np.abs(pr)), b).max(axis=1)
    band = TIE_REL * mag + 2.0 * bias_diff
    gap = s[:, :-1] - s[:, 1:]
    kk = gap[:, k - 1] <= band if k < E else np.zeros(T, dtype=bool)
    adj = np.any(gap <= band[:, None], axis=1) if depth > 1 else np.zeros(T, dtype=bool)
    return kk, adj


def valid_topk(r: "om.RouterOut", t: int, picks, bias_diff: float = 0.0) -> bool:
    """Is ``picks`` (best first) a correct top-k of token t's oracle scores
    under the tie band?"""
    g = [int(e) for e in picks]
    E = r.scores.shape[1]
    if len(set(g)) != len(g) or min(g) < 0 or max(g) >= E:
        return False
    s = r.scores[t]
    rest = np.setdiff1d(np.arange(E), g)
    top_rest = int(rest[np.argmax(s[rest])]) if rest.size else None
    band = tie_band(r, t, g + ([top_rest] if top_rest is not None else []), bias_diff)
    if any(s[g[j]] < s[g[j + 1]] - band for j in range(len(g) - 1)):
        return False
    return top_rest is None or s[g].min() >= s[top_rest] - band


def resolve_ranking(r: "om.RouterOut", gpu_lead: np.ndarray, bias_diff: float = 0.0
                    ) -> Dict[int, np.ndarray]:
    """The GPU's leading experts (its top k, then with redirection its
    candidates after them) for every token where they differ from the
    oracle's ranking, after checking that they are a valid ranking prefix
    under the tie band; a token whose GPU order is not valid fails the
    comparison."""
    gi = gpu_lead.astype(np.int64)
    ref = np.argsort(-r.scores, axis=1, kind="stable")[:, :gi.shape[1]]
    differ = np.nonzero(np.any(gi != ref, axis=1))[0]
    bad = [int(t) for t in differ if not valid_topk(r, int(t), gi[t], bias_diff)]
    assert not bad, (f"GPU expert ranking is not valid on tokens {bad[:10]}: "
                     f"gpu {gi[bad[:3]].tolist()} oracle {ref[bad[:3]].tolist()}")
    return {int(t): gi[t].copy() for t in differ}


def compare_routing(workload, gpu, orc):
    """After the tie orders are fixed, indices are bit-exact and weights
    within W_ATOL on every token."""
    r = orc["router"]
    gi = gpu["idx"].astype(np.int64)
    bad = np.nonzero(np.any(gi != r.idx, axis=1))[0]
    assert bad.size == 0, f"expert indices differ on tokens {bad[:10]}"
    err = np.abs(gpu["w"].astype(np.float64) - r.w)
    werr = float(err.max()) if err.size else 0.0
    assert werr <= W_ATOL, f"gate weight error {werr}"
    return {"w_err": werr}


def compare_stats(workload, gpu, orc):
    st = orc["stats"]
    assert np.array_equal(gpu["counts"].astype(np.int64), st["counts"]), "counts differ"
    assert int(gpu["n_dropped"][0]) == orc["dispatch"].n_dropped, "n_dropped differs"
    ferr = float(np.max(np.abs(gpu["f"] - st["f"]))) if st["f"].size else 0.0
    assert ferr <= FP_ATOL, f"f error {ferr}"
    perr = float(np.max(np.abs(gpu["p"] - st["p"]))) if st["p"].size else 0.0
    assert perr <= FP_ATOL, f"p error {perr}"
    if st["aux"] != 0:
        rel = abs(float(gpu["aux"][0]) - st["aux"]) / abs(st["aux"])
        assert rel <= AUX_RTOL, f"aux rel error {rel}"
    lr = abs(float(gpu["load_max_over_mean"][0]) - st["load_max_over_mean"])
    assert lr <= AUX_RTOL * max(st["load_max_over_mean"], 1e-30), f"load error {lr}"
    return {"p_err": perr}


def compare_y(workload, gpu_y, orc):
    """max |y_gpu - y_oracle| <= y_tol * RMS(y_oracle) on the oracle's rows."""
    rows = orc["rows"]
    yo = orc["y"]
    yg = gpu_y[rows].astype(np.float64)
    rms = float(np.sqrt(np.mean(yo ** 2))) if yo.size else 0.0
    d = np.abs(yg - yo)
    err = float(np.max(d)) if yo.size else 0.0
    tol = y_tol(workload)
    if yo.size:
        i = np.unravel_index(np.argmax(d), d.shape)
        assert err <= tol * rms, (f"y error {err:.3e} = {err / rms:.3e} x RMS > {tol} x RMS "
                                  f"at row {int(rows[i[0]])} col {int(i[1])}")
    return {"y_err_over_rms": err / rms if rms > 0 else 0.0}


def full_check(workload, T, inp, tokens=None, out_dtype=moe.DTYPE_FP32, ws=None,
               want_slots=False):
    """Layer through the ABI vs the oracle on the same inputs; returns a report."""
    redirect = workload.reroute_rounds > 0
    gpu = gpu_layer(workload, T, inp, out_dtype, ws=ws, want_slots=want_slots or redirect)
    r = oracle_route(workload, inp)
    bias_diff = 0.0
    if workload.quantile_balance:
        db = np.abs(gpu["select_bias"].astype(np.float64) - r.select_bias)
        bias_diff = float(db.max()) if db.size else 0.0
        assert bias_diff <= 1e-6, f"quantile bias differs by {bias_diff}"
    # with redirection a slot may take its token's next candidates down the
    # ranking: the GPU's candidates join its top k in the checked order
    lead = np.concatenate([gpu["idx"], gpu["cand_idx"]], axis=1) if redirect else gpu["idx"]
    ranking = resolve_ranking(r, lead, bias_diff)
    orc = oracle_layer(workload, inp, tokens, ranking=ranking, router=r)
    ties, near = tie_mask(r, workload.top_k, bias_diff)
    rep = {"ties": int(ties.sum()), "near": int(near.sum()), "resolved": len(ranking)}
    rep.update(compare_routing(workload, gpu, orc))
    rep.update(compare_stats(workload, gpu, orc))
    rep.update(compare_y(workload, gpu["y"], orc))
    return rep, gpu, orc


def sample_tokens(T, n, seed=7):
    g = np.random.default_rng(seed)
    if T <= n:
        return np.arange(T)
    s = set(g.choice(T, size=n, replace=False).tolist())
    s.update([0, T - 1])
    return np.array(sorted(s))
