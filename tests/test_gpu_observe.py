"""GPU parity of the monitoring set (drop ratio, gate entropy, size of the
selection bias, per-expert output mean / standard deviation / max) against
the fp64 oracle: through the whole layer on reduced-size workloads (the
oracle computes every token), through the stage call on the oracle's own
tensors, and the entropy, drop ratio and bias size at full sizes.

Tolerances: drop ratio 1e-7 absolute; gate entropy 1e-5 relative; bias size
1e-6 absolute (plus the quantile bias difference allowed by the routing
rules); per-expert output mean and standard deviation within the layer's y
tolerance (1e-2 x the expert's output RMS for bf16, 1e-4 for fp32), and the
largest magnitude within that plus the largest change that bf16 rounding
flips of h can make to one output element (computed from the data by
_flip_allowance: a maximum follows a single element, where the y tolerance
averages over the token's slots); 1e-5 x RMS when the stage call is fed the
oracle's own outputs, which checks the reductions exactly.  Tokens whose selection scores
tie within rounding are routed as the GPU routed them, after the check of
tests/parity.py that the GPU's order is a valid top-k."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle.moe_oracle as om
import sparse_mixture_experts_47_b300 as moe
from tests.parity import act_dtype, oracle_route, resolve_ranking, weights_dict, y_tol

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = {
    "tiny": (mi.workload("tiny"), 64),
    "switch_small": (mi.workload("switch").with_sizes(d_model=256, d_ff=512), 1000),
    "deepseek_small": (mi.workload("deepseek").with_sizes(d_model=256, n_experts=64, d_ff=128,
                                                          d_ff_shared=192), 200),
    "e896_small": (mi.workload("e896").with_sizes(d_model=128, d_ff=64), 2000),
    "mixtral_T1_split": (mi.workload("mixtral").with_sizes(d_model=1024, d_ff=2048), 1),
}


def _rms(a):
    a = np.asarray(a, dtype=np.float64)
    return float(np.sqrt(np.mean(a ** 2))) if a.size else 0.0


FLIP_REL = 2.0 ** -12


def _flip_allowance(x_rows, w1, w3, w2, act):
    """Largest change of one output element of an expert that bf16 rounding
    flips of its h can make (bf16 layer).  The GPU rounds an fp32 h; where
    the exact h lies within FLIP_REL (relative) of a bf16 rounding midpoint
    (far wider than the fp32 error of h), the two may round to neighbouring
    bf16 values, one unit apart.  Each such element f of a row moves output
    j by at most that unit times |w2[j, f]|; the allowance is the largest sum
    over the flippable elements of one row."""
    a = x_rows @ om._f64(w1).T
    h = om._silu(a) * (x_rows @ om._f64(w3).T) if act == "swiglu" else np.maximum(a, 0.0)
    _, ex = np.frexp(h)
    unit = np.ldexp(1.0, np.maximum(ex, -125) - 8)         # bf16 spacing at |h|
    mid = np.abs(np.abs(h - om.round_to_bf16(h)) - unit / 2)  # distance to the midpoint
    flippable = (mid <= FLIP_REL * np.abs(h)) & (h != 0)
    return float(np.max((flippable * unit) @ np.abs(om._f64(w2)).T)) if h.size else 0.0


def _check_scale(got, ref_out, E, tol, flip=None):
    """Mean and std within tol x the expert's output RMS; the largest
    magnitude follows a single element, so it also gets that element's
    rounding-flip allowance (``flip[e]``; none when the stage is fed the
    oracle's own outputs)."""
    for e in range(E):
        o = ref_out.get(e)
        if o is None or o.size == 0:
            assert got["expert_out_mean"][e] == 0 and got["expert_out_std"][e] == 0
            assert got["expert_out_max_abs"][e] == 0
            continue
        r = _rms(o)
        fa = 0.0 if flip is None else flip[e]
        assert abs(got["expert_out_mean"][e] - o.mean()) <= tol * r, e
        assert abs(got["expert_out_std"][e] - o.std()) <= tol * r, e
        assert abs(got["expert_out_max_abs"][e] - np.abs(o).max()) <= tol * r + fa, (e, fa)


@pytest.mark.parametrize("name", list(CASES))
def test_layer_observability_vs_oracle(name):
    w, T = CASES[name]
    inp = mi.generate(w, T, DEV)
    cfg = moe.config_for(w, T)
    out = moe.layer_forward(cfg, inp["x"], weights_dict(inp), observe=True)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    ob = {k: v.cpu().numpy().astype(np.float64) for k, v in out["observe"].items()}
    r = oracle_route(w, inp)
    bias_diff = 0.0
    if w.quantile_balance:
        bias_diff = float(np.max(np.abs(out["select_bias"].cpu().numpy() - r.select_bias)))
        assert bias_diff <= 1e-6
    # tokens whose scores tie within rounding take the GPU's (checked) order
    ranking = resolve_ranking(r, out["idx"].cpu().numpy(), bias_diff)
    orc = om.moe_forward(inp, w.top_k, w.act, w.capacity_factor, "probs", w.quantile_balance,
                         None, act_dtype(w), observe_outputs=True, ranking=ranking, router=r)
    ro = orc["observe"]
    assert abs(ob["drop_ratio"][0] - ro["drop_ratio"]) <= 1e-7
    assert abs(ob["gate_entropy"][0] - ro["gate_entropy"]) <= 1e-5 * ro["gate_entropy"]
    assert abs(ob["bias_mean_abs"][0] - ro["bias"]["mean_abs"]) <= 1e-6 + bias_diff
    assert abs(ob["bias_max_abs"][0] - ro["bias"]["max_abs"]) <= 1e-6 + bias_diff
    ref_out, flip = {}, {}
    x = om._f64(inp["x"])
    dp = orc["dispatch"]
    for e in range(w.n_experts):
        a, b = int(dp.offsets[e]), int(dp.offsets[e + 1])
        if a < b:
            rows = dp.perm[a:b] // w.top_k
            w3 = None if inp["w3"] is None else inp["w3"][e]
            ref_out[e] = om.expert_ffn(x[rows], inp["w1"][e], w3, inp["w2"][e], w.act,
                                       act_dtype(w))
            flip[e] = (_flip_allowance(x[rows], inp["w1"][e], w3, inp["w2"][e], w.act)
                       if w.dtype == "bf16" else 0.0)
    _check_scale(ob, ref_out, w.n_experts, y_tol(w), flip)


def test_observe_stage_on_oracle_tensors():
    rng = np.random.default_rng(11)
    T, E, k, d = 3000, 40, 3, 96
    probs = om.softmax(rng.normal(size=(T, E)) * 2)
    counts = rng.integers(0, 400, size=E)
    counts[5] = 0
    offsets = np.concatenate([[0], np.cumsum(counts)])
    rows = int(offsets[-1])
    outs = (rng.normal(size=(rows, d)) * rng.uniform(0.1, 3.0, size=(rows, 1))).astype(np.float32)
    bias = rng.uniform(-0.05, 0.05, size=E).astype(np.float32)
    cfg = moe.MoEConfig(T=rows, d_model=d, n_experts=E, top_k=1, d_ff=8)
    cfg_p = moe.MoEConfig(T=T, d_model=d, n_experts=E, top_k=k, d_ff=8)
    nd = torch.tensor([123], dtype=torch.int32, device=DEV)
    ob = moe.observe(cfg_p, probs=torch.tensor(probs, dtype=torch.float32, device=DEV),
                     select_bias=torch.tensor(bias, device=DEV), n_dropped=nd)
    ob2 = moe.observe(cfg, out_sorted=torch.tensor(outs, device=DEV),
                      offsets=torch.tensor(offsets, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    p32 = probs.astype(np.float32).astype(np.float64)
    ent = om.gate_entropy(p32)
    assert abs(float(ob["gate_entropy"][0]) - ent) <= 1e-5 * ent
    assert abs(float(ob["drop_ratio"][0]) - 123 / (T * k)) <= 1e-7
    bm = om.bias_magnitude(bias.astype(np.float64))
    assert abs(float(ob["bias_mean_abs"][0]) - bm["mean_abs"]) <= 1e-7
    assert float(ob["bias_max_abs"][0]) == bm["max_abs"]
    ref = {e: outs[offsets[e]:offsets[e + 1]].astype(np.float64) for e in range(E)
           if counts[e] > 0}
    got = {kk: v.cpu().numpy().astype(np.float64) for kk, v in ob2.items()}
    _check_scale(got, ref, E, 1e-5)
    assert got["expert_out_max_abs"][5] == 0.0


@pytest.mark.parametrize("name,T", [("e896", 16384), ("deepseek_cap", 8192)])
def test_observability_full_size(name, T):
    w = mi.workload(name)
    inp = mi.generate(w, T, DEV)
    cfg = moe.config_for(w, T)
    out = moe.layer_forward(cfg, inp["x"], weights_dict(inp), observe=True)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    ob = {k: v.cpu().numpy().astype(np.float64) for k, v in out["observe"].items()}
    r = om.route(inp["x"], inp["w_r"], w.top_k, inp.get("logit_bias"), inp.get("select_bias"),
                 "probs", w.quantile_balance)
    ent = om.gate_entropy(r.probs)
    assert abs(ob["gate_entropy"][0] - ent) <= 1e-5 * ent
    bm = om.bias_magnitude(r.select_bias)
    extra = 1e-6 if w.quantile_balance else 0.0
    assert abs(ob["bias_mean_abs"][0] - bm["mean_abs"]) <= 1e-6 + extra
    assert abs(ob["bias_max_abs"][0] - bm["max_abs"]) <= 1e-6 + extra
    nd = int(out["n_dropped"][0])
    assert abs(ob["drop_ratio"][0] - nd / (T * w.top_k)) <= 1e-7
    if w.capacity_factor > 0:
        assert nd > 0
    # experts with rows have positive scale, the others report zeros
    counts = out["counts"].cpu().numpy()
    assert np.all(ob["expert_out_std"][counts > 0] > 0)
    assert np.all(ob["expert_out_max_abs"][counts == 0] == 0)
    del inp
    torch.cuda.empty_cache()
