"""GPU parity of expert-choice routing (each expert takes its top-C tokens;
deepseekmodel.com TopKRouter discussion, iwashi.co routing table) against
the fp64 oracle: the selection stage on the oracle's probabilities
(bit-exact, ties by lower token index), the combine stage, and the whole
layer on reduced and full sizes.

Comparison: an expert's token set is bit-exact, with one freedom: where the
expert's column ties within rounding at its Cn-th largest value (within 1e-6
relative, the fp32 and fp64 routers), either token is a correct pick.  A GPU
set that differs from the oracle's is accepted only if no token outside it
has a probability above its smallest one by more than that band; the oracle
is then re-run with the GPU's accepted sets, and counts, n_unchosen, f, p,
aux and y are compared on every token: y within 1e-2 x RMS (bf16) / 1e-4 x
RMS (fp32); f, p 1e-6; aux 1e-5 relative."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle.moe_oracle as om
import sparse_mixture_experts_47_b300 as moe
from tests.conftest import load_golden
from tests.parity import FP_ATOL, TIE_REL, act_dtype, sample_tokens, weights_dict, y_tol

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ec_cfg(T, E, C):
    cfg = moe.MoEConfig(T=T, d_model=8, n_experts=E, top_k=1, d_ff=8,
                        capacity_factor=float(C) * E / T - 1e-6,
                        routing=moe.ROUTING_EXPERT_CHOICE)
    assert min(moe.capacity(cfg), T) == min(C, T)
    return cfg


def _stage_check(probs, C):
    T, E = probs.shape
    ref = om.expert_choice(probs, C)
    cfg = _ec_cfg(T, E, C)
    pt = torch.tensor(np.ascontiguousarray(probs.T), dtype=torch.float32, device=DEV)
    out = moe.expert_choice(cfg, pt)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    Cn = min(C, T)
    got = out["perm"].cpu().numpy().reshape(E, Cn)
    assert got.tolist() == ref.chosen.tolist()
    assert np.array_equal(out["row_w"].cpu().numpy().reshape(E, Cn),
                          ref.weight.astype(np.float32))
    assert out["offsets"].cpu().numpy().tolist() == ref.offsets.tolist()
    assert int(out["n_unchosen"][0]) == ref.n_unchosen
    # per-token lists: expert order, rows pointing back at the token
    ts = out["tok_start"].cpu().numpy()
    tr = out["tok_rows"].cpu().numpy()
    for t in range(T):
        rows = tr[ts[t]:ts[t + 1]]
        experts = rows // Cn
        assert np.all(np.diff(experts) > 0)
        assert np.all(got.reshape(-1)[rows] == t)
        assert set(experts.tolist()) == {e for e in range(E) if t in set(ref.chosen[e].tolist())}
    return out


def test_expert_choice_golden_case():
    g = load_golden("expert_choice_case.json")
    probs = np.array(g["probs"], dtype=np.float32).astype(np.float64)
    _stage_check(probs, g["C"])


@pytest.mark.parametrize("T,E,C", [(1000, 8, 250), (4097, 8, 1025), (3000, 64, 100),
                                    (2000, 896, 18), (5, 4, 9), (300, 16, 300)])
def test_expert_choice_stage_bit_exact(T, E, C):
    rng = np.random.default_rng(T * 7 + E)
    logits = rng.normal(size=(T, E)) * 2
    logits[::7] = np.round(logits[::7], 1)          # repeated values make exact ties
    probs = om.softmax(logits).astype(np.float32).astype(np.float64)
    _stage_check(probs, C)


@pytest.mark.parametrize("dtype", [moe.DTYPE_BF16, moe.DTYPE_FP32])
def test_combine_rows_stage(dtype):
    rng = np.random.default_rng(4)
    T, E, d, C = 300, 8, 64, 90
    probs = om.softmax(rng.normal(size=(T, E))).astype(np.float32).astype(np.float64)
    ref = om.expert_choice(probs, C)
    cfg = _ec_cfg(T, E, C)
    cfg = moe.MoEConfig(**{**cfg.__dict__, "d_model": d, "dtype": dtype})
    out = moe.expert_choice(cfg, torch.tensor(np.ascontiguousarray(probs.T), dtype=torch.float32,
                                              device=DEV))
    o = rng.normal(size=(E * C, d)).astype(np.float32)
    sh = rng.normal(size=(T, d)).astype(np.float32)
    y = moe.combine_rows(cfg, torch.tensor(o, device=DEV), out["row_w"], out["tok_start"],
                         out["tok_rows"], torch.tensor(sh, device=DEV)).cpu().numpy()
    o64, sh64 = o.astype(np.float64), sh.astype(np.float64)
    yr = sh64.copy()
    for e in range(E):
        for i, t in enumerate(ref.chosen[e]):
            yr[t] += ref.weight[e, i] * o64[e * C + i]
    assert np.max(np.abs(y - yr)) <= 1e-5 * np.sqrt(np.mean(yr ** 2))


def _resolve_chosen(probs, got_sets):
    """The GPU's token set of every expert whose set differs from the
    oracle's, after checking that it is a valid top-Cn of the expert's
    oracle probabilities under the tie band."""
    T, E = probs.shape
    chosen = {}
    for e, got in enumerate(got_sets):
        col = probs[:, e]
        g = np.sort(np.asarray(got, dtype=np.int64))
        Cn = g.shape[0]
        ref = np.sort(np.argsort(-col, kind="stable")[:Cn])
        if np.array_equal(g, ref):
            continue
        assert np.unique(g).shape[0] == Cn and g.min() >= 0 and g.max() < T, e
        rest = np.setdiff1d(np.arange(T), g)
        band = TIE_REL * max(col[g].max(), col[rest].max() if rest.size else 0.0)
        assert rest.size == 0 or col[g].min() >= col[rest].max() - band, (
            f"expert {e}: GPU token set is not a valid top-{Cn}")
        chosen[e] = g
    return chosen


def _layer_check(w, T, inp, tokens=None):
    cfg = moe.config_for(w, T)
    out = moe.layer_forward(cfg, inp["x"], weights_dict(inp), want_layout=True)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    probs = om.softmax(om.router_logits(inp["x"], inp["w_r"], inp.get("logit_bias")))
    offs = out["offsets"].cpu().numpy()
    perm = out["perm"].cpu().numpy()
    got_sets = [perm[offs[e]:offs[e + 1]] for e in range(w.n_experts)]
    chosen = _resolve_chosen(probs, got_sets)
    orc = om.moe_forward_expert_choice(inp, w.top_k, w.act, w.capacity_factor, tokens,
                                       act_dtype(w), chosen=chosen, probs=probs)
    ec = orc["ec"]
    assert offs.tolist() == ec.offsets.tolist()
    for e in range(w.n_experts):
        assert got_sets[e].tolist() == ec.chosen[e].tolist(), e
    st = orc["stats"]
    assert np.array_equal(out["counts"].cpu().numpy(), st["counts"])
    assert np.max(np.abs(out["f"].cpu().numpy() - st["f"])) <= FP_ATOL
    assert np.max(np.abs(out["p"].cpu().numpy() - st["p"])) <= FP_ATOL
    assert abs(float(out["aux"][0]) - st["aux"]) <= 1e-5 * st["aux"]
    assert int(out["n_dropped"][0]) == ec.n_unchosen
    rows = orc["rows"]
    yg = out["y"].float().cpu().numpy()[rows].astype(np.float64)
    rms = float(np.sqrt(np.mean(orc["y"] ** 2)))
    err = float(np.max(np.abs(yg - orc["y"])))
    assert err <= y_tol(w) * rms, (err / rms, y_tol(w))
    return {"resolved_experts": len(chosen), "y_err_over_rms": err / rms,
            "unchosen": ec.n_unchosen}


SMALL = {
    "mixtral_ec_small": (mi.workload("mixtral_ec").with_sizes(d_model=512, d_ff=1024), 300),
    "mixtral_ec_T3": (mi.workload("mixtral_ec").with_sizes(d_model=256, d_ff=512), 3),
    "tiny_ec": (mi.workload("tiny").with_sizes(capacity_factor=1.0, routing="expert"), 64),
    "deepseek_ec_small": (mi.workload("deepseek").with_sizes(
        d_model=256, n_experts=64, d_ff=128, d_ff_shared=192, capacity_factor=1.0,
        routing="expert", select_bias="none"), 400),
    "e896_ec_small": (mi.workload("e896").with_sizes(d_model=128, d_ff=64, capacity_factor=1.0,
                                                     routing="expert", quantile_balance=False),
                      2000),
    # 50 experts in a bf16 layer: the CUDA-core tiled router writes the
    # expert-major probabilities
    "deepseek_ec_E50": (mi.workload("deepseek").with_sizes(
        d_model=256, n_experts=50, d_ff=128, d_ff_shared=192, capacity_factor=1.0,
        routing="expert", select_bias="none"), 400),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_expert_choice_small(name):
    w, T = SMALL[name]
    inp = mi.generate(w, T, DEV)
    print(name, _layer_check(w, T, inp))


def test_layer_expert_choice_full_size():
    w = mi.workload("mixtral_ec")
    T = 4096
    inp = mi.generate(w, T, DEV)
    print(_layer_check(w, T, inp, sample_tokens(T, 96)))
