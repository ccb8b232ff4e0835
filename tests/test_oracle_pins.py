"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each ``pin_*`` function raises AssertionError on a mismatch.  The tests call
them on the oracle as written; ``test_planted_mistakes_are_caught`` plants a
plausible mistake in the oracle (on the CPU, by monkeypatching one function)
and checks that at least one pin fails, so the pins are known to bite.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

import oracle.moe_oracle as om
from tests.conftest import load_golden

RNG = np.random.default_rng(12345)


# ----------------------------------------------------------------- printed examples

def pin_top2_example():
    g = load_golden("top2_example.json")
    probs = np.array([g["probs"]])
    # x = log(p), W_r = I: the router logits are log(p), so softmax gives p back.
    r = om.route(np.log(probs), np.eye(8), g["k"])
    assert np.allclose(r.probs[0], probs[0], rtol=0, atol=1e-15)
    assert r.idx[0].tolist() == g["top_k_indices"]
    assert np.allclose(np.take(r.probs[0], r.idx[0]), g["top_k_probs"], atol=1e-15)
    exact = np.array(g["top_k_probs"]) / sum(g["top_k_probs"])
    assert np.allclose(r.w[0], exact, rtol=0, atol=1e-15)
    half_ulp = 0.5 * 10.0 ** (-g["weights_printed_decimals"])
    assert np.all(np.abs(r.w[0] - np.array(g["weights_printed"])) <= half_ulp + 1e-12)


def pin_aux_worked_example():
    g = load_golden("aux_worked_example.json")
    probs = np.array(g["probs"])
    T, E = probs.shape
    # Feed logits = log(probs): softmax returns the printed probabilities.
    r = om.route(np.log(probs), np.eye(E), g["k"])
    assert np.allclose(r.probs, probs, atol=1e-15)
    assert (r.idx[:, 0] + 1).tolist() == g["selected_expert_1based"]
    st = om.load_stats(r.probs, r.idx, E)
    assert np.allclose(st["f"], g["f"], atol=1e-15)
    assert np.allclose(st["p"], g["p"], atol=1e-15)
    assert abs(float(np.sum(st["f"] * st["p"])) - g["sum_f_times_p"]) < 1e-15
    assert abs(st["aux"] - g["aux"]) < 1e-14


def pin_selection_bias_example():
    g = load_golden("selection_bias_example.json")
    s = np.array([g["scores"]])
    b = np.array(g["bias"])
    assert np.allclose(s[0] + b, g["biased_printed"], atol=1e-15)
    unb = om.topk_desc(s, g["k"])[0]
    assert sorted((unb + 1).tolist()) == sorted(g["unbiased_top2_1based"])
    sel = om.topk_desc(s + b[None, :], g["k"])[0]
    assert (sel + 1).tolist() == g["biased_top2_1based"]
    w = om.renormalise(s, sel[None, :])[0]
    assert np.allclose(w, [0.50 / 1.20, 0.70 / 1.20], atol=1e-15)
    # Through the whole router: logits = log(score) give probs = score / 2.4;
    # the same bias on the probs picks the same two experts, weights unchanged.
    r = om.route(np.log(s), np.eye(4), g["k"], select_bias=b)
    assert (r.idx[0] + 1).tolist() == g["biased_top2_1based"]
    assert np.allclose(r.w[0], [0.50 / 1.20, 0.70 / 1.20], atol=1e-15)


# ----------------------------------------------------------------- closed forms and brute force

def pin_uniform_aux_is_one():
    # T = E tokens, token t prefers experts t, t+1, ... cyclically: every
    # expert gets the same count and, by symmetry, the same mean probability.
    for E, k in [(4, 1), (8, 2), (6, 3)]:
        base = np.array([3.0, 2.0, 1.0] + [0.0] * (E - 3))
        logits = np.stack([np.roll(base, t) for t in range(E)])
        r = om.route(logits, np.eye(E), k)
        st = om.load_stats(r.probs, r.idx, E)
        assert np.allclose(st["f"], 1.0 / E, atol=1e-15)
        assert abs(st["aux"] - 1.0) < 1e-12
        assert abs(st["load_max_over_mean"] - 1.0) < 1e-12


def pin_topk_bruteforce():
    for trial in range(200):
        E = int(RNG.integers(2, 9))
        k = int(RNG.integers(1, min(3, E) + 1))
        s = RNG.normal(size=(1, E))
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(s[0, list(c)]))
        idx = om.topk_desc(s, k)[0]
        assert set(idx.tolist()) == set(best)
        vals = s[0, idx]
        assert np.all(vals[:-1] >= vals[1:])
    # equal scores: lower index first
    idx = om.topk_desc(np.array([[1.0, 2.0, 2.0, 0.5, 2.0]]), 2)[0]
    assert idx.tolist() == [1, 2]


def pin_softmax_closed_forms():
    for _ in range(20):
        E = int(RNG.integers(1, 40))
        p = RNG.dirichlet(np.ones(E))
        assert np.allclose(om.softmax(np.log(p)[None, :])[0], p, atol=1e-14)
        l = RNG.normal(size=(3, E)) * 5
        ref = torch.softmax(torch.tensor(l, dtype=torch.float64), dim=-1).numpy()
        assert np.allclose(om.softmax(l), ref, atol=1e-15)
        assert np.allclose(om.softmax(l + 7.5), ref, atol=1e-14)


def pin_router_logits_layout():
    x = RNG.normal(size=(5, 7))
    w_r = RNG.normal(size=(3, 7))   # nn.Linear(7 -> 3).weight
    ref = Fnn.linear(torch.tensor(x), torch.tensor(w_r)).numpy()
    assert np.allclose(om.router_logits(x, w_r), ref, atol=1e-13)
    b = RNG.normal(size=3)
    assert np.allclose(om.router_logits(x, w_r, b), ref + b, atol=1e-13)


# ----------------------------------------------------------------- FFN reductions

def _torch_ffn(x, w1, w3, w2, act):
    """The pages' Expert module with torch.nn.functional, float64."""
    x, w1, w2 = (torch.tensor(np.asarray(a, dtype=np.float64)) for a in (x, w1, w2))
    if act == "swiglu":
        w3 = torch.tensor(np.asarray(w3, dtype=np.float64))
        return Fnn.linear(Fnn.silu(Fnn.linear(x, w1)) * Fnn.linear(x, w3), w2).numpy()
    return Fnn.linear(Fnn.relu(Fnn.linear(x, w1)), w2).numpy()


def _rand_layer(T, d, E, F, act, Fs=0):
    inp = {"x": RNG.normal(size=(T, d)), "w_r": RNG.normal(size=(E, d)) / math.sqrt(d),
           "w1": RNG.normal(size=(E, F, d)) / math.sqrt(d),
           "w3": RNG.normal(size=(E, F, d)) / math.sqrt(d) if act == "swiglu" else None,
           "w2": RNG.normal(size=(E, d, F)) / math.sqrt(F)}
    if Fs:
        inp["ws1"] = RNG.normal(size=(Fs, d)) / math.sqrt(d)
        inp["ws3"] = RNG.normal(size=(Fs, d)) / math.sqrt(d)
        inp["ws2"] = RNG.normal(size=(d, Fs)) / math.sqrt(Fs)
    return inp


def pin_single_expert_is_dense_ffn():
    for act in ("swiglu", "relu"):
        inp = _rand_layer(9, 12, 1, 20, act)
        out = om.moe_forward(inp, 1, act)
        ref = _torch_ffn(inp["x"], inp["w1"][0], None if inp["w3"] is None else inp["w3"][0],
                         inp["w2"][0], act)
        assert np.allclose(out["y"], ref, atol=1e-12)


def pin_identical_experts():
    inp = _rand_layer(11, 10, 5, 16, "swiglu")
    for key in ("w1", "w3", "w2"):
        inp[key] = np.repeat(inp[key][:1], 5, axis=0)
    ref = _torch_ffn(inp["x"], inp["w1"][0], inp["w3"][0], inp["w2"][0], "swiglu")
    for k in (1, 2, 3):
        out = om.moe_forward(inp, k, "swiglu")
        assert np.allclose(out["y"], ref, atol=1e-12)


def pin_all_experts_is_dense_mixture():
    T, d, E, F = 7, 10, 4, 12
    inp = _rand_layer(T, d, E, F, "swiglu")
    out = om.moe_forward(inp, E, "swiglu")
    probs = torch.softmax(Fnn.linear(torch.tensor(inp["x"]), torch.tensor(inp["w_r"])), -1).numpy()
    ref = sum(probs[:, e:e + 1] * _torch_ffn(inp["x"], inp["w1"][e], inp["w3"][e], inp["w2"][e], "swiglu")
              for e in range(E))
    assert np.allclose(out["y"], ref, atol=1e-12)


def pin_shared_expert_added():
    inp = _rand_layer(6, 8, 3, 10, "swiglu", Fs=14)
    base = om.moe_forward({k: v for k, v in inp.items() if not k.startswith("ws")}, 2, "swiglu")
    full = om.moe_forward(inp, 2, "swiglu")
    shared = _torch_ffn(inp["x"], inp["ws1"], inp["ws3"], inp["ws2"], "swiglu")
    assert np.allclose(full["y"], base["y"] + shared, atol=1e-12)


# ----------------------------------------------------------------- capacity and dispatch

def pin_capacity_cases():
    g = load_golden("capacity_cases.json")
    for c in g["cases"]:
        C = om.capacity(c["T"], c["k"], c["E"], c["capacity_factor"])
        assert C == c["C"]
        dp = om.dispatch(np.array(c["idx"]), c["E"], C)
        assert dp.counts.tolist() == c["counts"]
        assert dp.kept_counts.tolist() == c["kept_counts"]
        assert dp.offsets.tolist() == c["offsets"]
        assert dp.perm.tolist() == c["perm"]
        assert dp.inv.tolist() == c["inv"]
        assert dp.n_dropped == c["n_dropped"]
    # a fully dropped token has y = 0 (its FFN branch is zeroed, no renormalisation)
    c = g["cases"][1]
    T, E, k, d, F = c["T"], c["E"], c["k"], 6, 8
    inp = _rand_layer(T, d, E, F, "relu")
    # pin the routing to the case's idx: x = one-hot rows, W_r rows pick the scores
    score = np.full((T, E), -30.0)
    for t in range(T):
        for j, e in enumerate(c["idx"][t]):
            score[t, e] = 5.0 - j
    inp["x"] = np.concatenate([np.eye(T), np.zeros((T, d - T))], axis=1)
    inp["w_r"] = np.concatenate([score.T, np.zeros((E, d - T))], axis=1)
    out = om.moe_forward(inp, k, "relu", capacity_factor=c["capacity_factor"])
    assert out["router"].idx.tolist() == c["idx"]
    for t in c["fully_dropped_tokens"]:
        assert np.all(out["y"][t] == 0.0)
    # token 2 keeps slot 0 only: y = w[2,0] * FFN_{e}(x_2) with the original w
    e = c["idx"][2][0]
    ref = out["router"].w[2, 0] * _torch_ffn(inp["x"][2:3], inp["w1"][e], None, inp["w2"][e], "relu")[0]
    assert np.allclose(out["y"][2], ref, atol=1e-13)


def pin_capacity_switch_workload():
    # ceil(1.25 * 8192 * 1 / 8) = 1280
    assert om.capacity(8192, 1, 8, 1.25) == 1280
    assert om.capacity(100, 2, 8, 0.0) == 200


def pin_dispatch_invariants():
    for trial in range(30):
        T = int(RNG.integers(1, 300))
        E = int(RNG.integers(1, 40))
        k = int(RNG.integers(1, min(E, 8) + 1))
        idx = np.stack([RNG.permutation(E)[:k] for _ in range(T)])
        C = int(RNG.integers(1, T * k + 2))
        dp = om.dispatch(idx, E, C)
        assert dp.counts.sum() == T * k
        assert np.array_equal(dp.kept_counts, np.minimum(dp.counts, C))
        assert np.all(np.diff(dp.offsets) >= 0) and dp.offsets[-1] == dp.perm.shape[0]
        assert dp.n_dropped == T * k - dp.perm.shape[0]
        flat = idx.reshape(-1)
        for e in range(E):
            seg = dp.perm[dp.offsets[e]:dp.offsets[e + 1]]
            assert np.all(flat[seg] == e)
            assert np.all(np.diff(seg) > 0)                      # stable: f order
            assert np.array_equal(seg, np.nonzero(flat == e)[0][:C])   # first C kept
        kept = dp.inv >= 0
        assert np.array_equal(dp.inv[dp.perm], np.arange(dp.perm.shape[0]))
        assert kept.sum() == dp.perm.shape[0]


# ----------------------------------------------------------------- quantile balancing

def pin_quantile_vs_numpy():
    for _ in range(50):
        n = int(RNG.integers(1, 500))
        v = RNG.normal(size=n)
        q = float(RNG.uniform())
        assert abs(om.quantile_linear(v, q) - float(np.quantile(v, q, method="linear"))) < 1e-13
    v = np.array([3.0, 1.0, 2.0, 4.0])
    assert om.quantile_linear(v, 1.0) == 4.0 and om.quantile_linear(v, 0.0) == 1.0
    assert abs(om.quantile_linear(v, 0.5) - 2.5) < 1e-15


def pin_quantile_balance_share():
    T, E, k = 1000, 16, 2
    probs = om.softmax(RNG.normal(size=(T, E)) + np.log(np.arange(1, E + 1.0))[None, :] * -1.1)
    b = om.quantile_select_bias(probs, k)
    h = (T - 1) * (1 - k / E)
    expect_above = T - 1 - math.floor(h)
    for e in range(E):
        assert int(np.sum(probs[:, e] + b[e] > 0)) == expect_above
    r = om.route(np.log(probs), np.eye(E), k, quantile_balance=True)
    assert np.allclose(r.select_bias, b)
    before = om.load_stats(probs, om.topk_desc(probs, k), E)["load_max_over_mean"]
    after = om.load_stats(probs, r.idx, E)["load_max_over_mean"]
    assert after < before


def pin_round_to_bf16():
    # fp32-representable values: torch's float32 -> bfloat16 conversion rounds
    # to nearest even in one step, the same definition.
    v = (RNG.normal(size=5000) * np.exp(RNG.uniform(-30, 30, size=5000))).astype(np.float32)
    v = np.concatenate([v, np.float32([0.0, -0.0, 1.0, 3.0, 1e-40, -2.5e-39])])
    ref = torch.tensor(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(om.round_to_bf16(v.astype(np.float64)), ref)
    # ties go to the even neighbour (spacing 2^-7 on [1, 2))
    assert om.round_to_bf16(np.array([1 + 2.0 ** -8]))[0] == 1.0
    assert om.round_to_bf16(np.array([1 + 3 * 2.0 ** -8]))[0] == 1 + 2.0 ** -6
    assert om.round_to_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -30]))[0] == 1 + 2.0 ** -7


def pin_bf16_activation_ffn():
    # E = 1 with a bf16 intermediate: the page's Expert in a bf16 model stores
    # h in bf16 before w2; torch.nn.functional in float64 with h rounded by torch.
    inp = _rand_layer(13, 16, 1, 24, "swiglu")
    out = om.moe_forward(inp, 1, "swiglu", act_dtype="bf16")
    x, w1, w3, w2 = (torch.tensor(np.asarray(a, dtype=np.float64))
                     for a in (inp["x"], inp["w1"][0], inp["w3"][0], inp["w2"][0]))
    h = Fnn.silu(Fnn.linear(x, w1)) * Fnn.linear(x, w3)
    h = h.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    ref = Fnn.linear(h, w2).numpy()
    assert np.allclose(out["y"], ref, atol=1e-12)
    exact = om.moe_forward(inp, 1, "swiglu")
    assert not np.allclose(out["y"], exact["y"], atol=1e-6)   # the rounding is visible


PINS = [pin_top2_example, pin_aux_worked_example, pin_selection_bias_example,
        pin_uniform_aux_is_one, pin_topk_bruteforce, pin_softmax_closed_forms,
        pin_router_logits_layout, pin_single_expert_is_dense_ffn, pin_identical_experts,
        pin_all_experts_is_dense_mixture, pin_shared_expert_added, pin_capacity_cases,
        pin_capacity_switch_workload, pin_dispatch_invariants, pin_quantile_vs_numpy,
        pin_quantile_balance_share, pin_round_to_bf16, pin_bf16_activation_ffn]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ----------------------------------------------------------------- planted mistakes

def _mut_no_renorm(probs, idx):
    return np.take_along_axis(probs, idx, axis=1)


def _mut_f_over_T(probs, idx, E):
    T, k = idx.shape
    counts = np.bincount(idx.reshape(-1), minlength=E)
    f = counts / float(T)
    p = probs.mean(axis=0)
    return {"counts": counts, "f": f, "p": p, "aux": E * float(np.sum(f * p)),
            "load_max_over_mean": float(counts.max()) / (T * k / E)}


def _mut_topk_ascending(scores, k):
    return np.argsort(scores, axis=1, kind="stable")[:, :k]


def _mut_topk_unstable_ties(scores, k):
    # equal scores resolved toward the HIGHER expert index
    E = scores.shape[1]
    return (E - 1 - np.argsort(-scores[:, ::-1], axis=1, kind="stable"))[:, :k]


_ORIG_EXPERT_FFN = om.expert_ffn


def _mut_silu_on_w3(x_rows, w1, w3, w2, act):
    if act == "swiglu":
        return _ORIG_EXPERT_FFN(x_rows, w3, w1, w2, act)     # gate and up swapped
    return _ORIG_EXPERT_FFN(x_rows, w1, w3, w2, act)


def _mut_router_reversed_experts(x, w_r, logit_bias=None):
    lg = (om._f64(x) @ om._f64(w_r).T)[:, ::-1]     # wrong expert index mapping
    if logit_bias is not None:
        lg = lg + om._f64(logit_bias)[None, :]
    return lg


def _mut_router_sign(x, w_r, logit_bias=None):
    lg = -(om._f64(x) @ om._f64(w_r).T)             # wrong sign
    if logit_bias is not None:
        lg = lg + om._f64(logit_bias)[None, :]
    return lg


def _mut_drop_last(idx, E, C):
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E)
    order = np.argsort(flat, kind="stable")
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    rank = np.arange(T * k) - starts[flat[order]]
    keep_sorted = rank >= (counts[flat[order]] - C)            # keeps the LAST C
    perm = order[keep_sorted]
    kept = np.minimum(counts, C)
    inv = np.full(T * k, -1)
    inv[perm] = np.arange(perm.shape[0])
    return om.DispatchOut(counts, kept, np.concatenate([[0], np.cumsum(kept)]), perm, inv,
                          (inv >= 0).reshape(T, k), int(T * k - perm.shape[0]))


def _mut_quantile_wrong_q(probs, k):
    T, E = probs.shape
    return np.array([-om.quantile_linear(probs[:, e], k / E) for e in range(E)])


def _mut_quantile_floor_only(values, q):
    v = np.sort(np.asarray(values, dtype=np.float64))
    return float(v[int(math.floor((v.shape[0] - 1) * q))])


def _mut_softmax_no_max(logits):
    e = np.exp(logits)
    return e / e.sum(axis=0, keepdims=True)         # normalised over the wrong axis


def _mut_round_truncate(a):
    _, e = np.frexp(a)
    q = np.ldexp(1.0, np.maximum(e, -125) - 8)
    return np.trunc(a / q) * q                      # truncation instead of nearest-even


def _mut_capacity_floor(T, k, E, cf):
    return T * k if cf <= 0 else int(cf * T / E)    # drops k (one of the page variants)


MUTATIONS = [
    ("renormalise", _mut_no_renorm),
    ("load_stats", _mut_f_over_T),
    ("topk_desc", _mut_topk_ascending),
    ("topk_desc", _mut_topk_unstable_ties),
    ("expert_ffn", _mut_silu_on_w3),
    ("router_logits", _mut_router_reversed_experts),
    ("router_logits", _mut_router_sign),
    ("dispatch", _mut_drop_last),
    ("quantile_select_bias", _mut_quantile_wrong_q),
    ("quantile_linear", _mut_quantile_floor_only),
    ("softmax", _mut_softmax_no_max),
    ("capacity", _mut_capacity_floor),
    ("round_to_bf16", _mut_round_truncate),
]


@pytest.mark.parametrize("name,mut", MUTATIONS, ids=[f"{n}:{m.__name__}" for n, m in MUTATIONS])
def test_planted_mistakes_are_caught(monkeypatch, name, mut):
    monkeypatch.setattr(om, name, mut)
    failed = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError, TypeError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake in {name}"
