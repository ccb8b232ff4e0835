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


def pin_round_to_fp32():
    # nearest even at 24 significant bits, checked on values built from their
    # binary expansion (spacing 2^-23 on [1, 2)) and against torch's
    # float64 -> float32 conversion of random values over a wide range
    assert om.round_to_fp32(np.array([1 + 2.0 ** -24]))[0] == 1.0
    assert om.round_to_fp32(np.array([1 + 3 * 2.0 ** -24]))[0] == 1 + 2.0 ** -22
    assert om.round_to_fp32(np.array([1 + 2.0 ** -24 + 2.0 ** -40]))[0] == 1 + 2.0 ** -23
    assert om.round_to_fp32(np.array([-(2 + 2.0 ** -23)]))[0] == -2.0
    v = RNG.normal(size=4000) * np.exp(RNG.uniform(-60, 60, size=4000))
    ref = torch.tensor(v, dtype=torch.float64).to(torch.float32).to(torch.float64).numpy()
    assert np.array_equal(om.round_to_fp32(v), ref)


def pin_bf16_activation_ffn():
    # E = 1 with bf16 storage of the intermediate activation (reading R8):
    # h is a bf16 tensor before w2, the output row stays exact (gate weight 1
    # here); torch.nn.functional in float64 with h rounded by torch.
    inp = _rand_layer(13, 16, 1, 24, "swiglu")
    out = om.moe_forward(inp, 1, "swiglu", act_dtype="bf16")
    x, w1, w3, w2 = (torch.tensor(np.asarray(a, dtype=np.float64))
                     for a in (inp["x"], inp["w1"][0], inp["w3"][0], inp["w2"][0]))
    h = Fnn.silu(Fnn.linear(x, w1)) * Fnn.linear(x, w3)
    hb = h.to(torch.float32).to(torch.bfloat16).to(torch.float64)
    ref = Fnn.linear(hb, w2).numpy()
    assert np.allclose(out["y"], ref, atol=1e-12)
    # the output is not rounded: some element lies off the bf16 grid
    assert not np.array_equal(om.round_to_bf16(out["y"]), out["y"])
    exact = om.moe_forward(inp, 1, "swiglu")
    assert np.allclose(exact["y"], Fnn.linear(h, w2).numpy(), atol=1e-12)
    assert not np.allclose(out["y"], exact["y"], atol=1e-6)   # h's rounding is visible


def pin_bf16_mixture_exact_expert_outputs():
    # k = 2 of E = 3 with a shared expert, bf16 storage: each expert rounds
    # its h to bf16 (torch), and the expert outputs, the gate-weighted sum
    # and the shared expert's output are exact float64.
    inp = _rand_layer(11, 16, 3, 24, "swiglu", Fs=20)
    out = om.moe_forward(inp, 2, "swiglu", act_dtype="bf16")
    x = torch.tensor(np.asarray(inp["x"], dtype=np.float64))

    def bf(t):
        return t.to(torch.float32).to(torch.bfloat16).to(torch.float64)

    def expert(w1, w3, w2, rows):
        t = lambda a: torch.tensor(np.asarray(a, dtype=np.float64))
        h = bf(Fnn.silu(Fnn.linear(rows, t(w1))) * Fnn.linear(rows, t(w3)))
        return Fnn.linear(h, t(w2))

    r = out["router"]
    ref = np.zeros_like(out["y"])
    for tok in range(x.shape[0]):
        for j in range(2):
            e = int(r.idx[tok, j])
            o = expert(inp["w1"][e], inp["w3"][e], inp["w2"][e], x[tok:tok + 1])
            ref[tok] += r.w[tok, j] * o[0].numpy()
    ref += expert(inp["ws1"], inp["ws3"], inp["ws2"], x).numpy()
    assert np.allclose(out["y"], ref, atol=1e-12)


def _logit_layer(logits, F):
    """A layer whose router logits are ``logits`` exactly: x = logits,
    W_r = I (d = E), random experts of width F."""
    T, E = logits.shape
    return {"x": logits, "w_r": np.eye(E),
            "w1": RNG.normal(size=(E, F, E)) / math.sqrt(E),
            "w3": RNG.normal(size=(E, F, E)) / math.sqrt(E),
            "w2": RNG.normal(size=(E, E, F)) / math.sqrt(F)}


def pin_ranking_of_tied_tokens():
    # Token 0 has two experts with exactly equal scores: the plain rule puts
    # the lower index first (R5).  Giving the other order through ``ranking``
    # must equal routing on scores nudged to prefer it (the nudge is far below
    # every other gap and moves the weights by ~1e-12), for the top-k, the
    # capacity drops, the statistics and y; tokens not named keep the plain
    # order.
    lg = RNG.normal(size=(12, 4))
    lg[0, 1] = lg[0, 2] = lg[0].max() + 0.5              # experts 1 and 2 tie on token 0
    inp = _logit_layer(lg, 10)
    plain = om.moe_forward(inp, 1, "swiglu", capacity_factor=0.7)
    assert plain["router"].idx[0, 0] == 1
    alt = om.moe_forward(inp, 1, "swiglu", capacity_factor=0.7, ranking={0: [2]})
    nudged = dict(inp, x=lg.copy())
    nudged["x"][0, 2] += 1e-12
    ref = om.moe_forward(nudged, 1, "swiglu", capacity_factor=0.7)
    assert alt["router"].idx[0, 0] == 2
    assert alt["router"].idx.tolist() == ref["router"].idx.tolist()
    assert np.allclose(alt["router"].w, ref["router"].w, atol=1e-12)
    assert alt["dispatch"].perm.tolist() == ref["dispatch"].perm.tolist()
    assert alt["stats"]["counts"].tolist() == ref["stats"]["counts"].tolist()
    assert np.allclose(alt["y"], ref["y"], atol=1e-9)
    assert not np.allclose(alt["y"][0], plain["y"][0], atol=1e-6)
    # k = 2, with and without redirection: the given order of token 0 leads
    # its ranking, the rest of its ranking follows the scores
    lg2 = RNG.normal(size=(10, 5))
    lg2[0, 3] = lg2[0, 4] = lg2[0].max() + 1.0
    inp2 = _logit_layer(lg2, 8)
    n2 = dict(inp2, x=lg2.copy())
    n2["x"][0, 4] += 1e-12
    for rounds in (0, 1):
        a = om.moe_forward(inp2, 2, "swiglu", capacity_factor=0.6, reroute_rounds=rounds,
                           ranking={0: [4, 3]})
        b = om.moe_forward(n2, 2, "swiglu", capacity_factor=0.6, reroute_rounds=rounds)
        assert a["router"].idx.tolist() == b["router"].idx.tolist()
        assert np.allclose(a["router"].w, b["router"].w, atol=1e-12)
        assert a["dispatch"].perm.tolist() == b["dispatch"].perm.tolist()
        assert a["dispatch"].n_dropped == b["dispatch"].n_dropped
        assert np.allclose(a["y"], b["y"], atol=1e-9)
    # a selection bias makes experts 3 and 4 tie in score at the k-th place
    # of token 0 while their probabilities differ: the given order swaps
    # which one is selected, and its weights come from the probabilities
    lg3 = RNG.normal(size=(6, 5))
    lg3[0] = [3.0, -1.0, -2.0, 1.0, 0.5]
    inp3 = _logit_layer(lg3, 8)
    p0 = om.softmax(lg3)[0]
    b4 = p0[3] - p0[4]
    for _ in range(8):
        if p0[4] + b4 == p0[3]:
            break
        b4 = np.nextafter(b4, np.inf if p0[4] + b4 < p0[3] else -np.inf)
    assert p0[4] + b4 == p0[3]
    bias = np.array([0.0, 0.0, 0.0, 0.0, b4])
    inp3["select_bias"] = bias
    plain3 = om.moe_forward(inp3, 2, "swiglu")
    assert plain3["router"].idx[0].tolist() == [0, 3]
    a3 = om.moe_forward(inp3, 2, "swiglu", ranking={0: [0, 4]})
    n3 = dict(inp3, select_bias=bias + np.array([0, 0, 0, 0, 1e-15]))
    b3 = om.moe_forward(n3, 2, "swiglu")
    assert a3["router"].idx.tolist() == b3["router"].idx.tolist()
    assert np.array_equal(a3["router"].w, b3["router"].w)
    assert np.allclose(a3["y"], b3["y"], atol=1e-12)
    assert not np.allclose(a3["router"].w[0], plain3["router"].w[0], atol=1e-3)


def pin_expert_choice_given_set():
    # Expert 0's column ties exactly at its C-th value between tokens 2 and 5;
    # the lower token wins (R11).  Giving the other token through ``chosen``
    # equals expert choice on a column nudged to prefer it.
    T, E, C = 8, 3, 3
    probs = om.softmax(RNG.normal(size=(T, E)))
    col = np.array([0.9, 0.1, 0.5, 0.2, 0.8, 0.5, 0.05, 0.3])
    probs[:, 0] = col
    plain = om.expert_choice(probs, C)
    assert plain.chosen[0].tolist() == [0, 2, 4]
    alt = om.expert_choice(probs, C, chosen={0: [5, 0, 4]})
    nudged = probs.copy()
    nudged[5, 0] += 1e-15
    ref = om.expert_choice(nudged, C)
    assert alt.chosen.tolist() == ref.chosen.tolist()
    assert np.allclose(alt.weight, ref.weight, atol=1e-14)
    assert alt.n_unchosen == ref.n_unchosen


def pin_gate_entropy():
    # closed forms: a uniform router over E experts has entropy ln E, a
    # one-hot router 0; a general distribution against scipy.stats.entropy
    from scipy.stats import entropy as sp_entropy
    for E in (2, 8, 896):
        assert abs(om.gate_entropy(np.full((3, E), 1.0 / E)) - math.log(E)) < 1e-12
    assert om.gate_entropy(np.eye(5)) == 0.0
    p = om.softmax(RNG.normal(size=(7, 11)) * 3)
    ref = float(np.mean([sp_entropy(row) for row in p]))
    assert abs(om.gate_entropy(p) - ref) < 1e-12
    # through the layer: logits = log(p) give back p
    r = om.route(np.log(p), np.eye(11), 2)
    assert abs(om.gate_entropy(r.probs) - ref) < 1e-12


def pin_expert_output_scale():
    # constant outputs: mean c, std 0, max |c|; a +-a pattern: mean 0, std a
    c = om.expert_output_scale({0: np.full((3, 4), -2.5), 2: np.array([[1.5, -1.5], [-1.5, 1.5]])}, 3)
    assert c["mean"].tolist() == [-2.5, 0.0, 0.0]
    assert c["std"].tolist() == [0.0, 0.0, 1.5]
    assert c["max_abs"].tolist() == [2.5, 0.0, 1.5]
    # against torch's reductions of the same values (population std)
    o = RNG.normal(size=(5, 6))
    st = om.expert_output_scale({1: o}, 2)
    ot = torch.tensor(o)
    assert abs(st["mean"][1] - float(ot.mean())) < 1e-14
    assert abs(st["std"][1] - float(ot.std(unbiased=False))) < 1e-14
    assert st["max_abs"][1] == float(ot.abs().max())
    # through the layer: E = 1, no capacity: expert 0's outputs are the dense FFN
    inp = _rand_layer(9, 8, 1, 12, "relu")
    out = om.moe_forward(inp, 1, "relu", observe_outputs=True)
    x, w1, w2 = (torch.tensor(np.asarray(a, dtype=np.float64))
                 for a in (inp["x"], inp["w1"][0], inp["w2"][0]))
    dense = Fnn.linear(Fnn.relu(Fnn.linear(x, w1)), w2)
    ob = out["observe"]["expert_out"]
    assert abs(ob["mean"][0] - float(dense.mean())) < 1e-12
    assert abs(ob["std"][0] - float(dense.std(unbiased=False))) < 1e-12
    assert abs(ob["max_abs"][0] - float(dense.abs().max())) < 1e-12


def pin_observe_drop_and_bias():
    g = load_golden("capacity_cases.json")["cases"][0]
    idx = np.array(g["idx"])
    T, k = idx.shape
    E = g["E"]
    C = om.capacity(T, k, E, g["capacity_factor"])
    dp = om.dispatch(idx, E, C)
    probs = np.full((T, E), 1.0 / E)
    r = om.RouterOut(np.zeros((T, E)), probs, probs, idx, np.ones((T, k)) / k,
                     np.array([0.25, -0.5] + [0.0] * (E - 2)))
    ob = om.observe(r, dp, {}, E, k)
    assert ob["drop_ratio"] == g["n_dropped"] / (T * k)
    assert ob["bias"]["max_abs"] == 0.5 and abs(ob["bias"]["mean_abs"] - 0.75 / E) < 1e-15
    assert abs(ob["gate_entropy"] - math.log(E)) < 1e-12
    assert om.bias_magnitude(None) == {"mean_abs": 0.0, "max_abs": 0.0}


def _scores_from_ranking(ranking):
    ranking = np.asarray(ranking)
    T, E = ranking.shape
    sc = np.zeros((T, E))
    for t in range(T):
        sc[t, ranking[t]] = E - np.arange(E)
    return sc


def pin_reroute_cases():
    g = load_golden("reroute_cases.json")
    for c in g["cases"]:
        sc = _scores_from_ranking(c["ranking"])
        probs = om.softmax(sc)
        out = om.dispatch_reroute(sc, probs, c["k"], c["C"], c["rounds"])
        assert out.slot_expert.tolist() == c["slot_expert"], c["note"]
        assert out.slot_round.tolist() == c["slot_round"], c["note"]
        assert out.kept_counts.tolist() == c["kept_counts"], c["note"]
        assert out.perm.tolist() == c["perm"], c["note"]
        assert out.n_dropped == c["n_dropped"], c["note"]


def pin_reroute_invariants():
    rng = np.random.default_rng(21)
    for T, E, k, cf in [(200, 8, 1, 1.0), (150, 16, 2, 0.8), (90, 32, 4, 1.1), (60, 5, 2, 0.5)]:
        pop = 1.0 / np.arange(1, E + 1) ** 1.3
        sc = om.softmax(rng.normal(size=(T, E)) + np.log(pop)[None, :])
        C = om.capacity(T, k, E, cf)
        plain = om.dispatch(om.topk_desc(sc, k), E, C)
        r0 = om.dispatch_reroute(sc, sc, k, C, 0)
        # zero rounds is the plain capacity rule
        assert r0.perm.tolist() == plain.perm.tolist() and r0.n_dropped == plain.n_dropped
        assert r0.inv.tolist() == plain.inv.tolist()
        prev = r0.n_dropped
        top = om.topk_desc(sc, k)
        norm = np.take_along_axis(sc, top, axis=1).sum(axis=1)
        for R in (1, 2, 3):
            r = om.dispatch_reroute(sc, sc, k, C, R)
            assert np.all(r.kept_counts <= C)
            assert r.kept_counts.sum() + r.n_dropped == T * k
            assert r.n_dropped <= prev            # more rounds never drop more
            prev = r.n_dropped
            # every expert serves its first-choice slots exactly as the plain rule
            first = (r.slot_round == 0)
            assert np.array_equal(first, plain.keep)
            for t in range(T):
                served = [e for e in r.slot_expert[t] if e >= 0]
                assert len(served) == len(set(served))           # distinct experts
                for j in range(k):
                    e = r.slot_expert[t, j]
                    if r.slot_round[t, j] > 0:
                        assert e not in top[t]                  # redirected beyond top-k
                    if e >= 0:
                        assert abs(r.slot_w[t, j] - sc[t, e] / norm[t]) < 1e-15
                    else:
                        assert r.slot_w[t, j] == 0.0
            # grouped rows: each expert's rows are its served slots
            for e in range(E):
                a, b = r.offsets[e], r.offsets[e + 1]
                assert all(r.slot_expert.reshape(-1)[r.perm[a:b]] == e)
        # enough capacity: nothing overflows, nothing is redirected
        big = om.dispatch_reroute(sc, sc, k, T * k, 2)
        assert big.n_dropped == 0 and np.all(big.slot_round == 0)


def pin_expert_choice_case():
    g = load_golden("expert_choice_case.json")
    ec = om.expert_choice(np.array(g["probs"]), g["C"])
    assert ec.chosen.tolist() == g["chosen"]
    assert np.allclose(ec.weight, g["weight"], atol=1e-15)
    assert ec.n_unchosen == g["n_unchosen"]
    assert ec.offsets.tolist() == [0, 2, 4]


def pin_expert_choice_bruteforce():
    # every C-subset of a column: the chosen one has the largest sum, and among
    # equal sums the lexicographically smallest token set
    rng = np.random.default_rng(8)
    for T, E, C in [(6, 3, 2), (7, 2, 3), (5, 4, 5), (6, 2, 4)]:
        probs = om.softmax(np.round(rng.normal(size=(T, E)), 1))   # rounding makes ties
        ec = om.expert_choice(probs, C)
        for e in range(E):
            best = None
            for sub in itertools.combinations(range(T), min(C, T)):
                key = (-probs[list(sub), e].sum(), sorted(sub))
                # ties in the sum resolved by preferring the largest values of the
                # lowest tokens: compare the per-token sorted selection instead
                if best is None or key < best:
                    best = key
            chosen_vals = np.sort(probs[ec.chosen[e], e])
            best_vals = np.sort(probs[best[1], e])
            assert np.allclose(chosen_vals, best_vals, atol=1e-15)
            # the exact tie rule: a picked token is never beaten by an unpicked
            # one with a larger value, or an equal value and a lower index
            picked = set(ec.chosen[e].tolist())
            for t in picked:
                for u in set(range(T)) - picked:
                    assert probs[t, e] > probs[u, e] or (probs[t, e] == probs[u, e] and t < u)


def pin_expert_choice_full_capacity_is_dense_mixture():
    # C >= T: every expert takes every token, y = sum_e p_e FFN_e(x), which is
    # token choice with k = E (renormalised weights p / sum p = p)
    inp = _rand_layer(6, 8, 3, 10, "swiglu")
    ec = om.moe_forward_expert_choice(inp, 3, "swiglu", capacity_factor=1.0)
    assert ec["ec"].n_unchosen == 0 and ec["capacity"] == 6
    tc = om.moe_forward(inp, 3, "swiglu")
    assert np.allclose(ec["y"], tc["y"], atol=1e-12)


PINS = [pin_top2_example, pin_aux_worked_example, pin_selection_bias_example,
        pin_uniform_aux_is_one, pin_topk_bruteforce, pin_softmax_closed_forms,
        pin_router_logits_layout, pin_single_expert_is_dense_ffn, pin_identical_experts,
        pin_all_experts_is_dense_mixture, pin_shared_expert_added, pin_capacity_cases,
        pin_capacity_switch_workload, pin_dispatch_invariants, pin_quantile_vs_numpy,
        pin_quantile_balance_share, pin_round_to_bf16, pin_round_to_fp32,
        pin_bf16_activation_ffn, pin_bf16_mixture_exact_expert_outputs,
        pin_ranking_of_tied_tokens, pin_expert_choice_given_set,
        pin_gate_entropy, pin_expert_output_scale, pin_observe_drop_and_bias,
        pin_reroute_cases, pin_reroute_invariants, pin_expert_choice_case,
        pin_expert_choice_bruteforce, pin_expert_choice_full_capacity_is_dense_mixture]


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


def _mut_ffn_output_rounded(x_rows, w1, w3, w2, act, act_dtype="fp64"):
    a = x_rows @ om._f64(w1).T
    h = om._silu(a) * (x_rows @ om._f64(w3).T) if act == "swiglu" else np.maximum(a, 0.0)
    h = om.ACT_ROUNDING[act_dtype](h)
    return om.ACT_ROUNDING[act_dtype](h @ om._f64(w2).T)   # output row rounded too


def _mut_ffn_h_unrounded(x_rows, w1, w3, w2, act, act_dtype="fp64"):
    a = x_rows @ om._f64(w1).T
    h = om._silu(a) * (x_rows @ om._f64(w3).T) if act == "swiglu" else np.maximum(a, 0.0)
    return h @ om._f64(w2).T                                # h left at full precision


def _mut_round_fp32_truncate(a):
    v = np.asarray(a, dtype=np.float64)
    f = v.astype(np.float32).astype(np.float64)
    over = np.abs(f) > np.abs(v)                            # rounded away from zero
    return np.where(over, np.nextafter(f.astype(np.float32), np.float32(0)).astype(np.float64), f)


_ORIG_WITH_RANKING = om.with_ranking


def _mut_ranking_keeps_weights(r, ranking):
    out = _ORIG_WITH_RANKING(r, ranking)
    out.w = r.w.copy()                                      # weights not renormalised
    return out


def _mut_ranking_ignored(r, ranking):
    return r


def _mut_capacity_floor(T, k, E, cf):
    return T * k if cf <= 0 else int(cf * T / E)    # drops k (one of the page variants)


def _mut_entropy_log2(probs):
    p = np.asarray(probs, dtype=np.float64)
    safe = np.where(p > 0, p, 1.0)
    return float(np.mean(-np.sum(np.where(p > 0, p * np.log2(safe), 0.0), axis=1)))   # bits


def _mut_scale_sample_std(outputs, E):
    mean, std, mx = np.zeros(E), np.zeros(E), np.zeros(E)
    for e, o in outputs.items():
        mean[e], std[e], mx[e] = o.mean(), o.std(ddof=1), o.max()   # sample std, signed max
    return {"mean": mean, "std": std, "max_abs": mx}


_ORIG_REROUTE = om.dispatch_reroute


def _mut_reroute_same_candidate(scores, probs, k, C, rounds):
    # every unserved slot of a token takes the SAME next candidate
    T, E = scores.shape
    order = np.argsort(-scores, axis=1, kind="stable")
    top = order[:, :k]
    norm = np.take_along_axis(probs, top, axis=1).sum(axis=1)
    slot_e = top.copy()
    served = np.full((T, k), -1)
    rnd = np.full((T, k), -1)
    rows = [[] for _ in range(E)]
    nxt = np.full(T, k)
    for r in range(rounds + 1):
        if r > 0:
            for t in range(T):
                if nxt[t] < E and (served[t] < 0).any():
                    slot_e[t, served[t] < 0] = order[t, nxt[t]]
                    nxt[t] += 1
        for t in range(T):
            for j in range(k):
                e = int(slot_e[t, j])
                if served[t, j] < 0 and len(rows[e]) < C:
                    rows[e].append(t * k + j)
                    served[t, j], rnd[t, j] = e, r
    kept = np.array([len(x) for x in rows])
    perm = np.array([f for x in rows for f in x], dtype=np.int64)
    inv = np.full(T * k, -1)
    inv[perm] = np.arange(perm.shape[0])
    w = np.where(served >= 0, np.take_along_axis(probs, np.maximum(served, 0), axis=1)
                 / norm[:, None], 0.0)
    return om.RerouteOut(served, w, rnd, np.bincount(top.reshape(-1), minlength=E), kept,
                         np.concatenate([[0], np.cumsum(kept)]), perm, inv,
                         int(T * k - perm.shape[0]))


def _mut_reroute_renormalised(scores, probs, k, C, rounds):
    out = _ORIG_REROUTE(scores, probs, k, C, rounds)
    tot = out.slot_w.sum(axis=1, keepdims=True)
    out.slot_w = np.where(tot > 0, out.slot_w / np.where(tot > 0, tot, 1), 0)
    return out


def _mut_ec_ties_high(probs, C):
    T, E = probs.shape
    Cn = min(C, T)
    chosen = np.zeros((E, Cn), dtype=np.int64)
    weight = np.zeros((E, Cn))
    picked = np.zeros(T, dtype=bool)
    for e in range(E):
        order = (T - 1 - np.argsort(-probs[::-1, e], kind="stable"))   # ties: HIGHER token
        top = np.sort(order[:Cn])
        chosen[e], weight[e], picked[top] = top, probs[top, e], True
    return om.ExpertChoiceOut(chosen, weight, np.full(E, Cn), np.arange(E + 1) * Cn,
                              int(T - picked.sum()))


def _mut_ec_renormalised(probs, C):
    out = _ORIG_EC(probs, C)
    out.weight = out.weight / out.weight.sum(axis=1, keepdims=True)
    return out


_ORIG_EC = om.expert_choice

MUTATIONS = [
    ("gate_entropy", _mut_entropy_log2),
    ("expert_choice", _mut_ec_ties_high),
    ("expert_choice", _mut_ec_renormalised),
    ("dispatch_reroute", _mut_reroute_same_candidate),
    ("dispatch_reroute", _mut_reroute_renormalised),
    ("expert_output_scale", _mut_scale_sample_std),
    ("renormalise", _mut_no_renorm),
    ("load_stats", _mut_f_over_T),
    ("topk_desc", _mut_topk_ascending),
    ("topk_desc", _mut_topk_unstable_ties),
    ("expert_ffn", _mut_silu_on_w3),
    ("expert_ffn", _mut_ffn_output_rounded),
    ("expert_ffn", _mut_ffn_h_unrounded),
    ("round_to_fp32", _mut_round_fp32_truncate),
    ("with_ranking", _mut_ranking_keeps_weights),
    ("with_ranking", _mut_ranking_ignored),
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
