"""GPU parity of capacity overflow sent to the next-best experts (the
"dropped or redirected to the next best expert" rule of the waylandz.com
ch. 30 §30.5.2) against the fp64 oracle: the dispatch stage fed with the
oracle's rankings (bit-exact), and the whole layer on reduced-size and
full-size workloads under the comparison rules of tests/parity.py."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle.moe_oracle as om
import sparse_mixture_experts_47_b300 as moe
from tests.conftest import load_golden
from tests.parity import full_check, sample_tokens

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _stage(scores, probs, k, C, R, E):
    """Run moe_dispatch_reroute on the oracle's ranking of `scores`."""
    T = scores.shape[0]
    order = np.argsort(-scores, axis=1, kind="stable")
    top = order[:, :k]
    norm = np.take_along_axis(probs, top, axis=1).sum(axis=1, keepdims=True)
    # a capacity factor that gives exactly C
    cfg = moe.MoEConfig(T=T, d_model=8, n_experts=E, top_k=k, d_ff=8,
                        capacity_factor=float(C) * E / (T * k) - 1e-6, reroute_rounds=R)
    assert moe.capacity(cfg) == C
    nc = moe.reroute_candidates(cfg)
    cand = order[:, k:k + nc]
    t32 = lambda a, dt: torch.tensor(np.ascontiguousarray(a), dtype=dt, device=DEV)
    w = np.take_along_axis(probs, top, axis=1) / norm
    cw = np.take_along_axis(probs, cand, axis=1) / norm
    out = moe.dispatch_reroute(cfg, t32(top, torch.int32), t32(w, torch.float32),
                               t32(cand if nc else np.zeros((T, 1)), torch.int32),
                               t32(cw if nc else np.zeros((T, 1)), torch.float32))
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    return {kk: v.cpu().numpy() for kk, v in out.items()}, w, cw


def _compare(got, ref, E):
    assert got["slot_expert"].tolist() == ref.slot_expert.tolist()
    assert got["offsets"].tolist() == ref.offsets.tolist()
    n = int(ref.offsets[-1])
    assert got["perm"][:n].tolist() == ref.perm.tolist()
    assert got["inv"].tolist() == ref.inv.tolist()
    assert int(got["n_dropped"][0]) == ref.n_dropped
    assert got["counts"].tolist() == ref.counts.tolist()


def test_reroute_stage_golden_cases():
    for c in load_golden("reroute_cases.json")["cases"]:
        ranking = np.array(c["ranking"])
        T, E = ranking.shape
        sc = np.zeros((T, E))
        for t in range(T):
            sc[t, ranking[t]] = E - np.arange(E)
        probs = om.softmax(sc)
        ref = om.dispatch_reroute(sc, probs, c["k"], c["C"], c["rounds"])
        got, _, _ = _stage(sc, probs, c["k"], c["C"], c["rounds"], E)
        _compare(got, ref, E)
        assert got["slot_expert"].tolist() == c["slot_expert"]


@pytest.mark.parametrize("T,E,k,cf,R", [(1000, 8, 1, 1.25, 1), (3000, 8, 2, 1.0, 2),
                                        (2500, 64, 8, 1.0, 3), (777, 16, 4, 0.7, 4),
                                        (5000, 256, 8, 1.0, 1), (1, 4, 2, 0.5, 1)])
def test_reroute_stage_bit_exact(T, E, k, cf, R):
    rng = np.random.default_rng(T + E)
    pop = 1.0 / np.arange(1, E + 1) ** 1.2
    probs = om.softmax(rng.normal(size=(T, E)) + np.log(pop)[None, :] * 2)
    probs = probs.astype(np.float32).astype(np.float64)   # the values the kernel sees
    C = om.capacity(T, k, E, cf)
    ref = om.dispatch_reroute(probs, probs, k, C, R)
    got, w, cw = _stage(probs, probs, k, C, R, E)
    _compare(got, ref, E)
    # weights: the fp32 copies of the oracle's weights of the serving expert
    ok = ref.slot_expert >= 0
    assert np.array_equal(got["slot_w"][~ok], np.zeros((~ok).sum(), dtype=np.float32))
    assert np.max(np.abs(got["slot_w"][ok] - ref.slot_w[ok])) <= 1e-6


SMALL = {
    "switch_reroute_small": (mi.workload("switch_reroute").with_sizes(d_model=256, d_ff=512), 1000),
    "mixtral_cap_reroute_small": (mi.workload("mixtral_cap").with_sizes(
        d_model=512, d_ff=1024, reroute_rounds=2), 300),
    "deepseek_cap_reroute_small": (mi.workload("deepseek_cap").with_sizes(
        d_model=256, n_experts=64, d_ff=128, d_ff_shared=192, reroute_rounds=2), 400),
    # 16 slots and 16 candidates per token (the 32 the router can rank):
    # every expert of 32 ranked, and 32 of 64 on the tensor-core router with
    # the selection bias on the logits
    "mixtral_cap_reroute_k16": (mi.workload("mixtral_cap").with_sizes(
        d_model=256, n_experts=32, top_k=16, d_ff=256, reroute_rounds=1), 300),
    "deepseek_cap_reroute_k16_logits": (mi.workload("deepseek_cap").with_sizes(
        d_model=256, n_experts=64, top_k=16, d_ff=128, d_ff_shared=192, reroute_rounds=1,
        select_space="logits"), 300),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_reroute_small_full_oracle(name):
    w, T = SMALL[name]
    inp = mi.generate(w, T, DEV)
    rep, gpu, orc = full_check(w, T, inp, want_slots=True)
    print(name, rep)
    plain = om.moe_forward(inp, w.top_k, w.act, w.capacity_factor, w.select_space, False, [0],
                           "bf16")
    assert orc["dispatch"].n_dropped < plain["dispatch"].n_dropped   # redirection helps
    assert (orc["dispatch"].slot_round > 0).any()
    # the served expert and weight of every slot
    assert np.array_equal(gpu["slot_expert"], orc["dispatch"].slot_expert)
    assert np.max(np.abs(gpu["slot_w"] - orc["dispatch"].slot_w)) <= 1e-5


def test_layer_reroute_full_size():
    w = mi.workload("switch_reroute")
    T = 8192
    inp = mi.generate(w, T, DEV)
    rep, gpu, orc = full_check(w, T, inp, sample_tokens(T, 192))
    print(rep, "dropped", int(gpu["n_dropped"][0]))
    assert int(gpu["n_dropped"][0]) < 1997 // 2
