"""GPU parity of the layer and of each stage against the fp64 oracle, on
reduced-size versions of every workload (the oracle covers every token), the
pages' printed examples through the kernels, edge cases and determinism."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle.moe_oracle as om
import sparse_mixture_experts_47_b300 as moe
from tests.conftest import load_golden
from tests.parity import (FP_ATOL, W_ATOL, act_dtype, compare_y, full_check, gpu_layer,
                          oracle_layer, weights_dict, y_tol)

pytestmark = pytest.mark.gpu
DEV = "cuda"

SMALL = {
    "tiny": (mi.workload("tiny"), 64),
    "switch_small": (mi.workload("switch").with_sizes(d_model=256, d_ff=512), 1000),
    "mixtral_small": (mi.workload("mixtral").with_sizes(d_model=512, d_ff=1024), 300),
    "deepseek_small": (mi.workload("deepseek").with_sizes(d_model=256, n_experts=64, d_ff=128,
                                                          d_ff_shared=192), 200),
    "e896_small": (mi.workload("e896").with_sizes(d_model=128, d_ff=64), 2000),
    "mixtral_T1": (mi.workload("mixtral").with_sizes(d_model=256, d_ff=512), 1),
    "mixtral_T3": (mi.workload("mixtral").with_sizes(d_model=256, d_ff=512), 3),
    "mixtral_T17": (mi.workload("mixtral").with_sizes(d_model=256, d_ff=512), 17),
    "switch_ragged": (mi.workload("switch").with_sizes(d_model=136, d_ff=264), 333),
    # a few rows per expert: weights on the MMA's M side, reduction split
    # over CTAs (partial sums added by the activation and combine kernels)
    "mixtral_T1_split": (mi.workload("mixtral").with_sizes(d_model=1024, d_ff=2048), 1),
    "mixtral_T5_split": (mi.workload("mixtral").with_sizes(d_model=1024, d_ff=2048), 5),
    "switch_T20_split": (mi.workload("switch").with_sizes(d_model=1024, d_ff=2048), 20),
    "switch_T3_split": (mi.workload("switch").with_sizes(d_model=2048, d_ff=512), 3),
    "deepseek_T100_split": (mi.workload("deepseek").with_sizes(d_model=1024, n_experts=64,
                                                               d_ff=256, d_ff_shared=1024), 100),
    # about 75-280 rows per expert: 128-row tiles up, and a down projection on
    # tiles of up to 256 rows whose MMA N is the tile's row count rounded to
    # 16 (ragged widths, a split reduction, many experts, skewed loads)
    "mixtral_var": (mi.workload("mixtral").with_sizes(d_model=512, d_ff=1024), 1100),
    "switch_var_ragged": (mi.workload("switch").with_sizes(d_model=136, d_ff=264), 2080),
    "mixtral_var_split": (mi.workload("mixtral").with_sizes(d_model=1024, d_ff=2048), 584),
    "e896_var": (mi.workload("e896").with_sizes(d_model=128, d_ff=64), 8192),
    "deepseek_var": (mi.workload("deepseek").with_sizes(d_model=256, n_experts=64, d_ff=384,
                                                        d_ff_shared=192), 1200),
    # about 525 rows per expert and a reduction of 8192: the down projection
    # on tiles of 256 rows, two M = 128 MMAs per weight stage (ragged tails)
    "mixtral_wide": (mi.workload("mixtral").with_sizes(d_model=2048, d_ff=8192), 2100),
    # capacity factor 1.0 with k > 1: overflow dropped in (t, j) order
    "mixtral_cap_small": (mi.workload("mixtral_cap").with_sizes(d_model=512, d_ff=1024), 300),
    "deepseek_cap_small": (mi.workload("deepseek_cap").with_sizes(
        d_model=256, n_experts=64, d_ff=128, d_ff_shared=192), 400),
    # router paths by expert count: 8 < E <= 32 (W_r slices in shared memory,
    # 16 and 32 lanes per token), E > 32 not a multiple of 4 in a bf16 layer
    # (the CUDA-core tiled router), and an fp32 layer with E > 32
    "mixtral_E12": (mi.workload("mixtral").with_sizes(d_model=256, n_experts=12, d_ff=512), 300),
    "mixtral_E24_k3": (mi.workload("mixtral").with_sizes(d_model=512, n_experts=24, top_k=3,
                                                         d_ff=256), 400),
    "deepseek_E50": (mi.workload("deepseek").with_sizes(d_model=256, n_experts=50, d_ff=128,
                                                        d_ff_shared=192), 300),
    "tiny_E40": (mi.workload("tiny").with_sizes(n_experts=40, top_k=3), 200),
    "e896_E50": (mi.workload("e896").with_sizes(d_model=128, n_experts=50, d_ff=64), 600),
    # top-k at its largest (16): 32 experts on one warp per token, and 64
    # experts on the tensor-core router with the selection bias
    "mixtral_E32_k16": (mi.workload("mixtral").with_sizes(d_model=256, n_experts=32, top_k=16,
                                                          d_ff=256), 200),
    "deepseek_E64_k16": (mi.workload("deepseek").with_sizes(d_model=256, n_experts=64, top_k=16,
                                                            d_ff=128, d_ff_shared=192), 300),
    # the selection bias added to the logits instead of the probabilities, on
    # each router path: 8 experts, 24 (W_r slices in shared memory), 50 (the
    # CUDA-core tiled router), 64 (tensor cores), and an fp32 layer
    "mixtral_logits": (mi.workload("mixtral").with_sizes(
        d_model=256, d_ff=512, select_bias="uniform", select_space="logits"), 300),
    "mixtral_E24_logits": (mi.workload("mixtral").with_sizes(
        d_model=256, n_experts=24, top_k=3, d_ff=256, select_bias="uniform",
        select_space="logits"), 300),
    "deepseek_E50_logits": (mi.workload("deepseek").with_sizes(
        d_model=256, n_experts=50, d_ff=128, d_ff_shared=192, select_space="logits"), 300),
    "deepseek_logits": (mi.workload("deepseek").with_sizes(
        d_model=256, n_experts=64, d_ff=128, d_ff_shared=192, select_space="logits"), 300),
    "tiny_E40_logits": (mi.workload("tiny").with_sizes(n_experts=40, top_k=3, select_bias="uniform",
                                                       select_space="logits"), 200),
    # a capacity of 4 rows per expert (capacity factor 0.05): almost every
    # slot dropped, four rows per expert kept
    "mixtral_cap_tiny": (mi.workload("mixtral_cap").with_sizes(d_model=256, d_ff=512,
                                                               capacity_factor=0.05), 300),
    # degenerate expert counts: one expert (a dense FFN: every probability 1,
    # every gate weight 1), and k = E (every token to every expert)
    "mixtral_E1": (mi.workload("mixtral").with_sizes(d_model=256, n_experts=1, top_k=1, d_ff=512),
                   300),
    "tiny_E1": (mi.workload("tiny").with_sizes(n_experts=1, top_k=1), 64),
    "mixtral_kE": (mi.workload("mixtral").with_sizes(d_model=256, n_experts=4, top_k=4, d_ff=256),
                   200),
    # the largest expert count (1024) with the largest k (16), with the
    # selection bias; and quantile balancing over 1024 experts
    "deepseek_E1024_k16": (mi.workload("deepseek").with_sizes(
        d_model=256, n_experts=1024, top_k=16, d_ff=64, d_ff_shared=128), 2048),
    "e896_E1024": (mi.workload("e896").with_sizes(d_model=128, n_experts=1024, d_ff=64), 4096),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_small_full_oracle(name):
    w, T = SMALL[name]
    inp = mi.generate(w, T, DEV)
    rep, gpu, orc = full_check(w, T, inp)
    print(name, rep)
    if w.capacity_factor > 0 and T >= 16:
        assert orc["dispatch"].n_dropped > 0          # the skewed expert overflows


@pytest.mark.parametrize("name,T", [("mixtral_small", 3000), ("switch_small", 2000)])
def test_every_token_to_one_expert(name, T):
    """Router collapse: a logit offset of +10 on expert 0 sends every token
    there first (k = 2: one 3000-row group on SM-pair tiles and the second
    choices spread over the rest; k = 1 with capacity 1.25: one expert full,
    the rest of the batch dropped and seven experts empty)."""
    w, _ = SMALL[name]
    inp = mi.generate(w, T, DEV)
    lb = torch.zeros(w.n_experts, dtype=torch.float32, device=DEV)
    lb[0] = 10.0
    inp["logit_bias"] = lb
    rep, gpu, orc = full_check(w, T, inp)
    print(name, rep)
    assert np.all(gpu["idx"][:, 0] == 0)
    counts = orc["stats"]["counts"]
    assert counts[0] == T
    if w.capacity_factor > 0:
        assert int(gpu["n_dropped"][0]) == T - om.capacity(T, w.top_k, w.n_experts,
                                                            w.capacity_factor)


def test_layer_deterministic():
    w, T = SMALL["deepseek_small"]
    inp = mi.generate(w, T, DEV)
    a = gpu_layer(w, T, inp)
    b = gpu_layer(w, T, inp)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_bf16_output_matches_fp32_output():
    w, T = SMALL["mixtral_small"]
    inp = mi.generate(w, T, DEV)
    a = gpu_layer(w, T, inp, moe.DTYPE_FP32)
    b = gpu_layer(w, T, inp, moe.DTYPE_BF16)
    ref = torch.tensor(a["y"]).to(torch.bfloat16).float().numpy()
    assert np.array_equal(ref, b["y"])


@pytest.mark.parametrize("name,T", [("mixtral_small", 300), ("mixtral_small", 2000),
                                    ("deepseek_small", 200), ("deepseek_small", 5000)])
def test_batch_invariance(name, T):
    """A token's routing does not depend on the batch it comes in (the
    pages' batch=1 vs batch=64 check): indices and gate weights are
    bit-identical, outputs agree within the layer's y tolerance (GEMM tiling
    differs)."""
    w, _ = SMALL[name]
    inp = mi.generate(w, T, DEV)
    big = gpu_layer(w, T, inp)
    rms = float(np.sqrt(np.mean(big["y"].astype(np.float64) ** 2)))
    for t in (1, 16):
        sub = dict(inp)
        sub["x"] = inp["x"][:t].contiguous()
        small = gpu_layer(w, t, sub)
        assert np.array_equal(small["idx"], big["idx"][:t])
        assert np.array_equal(small["w"], big["w"][:t])
        assert np.max(np.abs(small["y"] - big["y"][:t])) <= y_tol(w) * rms


def test_layer_graph_and_pipeline_match_eager():
    """The captured layer (LayerGraph) and the copy-overlapped pipeline
    (LayerPipeline) give exactly the eager call's outputs, batch by batch."""
    w, T = SMALL["mixtral_small"]
    inp = mi.generate(w, T, DEV)
    cfg = moe.config_for(w, T, moe.DTYPE_BF16)
    wts = weights_dict(inp)
    g = torch.Generator(device=DEV)
    g.manual_seed(11)
    batches = [torch.randn(inp["x"].shape, generator=g, device=DEV).to(inp["x"].dtype)
               for _ in range(5)]
    eager = [moe.layer_forward(cfg, b, wts)["y"].float().cpu() for b in batches]
    graph = moe.LayerGraph(cfg, batches[0].clone(), wts)
    for b, ref in zip(batches, eager):
        graph.x.copy_(b)
        assert torch.equal(graph.replay()["y"].float().cpu(), ref)
    xs = [b.cpu().pin_memory() for b in batches]
    for overlap in (True, False):      # three streams, and the one-stream path
        pipe = moe.LayerPipeline(cfg, wts, DEV)
        pipe.OVERLAP_MIN_BYTES = 0 if overlap else 1 << 62
        ys = [torch.empty((T, w.d_model), dtype=torch.bfloat16).pin_memory() for _ in batches]
        pipe.run(xs, ys)
        torch.cuda.synchronize()
        assert moe.device_status() == 0
        for y, ref in zip(ys, eager):
            assert torch.equal(y.float(), ref)


def test_empty_batch():
    w = mi.workload("mixtral").with_sizes(d_model=64, d_ff=64)
    inp = mi.generate(w, 4, DEV)
    inp["x"] = inp["x"][:0]
    out = gpu_layer(w, 0, inp)
    assert out["y"].shape == (0, 64)
    assert out["counts"].sum() == 0 and out["n_dropped"][0] == 0


# ------------------------------------------------------------------ printed examples through the kernels

def _router(E, k, logits, select_bias=None, d=None):
    T = logits.shape[0]
    d = d or max(4, E)
    x = torch.zeros((T, d), dtype=torch.float32)
    x[:, :E] = torch.tensor(logits, dtype=torch.float32)
    w_r = torch.zeros((E, d), dtype=torch.float32)
    w_r[:, :E] = torch.eye(E)
    cfg = moe.MoEConfig(T=T, d_model=d, n_experts=E, top_k=k, d_ff=4, dtype=moe.DTYPE_FP32)
    sb = None if select_bias is None else torch.tensor(select_bias, dtype=torch.float32, device=DEV)
    return cfg, moe.router_topk(cfg, x.to(DEV), w_r.to(DEV), select_bias=sb, want_probs=True)


def test_top2_example_through_router():
    g = load_golden("top2_example.json")
    cfg, r = _router(8, 2, np.log(np.array([g["probs"]])))
    assert r["idx"][0].tolist() == g["top_k_indices"]
    exact = np.array(g["top_k_probs"]) / sum(g["top_k_probs"])
    assert np.allclose(r["w"][0].cpu().numpy(), exact, atol=1e-6)


def test_aux_example_through_router_and_stats():
    g = load_golden("aux_worked_example.json")
    probs = np.array(g["probs"])
    cfg, r = _router(2, 1, np.log(probs))
    assert (r["idx"][:, 0].cpu().numpy() + 1).tolist() == g["selected_expert_1based"]
    st = moe.load_stats(cfg, r["idx"], r["probs"])
    assert np.allclose(st["f"].cpu().numpy(), g["f"], atol=1e-7)
    assert np.allclose(st["p"].cpu().numpy(), g["p"], atol=1e-7)
    assert abs(float(st["aux"][0]) - g["aux"]) < 1e-6
    assert np.allclose(r["p"].cpu().numpy(), g["p"], atol=1e-7)


def test_selection_bias_example_through_router():
    g = load_golden("selection_bias_example.json")
    cfg, r = _router(4, 2, np.log(np.array([g["scores"]])), select_bias=g["bias"])
    assert (r["idx"][0].cpu().numpy() + 1).tolist() == g["biased_top2_1based"]
    assert np.allclose(r["w"][0].cpu().numpy(), [0.5 / 1.2, 0.7 / 1.2], atol=1e-6)


# ------------------------------------------------------------------ stages fed with oracle inputs

def _idx_cases():
    """The golden capacity cases plus skewed random assignments (expert e drawn
    with weight (e+1)^-1.2, k distinct experts per token)."""
    rng = np.random.default_rng(3)
    g = load_golden("capacity_cases.json")
    cases = [(c["E"], c["k"], c["capacity_factor"], np.array(c["idx"])) for c in g["cases"]]
    for T, E, k, cf in [(1000, 8, 1, 1.25), (777, 64, 8, 1.0), (3000, 896, 8, 1.5),
                        (4097, 8, 2, 0.0), (1, 4, 2, 1.0), (2500, 300, 3, 0.9)]:
        pop = 1.0 / np.arange(1, E + 1) ** 1.2
        pop /= pop.sum()
        idx = np.stack([rng.choice(E, size=k, replace=False, p=pop) for _ in range(T)])
        cases.append((E, k, cf, idx))
    return cases


IDX_CASES = _idx_cases()


@pytest.mark.parametrize("case", list(range(8)))
def test_dispatch_stage_bit_exact(case):
    E, k, cf, idx = IDX_CASES[case]
    T = idx.shape[0]
    C = om.capacity(T, k, E, cf)
    ref = om.dispatch(idx, E, C)
    cfg = moe.MoEConfig(T=T, d_model=8, n_experts=E, top_k=k, d_ff=8, capacity_factor=cf)
    assert moe.capacity(cfg) == C
    out = moe.dispatch(cfg, torch.tensor(idx, dtype=torch.int32, device=DEV))
    n = int(ref.offsets[-1])
    assert out["counts"].cpu().numpy().tolist() == ref.counts.tolist()
    assert out["offsets"].cpu().numpy().tolist() == ref.offsets.tolist()
    assert out["perm"][:n].cpu().numpy().tolist() == ref.perm.tolist()
    assert out["inv"].cpu().numpy().tolist() == ref.inv.tolist()
    assert int(out["n_dropped"][0]) == ref.n_dropped


def test_bad_index_reported_not_faulted():
    cfg = moe.MoEConfig(T=4, d_model=8, n_experts=4, top_k=1, d_ff=8)
    idx = torch.tensor([[0], [5], [1], [-2]], dtype=torch.int32, device=DEV)
    out = moe.dispatch(cfg, idx)
    assert moe.device_status() == -1
    assert out["inv"].cpu().numpy().tolist()[1] == -1 and out["inv"].cpu().numpy().tolist()[3] == -1
    assert moe.device_status() == 0


def test_load_stats_stage_vs_oracle():
    rng = np.random.default_rng(5)
    T, E, k = 999, 40, 3
    probs = om.softmax(rng.normal(size=(T, E)) * 2)
    idx = om.topk_desc(probs, k)
    ref = om.load_stats(probs, idx, E)
    cfg = moe.MoEConfig(T=T, d_model=8, n_experts=E, top_k=k, d_ff=8)
    st = moe.load_stats(cfg, torch.tensor(idx, dtype=torch.int32, device=DEV),
                        torch.tensor(probs, dtype=torch.float32, device=DEV))
    assert st["counts"].cpu().numpy().tolist() == ref["counts"].tolist()
    assert np.max(np.abs(st["f"].cpu().numpy() - ref["f"])) <= FP_ATOL
    assert np.max(np.abs(st["p"].cpu().numpy() - ref["p"])) <= FP_ATOL
    assert abs(float(st["aux"][0]) - ref["aux"]) <= 1e-5 * ref["aux"]
    assert abs(float(st["load_max_over_mean"][0]) - ref["load_max_over_mean"]) <= 1e-5


@pytest.mark.parametrize("name", ["tiny", "mixtral_small", "switch_ragged", "deepseek_small",
                                  "mixtral_T1_split", "switch_T20_split"])
def test_expert_ffn_and_combine_stages(name):
    w, T = SMALL[name]
    inp = mi.generate(w, T, DEV)
    orc = oracle_layer(w, inp)
    dp = orc["dispatch"]
    cfg = moe.config_for(w, T)
    perm = torch.tensor(dp.perm, dtype=torch.int32, device=DEV)
    offs = torch.tensor(dp.offsets, dtype=torch.int32, device=DEV)
    out = moe.expert_ffn(cfg, inp["x"], perm, offs, inp["w1"], inp["w3"], inp["w2"])
    got = out[:dp.perm.shape[0]].cpu().numpy().astype(np.float64)
    x = om._f64(inp["x"])
    E = w.n_experts
    ref = np.zeros_like(got)
    for e in range(E):
        a, b = int(dp.offsets[e]), int(dp.offsets[e + 1])
        if a == b:
            continue
        rows = dp.perm[a:b] // w.top_k
        ref[a:b] = om.expert_ffn(x[rows], inp["w1"][e], None if inp["w3"] is None else inp["w3"][e],
                                 inp["w2"][e], w.act, act_dtype(w))
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got - ref)))
    assert err <= y_tol(w) * rms, (err / rms, y_tol(w))
    # combine with the oracle's expert outputs (rounded to fp32) and weights
    shared = None
    if w.d_ff_shared:
        shared_ref = om.expert_ffn(x, inp["ws1"], inp["ws3"], inp["ws2"], "swiglu", act_dtype(w))
        shared = torch.tensor(shared_ref, dtype=torch.float32, device=DEV)
    y = moe.combine(cfg, torch.tensor(ref, dtype=torch.float32, device=DEV),
                    torch.tensor(dp.inv, dtype=torch.int32, device=DEV),
                    torch.tensor(orc["router"].w, dtype=torch.float32, device=DEV), shared)
    yo = orc["y"]
    assert np.max(np.abs(y.cpu().numpy() - yo)) <= 1e-5 * float(np.sqrt(np.mean(yo ** 2)))


def test_kernels_loaded_for_sm_103a():
    assert moe.kernel_binary_version() == 103
