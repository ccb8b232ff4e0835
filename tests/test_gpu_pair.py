"""GPU parity of the grouped GEMM's SM-pair geometry: tiles of 256 token rows
on a cluster of two CTAs (two SMs) running one tcgen05.mma.cta_group::2 of
M = 256, each CTA staging its own 128 rows and half of the weight tile.

Reduced layers, with the pair tiles forced wherever the geometry allows
(moe_debug_set_pair_tiles(1)), against the fp64 oracle on every token:
SwiGLU and ReLU up projections, the down projection, ragged experts (partial
last tiles, experts whose rows end inside a CTA's half), capacity, a shared
expert.  The full-size Mixtral workloads, where the library picks the pair
tiles by itself, are covered by test_gpu_full.py."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import sparse_mixture_experts_47_b300 as moe
from tests.parity import full_check, gpu_layer

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = {
    # 1000 tokens x top-2 over 8 experts: about 250 rows each, ragged tails
    "mixtral_T1000": (mi.workload("mixtral").with_sizes(d_model=512, d_ff=2048), 1000),
    "mixtral_T2048": (mi.workload("mixtral").with_sizes(d_model=768, d_ff=1536), 2048),
    # ReLU, capacity 1.25 with a hot expert 0, 3 output-column tiles of 256
    "switch_T3000": (mi.workload("switch").with_sizes(d_model=256, d_ff=768), 3000),
    # 16 experts of about 350 rows, uneven under the selection bias (tiles
    # that end inside the first CTA's half), plus a shared expert over all
    # 700 tokens
    "deepseek_T700": (mi.workload("deepseek").with_sizes(d_model=512, n_experts=16, d_ff=512,
                                                         d_ff_shared=512), 700),
    # widths that fill no tile: the last K block (520 = 8 x 64 + 8), the last
    # SwiGLU column tile (1000 = 7 x 128 + 104) and the last down tile
    # (520 = 2 x 256 + 8) are partial
    "mixtral_ragged_T1100": (mi.workload("mixtral").with_sizes(d_model=520, d_ff=1000), 1100),
    # the same widths with the down projection on pairs too (375 rows per expert)
    "mixtral_ragged_T1500": (mi.workload("mixtral").with_sizes(d_model=520, d_ff=1000), 1500),
}


@pytest.fixture
def pair_tiles():
    moe.debug_set_pair_tiles(1)
    moe.debug_set_var_up_tiles(-1)      # token rows on the M side for the up projection too
    try:
        yield
    finally:
        moe.debug_set_pair_tiles(0)
        moe.debug_set_var_up_tiles(0)


@pytest.mark.parametrize("name", list(CASES))
def test_pair_tiles_vs_oracle(name, pair_tiles):
    w, T = CASES[name]
    cfg = moe.config_for(w, T)
    plan = moe.ffn_plan(cfg)
    assert plan["rows_per_tile"] == 0 and plan["up_pair"] == 1
    # the down projection takes pairs unless its per-tile-width geometry applies
    assert plan["down_pair"] == 1 or plan["down_rows_per_tile"] == 256
    if w.d_ff_shared:
        sh = moe.ffn_plan(cfg, shared=True)
        assert sh["up_pair"] == 1 and sh["down_pair"] == 1
    inp = mi.generate(w, T, DEV)
    rep, gpu, _ = full_check(w, T, inp)
    assert moe.device_status() == 0
    print(name, rep)
    if w.capacity_factor > 0:
        assert int(gpu["n_dropped"][0]) > 0


@pytest.mark.parametrize("name", ["mixtral_ragged_T1100", "mixtral_ragged_T1500"])
def test_ragged_widths_one_sm_tiles(name):
    """The same ragged layer on the one-SM tiles, against the oracle."""
    w, T = CASES[name]
    moe.debug_set_pair_tiles(-1)
    moe.debug_set_var_up_tiles(-1)
    try:
        plan = moe.ffn_plan(moe.config_for(w, T))
        assert plan["up_pair"] == 0 and plan["rows_per_tile"] == 0
        inp = mi.generate(w, T, DEV)
        rep, _, _ = full_check(w, T, inp)
        assert moe.device_status() == 0
        print(name, rep)
    finally:
        moe.debug_set_pair_tiles(0)
        moe.debug_set_var_up_tiles(0)


def test_pair_tiles_match_one_sm_tiles(pair_tiles):
    """The same layer with and without the pair tiles: the MMAs accumulate
    the same K steps in the same order, so the outputs are expected to agree
    to the last bit; the report prints the largest difference, and the test
    holds them to the y tolerance of a bf16 layer."""
    w, T = CASES["mixtral_T2048"]
    inp = mi.generate(w, T, DEV)
    a = gpu_layer(w, T, inp)
    moe.debug_set_pair_tiles(-1)
    assert moe.ffn_plan(moe.config_for(w, T))["up_pair"] == 0
    b = gpu_layer(w, T, inp)
    torch.cuda.synchronize()
    assert np.array_equal(a["idx"], b["idx"])
    diff = float(np.max(np.abs(a["y"].astype(np.float64) - b["y"])))
    rms = float(np.sqrt(np.mean(b["y"].astype(np.float64) ** 2)))
    print(f"pair vs one-SM tiles: max |dy| = {diff:.3e} (RMS {rms:.3e})")
    assert diff <= 1e-2 * rms


def test_pair_tiles_in_a_captured_graph(pair_tiles):
    """The layer captured in a CUDA graph (LayerGraph) with the SM-pair
    kernels (clusters of two CTAs) gives exactly the eager call's outputs,
    batch by batch; so does the copy-overlapped pipeline."""
    w, T = CASES["mixtral_T1000"]
    inp = mi.generate(w, T, DEV)
    cfg = moe.config_for(w, T, moe.DTYPE_BF16)
    assert moe.ffn_plan(cfg)["up_pair"] == 1
    wts = {k: inp.get(k) for k in moe._WEIGHT_KEYS}
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    batches = [torch.randn(inp["x"].shape, generator=g, device=DEV).to(inp["x"].dtype)
               for _ in range(3)]
    eager = [moe.layer_forward(cfg, b, wts)["y"].float().cpu() for b in batches]
    graph = moe.LayerGraph(cfg, batches[0].clone(), wts)
    for b, ref in zip(batches, eager):
        graph.x.copy_(b)
        assert torch.equal(graph.replay()["y"].float().cpu(), ref)
    xs = [b.cpu().pin_memory() for b in batches]
    pipe = moe.LayerPipeline(cfg, wts, DEV)
    pipe.OVERLAP_MIN_BYTES = 0
    ys = [torch.empty((T, w.d_model), dtype=torch.bfloat16).pin_memory() for _ in batches]
    pipe.run(xs, ys)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    for y, ref in zip(ys, eager):
        assert torch.equal(y.float(), ref)
