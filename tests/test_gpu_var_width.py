"""GPU parity of the up projection on the per-tile-width geometry: weights on
the MMA's M side (128 rows of W1, plus the same 128 rows of W3 for SwiGLU),
up to 256 of one expert's token rows on its N side, the N being that count
rounded up to 16 for each tile.  SwiGLU fills the 512 TMEM columns with the
W1 and W3 parts of one tile, so its epilogue does not overlap the next tile.

Reduced layers with the geometry forced (moe_debug_set_var_up_tiles(1))
against the fp64 oracle on every token: one tile per expert, experts of more
than 256 rows (a full tile and a ragged one), widths that fill no tile, ReLU,
capacity, a shared expert, a split reduction; and the same layer on
128-row token tiles.  The library does not pick this geometry for the up
projection by itself (the down projection's own choice of it is covered by
the parity cases with about 75-280 rows per expert).

The element-wise check of h (every element within half a bf16 spacing plus
a derived accumulation allowance of its exact value) runs on both this
geometry and the token-row tiles."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle.moe_oracle as om
import sparse_mixture_experts_47_b300 as moe
from tests.parity import full_check, gpu_layer, y_tol

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = {
    # about 250 rows per expert: one tile each, N up to 256
    "mixtral_T1000": (mi.workload("mixtral").with_sizes(d_model=512, d_ff=2048), 1000),
    # about 275 rows per expert: a tile of 256 and one of about 19 (N = 32);
    # K = 520 (a partial K block) and F = 1000 (a partial last column tile)
    "mixtral_ragged_T1100": (mi.workload("mixtral").with_sizes(d_model=520, d_ff=1000), 1100),
    # ReLU (two accumulators of 256 columns), capacity 1.25 with a hot expert
    "switch_T3000": (mi.workload("switch").with_sizes(d_model=256, d_ff=768), 3000),
    # 16 uneven experts and a shared expert over all 700 tokens (tiles of
    # 256, 256 and 188 rows of one group)
    "deepseek_T700": (mi.workload("deepseek").with_sizes(d_model=512, n_experts=16, d_ff=512,
                                                         d_ff_shared=512), 700),
    # 4 experts of about 300 rows in 64 tiles for 148 SMs: the reduction
    # (K = 1024) split in two, the pre-activation partial sums added by the
    # activation kernel
    "mixtral_split_T600": (mi.workload("mixtral").with_sizes(d_model=1024, n_experts=4,
                                                             d_ff=1024), 600),
    # 896 experts of about 74 rows, F = 64 (one partial column tile)
    "e896_T8192": (mi.workload("e896").with_sizes(d_model=128, d_ff=64), 8192),
}


@pytest.fixture
def var_up():
    moe.debug_set_var_up_tiles(1)
    try:
        yield
    finally:
        moe.debug_set_var_up_tiles(0)


@pytest.mark.parametrize("name", list(CASES))
def test_var_width_up_vs_oracle(name, var_up):
    w, T = CASES[name]
    cfg = moe.config_for(w, T)
    plan = moe.ffn_plan(cfg)
    assert plan["rows_per_tile"] == 256 and plan["up_pair"] == 0
    if w.d_ff_shared:
        assert moe.ffn_plan(cfg, shared=True)["rows_per_tile"] == 256
    inp = mi.generate(w, T, DEV)
    rep, gpu, _ = full_check(w, T, inp)
    assert moe.device_status() == 0
    print(name, plan, rep)
    if name == "mixtral_split_T600":
        assert plan["up_splits"] == 2
    if w.capacity_factor > 0:
        assert int(gpu["n_dropped"][0]) > 0


def test_var_width_up_matches_token_row_tiles(var_up):
    """The same layer on the per-tile-width geometry and on 128-row token
    tiles: identical routing, outputs within the bf16 layer's tolerance."""
    w, T = CASES["mixtral_ragged_T1100"]
    inp = mi.generate(w, T, DEV)
    a = gpu_layer(w, T, inp)
    moe.debug_set_var_up_tiles(-1)
    moe.debug_set_pair_tiles(-1)
    try:
        assert moe.ffn_plan(moe.config_for(w, T))["rows_per_tile"] == 0
        b = gpu_layer(w, T, inp)
    finally:
        moe.debug_set_pair_tiles(0)
    assert np.array_equal(a["idx"], b["idx"])
    diff = float(np.max(np.abs(a["y"].astype(np.float64) - b["y"])))
    rms = float(np.sqrt(np.mean(b["y"].astype(np.float64) ** 2)))
    print(f"per-tile width vs 128-row tiles: max |dy| = {diff:.3e} (RMS {rms:.3e})")
    assert diff <= y_tol(w) * rms


def _gpu_h(w, T, inp):
    """The bf16 activation h of every dispatched row, read through the
    expert FFN entry point with W2 set to a block of the identity (each
    expert output column then holds one h feature exactly: one product by
    1.0 in an fp32 sum of zeros), d_model features per call."""
    cfg = moe.config_for(w, T)
    r = moe.router_topk(cfg, inp["x"], inp["w_r"], inp.get("logit_bias"), inp.get("select_bias"))
    dp = moe.dispatch(cfg, r["idx"])
    off = dp["offsets"].cpu().numpy().astype(np.int64)
    R, E, F, d = int(off[-1]), w.n_experts, w.d_ff, w.d_model
    h = np.empty((R, F))
    for c0 in range(0, F, d):
        n = min(d, F - c0)
        w2 = torch.zeros((E, d, F), dtype=inp["w2"].dtype, device=DEV)
        i = torch.arange(n, device=DEV)
        w2[:, i, c0 + i] = 1
        out = moe.expert_ffn(cfg, inp["x"], dp["perm"], dp["offsets"], inp["w1"], inp.get("w3"),
                             w2)
        torch.cuda.synchronize()
        assert moe.device_status() == 0
        h[:, c0:c0 + n] = out[:R, :n].cpu().numpy()
    return h, dp["perm"].cpu().numpy().astype(np.int64)[:R], off


H_CASES = {
    # K = 2048 split in four (32 tiles), F = 256
    "mixtral_split4_T1200": (mi.workload("mixtral").with_sizes(d_model=2048, d_ff=256), 1200),
    "mixtral_ragged_T1100": CASES["mixtral_ragged_T1100"],
    "e896_T8192": CASES["e896_T8192"],
}


@pytest.mark.parametrize("policy", [1, -1], ids=["var_width", "token_rows"])
@pytest.mark.parametrize("name", list(H_CASES))
def test_h_is_the_rounding_of_the_exact_activation(name, policy):
    """Every element of h is within half a bf16 spacing, plus the error that
    the fp32 accumulation can carry into it, of its exact (fp64) value.

    With S_a = sum_i |x_i| |W1[f, i]| (S_b the same for W3) and K the
    reduction length, each MMA step of K = 16 is taken to add at most 2^-22
    of the magnitudes it sums (two fp32 units, truncation allowed), and split
    partial sums are added in fp32: |a - a_exact| <= E_a = (K/16 2^-22 +
    8 2^-24) S_a.  To first order h = silu(a) b moves by at most
    1.1 |b| E_a + |silu(a)| E_b (|silu'| <= 1.1), and the fp32 SiLU and
    product add 2^-20 |h|.  The test allows four times the first-order
    terms.  A K block of 64, a split's partial sum or a token row gone
    missing moves a by about 8 / K of S_a (K = 2048: 0.4 %), tens of times
    this allowance (a K block zeroed in a CPU model of the computation puts
    over 97 % of the elements past it)."""
    w, T = H_CASES[name]
    moe.debug_set_var_up_tiles(policy)
    try:
        assert moe.ffn_plan(moe.config_for(w, T))["rows_per_tile"] == (256 if policy > 0 else 0)
        inp = mi.generate(w, T, DEV)
        hg, perm, off = _gpu_h(w, T, inp)
    finally:
        moe.debug_set_var_up_tiles(0)
    hx, allow = _exact_h_and_allowance(w, inp, perm, off)
    big = np.maximum(np.abs(hx), np.abs(hg))
    _, ex = np.frexp(big)
    q = np.ldexp(1.0, np.maximum(ex, -125) - 8)          # bf16 spacing there
    diff = np.abs(hg - hx)
    over = diff / (0.5 * q + allow)
    ref = om.round_to_bf16(hx)
    print(f"{name} policy {policy}: {int((hg != ref).sum())} of {hg.size} elements differ from "
          f"the rounded exact value; largest error / allowance {over.max():.3f}")
    assert over.max() <= 1.0, np.unravel_index(over.argmax(), over.shape)


def _exact_h_and_allowance(w, inp, perm, off):
    """The exact h of every dispatched row (fp64) and its error allowance
    beyond half a bf16 spacing."""
    x = inp["x"].float().cpu().numpy().astype(np.float64)
    R = int(off[-1])
    hx = np.empty((R, w.d_ff))
    allow = np.empty((R, w.d_ff))
    eps = (w.d_model / 16 * 2.0 ** -22 + 8 * 2.0 ** -24)
    for e in range(w.n_experts):
        lo, hi = off[e], off[e + 1]
        if hi == lo:
            continue
        xr = x[perm[lo:hi] // w.top_k]
        w1 = inp["w1"][e].float().cpu().numpy().astype(np.float64)
        w3 = inp["w3"][e].float().cpu().numpy().astype(np.float64)
        a, b = xr @ w1.T, xr @ w3.T
        silu = a / (1.0 + np.exp(-a))
        hx[lo:hi] = silu * b
        ea, eb = eps * (np.abs(xr) @ np.abs(w1).T), eps * (np.abs(xr) @ np.abs(w3).T)
        allow[lo:hi] = (4.0 * (1.1 * np.abs(b) * ea + np.abs(silu) * eb)
                        + 2.0 ** -20 * np.abs(hx[lo:hi]))
    return hx, allow
