"""GPU check of the quantile bias b_e = -(v_lo + frac (v_hi - v_lo)), v_lo and
v_hi the order statistics of rank lo and lo + 1 of the probabilities of expert
e over the batch (h = (T - 1) q, q = 1 - k/E, lo = floor h, frac = h - lo;
"Kimi K3 -> Quantile Balancing").

The bias is recomputed with numpy from the very probabilities the router
returned (fp32), so the comparison is exact up to the last rounding of the
interpolation.  The columns are built (x = logits, W_r = I, an fp32 router)
to drive every path of the selection: the counted top-tail path, ties at the
threshold, a column whose sampled positions hold its largest values (too few
candidates above the sample's threshold) and a column with more than 2048
equal candidates (too many), both of which fall back to the full select, a
column with 700 equal largest values (the radix select on the candidates);
and batches below the top-tail path's size or with a wide tail."""
import dataclasses

import numpy as np
import pytest
import torch

import moe_inputs as mi
import sparse_mixture_experts_47_b300 as moe

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _expected_bias(probs, k):
    T, E = probs.shape
    h = (T - 1) * (1.0 - k / E)
    lo = int(np.floor(h))
    frac = np.float32(h - lo)
    col = np.sort(probs.astype(np.float32), axis=0)
    v_lo = col[lo].astype(np.float64)
    v_hi = col[min(lo + 1, T - 1)].astype(np.float64)
    return -(v_lo + np.float64(frac) * (v_hi - v_lo))


def _logits(T, E, kind, seed):
    g = np.random.default_rng(seed)
    lg = g.normal(size=(T, E))
    if kind == "ties":
        # 512 distinct rows, each repeated: every column holds groups of
        # equal probabilities, at the threshold too
        lg = lg[np.arange(T) % 512]
    elif kind == "sampled_top":
        step = T // 1024                                # every sampled token among them
        # expert 3: the sampled tokens hold the column's largest values, so
        # the sample's threshold admits too few
        lg[:, 3] = -4.0
        lg[::step, 3] = 6.0 + g.random(lg[::step, 3].shape)
        # expert 5: 3000 identical rows (none of them sampled) share the
        # column's largest value: too many candidates
        rows = g.choice(np.flatnonzero(np.arange(T) % step != 0), 3700, replace=False)
        same = g.normal(size=E)
        same[3], same[5], same[7] = -4.0, 5.0, -4.0
        lg[:, 5] = np.minimum(lg[:, 5], 0.0)
        lg[rows[:3000]] = same
        # expert 7: 700 other identical rows share its largest value: a
        # candidate set the counting step cannot hold (more than 512 equal)
        same7 = g.normal(size=E)
        same7[3], same7[5], same7[7] = -4.0, 0.0, 5.0
        lg[:, 7] = np.minimum(lg[:, 7], 0.0)
        lg[rows[3000:]] = same7
    return lg.astype(np.float32)


@pytest.mark.parametrize("T,E,k,kind", [(16384, 896, 8, "normal"), (8192, 512, 8, "ties"),
                                        (8192, 896, 8, "sampled_top"),
                                        (2000, 896, 8, "normal"), (6000, 64, 8, "normal")])
def test_quantile_bias_exact(T, E, k, kind):
    lg = _logits(T, E, kind, seed=T + E)
    cfg = moe.MoEConfig(T=T, d_model=E, n_experts=E, top_k=k, d_ff=8, dtype=moe.DTYPE_FP32,
                        quantile_balance=1)
    x = torch.tensor(lg, device=DEV)
    w_r = torch.eye(E, dtype=torch.float32, device=DEV)
    r = moe.router_topk(cfg, x, w_r, want_probs=True)
    torch.cuda.synchronize()
    assert moe.device_status() == 0
    probs = r["probs"].cpu().numpy()
    got = r["select_bias"].cpu().numpy().astype(np.float64)
    exp = _expected_bias(probs, k)
    err = np.abs(got - exp)
    # one rounding of the fp32 interpolation
    assert np.all(err <= 2.0 ** -23 * np.abs(exp) + 1e-30), (float(err.max()), int(err.argmax()))
    if kind == "sampled_top":
        assert got[3] < got[0] and got[5] == -probs[:, 5].max() and got[7] == -probs[:, 7].max()
