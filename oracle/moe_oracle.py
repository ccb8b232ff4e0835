"""fp64 CPU oracle for the forward pass of a token-choice sparse MoE FFN layer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA library and reads the
same stored input values (bf16 or fp32), widened exactly to float64.

Every step is the plain definition from the pages, written out in float64 with
numpy; a library matmul, exp, sort or floor serves as a step, with no blocking,
fusion or reordering beyond the definition.  Sources (page title, section):

[MoE-ch30]  "Mixture of Experts", LLM Transformer book (waylandz.com), ch. 30:
            §30.2.3 router (linear -> softmax -> top-k -> renormalise),
            §30.2.4 SwiGLU expert, §30.2.6 load-balancing loss,
            §30.4.5 shared expert, §30.5.2 capacity, §30.6.1 MoELayer.
[MoE-guide] "Mixture of Experts guide" (ai-native-b2y.pages.dev):
            "MoEの核心：ルーターの仕組み", "解決策1：補助損失".
[MoE-memo]  "Mixture of Experts (MoE) memo" (iwashi.co): "補助損失" worked
            example, "DeepSeek-V3のアプローチ → Aux-loss-free（バイアス）",
            "Kimi K3 → Quantile Balancing".
[MoE-prac]  "混合エキスパートモデル（MoE）実践" (deepseekmodel.com):
            "ルーティングの数学的な形" (TopKRouter), "capacity factor、token
            dropping", "ロードバランシング損失" (BiasBalancedRouter),
            "expert parallelism と all-to-all" (stable grouping by expert).

Readings where the pages are silent or disagree (each restated where used):
  R1  f_e = count_e / (T*k): fraction of all routed assignments, so sum f = 1
      and uniform routing gives aux = 1 for every k.
  R2  aux is returned without the 0.01 coefficient.
  R3  f counts router assignments before capacity drops; p is the mean of the
      unbiased softmax probability over all T tokens.
  R4  the selection bias is added to the softmax probabilities (default) or,
      on request, to the logits; weights always come from the unbiased probs.
  R5  top-k order is descending score; exactly equal scores: lower expert
      index first.
  R6  capacity C = ceil(cf*T*k/E); per expert the first C assignments in
      flattened (t*k + j) order are kept, the rest dropped; a dropped slot
      contributes 0 and the surviving weights are not renormalised.
  R7  quantile bias b_e = -Q(probs[:, e], 1 - k/E) with Q the linear
      interpolation between order statistics (h = (T-1) q).
  R10 capacity overflow redirected to the next-best expert (ch30 §30.5.2):
      round 0 is R6; in each further round, unserved slots take their
      token's next unused experts down the full score ranking and are
      served in (t*k + j) order by experts with room; the weight of a slot
      served by expert e is p[t, e] over the token's top-k probability sum.
  R11 expert-choice routing (prac, memo routing table): each expert takes
      the min(C, T) tokens with the largest softmax probability for it (ties
      by lower token index), C = ceil(cf*T*k/E); weight probs[t, e], not
      renormalised; a token picked by no expert gets routed output 0.
  R9  observability (prac, scale drift): gate entropy is the mean over
      tokens of -sum_e p ln p in nats; an expert's output scale is the mean,
      population standard deviation and largest magnitude over all elements
      of its output tensor (its kept rows' FFN outputs, before the gate
      weight); bias size is mean and max |b_e| of the selection bias in
      effect.
  R8  the layer's intermediate activation is stored in the layer dtype: for
      a bf16 layer the expert's intermediate activation h (the input of W2)
      is a bf16 tensor, rounded once, to nearest even, from its exact value
      before the down projection.  The pages run the model in
      torch.bfloat16 ([MoE-ch30] §30.6.3), and the Switch workload is
      specified with bf16 weights and activations, so the down projection
      takes a bf16 operand.  Everything after it (each expert's output row,
      the gate-weighted sum, the shared expert's output, y) stays exact
      float64: the layer's output is compared in fp32 against a bound of
      1e-2 x RMS, and a bf16 rounding of an expert output alone moves it by
      up to 2^-8 of its magnitude, which at a few RMS is that whole bound.

Pins (tests/test_oracle_pins.py): the printed worked examples (top-2
renormalisation, 4-token aux loss, selection-bias example), brute-force top-k
over all subsets, softmax of log-probabilities, E=1 and k=E reductions to a
dense FFN / dense mixture computed with torch.nn.functional, identical experts,
numpy.quantile, a hand-built capacity case, and dispatch invariants.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, Optional, Sequence

import numpy as np

__all__ = [
    "router_logits", "softmax", "topk_desc", "renormalise", "route",
    "quantile_linear", "quantile_select_bias", "capacity", "dispatch",
    "expert_ffn", "load_stats", "moe_forward", "RouterOut", "DispatchOut", "round_to_bf16",
    "round_to_fp32", "gate_entropy", "expert_output_scale", "bias_magnitude", "observe",
    "dispatch_reroute", "RerouteOut", "expert_choice", "ExpertChoiceOut",
    "moe_forward_expert_choice", "with_ranking",
]


def _f64(a) -> np.ndarray:
    """Widen a torch tensor or array to float64 (exact for fp32/bf16 inputs)."""
    if hasattr(a, "detach"):
        a = a.detach().cpu()
        if str(a.dtype) == "torch.bfloat16":
            a = a.float()
        a = a.numpy()
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# Router: [MoE-ch30] §30.2.3 steps 1-4, [MoE-prac] TopKRouter.forward
# --------------------------------------------------------------------------

def router_logits(x, w_r, logit_bias=None) -> np.ndarray:
    """logits[t, e] = sum_i x[t, i] * W_r[e, i]  (+ logit_bias[e]).

    The router is a bias-free linear layer hidden -> E ([MoE-ch30] §30.2.3
    step 1, [MoE-prac] "ルーターが bias を持たない").  W_r is stored like an
    nn.Linear weight, [E, d].  ``logit_bias`` is a fixed per-expert offset
    that the synthetic workloads use to skew expert popularity.
    """
    lg = _f64(x) @ _f64(w_r).T
    if logit_bias is not None:
        lg = lg + _f64(logit_bias)[None, :]
    return lg


def softmax(logits: np.ndarray) -> np.ndarray:
    """probs = exp(l - max) / sum exp(l - max) over the expert axis (step 2)."""
    m = logits.max(axis=1, keepdims=True)
    e = np.exp(logits - m)
    return e / e.sum(axis=1, keepdims=True)


def topk_desc(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores per row, largest first (step 3).

    Reading R5: exactly equal scores are ordered by lower expert index.  A
    stable ascending sort of the negated scores gives exactly that order.
    """
    order = np.argsort(-scores, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def renormalise(probs: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """w[t, j] = probs[t, idx[t, j]] / sum_j' probs[t, idx[t, j']] (step 4).

    [MoE-ch30] §30.2.3 step 4; [MoE-prac] calls this the step that must not
    be skipped.  With a selection bias the weights still come from the
    unbiased probabilities ([MoE-memo] aux-loss-free section, [MoE-prac]
    BiasBalancedRouter).
    """
    sel = np.take_along_axis(probs, idx, axis=1)
    return sel / sel.sum(axis=1, keepdims=True)


def quantile_linear(values: np.ndarray, q: float) -> float:
    """Q(values, q) by linear interpolation between order statistics.

    Sort ascending into v_(0..n-1); h = (n-1) q; Q = v_(floor h) +
    (h - floor h) (v_(floor h + 1) - v_(floor h)).  Reading R7.
    """
    v = np.sort(np.asarray(values, dtype=np.float64))
    n = v.shape[0]
    h = (n - 1) * q
    lo = int(math.floor(h))
    if lo >= n - 1:
        return float(v[n - 1])
    return float(v[lo] + (h - lo) * (v[lo + 1] - v[lo]))


def quantile_select_bias(probs: np.ndarray, k: int) -> np.ndarray:
    """Per-batch quantile balancing: b_e = -Q(probs[:, e], 1 - k/E).

    [MoE-memo] "Kimi K3 → Quantile Balancing" sets, per expert, the bias
    that makes the target share of tokens enter the top-k, read off the
    score distribution instead of stepping it.  With b_e at the (1 - k/E)
    quantile, about a k/E share of each expert's column has probs + b > 0.
    """
    T, E = probs.shape
    q = 1.0 - k / E
    return np.array([-quantile_linear(probs[:, e], q) for e in range(E)])


@dataclass
class RouterOut:
    logits: np.ndarray        # [T, E] float64
    probs: np.ndarray         # [T, E] unbiased softmax
    scores: np.ndarray        # [T, E] the values top-k ran on
    idx: np.ndarray           # [T, k] int64, descending score
    w: np.ndarray             # [T, k] renormalised gate weights
    select_bias: Optional[np.ndarray]   # [E] bias used for selection


def with_ranking(r: RouterOut, ranking: Dict[int, Sequence[int]]) -> RouterOut:
    """The router's result with the leading experts of some tokens given.

    Where two selection scores are equal to within rounding, either order
    is a correct top-k (reading R5 fixes only exactly equal scores), and a
    device computing the scores in fp32 may take the other one.
    ``ranking[t]`` lists token t's experts best first (at least k of them);
    its first k become the token's slots, in that order, and their weights
    are renormalised from the unbiased probabilities as in ``route``.  The
    caller checks that the scores allow the order before passing it.
    """
    idx, w = r.idx.copy(), r.w.copy()
    k = idx.shape[1]
    for t, lead in ranking.items():
        row = np.asarray(lead, dtype=np.int64)[:k]
        idx[t] = row
        w[t] = renormalise(r.probs[t:t + 1], row[None, :])[0]
    return RouterOut(r.logits, r.probs, r.scores, idx, w, r.select_bias)


def route(x, w_r, k: int, logit_bias=None, select_bias=None,
          select_space: str = "probs", quantile_balance: bool = False
          ) -> RouterOut:
    """Router linear -> softmax -> (bias for selection) -> top-k -> renorm.

    Reading R4: the selection bias goes on the probs ([MoE-prac]
    BiasBalancedRouter adds it to the softmax output) unless
    ``select_space == "logits"``.
    """
    logits = router_logits(x, w_r, logit_bias)
    probs = softmax(logits)
    base = probs if select_space == "probs" else logits
    bias = None
    if quantile_balance:
        bias = quantile_select_bias(probs, k)
    elif select_bias is not None:
        bias = _f64(select_bias)
    scores = base if bias is None else base + bias[None, :]
    idx = topk_desc(scores, k)
    w = renormalise(probs, idx)
    return RouterOut(logits, probs, scores, idx, w, bias)


# --------------------------------------------------------------------------
# Capacity and dispatch: [MoE-prac] "capacity factor、token dropping",
# "expert parallelism と all-to-all" (stable grouping by expert)
# --------------------------------------------------------------------------

def capacity(T: int, k: int, E: int, capacity_factor: float) -> int:
    """C = ceil(cf * k * T / E) ([MoE-prac] capacity section); no limit
    (returns T*k) when cf <= 0.  Reading R6 picks this among the pages'
    variants."""
    if capacity_factor <= 0:
        return T * k
    return int(math.ceil(float(capacity_factor) * T * k / E))


@dataclass
class DispatchOut:
    counts: np.ndarray        # [E] assignments per expert before drops
    kept_counts: np.ndarray   # [E] min(counts, C)
    offsets: np.ndarray       # [E+1] exclusive scan of kept_counts
    perm: np.ndarray          # [sum kept] flat slot (t*k+j) of each sorted row
    inv: np.ndarray           # [T*k] sorted row of each flat slot, -1 if dropped
    keep: np.ndarray          # [T, k] bool
    n_dropped: int


def dispatch(idx: np.ndarray, E: int, C: int) -> DispatchOut:
    """Group the T*k assignments by expert, stably, and apply capacity.

    Flatten (t, j) to f = t*k + j; order the slots by expert, keeping the f
    order inside each expert (the stable argsort of [MoE-prac]'s dispatch);
    within an expert the slot of rank r (0-based, in f order) is kept iff
    r < C (reading R6: drops go in token-index order).
    """
    T, k = idx.shape
    flat = idx.reshape(-1)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    order = np.argsort(flat, kind="stable")          # slots grouped by expert
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    rank_sorted = np.arange(T * k) - starts[flat[order]]
    keep_sorted = rank_sorted < C
    perm = order[keep_sorted]
    kept_counts = np.minimum(counts, C)
    offsets = np.concatenate([[0], np.cumsum(kept_counts)]).astype(np.int64)
    inv = np.full(T * k, -1, dtype=np.int64)
    inv[perm] = np.arange(perm.shape[0])
    keep = (inv >= 0).reshape(T, k)
    return DispatchOut(counts, kept_counts, offsets, perm.astype(np.int64), inv,
                       keep, int(T * k - perm.shape[0]))


@dataclass
class RerouteOut:
    slot_expert: np.ndarray   # [T, k] expert serving each slot, -1 if dropped
    slot_w: np.ndarray        # [T, k] gate weight of that expert (0 if dropped)
    slot_round: np.ndarray    # [T, k] round that placed the slot (0 = first choice)
    counts: np.ndarray        # [E] first-choice assignments (before capacity)
    kept_counts: np.ndarray   # [E] rows served per expert (<= C)
    offsets: np.ndarray       # [E+1]
    perm: np.ndarray          # [sum kept] flat slot of each grouped row
    inv: np.ndarray           # [T*k] grouped row of each slot, -1 if dropped
    n_dropped: int


def dispatch_reroute(scores: np.ndarray, probs: np.ndarray, k: int, C: int, rounds: int,
                     ranking: Optional[Dict[int, Sequence[int]]] = None) -> RerouteOut:
    """Capacity with overflow redirected to the next-best expert ([MoE-ch30]
    §30.5.2: tokens beyond an expert's capacity are dropped or sent to the
    next-best expert).  Reading R10:

    * each token ranks all experts by its selection score (descending,
      exactly equal scores by lower index); its first k are its slots;
    * round 0 is the plain capacity rule: slots in flattened (t*k + j) order,
      a slot is served by its expert while that expert has fewer than C rows;
    * in each of ``rounds`` further rounds, every slot still unserved takes
      its token's next unused expert down the ranking (a token's unserved
      slots in j order take consecutive candidates), and the slots are then
      served, again in (t*k + j) order, by experts that still have room;
    * slots unserved after the last round are dropped (output 0);
    * a slot served by expert e carries the weight p[t, e] / sum of the
      token's top-k probabilities: the normaliser of the plain top-k, so that
      capacity decisions never rescale the other slots (as for drops, R6);
    * an expert's rows are grouped in the order they were served: round 0 in
      (t*k + j) order, then round 1, and so on.

    ``ranking[t]`` (as in ``with_ranking``) fixes the leading experts of
    token t's ranking where its scores tie within rounding; the rest of the
    ranking follows the scores.
    """
    T, E = scores.shape
    order = np.argsort(-scores, axis=1, kind="stable")        # full ranking per token
    for t, lead in (ranking or {}).items():
        lead = [int(e) for e in lead]
        order[t] = lead + [int(e) for e in order[t] if int(e) not in set(lead)]
    top = order[:, :k]
    norm = np.take_along_axis(probs, top, axis=1).sum(axis=1)
    counts = np.bincount(top.reshape(-1), minlength=E).astype(np.int64)
    slot_e = top.copy()
    served = np.full((T, k), -1, dtype=np.int64)      # expert serving the slot
    rnd = np.full((T, k), -1, dtype=np.int64)
    rows: list = [[] for _ in range(E)]                 # served slots per expert, in order
    nxt = np.full(T, k, dtype=np.int64)                 # next candidate position per token
    for r in range(rounds + 1):
        if r > 0:
            for t in range(T):
                for j in range(k):
                    if served[t, j] >= 0:
                        continue
                    if nxt[t] < E:
                        slot_e[t, j] = order[t, nxt[t]]
                        nxt[t] += 1
                    else:
                        slot_e[t, j] = -1                # no candidate left
        for t in range(T):
            for j in range(k):
                e = int(slot_e[t, j])
                if served[t, j] >= 0 or e < 0:
                    continue
                if len(rows[e]) < C:
                    rows[e].append(t * k + j)
                    served[t, j] = e
                    rnd[t, j] = r
    kept = np.array([len(rows[e]) for e in range(E)], dtype=np.int64)
    offsets = np.concatenate([[0], np.cumsum(kept)]).astype(np.int64)
    perm = np.array([f for e in range(E) for f in rows[e]], dtype=np.int64)
    inv = np.full(T * k, -1, dtype=np.int64)
    inv[perm] = np.arange(perm.shape[0])
    w = np.zeros((T, k))
    for t in range(T):
        for j in range(k):
            if served[t, j] >= 0:
                w[t, j] = probs[t, served[t, j]] / norm[t]
    return RerouteOut(served, w, rnd, counts, kept, offsets, perm, inv,
                      int(T * k - perm.shape[0]))


@dataclass
class ExpertChoiceOut:
    chosen: np.ndarray        # [E, Cn] tokens each expert picked, ascending token index
    weight: np.ndarray        # [E, Cn] their gate weights probs[t, e]
    counts: np.ndarray        # [E] Cn = min(C, T) for every expert
    offsets: np.ndarray       # [E+1] e * Cn
    n_unchosen: int           # tokens no expert picked (their routed output is 0)


def expert_choice(probs: np.ndarray, C: int,
                  chosen: Optional[Dict[int, Sequence[int]]] = None) -> ExpertChoiceOut:
    """Expert-choice routing ([MoE-prac] TopKRouter discussion: each expert
    picks the top-C tokens for its capacity, so every expert is exactly
    full; [MoE-memo] routing table: each expert chooses its top tokens).
    Reading R11: the scores are the router's softmax probabilities (the same
    router as token choice); expert e takes the min(C, T) tokens with the
    largest probs[:, e], exactly equal values by lower token index; the gate
    weight of (t, e) is probs[t, e] with no renormalisation; a token may be
    picked by any number of experts, including none.

    ``chosen[e]`` gives expert e's Cn tokens where its column ties within
    rounding at the Cn-th value (either token is a correct pick there); the
    caller checks that the values allow the set before passing it."""
    T, E = probs.shape
    Cn = min(C, T)
    picks = np.zeros((E, Cn), dtype=np.int64)
    weight = np.zeros((E, Cn))
    picked = np.zeros(T, dtype=bool)
    for e in range(E):
        if chosen is not None and e in chosen:
            top = np.sort(np.asarray(chosen[e], dtype=np.int64))
            assert top.shape[0] == Cn
        else:
            order = np.argsort(-probs[:, e], kind="stable")   # ties: lower token first
            top = np.sort(order[:Cn])
        picks[e] = top
        weight[e] = probs[top, e]
        picked[top] = True
    return ExpertChoiceOut(picks, weight, np.full(E, Cn, dtype=np.int64),
                           np.arange(E + 1, dtype=np.int64) * Cn, int(T - picked.sum()))


def moe_forward_expert_choice(inp: Dict, k: int, act: str, capacity_factor: float = 1.0,
                              tokens: Optional[Sequence[int]] = None,
                              act_dtype: str = "fp64",
                              chosen: Optional[Dict[int, Sequence[int]]] = None,
                              probs: Optional[np.ndarray] = None) -> Dict:
    """Layer forward with expert-choice routing (reading R11):
    y[t] = sum over experts e that picked t of probs[t, e] FFN_e(x[t]) +
    shared(x[t]), with capacity C = ceil(cf * T * k / E) (k = average number
    of experts per token).  f, p and aux use the experts' actual loads:
    f_e = Cn / (T k).  ``chosen`` is passed to ``expert_choice``; ``probs``,
    when given, is this module's softmax of the router logits for the same
    inputs, computed earlier."""
    x = _f64(inp["x"])
    T = x.shape[0]
    E = inp["w_r"].shape[0]
    if probs is None:
        probs = softmax(router_logits(x, inp["w_r"], inp.get("logit_bias")))
    C = capacity(T, k, E, capacity_factor)
    ec = expert_choice(probs, C, chosen)
    f = ec.counts / float(T * k) if T else np.zeros(E)
    p = probs.mean(axis=0) if T else np.zeros(E)
    stats = {"counts": ec.counts, "f": f, "p": p, "aux": E * float(np.sum(f * p)),
             "load_max_over_mean": (float(ec.counts.max()) / (T * k / float(E))) if T else 0.0}
    rows = np.arange(T) if tokens is None else np.asarray(sorted(set(int(t) for t in tokens)))
    pos = {int(t): i for i, t in enumerate(rows)}
    y = np.zeros((rows.shape[0], x.shape[1]))
    for e in range(E):
        sel = [(n, int(t)) for n, t in enumerate(ec.chosen[e]) if int(t) in pos]
        if not sel:
            continue
        tt = np.array([t for _, t in sel])
        out = expert_ffn(x[tt], inp["w1"][e], None if inp.get("w3") is None else inp["w3"][e],
                         inp["w2"][e], act, act_dtype)
        for i, (n, t) in enumerate(sel):
            y[pos[t]] += ec.weight[e, n] * out[i]
    if inp.get("ws1") is not None:
        sh = expert_ffn(x[rows], inp["ws1"], inp["ws3"], inp["ws2"], "swiglu", act_dtype)
        y += sh
    return {"probs": probs, "ec": ec, "stats": stats, "capacity": C, "rows": rows, "y": y}


# --------------------------------------------------------------------------
# Expert FFN: [MoE-ch30] §30.2.4 / §30.6.1 Expert
# --------------------------------------------------------------------------

def _silu(a: np.ndarray) -> np.ndarray:
    return a / (1.0 + np.exp(-a))


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits: for |a| in [2^(e-1), 2^e) the spacing is
    2^(e-8); below the smallest normal 2^-126 the spacing is 2^-133.
    """
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)
    e = np.maximum(e, -125)
    q = np.ldexp(1.0, e - 8)
    return np.round(a / q) * q


def round_to_fp32(a: np.ndarray) -> np.ndarray:
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


ACT_ROUNDING = {"fp64": lambda a: a, "fp32": round_to_fp32, "bf16": round_to_bf16}


def expert_ffn(x_rows: np.ndarray, w1, w3, w2, act: str, act_dtype: str = "fp64") -> np.ndarray:
    """One expert on the rows x_rows [n, d] (float64).

    SwiGLU: w2(silu(w1 x) * w3 x)  ([MoE-ch30] §30.2.4), ReLU: w2(relu(w1 x)).
    Weights are nn.Linear-shaped: w1, w3 [F, d], w2 [d, F]; no biases.
    ``act_dtype`` is the layer's storage type of the intermediate activation
    h (reading R8): h is rounded once to it; "fp64" keeps it exact.  The
    expert's output row is exact.  Products and sums are exact.
    """
    a = x_rows @ _f64(w1).T
    if act == "swiglu":
        h = _silu(a) * (x_rows @ _f64(w3).T)
    elif act == "relu":
        h = np.maximum(a, 0.0)
    else:
        raise ValueError(act)
    h = ACT_ROUNDING[act_dtype](h)
    return h @ _f64(w2).T


# --------------------------------------------------------------------------
# Load statistics: [MoE-ch30] §30.2.6, [MoE-memo] 補助損失, [MoE-prac]
# load_balance_loss
# --------------------------------------------------------------------------

def load_stats(probs: np.ndarray, idx: np.ndarray, E: int) -> Dict[str, np.ndarray]:
    """f, p, aux = E * sum_e f_e p_e, and the load max/mean ratio.

    f_e = (number of (t, j) with idx = e) / (T*k)   (reading R1, before drops)
    p_e = mean over tokens of probs[t, e]
    """
    T, k = idx.shape
    counts = np.bincount(idx.reshape(-1), minlength=E).astype(np.int64)
    f = counts / float(T * k)
    p = probs.mean(axis=0)
    aux = E * float(np.sum(f * p))
    mean_load = T * k / float(E)
    return {"counts": counts, "f": f, "p": p, "aux": aux,
            "load_max_over_mean": float(counts.max()) / mean_load}


# --------------------------------------------------------------------------
# Observability: [MoE-prac] "エキスパート間のスケールドリフト" (monitor each
# expert's output mean, standard deviation and maximum; the minimum set of
# MoE metrics: drop ratio, per-expert load, per-expert output scale, the
# size of the bias term and the gate entropy)
# --------------------------------------------------------------------------

def gate_entropy(probs: np.ndarray) -> float:
    """Mean over tokens of the router distribution's entropy, in nats:
    H_t = -sum_e p[t, e] ln p[t, e], with 0 ln 0 = 0 (reading R9)."""
    p = np.asarray(probs, dtype=np.float64)
    if p.shape[0] == 0:
        return 0.0
    safe = np.where(p > 0, p, 1.0)
    return float(np.mean(-np.sum(np.where(p > 0, p * np.log(safe), 0.0), axis=1)))


def expert_output_scale(outputs: Dict[int, np.ndarray], E: int) -> Dict[str, np.ndarray]:
    """Per expert, over every element of its output tensor (the FFN outputs
    of its kept rows, before the gate weight): mean, standard deviation
    (population) and largest magnitude; zeros for an expert without rows
    (reading R9)."""
    mean, std, mx = np.zeros(E), np.zeros(E), np.zeros(E)
    for e, o in outputs.items():
        o = np.asarray(o, dtype=np.float64)
        if o.size == 0:
            continue
        mean[e] = o.mean()
        std[e] = o.std()
        mx[e] = np.abs(o).max()
    return {"mean": mean, "std": std, "max_abs": mx}


def bias_magnitude(bias: Optional[np.ndarray]) -> Dict[str, float]:
    """Size of the selection bias in effect: mean and largest |b_e| (0
    without a bias)."""
    if bias is None:
        return {"mean_abs": 0.0, "max_abs": 0.0}
    b = np.abs(np.asarray(bias, dtype=np.float64))
    return {"mean_abs": float(b.mean()), "max_abs": float(b.max())}


def observe(r: "RouterOut", dp: "DispatchOut", outputs: Dict[int, np.ndarray], E: int,
            k: int) -> Dict:
    """The pages' MoE observability set for one batch."""
    T = r.probs.shape[0]
    return {"drop_ratio": dp.n_dropped / float(T * k) if T else 0.0,
            "gate_entropy": gate_entropy(r.probs),
            "bias": bias_magnitude(r.select_bias),
            "expert_out": expert_output_scale(outputs, E)}


# --------------------------------------------------------------------------
# Whole layer: [MoE-ch30] §30.6.1 MoELayer.forward, §30.4.5 shared expert
# --------------------------------------------------------------------------

def moe_forward(inp: Dict, k: int, act: str, capacity_factor: float = 0.0,
                select_space: str = "probs", quantile_balance: bool = False,
                tokens: Optional[Sequence[int]] = None, act_dtype: str = "fp64",
                observe_outputs: bool = False, reroute_rounds: int = 0,
                ranking: Optional[Dict[int, Sequence[int]]] = None,
                router: Optional[RouterOut] = None) -> Dict:
    """Forward of the token-choice MoE layer.

    y[t] = sum_j keep[t,j] * w[t,j] * FFN_{idx[t,j]}(x[t]) + shared(x[t]).
    Routing, dispatch and statistics are computed for all T tokens (capacity
    couples them); y is computed for ``tokens`` only (all when None), since
    each token's output depends on nothing else once its slots are known.
    ``act_dtype`` is the storage type of the experts' intermediate
    activation (reading R8).  ``observe_outputs`` adds the observability set
    (needs every token: ``tokens`` None).  ``reroute_rounds`` > 0 sends
    capacity overflow to the next-best experts (reading R10) instead of
    dropping it.  ``ranking`` fixes the order of tokens whose scores tie
    within rounding (``with_ranking``); ``router``, when given, is this
    module's ``route`` of the same inputs and options, computed earlier.
    """
    x = _f64(inp["x"])
    T = x.shape[0]
    E = inp["w_r"].shape[0]
    r = router if router is not None else route(
        x, inp["w_r"], k, inp.get("logit_bias"), inp.get("select_bias"), select_space,
        quantile_balance)
    if ranking:
        r = with_ranking(r, ranking)
    C = capacity(T, k, E, capacity_factor)
    if reroute_rounds > 0:
        dp = dispatch_reroute(r.scores, r.probs, k, C, reroute_rounds, ranking)
        slot_e, slot_w = dp.slot_expert, dp.slot_w
    else:
        dp = dispatch(r.idx, E, C)
        slot_e, slot_w = np.where(dp.keep, r.idx, -1), r.w
    st = load_stats(r.probs, r.idx, E)
    rows = np.arange(T) if tokens is None else np.asarray(sorted(set(int(t) for t in tokens)))
    y = np.zeros((rows.shape[0], x.shape[1]))
    pos = {int(t): i for i, t in enumerate(rows)}
    groups: Dict[int, list] = {}
    for t in rows:
        for j in range(k):
            if slot_e[t, j] >= 0:
                groups.setdefault(int(slot_e[t, j]), []).append((int(t), j))
    outputs: Dict[int, np.ndarray] = {}
    for e, tj in sorted(groups.items()):
        tt = np.array([t for t, _ in tj])
        ww = np.array([slot_w[t, j] for t, j in tj])
        out = expert_ffn(x[tt], inp["w1"][e], None if inp.get("w3") is None else inp["w3"][e],
                         inp["w2"][e], act, act_dtype)
        outputs[e] = out
        for n, (t, _) in enumerate(tj):
            y[pos[int(t)]] += ww[n] * out[n]
    if inp.get("ws1") is not None:
        sh = expert_ffn(x[rows], inp["ws1"], inp["ws3"], inp["ws2"], "swiglu", act_dtype)
        y += sh
    res = {"router": r, "dispatch": dp, "stats": st, "capacity": C, "rows": rows, "y": y}
    if observe_outputs:
        assert tokens is None, "observability needs every token"
        res["observe"] = observe(r, dp, outputs, E, k)
    return res
