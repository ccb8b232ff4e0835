"""Token-choice sparse MoE FFN layer forward on B300 (sm_103a).

A thin ctypes binding over the C ABI of ``libmoe_b300.so`` (declared in
``include/moe.h``): every step of the layer runs in the library's CUDA
kernels.  This module only marshals arguments: it allocates outputs and the
workspace with torch on the input's device and passes raw device pointers and
torch's current CUDA stream.  There is no CPU path; the import fails if the
library has not been built (``python sparse_mixture_experts_47_b300/build.py``).
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Dict, Optional

import torch

__all__ = [
    "MoEConfig", "MoEError", "lib", "capacity", "workspace_size", "router_topk", "dispatch",
    "expert_ffn", "combine", "load_stats", "layer_forward", "device_status", "Workspace",
    "LayerGraph", "LayerPipeline", "observe", "OBS_KEYS", "dispatch_reroute", "reroute_candidates",
    "ROUTING_TOKEN_CHOICE", "ROUTING_EXPERT_CHOICE", "expert_choice", "expert_choice_rows",
    "combine_rows",
    "ACT_RELU", "ACT_SWIGLU", "DTYPE_FP32", "DTYPE_BF16", "SELECT_PROBS", "SELECT_LOGITS",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_b300.so")

ACT_RELU, ACT_SWIGLU = 0, 1
DTYPE_FP32, DTYPE_BF16 = 0, 1
SELECT_PROBS, SELECT_LOGITS = 0, 1
ROUTING_TOKEN_CHOICE, ROUTING_EXPERT_CHOICE = 0, 1

MOE_OK = 0
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED",
          -3: "MOE_ERR_WORKSPACE", -4: "MOE_ERR_CUDA", -5: "MOE_ERR_DEVICE_TIMEOUT",
          -6: "MOE_ERR_TOO_LARGE"}


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {status} ({STATUS.get(status, '?')}: "
                         f"{lib.moe_strerror(status).decode()})")
        self.status = status


class _Config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("d_ff", ctypes.c_int32), ("act", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("d_ff_shared", ctypes.c_int32),
                ("select_space", ctypes.c_int32), ("quantile_balance", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("reroute_rounds", ctypes.c_int32),
                ("routing", ctypes.c_int32)]


class _Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_r", "logit_bias", "select_bias", "w1", "w3", "w2", "ws1", "ws3", "ws2")]


class _Outputs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("y", "topk_idx", "topk_w", "counts", "n_dropped", "f", "p", "aux",
                 "load_max_over_mean", "select_bias_out", "counts_unbiased", "slot_expert",
                 "slot_w", "offsets", "perm", "cand_idx")]


OBS_KEYS = ("drop_ratio", "gate_entropy", "bias_mean_abs", "bias_max_abs", "expert_out_mean",
            "expert_out_std", "expert_out_max_abs")


class _Observability(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in OBS_KEYS]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python sparse_mixture_experts_47_b300/build.py`")
    L = ctypes.CDLL(LIB_PATH)
    P, I, Z, V = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    C = ctypes.POINTER(_Config)
    L.moe_capacity.argtypes = [C]; L.moe_capacity.restype = ctypes.c_int64
    L.moe_workspace_size.argtypes = [C]; L.moe_workspace_size.restype = Z
    L.moe_router_topk.argtypes = [C] + [P] * 10 + [Z, V]; L.moe_router_topk.restype = I
    L.moe_dispatch.argtypes = [C] + [P] * 7 + [Z, V]; L.moe_dispatch.restype = I
    L.moe_dispatch_static.argtypes = [C] + [P] * 6 + [V]; L.moe_dispatch_static.restype = I
    L.moe_dispatch_reroute.argtypes = [C] + [P] * 12 + [Z, V]
    L.moe_dispatch_reroute.restype = I
    L.moe_reroute_candidates.argtypes = [C]; L.moe_reroute_candidates.restype = ctypes.c_int64
    L.moe_expert_choice_rows.argtypes = [C]; L.moe_expert_choice_rows.restype = ctypes.c_int64
    L.moe_ffn_plan.argtypes = [C, ctypes.c_int32, ctypes.c_void_p]; L.moe_ffn_plan.restype = I
    L.moe_expert_choice.argtypes = [C] + [P] * 9 + [Z, V]; L.moe_expert_choice.restype = I
    L.moe_combine_rows.argtypes = [C] + [P] * 6 + [V]; L.moe_combine_rows.restype = I
    L.moe_expert_ffn.argtypes = [C] + [P] * 8 + [Z, V]; L.moe_expert_ffn.restype = I
    L.moe_combine.argtypes = [C] + [P] * 5 + [V]; L.moe_combine.restype = I
    L.moe_load_stats.argtypes = [C] + [P] * 8 + [Z, V]; L.moe_load_stats.restype = I
    L.moe_layer_forward.argtypes = [C, P, ctypes.POINTER(_Weights), ctypes.POINTER(_Outputs),
                                    P, Z, V]
    L.moe_layer_forward.restype = I
    L.moe_layer_forward_observed.argtypes = [C, P, ctypes.POINTER(_Weights),
                                             ctypes.POINTER(_Outputs),
                                             ctypes.POINTER(_Observability), P, Z, V]
    L.moe_layer_forward_observed.restype = I
    L.moe_observe.argtypes = [C] + [P] * 5 + [ctypes.POINTER(_Observability), P, Z, V]
    L.moe_observe.restype = I
    L.moe_device_status.argtypes = [V]; L.moe_device_status.restype = I
    L.moe_strerror.argtypes = [I]; L.moe_strerror.restype = ctypes.c_char_p
    L.moe_kernel_launches.argtypes = []; L.moe_kernel_launches.restype = ctypes.c_int64
    L.moe_kernel_binary_version.argtypes = [P]; L.moe_kernel_binary_version.restype = I
    L.moe_debug_set_wait_hooks.argtypes = [ctypes.c_uint64, ctypes.c_int32]
    L.moe_debug_set_wait_hooks.restype = I
    L.moe_debug_set_pair_tiles.argtypes = [ctypes.c_int32]
    L.moe_debug_set_pair_tiles.restype = I
    L.moe_debug_set_var_up_tiles.argtypes = [ctypes.c_int32]
    L.moe_debug_set_var_up_tiles.restype = I
    L.moe_stage_timing_enable.argtypes = [I]; L.moe_stage_timing_enable.restype = I
    L.moe_stage_timing_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_int64)]
    L.moe_stage_timing_read.restype = I
    return L


lib = _load()


@dataclasses.dataclass
class MoEConfig:
    T: int
    d_model: int
    n_experts: int
    top_k: int
    d_ff: int
    act: int = ACT_SWIGLU
    dtype: int = DTYPE_BF16
    capacity_factor: float = 0.0
    d_ff_shared: int = 0
    select_space: int = SELECT_PROBS
    quantile_balance: int = 0
    out_dtype: int = DTYPE_FP32
    reroute_rounds: int = 0
    routing: int = 0

    def c(self) -> _Config:
        return _Config(*(getattr(self, f.name) for f in dataclasses.fields(self)))

    def with_T(self, T: int) -> "MoEConfig":
        return dataclasses.replace(self, T=T)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == DTYPE_FP32 else torch.bfloat16


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(fn: str, rc: int):
    if rc != MOE_OK:
        raise MoEError(fn, rc)


def capacity(cfg: MoEConfig) -> int:
    return int(lib.moe_capacity(ctypes.byref(cfg.c())))


def workspace_size(cfg: MoEConfig) -> int:
    return int(lib.moe_workspace_size(ctypes.byref(cfg.c())))


class Workspace:
    """A device byte buffer reused across calls (grows on demand)."""

    def __init__(self, device):
        self.device = torch.device(device)
        self.buf = torch.empty(0, dtype=torch.uint8, device=self.device)

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


def _ws(cfg, device, workspace):
    n = workspace_size(cfg)
    buf = (workspace or Workspace(device)).get(n)
    return buf, buf.numel()


def router_topk(cfg: MoEConfig, x, w_r, logit_bias=None, select_bias=None, want_probs=False,
                want_p=True, workspace: Optional[Workspace] = None) -> Dict[str, torch.Tensor]:
    dev = x.device
    T, E, k = cfg.T, cfg.n_experts, cfg.top_k
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    w = torch.empty((T, k), dtype=torch.float32, device=dev)
    probs = torch.empty((T, E), dtype=torch.float32, device=dev) if want_probs else None
    p = torch.empty(E, dtype=torch.float32, device=dev) if want_p else None
    sb = torch.empty(E, dtype=torch.float32, device=dev) if cfg.quantile_balance else None
    buf, nb = _ws(cfg, dev, workspace)
    _check("moe_router_topk", lib.moe_router_topk(
        ctypes.byref(cfg.c()), _ptr(x), _ptr(w_r), _ptr(logit_bias), _ptr(select_bias),
        _ptr(idx), _ptr(w), _ptr(probs), _ptr(p), _ptr(sb), _ptr(buf), nb, _stream(dev)))
    return {"idx": idx, "w": w, "probs": probs, "p": p, "select_bias": sb}


def dispatch(cfg: MoEConfig, idx, workspace: Optional[Workspace] = None) -> Dict[str, torch.Tensor]:
    dev = idx.device
    Tk, E = cfg.T * cfg.top_k, cfg.n_experts
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.full((max(Tk, 1),), -7, dtype=torch.int32, device=dev)
    inv = torch.full((max(Tk, 1),), -7, dtype=torch.int32, device=dev)
    nd = torch.empty(1, dtype=torch.int32, device=dev)
    buf, nb = _ws(cfg, dev, workspace)
    _check("moe_dispatch", lib.moe_dispatch(
        ctypes.byref(cfg.c()), _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(inv),
        _ptr(nd), _ptr(buf), nb, _stream(dev)))
    return {"counts": counts, "offsets": offsets, "perm": perm[:Tk], "inv": inv[:Tk],
            "n_dropped": nd}


def reroute_candidates(cfg: MoEConfig) -> int:
    """Candidates per token that redirection of capacity overflow uses."""
    return int(lib.moe_reroute_candidates(ctypes.byref(cfg.c())))


def dispatch_reroute(cfg: MoEConfig, idx, w, cand_idx, cand_w,
                     workspace: Optional[Workspace] = None) -> Dict[str, torch.Tensor]:
    """Dispatch with capacity overflow sent to the next-best experts
    (``cfg.reroute_rounds`` rounds); ``cand_idx``/``cand_w`` [T, nc] are each
    token's experts after its top k and their weights."""
    dev = idx.device
    T, k, E = cfg.T, cfg.top_k, cfg.n_experts
    Tk = T * k
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.full((max(Tk, 1),), -7, dtype=torch.int32, device=dev)
    inv = torch.full((max(Tk, 1),), -7, dtype=torch.int32, device=dev)
    se = torch.empty((max(T, 1), k), dtype=torch.int32, device=dev)
    sw = torch.empty((max(T, 1), k), dtype=torch.float32, device=dev)
    nd = torch.empty(1, dtype=torch.int32, device=dev)
    buf, nb = _ws(cfg, dev, workspace)
    _check("moe_dispatch_reroute", lib.moe_dispatch_reroute(
        ctypes.byref(cfg.c()), _ptr(idx), _ptr(w), _ptr(cand_idx), _ptr(cand_w), _ptr(counts),
        _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(se), _ptr(sw), _ptr(nd), _ptr(buf), nb,
        _stream(dev)))
    return {"counts": counts, "offsets": offsets, "perm": perm[:Tk], "inv": inv[:Tk],
            "slot_expert": se[:T], "slot_w": sw[:T], "n_dropped": nd}


class _FfnPlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "rows_per_tile", "up_splits", "down_splits", "up_n", "down_n", "down_rows_per_tile",
        "down_halves", "up_pair", "down_pair")]


def ffn_plan(cfg: MoEConfig, shared: bool = False) -> Dict[str, int]:
    """The grouped-GEMM geometry the library picks for ``cfg`` (host only):
    see ``moe_ffn_plan`` in moe.h."""
    info = _FfnPlanInfo()
    _check("moe_ffn_plan", lib.moe_ffn_plan(ctypes.byref(cfg.c()), 1 if shared else 0,
                                             ctypes.byref(info)))
    return {n: int(getattr(info, n)) for n, _ in _FfnPlanInfo._fields_}


def expert_choice_rows(cfg: MoEConfig) -> int:
    """Rows each expert takes under expert choice, min(C, T)."""
    return int(lib.moe_expert_choice_rows(ctypes.byref(cfg.c())))


def expert_choice(cfg: MoEConfig, probs_t, workspace: Optional[Workspace] = None
                  ) -> Dict[str, torch.Tensor]:
    """Expert-choice selection from expert-major probabilities ``probs_t``
    [E, T]: every expert takes its top ``expert_choice_rows(cfg)`` tokens."""
    dev = probs_t.device
    T, E = cfg.T, cfg.n_experts
    R = E * expert_choice_rows(cfg)
    perm = torch.full((max(R, 1),), -7, dtype=torch.int32, device=dev)
    row_w = torch.zeros(max(R, 1), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    tok_start = torch.empty(T + 1, dtype=torch.int32, device=dev)
    tok_rows = torch.full((max(R, 1),), -7, dtype=torch.int32, device=dev)
    nu = torch.empty(1, dtype=torch.int32, device=dev)
    buf, nb = _ws(cfg, dev, workspace)
    _check("moe_expert_choice", lib.moe_expert_choice(
        ctypes.byref(cfg.c()), _ptr(probs_t), _ptr(perm), _ptr(row_w), _ptr(counts),
        _ptr(offsets), _ptr(tok_start), _ptr(tok_rows), _ptr(nu), _ptr(buf), nb, _stream(dev)))
    return {"perm": perm[:R], "row_w": row_w[:R], "counts": counts, "offsets": offsets,
            "tok_start": tok_start, "tok_rows": tok_rows[:R], "n_unchosen": nu}


def combine_rows(cfg: MoEConfig, out_sorted, row_w, tok_start, tok_rows,
                 shared_out=None) -> torch.Tensor:
    """y[t] = sum over token t's rows r of row_w[r] out_sorted[r] (+ shared)."""
    dev = out_sorted.device
    ydt = torch.float32 if cfg.out_dtype == DTYPE_FP32 else torch.bfloat16
    y = torch.empty((cfg.T, cfg.d_model), dtype=ydt, device=dev)
    _check("moe_combine_rows", lib.moe_combine_rows(
        ctypes.byref(cfg.c()), _ptr(out_sorted), _ptr(row_w), _ptr(tok_start), _ptr(tok_rows),
        _ptr(shared_out), _ptr(y), _stream(dev)))
    return y


def expert_ffn(cfg: MoEConfig, x, perm, offsets, w1, w3, w2,
               workspace: Optional[Workspace] = None) -> torch.Tensor:
    dev = x.device
    rows = (cfg.n_experts * expert_choice_rows(cfg) if cfg.routing == ROUTING_EXPERT_CHOICE
            else cfg.T * cfg.top_k)
    out = torch.zeros((max(rows, 1), cfg.d_model), dtype=torch.float32, device=dev)
    buf, nb = _ws(cfg, dev, workspace)
    _check("moe_expert_ffn", lib.moe_expert_ffn(
        ctypes.byref(cfg.c()), _ptr(x), _ptr(perm), _ptr(offsets), _ptr(w1), _ptr(w3), _ptr(w2),
        _ptr(out), _ptr(buf), nb, _stream(dev)))
    return out


def combine(cfg: MoEConfig, out_sorted, inv, topk_w, shared_out=None) -> torch.Tensor:
    dev = out_sorted.device
    ydt = torch.float32 if cfg.out_dtype == DTYPE_FP32 else torch.bfloat16
    y = torch.empty((cfg.T, cfg.d_model), dtype=ydt, device=dev)
    _check("moe_combine", lib.moe_combine(
        ctypes.byref(cfg.c()), _ptr(out_sorted), _ptr(inv), _ptr(topk_w), _ptr(shared_out),
        _ptr(y), _stream(dev)))
    return y


def load_stats(cfg: MoEConfig, idx, probs, workspace: Optional[Workspace] = None):
    dev = probs.device
    E = cfg.n_experts
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    f = torch.empty(E, dtype=torch.float32, device=dev)
    p = torch.empty(E, dtype=torch.float32, device=dev)
    aux = torch.empty(1, dtype=torch.float32, device=dev)
    load = torch.empty(1, dtype=torch.float32, device=dev)
    buf, nb = _ws(cfg, dev, workspace)
    _check("moe_load_stats", lib.moe_load_stats(
        ctypes.byref(cfg.c()), _ptr(idx), _ptr(probs), _ptr(counts), _ptr(f), _ptr(p),
        _ptr(aux), _ptr(load), _ptr(buf), nb, _stream(dev)))
    return {"counts": counts, "f": f, "p": p, "aux": aux, "load_max_over_mean": load}


_WEIGHT_KEYS = ("w_r", "logit_bias", "select_bias", "w1", "w3", "w2", "ws1", "ws3", "ws2")


def _obs_tensors(cfg: MoEConfig, dev, obs: Optional[Dict]) -> Dict[str, torch.Tensor]:
    o = dict(obs or {})
    for key in OBS_KEYS:
        if o.get(key) is None:
            n = cfg.n_experts if key.startswith("expert_out") else 1
            o[key] = torch.empty(n, dtype=torch.float32, device=dev)
    return o


def layer_forward(cfg: MoEConfig, x, weights: Dict[str, Optional[torch.Tensor]],
                  workspace: Optional[Workspace] = None, outputs: Optional[Dict] = None,
                  want_unbiased_counts: bool = False, observe: bool = False,
                  observed: Optional[Dict] = None,
                  want_slots: bool = False, want_layout: bool = False
                  ) -> Dict[str, torch.Tensor]:
    """The whole layer on torch's current stream.  ``weights`` holds device
    tensors under the keys w_r, logit_bias, select_bias, w1, w3, w2, ws1,
    ws3, ws2 (missing or None = absent).  ``outputs`` may pass preallocated
    output tensors (same keys as the returned dict).  ``observe`` adds the
    monitoring set (``OBS_KEYS``: drop ratio, gate entropy, bias size,
    per-expert output mean/std/max) under the key "observe"; ``observed``
    may pass its preallocated tensors.  ``want_slots`` adds each slot's
    serving expert and gate weight (with redirection also each token's
    candidate experts after its top k); ``want_layout`` the grouped layout
    (offsets [E+1], perm [rows])."""
    dev = x.device
    T, E, k, d = cfg.T, cfg.n_experts, cfg.top_k, cfg.d_model
    o = dict(outputs or {})
    ydt = torch.float32 if cfg.out_dtype == DTYPE_FP32 else torch.bfloat16

    def need(key, shape, dtype):
        if o.get(key) is None:
            o[key] = torch.empty(shape, dtype=dtype, device=dev)

    need("y", (T, d), ydt)
    need("idx", (T, k), torch.int32)
    need("w", (T, k), torch.float32)
    need("counts", (E,), torch.int32)
    need("n_dropped", (1,), torch.int32)
    need("f", (E,), torch.float32)
    need("p", (E,), torch.float32)
    need("aux", (1,), torch.float32)
    need("load_max_over_mean", (1,), torch.float32)
    if cfg.quantile_balance:
        need("select_bias", (E,), torch.float32)
    if want_unbiased_counts:
        need("counts_unbiased", (E,), torch.int32)
    if want_slots:
        need("slot_expert", (T, k), torch.int32)
        need("slot_w", (T, k), torch.float32)
        if cfg.reroute_rounds > 0:
            need("cand_idx", (T, max(reroute_candidates(cfg), 1)), torch.int32)
    if want_layout:
        need("offsets", (E + 1,), torch.int32)
        rows = E * expert_choice_rows(cfg) if cfg.routing == ROUTING_EXPERT_CHOICE else T * k
        need("perm", (rows,), torch.int32)
    W = _Weights(*(_ptr(weights.get(key)) for key in _WEIGHT_KEYS))
    O = _Outputs(_ptr(o["y"]), _ptr(o["idx"]), _ptr(o["w"]), _ptr(o["counts"]),
                 _ptr(o["n_dropped"]), _ptr(o["f"]), _ptr(o["p"]), _ptr(o["aux"]),
                 _ptr(o["load_max_over_mean"]), _ptr(o.get("select_bias")),
                 _ptr(o.get("counts_unbiased")), _ptr(o.get("slot_expert")),
                 _ptr(o.get("slot_w")), _ptr(o.get("offsets")), _ptr(o.get("perm")),
                 _ptr(o.get("cand_idx")))
    buf, nb = _ws(cfg, dev, workspace)
    if observe or observed is not None:
        ob = _obs_tensors(cfg, dev, observed)
        OB = _Observability(*(_ptr(ob[key]) for key in OBS_KEYS))
        _check("moe_layer_forward_observed", lib.moe_layer_forward_observed(
            ctypes.byref(cfg.c()), _ptr(x), ctypes.byref(W), ctypes.byref(O), ctypes.byref(OB),
            _ptr(buf), nb, _stream(dev)))
        o["observe"] = ob
        return o
    _check("moe_layer_forward", lib.moe_layer_forward(
        ctypes.byref(cfg.c()), _ptr(x), ctypes.byref(W), ctypes.byref(O), _ptr(buf), nb,
        _stream(dev)))
    return o


def observe(cfg: MoEConfig, probs=None, out_sorted=None, offsets=None, select_bias=None,
            n_dropped=None, workspace: Optional[Workspace] = None) -> Dict[str, torch.Tensor]:
    """The monitoring set from stored tensors (stage form of the layer's
    ``observe``): gate entropy from ``probs`` [T, E], per-expert output
    scale from ``out_sorted`` [rows, d] fp32 grouped by ``offsets`` [E+1],
    bias size from ``select_bias``, drop ratio from ``n_dropped``."""
    dev = next(t.device for t in (probs, out_sorted, select_bias, n_dropped) if t is not None)
    ob = _obs_tensors(cfg, dev, None)
    OB = _Observability(*(_ptr(ob[key]) for key in OBS_KEYS))
    buf, nb = _ws(cfg, dev, workspace)
    _check("moe_observe", lib.moe_observe(
        ctypes.byref(cfg.c()), _ptr(probs), _ptr(out_sorted), _ptr(offsets), _ptr(select_bias),
        _ptr(n_dropped), ctypes.byref(OB), _ptr(buf), nb, _stream(dev)))
    return ob


class LayerGraph:
    """One ``layer_forward`` captured into a CUDA graph on fixed buffers.

    An eager ``layer_forward`` costs host time for argument checks,
    tensor-map encoding and about fifteen kernel launches; for small batches
    that host time is longer than the kernels themselves.  A graph replays
    the same kernels with a single launch.  The graph reads ``x`` and the
    weights from the tensors given here and writes the same output tensors on
    every replay: copy a new batch into ``self.x`` (same shape) before
    ``replay()``.  The capture itself runs no kernels; a first eager call
    made before it initialises the outputs and the kernels' attributes."""

    def __init__(self, cfg: MoEConfig, x, weights: Dict[str, Optional[torch.Tensor]],
                 workspace: Optional[Workspace] = None, outputs: Optional[Dict] = None,
                 warm: bool = True):
        """``warm=False`` skips the eager call; ``outputs`` must then hold
        every output tensor of an earlier ``layer_forward`` of this ``cfg``
        on the same workspace."""
        self.cfg, self.x, self.weights = cfg, x, dict(weights)
        self.workspace = workspace or Workspace(x.device)
        if warm or outputs is None:
            self.outputs = layer_forward(cfg, x, self.weights, workspace=self.workspace,
                                         outputs=outputs)
        else:
            self.outputs = outputs
        torch.cuda.synchronize(x.device)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, capture_error_mode="relaxed"):
            layer_forward(cfg, x, self.weights, workspace=self.workspace, outputs=self.outputs)

    def replay(self) -> Dict[str, torch.Tensor]:
        """Enqueue the captured layer on torch's current stream."""
        self.graph.replay()
        return self.outputs


class LayerPipeline:
    """The layer over a sequence of host batches, copies overlapped.

    Each batch goes host→device, through one replay of a captured layer, and
    its output back device→host.  The three run on separate CUDA streams
    with two device buffers per side, so the copy in of batch i+1 and the
    copy out of batch i-1 overlap the layer on batch i.  Host tensors should
    be pinned, shaped [T, d] in the layer dtype (inputs) and the output dtype
    (outputs).  Batches under a megabyte run copies and layer in sequence on
    the current stream instead."""

    def __init__(self, cfg: MoEConfig, weights: Dict[str, Optional[torch.Tensor]], device,
                 workspace: Optional[Workspace] = None):
        dev = torch.device(device)
        self.cfg = cfg
        self.workspace = workspace or Workspace(dev)
        xs = [torch.zeros((cfg.T, cfg.d_model), dtype=cfg.torch_dtype, device=dev)
              for _ in range(2)]
        # both graphs share the workspace: they never run at the same time
        self.graphs = [LayerGraph(cfg, x, weights, workspace=self.workspace) for x in xs]
        self.streams = [torch.cuda.Stream(dev) for _ in range(3)]     # in, layer, out
        self.ev = [[torch.cuda.Event() for _ in range(2)] for _ in range(3)]

    # Below this batch size (bytes in) the copies take a few microseconds and
    # the cross-stream waits cost more than the overlap saves: one stream.
    OVERLAP_MIN_BYTES = 1 << 20

    def run(self, xs_host, ys_host) -> None:
        """Enqueue batch i = xs_host[i] -> ys_host[i] for every i (no host
        synchronisation; synchronise the device before reading ys_host)."""
        s_in, s_layer, s_out = self.streams
        ev_in, ev_layer, ev_out = self.ev
        cur = torch.cuda.current_stream(s_in.device)
        g0 = self.graphs[0]
        if g0.x.numel() * g0.x.element_size() < self.OVERLAP_MIN_BYTES:
            for xh, yh in zip(xs_host, ys_host):
                g0.x.copy_(xh, non_blocking=True)
                g0.replay()
                yh.copy_(g0.outputs["y"], non_blocking=True)
            return
        for s in self.streams:
            s.wait_stream(cur)
        for i, (xh, yh) in enumerate(zip(xs_host, ys_host)):
            b = i % 2
            g = self.graphs[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_layer[b])      # batch i-2 has read this buffer
                g.x.copy_(xh, non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(s_layer):
                s_layer.wait_event(ev_in[b])
                if i >= 2:
                    s_layer.wait_event(ev_out[b])     # batch i-2's output is copied out
                g.replay()
                ev_layer[b].record(s_layer)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_layer[b])
                yh.copy_(g.outputs["y"], non_blocking=True)
                ev_out[b].record(s_out)
        for s in self.streams:
            cur.wait_stream(s)


STAGES = ("router", "dispatch", "stats", "gather", "up", "down", "shared", "combine")


def kernel_launches() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib.moe_kernel_launches())


def kernel_binary_version() -> int:
    """Architecture of the library's kernels as the CUDA runtime loads them on
    the current device (103 for sm_103a)."""
    v = ctypes.c_int32(0)
    _check("moe_kernel_binary_version", lib.moe_kernel_binary_version(ctypes.byref(v)))
    return int(v.value)


def debug_set_wait_hooks(main_loop_limit_ns: int = 2_000_000_000, stall_mma: bool = False
                         ) -> None:
    """Test hook of the GEMM's bounded waits on the current device (see
    moe_debug_set_wait_hooks); the defaults restore normal operation."""
    _check("moe_debug_set_wait_hooks",
           lib.moe_debug_set_wait_hooks(int(main_loop_limit_ns), int(bool(stall_mma))))


def debug_set_pair_tiles(policy: int = 0) -> None:
    """Switch of the 256-row SM-pair GEMM tiles (see moe_debug_set_pair_tiles):
    0 the library's rule, -1 never, 1 for every projection with token rows on
    the MMA's M side."""
    _check("moe_debug_set_pair_tiles", lib.moe_debug_set_pair_tiles(int(policy)))


def debug_set_var_up_tiles(policy: int = 0) -> None:
    """Switch of the up projection's per-tile-width geometry (see
    moe_debug_set_var_up_tiles): 1 wherever the experts average more than 64
    rows, 0 (the default) and -1 never."""
    _check("moe_debug_set_var_up_tiles", lib.moe_debug_set_var_up_tiles(int(policy)))


def stage_timing(on: bool) -> None:
    _check("moe_stage_timing_enable", lib.moe_stage_timing_enable(int(on)))


def stage_times():
    """(summed ms per stage, number of timed layer calls); blocks the host."""
    ms = (ctypes.c_double * len(STAGES))()
    calls = ctypes.c_int64(0)
    _check("moe_stage_timing_read", lib.moe_stage_timing_read(ms, ctypes.byref(calls)))
    return dict(zip(STAGES, list(ms))), int(calls.value)


def device_status(device=None) -> int:
    return int(lib.moe_device_status(_stream(device or torch.cuda.current_device())))


def config_for(workload, T: int, out_dtype: int = DTYPE_FP32) -> MoEConfig:
    """MoEConfig of a workload description (an object with the fields of
    ``moe_inputs.MoEWorkload``) at T tokens."""
    return MoEConfig(
        T=T, d_model=workload.d_model, n_experts=workload.n_experts, top_k=workload.top_k,
        d_ff=workload.d_ff, act=ACT_SWIGLU if workload.act == "swiglu" else ACT_RELU,
        dtype=DTYPE_FP32 if workload.dtype == "fp32" else DTYPE_BF16,
        capacity_factor=float(workload.capacity_factor), d_ff_shared=workload.d_ff_shared,
        select_space=SELECT_LOGITS if getattr(workload, "select_space", "probs") == "logits"
        else SELECT_PROBS, quantile_balance=int(bool(workload.quantile_balance)),
        out_dtype=out_dtype, reroute_rounds=int(getattr(workload, "reroute_rounds", 0)),
        routing=ROUTING_EXPERT_CHOICE if getattr(workload, "routing", "token") == "expert"
        else ROUTING_TOKEN_CHOICE)
