"""Seeded synthetic inputs for the token-choice sparse MoE FFN layer.

This module is shared by the oracle side and the CUDA side. It only draws
random numbers and fixes shapes; it holds none of the layer's arithmetic
(no router, softmax, selection, FFN or statistics).

Workloads (the model shapes the pages discuss; no dataset is involved):

* ``tiny``     fp32, T=64, d=64, E=4, k=2, SwiGLU d_ff=128, no capacity.
* ``switch``   Switch-Transformer-style top-1: bf16, T=8192, d=1024, E=8, k=1,
               ReLU d_ff=4096, capacity factor 1.25, constant logit offset
               on expert 0 so that it wins about 40 % of the tokens.
* ``mixtral``  Mixtral-8x7B-shaped: bf16, d=4096, E=8, k=2, SwiGLU d_ff=14336,
               T in {1, 16, 4096, 16384}.
* ``deepseek`` DeepSeek-V3-shaped: bf16, d=7168, 256 routed SwiGLU experts with
               d_ff=2048, k=8, one always-on shared SwiGLU expert d_ff=2048,
               fixed selection bias ~ U(-0.05, 0.05), T in {128, 8192}.
* ``e896``     very sparse: bf16, T=16384, d=4096, E=896, k=8, SwiGLU d_ff=512,
               Zipf(1.1) popularity via logit offsets -1.1*ln(e+1),
               per-batch quantile selection bias.
* ``switch_reroute`` the Switch workload with capacity overflow sent to the
               next-best expert (one round) instead of being dropped.
* ``mixtral_ec`` the Mixtral-shaped layer with expert-choice routing: every
               expert takes its C = T k / E top tokens (capacity factor 1.0).
* ``mixtral_cap``, ``deepseek_cap``  the Mixtral- and DeepSeek-shaped layers
               (same seeds, so the same weights and tokens) with a capacity
               factor of 1.0, the value the capacity section gives for k = 2
               and for fine-grained experts: overflow beyond
               C = ceil(T k / E) per expert is dropped in (t, j) order.

Value recipe: x ~ N(0,1); router weight W_r ~ N(0, 1/d) in fp32; expert
weights ~ N(0, 1/fan_in), drawn in fp32 and rounded to bf16 (round to nearest
even) for the bf16 workloads.  Weights are stored like ``nn.Linear`` weights,
[out_features, in_features]: W1, W3 as [E, d_ff, d] and W2 as [E, d, d_ff].

Every tensor has its own generator stream, so the weights of a workload do
not depend on T, and x for a given T does not depend on the device's other
draws.  Streams are torch's Philox (CUDA) or MT19937 (CPU) generator, so the
same seed gives different numbers on the two device kinds; a test always uses
one device's draw for both the oracle and the kernels.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Sequence

import torch

__all__ = ["MoEWorkload", "WORKLOADS", "workload", "generate", "EXPERT0_LOGIT_OFFSET"]

# Logit offset c on expert 0 such that P(l0 + c > max of 7 iid N(0,1)) = 0.40
# when the router logits are ~N(0,1) (x ~ N(0,1), W_r ~ N(0, 1/d)).
EXPERT0_LOGIT_OFFSET = 1.0443


@dataclasses.dataclass(frozen=True)
class MoEWorkload:
    name: str
    seed: int
    d_model: int
    n_experts: int
    top_k: int
    d_ff: int
    act: str                      # "swiglu" | "relu"
    dtype: str                    # "fp32" | "bf16"
    tokens: Sequence[int]         # the T values the workload is run at
    capacity_factor: float = 0.0  # <= 0: no capacity limit
    d_ff_shared: int = 0          # 0: no shared expert
    logit_offset: str = "none"    # "none" | "expert0" | "zipf"
    select_bias: str = "none"     # "none" | "uniform"
    quantile_balance: bool = False
    reroute_rounds: int = 0       # capacity overflow: 0 dropped, R > 0 redirected
    routing: str = "token"        # "token" (token choice) | "expert" (expert choice)
    select_space: str = "probs"   # "probs" | "logits": what the selection bias is added to

    def with_sizes(self, **kw) -> "MoEWorkload":
        """A reduced copy (same recipe, smaller shapes) for small test cases."""
        return dataclasses.replace(self, **kw)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "fp32" else torch.bfloat16


WORKLOADS: Dict[str, MoEWorkload] = {
    "tiny": MoEWorkload("tiny", 0, 64, 4, 2, 128, "swiglu", "fp32", (64,)),
    "switch": MoEWorkload("switch", 1, 1024, 8, 1, 4096, "relu", "bf16", (8192,),
                          capacity_factor=1.25, logit_offset="expert0"),
    "mixtral": MoEWorkload("mixtral", 2, 4096, 8, 2, 14336, "swiglu", "bf16",
                           (1, 16, 4096, 16384)),
    "deepseek": MoEWorkload("deepseek", 3, 7168, 256, 8, 2048, "swiglu", "bf16",
                            (128, 8192), d_ff_shared=2048, select_bias="uniform"),
    "e896": MoEWorkload("e896", 4, 4096, 896, 8, 512, "swiglu", "bf16", (16384,),
                        logit_offset="zipf", quantile_balance=True),
    "mixtral_cap": MoEWorkload("mixtral_cap", 2, 4096, 8, 2, 14336, "swiglu", "bf16",
                               (4096, 16384), capacity_factor=1.0),
    "deepseek_cap": MoEWorkload("deepseek_cap", 3, 7168, 256, 8, 2048, "swiglu", "bf16",
                                (8192,), capacity_factor=1.0, d_ff_shared=2048,
                                select_bias="uniform"),
    "switch_reroute": MoEWorkload("switch_reroute", 1, 1024, 8, 1, 4096, "relu", "bf16",
                                  (8192,), capacity_factor=1.25, logit_offset="expert0",
                                  reroute_rounds=1),
    "mixtral_ec": MoEWorkload("mixtral_ec", 2, 4096, 8, 2, 14336, "swiglu", "bf16",
                              (4096, 16384), capacity_factor=1.0, routing="expert"),
}


def workload(name: str) -> MoEWorkload:
    return WORKLOADS[name]


# Stream ids: one independent generator per tensor.
_STREAMS = {"x": 1, "w_r": 2, "w1": 3, "w3": 4, "w2": 5, "ws1": 6, "ws3": 7,
            "ws2": 8, "select_bias": 9}


def _gen(device: torch.device, seed: int, stream: str) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + _STREAMS[stream] * 7919)
    return g


def _normal(shape, std, g, device, dtype, chunk_leading: bool = False):
    """N(0, std^2) drawn in fp32 and rounded to ``dtype``.

    With ``chunk_leading`` the leading dimension is drawn one slice at a time
    from the same stream, which bounds the fp32 temporary for multi-GB
    expert-weight stacks.
    """
    out = torch.empty(shape, dtype=dtype, device=device)
    if chunk_leading:
        for i in range(shape[0]):
            tmp = torch.randn(shape[1:], generator=g, device=device, dtype=torch.float32)
            out[i].copy_(tmp.mul_(std))
    else:
        tmp = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        out.copy_(tmp.mul_(std))
    return out


def generate(w: MoEWorkload, T: int, device="cpu", with_experts: bool = True
             ) -> Dict[str, Optional[torch.Tensor]]:
    """Draw the inputs of workload ``w`` at ``T`` tokens on ``device``.

    Returns a dict with keys x [T,d], w_r [E,d] fp32, logit_bias [E] fp32 or
    None, select_bias [E] fp32 or None, w1 [E,F,d], w3 [E,F,d] or None (ReLU),
    w2 [E,d,F], ws1/ws3 [Fs,d] and ws2 [d,Fs] or None.  Expert tensors are
    skipped (None) with ``with_experts=False``.
    """
    device = torch.device(device)
    d, E, F, Fs = w.d_model, w.n_experts, w.d_ff, w.d_ff_shared
    dt = w.torch_dtype
    out: Dict[str, Optional[torch.Tensor]] = {}
    out["x"] = _normal((T, d), 1.0, _gen(device, w.seed, "x"), device, dt)
    out["w_r"] = _normal((E, d), 1.0 / math.sqrt(d), _gen(device, w.seed, "w_r"),
                         device, torch.float32)
    if w.logit_offset == "expert0":
        lb = torch.zeros(E, dtype=torch.float32)
        lb[0] = EXPERT0_LOGIT_OFFSET
        out["logit_bias"] = lb.to(device)
    elif w.logit_offset == "zipf":
        # Zipf(s=1.1) popularity: logit offset -s*ln(rank), expert e has rank e+1.
        r = torch.arange(1, E + 1, dtype=torch.float64)
        out["logit_bias"] = (-1.1 * torch.log(r)).to(torch.float32).to(device)
    else:
        out["logit_bias"] = None
    if w.select_bias == "uniform":
        g = _gen(device, w.seed, "select_bias")
        u = torch.rand(E, generator=g, device=device, dtype=torch.float32)
        out["select_bias"] = (u * 0.1 - 0.05)
    else:
        out["select_bias"] = None
    if not with_experts:
        for k in ("w1", "w3", "w2", "ws1", "ws3", "ws2"):
            out[k] = None
        return out
    big = E * F * d > (1 << 26)
    out["w1"] = _normal((E, F, d), 1.0 / math.sqrt(d), _gen(device, w.seed, "w1"), device, dt, big)
    out["w3"] = (_normal((E, F, d), 1.0 / math.sqrt(d), _gen(device, w.seed, "w3"), device, dt, big)
                 if w.act == "swiglu" else None)
    out["w2"] = _normal((E, d, F), 1.0 / math.sqrt(F), _gen(device, w.seed, "w2"), device, dt, big)
    if Fs > 0:
        out["ws1"] = _normal((Fs, d), 1.0 / math.sqrt(d), _gen(device, w.seed, "ws1"), device, dt)
        out["ws3"] = _normal((Fs, d), 1.0 / math.sqrt(d), _gen(device, w.seed, "ws3"), device, dt)
        out["ws2"] = _normal((d, Fs), 1.0 / math.sqrt(Fs), _gen(device, w.seed, "ws2"), device, dt)
    else:
        out["ws1"] = out["ws3"] = out["ws2"] = None
    return out
