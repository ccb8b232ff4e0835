"""GPU parity at the workloads' full sizes, in the configuration bench.py
times: routing, dispatch and statistics are compared on every token; layer
outputs on a seeded sample of tokens that the oracle computes one by one."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
import oracle.moe_oracle as om
from tests.parity import full_check, gpu_layer, sample_tokens, tie_mask

pytestmark = pytest.mark.gpu
DEV = "cuda"

FULL = [("switch", 8192, None), ("mixtral", 1, None), ("mixtral", 16, None),
        ("mixtral", 4096, 192), ("mixtral", 16384, 192), ("deepseek", 128, None),
        ("deepseek", 8192, 96), ("e896", 16384, 96), ("mixtral_cap", 4096, 192),
        ("mixtral_cap", 16384, 192), ("deepseek_cap", 8192, 96)]


@pytest.mark.parametrize("name,T,n_sample", FULL, ids=[f"{n}-T{T}" for n, T, _ in FULL])
def test_layer_full_size(name, T, n_sample):
    w = mi.workload(name)
    inp = mi.generate(w, T, DEV)
    tokens = None if n_sample is None else sample_tokens(T, n_sample)
    rep, gpu, orc = full_check(w, T, inp, tokens)
    print(name, T, rep)
    if w.capacity_factor > 0:
        assert int(gpu["n_dropped"][0]) > 0
    if name == "switch":
        C = om.capacity(T, w.top_k, w.n_experts, w.capacity_factor)
        assert C == 1280
        print("dropped", int(gpu["n_dropped"][0]), "expert-0 share", orc["stats"]["f"][0])
    if name == "e896":
        # the plain top-k without the bias, for the load ratio before
        # balancing: a token whose k-th and (k+1)-th probabilities tie within
        # the band may count for either expert, which moves two counts by one
        un = gpu_layer(w, T, inp, want_unbiased=True)
        r = orc["router"]
        plain = om.topk_desc(r.probs, w.top_k)
        ref_unb = np.bincount(plain.reshape(-1), minlength=w.n_experts)
        ru = om.RouterOut(r.logits, r.probs, r.probs, plain, om.renormalise(r.probs, plain), None)
        unb_ties = int(tie_mask(ru, w.top_k)[0].sum())
        diff = np.abs(un["counts_unbiased"].astype(np.int64) - ref_unb).sum()
        assert diff <= 2 * unb_ties, (diff, unb_ties)
        mean = T * w.top_k / w.n_experts
        print("load max/mean before", ref_unb.max() / mean, "after",
              orc["stats"]["load_max_over_mean"])
        assert orc["stats"]["load_max_over_mean"] < ref_unb.max() / mean
    del inp
    torch.cuda.empty_cache()
