"""Failure detection on the GPU without a fault: the tensor-core GEMM's
bounded waits.  A test hook makes the MMA issuer of every GEMM CTA wait on a
barrier phase that nothing completes, with the main-loop limit at 1 ms; the
wait runs out, the kernel flags MOE_ERR_DEVICE_TIMEOUT, drains its own copies
and MMAs, frees its tensor memory and returns.  The host reads the status,
and the next call, with the hooks back to normal, runs on the same context and
matches the oracle.  The SM-pair tiles (a cluster of two CTAs) take the same
path in both CTAs: the CTA without the MMA issuer runs out of its own waits."""
import pytest
import torch

import moe_inputs as mi
import sparse_mixture_experts_47_b300 as moe
from tests.parity import full_check, weights_dict

pytestmark = pytest.mark.gpu
DEV = "cuda"
MOE_ERR_DEVICE_TIMEOUT = -5


@pytest.mark.parametrize("sizes,T,pair,rows", [
    ({"d_model": 256, "d_ff": 512}, 300, 0, 64),      # swapped, 64 token rows
    ({"d_model": 1024, "d_ff": 2048}, 5, 0, 16),      # swapped, split
    ({"d_model": 512, "d_ff": 2048}, 1000, 1, 0),     # 256-row tiles on SM pairs
    ({"d_model": 512, "d_ff": 1024}, 1100, 0, 256),   # the MMA N set per tile (forced)
], ids=["swapped64", "swapped", "pair", "var_width"])
def test_expired_wait_is_reported_and_the_context_stays_usable(sizes, T, pair, rows):
    w = mi.workload("mixtral").with_sizes(**sizes)
    inp = mi.generate(w, T, DEV)
    cfg = moe.config_for(w, T)
    moe.debug_set_pair_tiles(pair)
    moe.debug_set_var_up_tiles(1 if rows == 256 else 0)
    try:
        plan = moe.ffn_plan(cfg)
        assert plan["up_pair"] == pair and plan["rows_per_tile"] == rows
        full_check(w, T, inp)                              # a healthy call first
        assert moe.device_status() == 0
        moe.debug_set_wait_hooks(1_000_000, True)
        try:
            moe.layer_forward(cfg, inp["x"], weights_dict(inp))
            torch.cuda.synchronize()
            assert moe.device_status() == MOE_ERR_DEVICE_TIMEOUT
            assert moe.device_status() == 0                # read and cleared
        finally:
            moe.debug_set_wait_hooks()
        rep, _, _ = full_check(w, T, inp)
        print(rep)
        assert moe.device_status() == 0
    finally:
        moe.debug_set_pair_tiles(0)
        moe.debug_set_var_up_tiles(0)


def test_hook_arguments_checked():
    with pytest.raises(moe.MoEError):
        moe.debug_set_wait_hooks(0, False)
