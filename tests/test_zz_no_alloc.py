"""moe_dispatch_static: dispatch for callers that cannot allocate device memory.

A caller inside a host framework that passes it only inputs and outputs, or a
service that forbids device allocations once it is running, has no workspace
to give moe_dispatch.  moe_dispatch_static keeps its scratch in a fixed array
compiled into the library instead.  These tests call it through the C ABI and
check it against moe_dispatch (which uses a caller-provided workspace) on the
same inputs, bit for bit, on two calls in a row, so a stale scratch from the
previous call would show.  The file is named to run last.
"""
import ctypes

import numpy as np
import pytest
import torch

import sparse_mixture_experts_47_b300 as moe

pytestmark = pytest.mark.gpu
DEV = "cuda"

MOE_ERR_TOO_LARGE = -6


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _outputs(cfg):
    Tk, E = cfg.T * cfg.top_k, cfg.n_experts
    full = lambda n: torch.full((n,), -7, dtype=torch.int32, device=DEV)
    return {"counts": full(E), "offsets": full(E + 1), "perm": full(max(Tk, 1)),
            "inv": full(max(Tk, 1)), "n_dropped": full(1)}


def _call(cfg, idx, o):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return moe.lib.moe_dispatch_static(ctypes.byref(cfg.c()), _ptr(idx), _ptr(o["counts"]),
                                       _ptr(o["offsets"]), _ptr(o["perm"]), _ptr(o["inv"]),
                                       _ptr(o["n_dropped"]), stream)


def _dispatch_static(cfg, idx):
    o = _outputs(cfg)
    rc = _call(cfg, idx, o)
    Tk = cfg.T * cfg.top_k
    return rc, dict(o, perm=o["perm"][:Tk], inv=o["inv"][:Tk])


def _skewed_idx(rng, T, E, k):
    pop = 1.0 / np.arange(1, E + 1) ** 1.1
    pop /= pop.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=pop) for _ in range(T)])


# Every case spans more than one 1024-slot chunk, so each one goes through the
# per-chunk histograms and bases held in the static scratch.  The last one
# needs exactly its 2 MiB: 2 * ceil(32768*8/1024) * 1024 * 4 bytes.
CASES = [(1025, 8, 1, 1.25), (513, 4, 2, 0.0), (4097, 8, 2, 0.0), (3000, 896, 8, 1.0),
         (777, 64, 8, 1.5), (32768, 1024, 8, 1.0)]


@pytest.mark.parametrize("T,E,k,cf", CASES)
def test_matches_workspace_dispatch_on_two_calls(T, E, k, cf):
    assert T * k > 1024
    rng = np.random.default_rng(T + E + k)
    cfg = moe.MoEConfig(T=T, d_model=8, n_experts=E, top_k=k, d_ff=8, capacity_factor=cf)
    for call in range(2):
        idx = torch.tensor(_skewed_idx(rng, T, E, k), dtype=torch.int32, device=DEV)
        rc, got = _dispatch_static(cfg, idx)
        assert rc == 0, moe.lib.moe_strerror(rc)
        ref = moe.dispatch(cfg, idx)
        torch.cuda.synchronize()
        assert moe.device_status() == 0
        n = int(ref["offsets"][-1])
        for key in ("counts", "offsets", "inv", "n_dropped"):
            assert torch.equal(got[key], ref[key]), (call, key)
        assert torch.equal(got["perm"][:n], ref["perm"][:n]), call


def test_allocates_no_device_memory():
    """After a first call on the device (which looks up the array's address
    and loads the kernels), a call changes neither the memory torch's
    allocator holds nor the device's free memory."""
    T, E, k = 4097, 64, 4
    rng = np.random.default_rng(1)
    cfg = moe.MoEConfig(T=T, d_model=8, n_experts=E, top_k=k, d_ff=8, capacity_factor=1.0)
    idx = torch.tensor(_skewed_idx(rng, T, E, k), dtype=torch.int32, device=DEV)
    o = _outputs(cfg)
    assert _call(cfg, idx, o) == 0
    torch.cuda.synchronize()
    ref = {key: v.clone() for key, v in o.items()}
    for v in o.values():
        v.fill_(-7)
    torch.cuda.synchronize()
    held, free = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
    assert _call(cfg, idx, o) == 0
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == held
    assert torch.cuda.mem_get_info()[0] == free
    for key in ref:
        assert torch.equal(o[key], ref[key]), key
    assert moe.device_status() == 0


def test_rejects_problem_beyond_its_scratch():
    # 2 * ceil(T*k/1024) * E * 4 bytes = 2 * 293 * 1024 * 4 > 2 MiB
    T, E = 300000, 1024
    cfg = moe.MoEConfig(T=T, d_model=8, n_experts=E, top_k=1, d_ff=8)
    idx = torch.zeros((T, 1), dtype=torch.int32, device=DEV)
    rc, _ = _dispatch_static(cfg, idx)
    assert rc == MOE_ERR_TOO_LARGE
    assert b"fixed scratch" in moe.lib.moe_strerror(rc)
