"""The C-ABI library on a machine without a GPU: it loads, exports every entry
point include/moe.h declares, and its host-only logic (capacity, workspace
sizing, argument validation, error strings) behaves; no kernel is launched."""
import ctypes
import os
import re
import subprocess

import pytest

import moe_inputs as mi
import sparse_mixture_experts_47_b300 as moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert "moe_layer_forward" in names and len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (moe_[a-z_0-9]+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert getattr(moe.lib, n) is not None


def test_built_for_sm_103a():
    # the build compiles for sm_103a only (the GPU tests ask the CUDA runtime
    # which architecture the loaded kernels carry)
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_moe_build", os.path.join(ROOT, "sparse_mixture_experts_47_b300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    flags = " ".join(b.NVCC_FLAGS)
    assert "-gencode arch=compute_103a,code=sm_103a" in flags
    assert flags.count("-gencode") == 1 and "-arch" not in flags


def mixtral(T=16384):
    return moe.MoEConfig(T=T, d_model=4096, n_experts=8, top_k=2, d_ff=14336)


def test_capacity_host_logic():
    sw = moe.MoEConfig(T=8192, d_model=1024, n_experts=8, top_k=1, d_ff=4096, act=moe.ACT_RELU,
                       capacity_factor=1.25)
    assert moe.capacity(sw) == 1280
    assert moe.capacity(mixtral(100)) == 200          # no limit: T*k
    odd = moe.MoEConfig(T=4, d_model=8, n_experts=3, top_k=2, d_ff=8, capacity_factor=0.75)
    assert moe.capacity(odd) == 2


def test_workspace_size_scales():
    a = moe.workspace_size(mixtral(4096))
    b = moe.workspace_size(mixtral(16384))
    assert 0 < a < b
    # the grouped intermediates dominate: x_sorted + h (bf16) + out_sorted (fp32)
    Tk = 16384 * 2
    assert b >= Tk * (4096 * 2 + 14336 * 2 + 4096 * 4)
    assert moe.workspace_size(moe.MoEConfig(T=0, d_model=64, n_experts=4, top_k=2, d_ff=128)) > 0


@pytest.mark.parametrize("field,value", [
    ("n_experts", 0), ("n_experts", 1025), ("top_k", 0), ("top_k", 17), ("d_model", 12),
    ("d_ff", 0), ("act", 5), ("dtype", 3), ("T", -1), ("select_space", 2), ("out_dtype", 7)])
def test_invalid_config_rejected_without_launch(field, value):
    cfg = mixtral(16)
    setattr(cfg, field, value)
    assert moe.workspace_size(cfg) == 0
    rc = moe.lib.moe_router_topk(ctypes.byref(cfg.c()), *([None] * 10), 0, None)
    assert rc == -1


def test_null_pointers_and_small_workspace_rejected():
    cfg = mixtral(16)
    c = ctypes.byref(cfg.c())
    fake = ctypes.c_void_p(1 << 20)                       # never dereferenced on the host
    assert moe.lib.moe_router_topk(c, None, fake, None, None, fake, fake, None, None, None,
                                   fake, 1 << 40, None) == -1
    assert moe.lib.moe_router_topk(c, fake, fake, None, None, fake, fake, None, None, None,
                                   fake, 16, None) == -3
    misaligned = ctypes.c_void_p((1 << 20) + 4)
    assert moe.lib.moe_combine(c, misaligned, fake, fake, None, fake, None) == -1
    qcfg = moe.MoEConfig(T=16, d_model=64, n_experts=32, top_k=2, d_ff=64, quantile_balance=1,
                         select_space=moe.SELECT_LOGITS)
    assert moe.lib.moe_router_topk(ctypes.byref(qcfg.c()), *([fake] * 10), 1 << 40, None) == -2


def test_strerror():
    for s in (0, -1, -2, -3, -4, -5):
        assert moe.lib.moe_strerror(s)
    assert moe.lib.moe_strerror(-99) == b"unknown status"


def _plan(name, T, **sizes):
    w = mi.workload(name)
    if sizes:
        w = w.with_sizes(**sizes)
    return moe.ffn_plan(moe.config_for(w, T))


def test_ffn_plan_geometries():
    """The GEMM geometry follows the rows per expert (host logic, no GPU):
    the choices behind the measured results of the bench workloads."""
    big = _plan("mixtral", 16384)            # 4096 rows per expert, reduction 14336 down
    assert (big["rows_per_tile"], big["up_n"], big["down_n"]) == (0, 256, 256)
    assert (big["down_rows_per_tile"], big["down_halves"]) == (0, 2)
    assert big["up_splits"] == big["down_splits"] == 1
    assert big["up_pair"] == 1 and big["down_pair"] == 0  # up on SM pairs, down one-SM 256 rows
    one = _plan("mixtral", 1)                # 2 rows: swap-AB, split down projection
    assert one["rows_per_tile"] == 16 and one["down_rows_per_tile"] == 16
    assert one["up_splits"] == 1 and one["down_splits"] > 1
    e896 = _plan("e896", 16384)              # about 146 rows per expert
    assert (e896["rows_per_tile"], e896["down_rows_per_tile"], e896["down_halves"]) == (0, 256, 1)
    assert e896["up_pair"] == 1 and e896["down_pair"] == 0   # balanced loads: SM pairs
    ds = _plan("deepseek", 8192)             # 256 rows per expert, reduction 2048 down
    assert (ds["rows_per_tile"], ds["down_rows_per_tile"], ds["down_halves"]) == (0, 0, 1)
    assert ds["up_pair"] == ds["down_pair"] == 0            # uneven experts: one-SM tiles
    dsc = _plan("deepseek_cap", 8192)
    assert dsc["up_pair"] == dsc["down_pair"] == 0
    assert _plan("switch", 8192)["up_pair"] == 1            # 1024 rows per expert
    sw = _plan("switch", 8192)               # 288 down tiles of N = 256: one round of SMs
    assert (sw["rows_per_tile"], sw["down_n"]) == (0, 256)
    shared = moe.ffn_plan(moe.config_for(mi.workload("deepseek"), 8192), shared=True)
    assert shared["rows_per_tile"] == 0 and shared["up_pair"] == 1


@pytest.mark.parametrize("name,T,rows,splits", [
    ("mixtral", 16, 16, (1, 1)),      # 4 rows per expert
    ("mixtral", 1, 16, (1, 2)),       # 64 down tiles: the reduction split in two
    ("switch", 1, 16, (2, 8)),        # one row, one expert: both reductions split
    ("deepseek", 128, 16, (1, 1)),    # 4 rows per expert over 256 experts
    ("e896", 4096, 64, (1, 1)),       # 36 rows per expert
])
def test_ffn_plan_swapped_tiles_for_few_rows(name, T, rows, splits):
    """A few rows per expert: weights on the MMA's M side, the token rows on
    its N side, and the reduction split only while the tiles do not fill the
    SMs once."""
    p = _plan(name, T)
    assert p["rows_per_tile"] == rows and p["down_rows_per_tile"] == rows
    assert (p["up_splits"], p["down_splits"]) == splits
    assert p["down_halves"] == 1 and p["up_pair"] == p["down_pair"] == 0


def test_pair_tiles_switch():
    """moe_debug_set_pair_tiles: -1 keeps the one-SM tiles, 1 takes the SM
    pairs wherever token rows are on the M side with N = 256 and no split."""
    try:
        moe.debug_set_pair_tiles(-1)
        assert _plan("mixtral", 16384)["up_pair"] == 0
        assert _plan("mixtral", 16384)["down_halves"] == 2          # one-SM 256-row tiles
        moe.debug_set_pair_tiles(1)
        p = _plan("mixtral", 1000, d_model=512, d_ff=2048)          # 250 rows per expert
        assert p["up_pair"] == p["down_pair"] == 1
        assert _plan("mixtral", 16)["up_pair"] == 0                 # swapped tiles stay
        with pytest.raises(moe.MoEError):
            moe.debug_set_pair_tiles(2)
    finally:
        moe.debug_set_pair_tiles(0)


def test_var_up_tiles_switch():
    """moe_debug_set_var_up_tiles: 1 takes the per-tile-width geometry for the
    up projection wherever the experts average more than 64 rows; the down
    projection keeps its own rule; 0 and -1 keep token-row tiles."""
    try:
        moe.debug_set_var_up_tiles(1)
        p = _plan("e896", 16384)
        assert (p["rows_per_tile"], p["up_pair"], p["down_rows_per_tile"]) == (256, 0, 256)
        assert p["up_splits"] == 1
        p = _plan("mixtral", 4096)                                   # 1024 rows per expert
        assert (p["rows_per_tile"], p["up_pair"], p["down_rows_per_tile"]) == (256, 0, 0)
        assert _plan("mixtral", 16)["rows_per_tile"] == 16           # swapped tiles stay
        with pytest.raises(moe.MoEError):
            moe.debug_set_var_up_tiles(2)
        moe.debug_set_var_up_tiles(-1)
        assert _plan("e896", 16384)["rows_per_tile"] == 0
    finally:
        moe.debug_set_var_up_tiles(0)
    assert _plan("mixtral", 4096)["rows_per_tile"] == 0
    assert _plan("e896", 16384)["rows_per_tile"] == 0


def test_ffn_plan_rejects_fp32_and_missing_shared_expert():
    with pytest.raises(moe.MoEError):
        moe.ffn_plan(moe.config_for(mi.workload("tiny"), 64))             # fp32 layer
    with pytest.raises(moe.MoEError):
        moe.ffn_plan(moe.config_for(mi.workload("mixtral"), 64), shared=True)
