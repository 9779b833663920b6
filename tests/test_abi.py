"""The C-ABI library loads and exports every symbol include/moe.h declares;
host-side argument checks and the capacity rule work without a GPU (no
compute call is made here)."""
import ctypes
import os
import re

import pytest

import oracle
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import build as moe_build
from sparsely_gated_mixture_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return B.lib()


def declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            text = open(os.path.join(ROOT, "include", h)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(moe_\w+)\s*\(", text, re.M))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"moe_gate", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward",
            "moe_aux_loss"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(B.EXPORTS) >= names


def test_capacity_matches_oracle(lib):
    for w in wl.WORKLOADS.values():
        assert B.moe_capacity(B.config_for(w)) == oracle.capacity(w.T, w.E, w.k, w.cf, w.min_cap)
    odd = wl.Workload("odd", T=7, d=8, E=5, d_ff=8, k=3, cf=0.3, mode=wl.TOPK, dtype="bf16",
                      noisy=False)
    assert B.moe_capacity(B.config_for(odd)) == oracle.capacity(7, 5, 3, 0.3, 1)


def test_workspace_and_status_strings(lib):
    for w in wl.WORKLOADS.values():
        assert B.moe_workspace_size(B.config_for(w)) > 0
    assert B.moe_status_string(0) == "ok"
    assert "non-finite" in B.moe_status_string(4)


@pytest.mark.parametrize("field,value,status", [
    ("k", 0, 1), ("k", 17, 1), ("E", 0, 1), ("T", 0, 1), ("capacity_factor", 0.0, 1),
    ("capacity_factor", float("nan"), 1), ("gate_mode", 2, 1), ("act_dtype", 5, 1),
    ("min_capacity", 0, 1), ("E", 2048, 2)])
def test_bad_config_rejected(lib, field, value, status):
    cfg = B.config(64, 32, 16, 64, 2, 1.0)
    setattr(cfg, field, value)
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == status


def test_switch_needs_k1(lib):
    cfg = B.config(64, 32, 16, 64, 2, 1.0, gate_mode=B.MOE_GATE_SWITCH)
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == 1


def test_null_and_misaligned_pointers_rejected_on_host(lib):
    cfg = B.config(64, 32, 16, 64, 2, 1.0)
    fake = 1 << 20  # never dereferenced: the checks fail first
    # NULL x
    assert lib.moe_gate(ctypes.byref(cfg), None, fake, None, None, None, fake, fake, fake, fake,
                        None) == 1
    # misaligned x
    assert lib.moe_gate(ctypes.byref(cfg), fake + 4, fake, None, None, None, fake, fake, fake,
                        fake, None) == 1
    # noise weights without noise
    assert lib.moe_gate(ctypes.byref(cfg), fake, fake, fake, None, None, fake, fake, fake, fake,
                        None) == 1
    # misaligned workspace
    assert lib.moe_aux_loss(ctypes.byref(cfg), fake + 16, fake, None, None, None) == 1
