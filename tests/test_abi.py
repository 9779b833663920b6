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


# ----------------------------------------------------------------------------- widened layers


def _hier(**kw):
    base = dict(T=64, d=32, a=4, b=8, k_primary=2, k_secondary=2, d_ff=64, capacity_factor=1.0,
                min_capacity=1, act_dtype=B.MOE_BF16)
    base.update(kw)
    return B.moe_hier_config(*(base[f] for f, _ in B.moe_hier_config._fields_))


@pytest.mark.parametrize("kw,status", [
    (dict(), 0), (dict(k_primary=5), 1), (dict(k_secondary=9), 1), (dict(a=0), 1),
    (dict(k_primary=0), 1), (dict(a=9, k_primary=9), 2), (dict(b=16, k_secondary=9), 2),
    (dict(a=33, b=32), 2), (dict(k_primary=4, k_secondary=8, b=8), 2), (dict(T=0), 1),
    (dict(capacity_factor=0.0), 1), (dict(act_dtype=7), 1)])
def test_hier_config_checks(lib, kw, status):
    n = ctypes.c_size_t()
    assert lib.moe_hier_workspace_size(ctypes.byref(_hier(**kw)), ctypes.byref(n)) == status
    if status == 0:
        assert n.value > 0


def test_hier_pointers_rejected_on_host(lib):
    cfg = _hier()
    f = 1 << 20  # never dereferenced: the checks fail first
    args = [f, f, None, None, f, None, None, f, None, f, None, f, None, None, None, None, None, f,
            None]
    bad = list(args)
    bad[0] = None  # x
    assert lib.moe_forward_hier(ctypes.byref(cfg), *bad) == 1
    bad = list(args)
    bad[1] = f + 4  # misaligned Wp
    assert lib.moe_forward_hier(ctypes.byref(cfg), *bad) == 1
    bad = list(args)
    bad[2] = f  # primary noise weights without noise
    assert lib.moe_forward_hier(ctypes.byref(cfg), *bad) == 1
    bad = list(args)
    bad[17] = f + 64  # workspace not 256-byte aligned
    assert lib.moe_forward_hier(ctypes.byref(cfg), *bad) == 1


def test_balanced_checks_on_host(lib):
    cfg = B.config(64, 32, 16, 64, 2, 1.0)
    n = ctypes.c_size_t()
    assert lib.moe_balanced_workspace_size(ctypes.byref(cfg), ctypes.byref(n)) == 0
    assert n.value > 0
    bad_cfg = B.config(64, 32, 16, 64, 17, 1.0)
    assert lib.moe_balanced_workspace_size(ctypes.byref(bad_cfg), ctypes.byref(n)) == 1
    f = 1 << 20
    # loss requested without thresholds
    assert lib.moe_forward_balanced(ctypes.byref(cfg), f, f, None, None, f, None, f, None, f, f,
                                    None, f, None) == 1
    # NULL Wg
    assert lib.moe_forward_balanced(ctypes.byref(cfg), f, None, None, None, f, None, f, None, f,
                                    None, None, f, None) == 1


def test_backward_checks_on_host(lib):
    cfg = B.config(64, 64, 8, 128, 2, 1.25)
    assert B.moe_backward_workspace_size(cfg) > 0
    f = 1 << 20  # never dereferenced: the checks fail first
    F = ctypes.c_float
    #       x  Wg Wn    noise W1 W2 b2    idx   gate  pos   keep  dy
    args = [f, f, None, None, f, f, None, None, None, None, None, f,
            F(0.0), F(0.0), F(0.0),
            #  dx dWg dWn  dbias dW1 db1  dW2 db2   dgate ws  bws stream
            f, f, None, None, f, None, f, None, None, f, f, None]
    bad = list(args)
    bad[11] = None  # dy
    assert lib.moe_backward(ctypes.byref(cfg), *bad) == 1
    bad = list(args)
    bad[2], bad[3] = f, f  # noise weights without their gradient
    assert lib.moe_backward(ctypes.byref(cfg), *bad) == 1
    bad = list(args)
    bad[12] = F(float("nan"))  # loss weight
    assert lib.moe_backward(ctypes.byref(cfg), *bad) == 1
    bad = list(args)
    bad[25] = f + 16  # backward workspace not 256-byte aligned
    assert lib.moe_backward(ctypes.byref(cfg), *bad) == 1
    f32 = B.config(64, 64, 8, 128, 2, 1.25, act_dtype=B.MOE_F32)
    assert B.moe_backward_workspace_size(f32) > B.moe_backward_workspace_size(cfg)  # fp32 rows
    bad = list(args)
    bad[15] = None  # dx
    assert lib.moe_backward(ctypes.byref(f32), *bad) == 1
    #        x  Wg Wn    noise idx   gate  dgate wl      wa      dWg dWn   db    dxg   ws bws st
    gargs = [f, f, None, None, None, None, f, F(0.0), F(0.0), f, None, None, None, f, f, None]
    bad = list(gargs)
    bad[9] = None  # dWg
    assert lib.moe_gate_backward(ctypes.byref(f32), *bad) == 1
    bad = list(gargs)
    bad[6] = None  # dgate
    assert lib.moe_gate_backward(ctypes.byref(cfg), *bad) == 1


def test_threshold_checks_on_host(lib):
    cfg = B.config(64, 32, 16, 64, 4, 1.0)
    assert B.moe_threshold_workspace_size(cfg) > 0
    # the bound on picks sizes the row buffers
    assert (B.moe_threshold_workspace_size(B.config(64, 32, 16, 64, 8, 1.0))
            > B.moe_threshold_workspace_size(cfg))
    n = ctypes.c_size_t()
    assert lib.moe_threshold_workspace_size(ctypes.byref(B.config(64, 32, 16, 64, 17, 1.0)),
                                            ctypes.byref(n)) == 1  # k > E
    assert lib.moe_threshold_workspace_size(ctypes.byref(B.config(64, 32, 32, 64, 17, 1.0)),
                                            ctypes.byref(n)) == 2  # k > 16
    f = 1 << 20  # never dereferenced: the checks fail first
    #       x  Wg bias  thr W1 b1    W2 b2    y  idx   gate  mask  ws stream
    args = [f, f, None, f, f, None, f, None, f, None, None, None, f, None]
    bad = list(args)
    bad[3] = None  # thresholds are required
    assert lib.moe_forward_threshold(ctypes.byref(cfg), *bad) == 1
    bad = list(args)
    bad[11] = f + 4  # misaligned mask
    assert lib.moe_forward_threshold(ctypes.byref(cfg), *bad) == 1
    bad = list(args)
    bad[12] = f + 128  # workspace not 256-byte aligned
    assert lib.moe_forward_threshold(ctypes.byref(cfg), *bad) == 1


def test_python_wrappers_reach_the_library(lib):
    """Each wrapper added for the threshold mask and expert parallelism passes
    its arguments through: arguments the host checks reject come back as
    MoEError with the library's status (no GPU work is enqueued)."""
    f = 1 << 20  # never dereferenced: the checks fail first
    cfg = B.config(64, 32, 16, 64, 4, 1.0)
    cases = [
        (lambda: B.moe_forward_threshold(cfg, f, f, None, None, f, None, f, None, f, f,
                                         stream=0), 1),
        (lambda: B.moe_expert_counts(cfg, None, f, f, stream=0), 1),
        (lambda: B.moe_dispatch_ranked(cfg, 0, f, 2, 0, f, f, f, f, f, f, f, f, f, f, f,
                                       stream=0), 1),
        (lambda: B.moe_dispatch_ranked(cfg, 10, f, 2, 2, f, f, f, f, f, f, f, f, f, f, f,
                                       stream=0), 1),
        (lambda: B.moe_aux_totals(cfg, f + 16, f, stream=0), 1),
        (lambda: B.moe_aux_from_totals(cfg, 0, f, f, f, stream=0), 1),
    ]
    for call, status in cases:
        with pytest.raises(B.MoEError) as e:
            call()
        assert e.value.status == status
