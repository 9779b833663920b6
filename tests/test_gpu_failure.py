"""Failure detection on the GPU without a GPU fault: a bounded wait inside the
tensor-core kernels is made to run out (MOE_WAIT_LIMIT_NS=0, so the first
wait that is not already satisfied gives up), the call reports
MOE_ERR_TIMEOUT through the status word, and the same process then runs the
layer normally and matches the oracle."""
import numpy as np
import pytest

from gpu_harness import oracle_gate, reconcile_selection, run_forward, to_device
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_wait_timeout_reported_and_context_survives(monkeypatch):
    # Long K (4096) so that the first accumulator wait of every tensor-core
    # kernel spans many pipeline stages and cannot be satisfied at once.
    w = wl.WORKLOADS["top2_large_experts"].with_(T=256, d_ff=4096)
    inp = wl.generate(w, seed=31)
    d = to_device(w, inp)
    monkeypatch.setenv("MOE_WAIT_LIMIT_NS", "0")
    res = run_forward(w, d)
    assert res["status"] == 5, B.STATUS_NAMES.get(res["status"], res["status"])  # MOE_ERR_TIMEOUT
    monkeypatch.delenv("MOE_WAIT_LIMIT_NS")
    res = run_forward(w, d)
    assert res["status"] == 0, (B.STATUS_NAMES[res["status"]], res["detail"])
    ref = oracle_gate(inp)
    _, ties, bad = reconcile_selection(ref["H"], ref["idx"], res["idx"])
    assert not bad
