"""Benchmark of the MoE layer forward path on GB300.

One step = one pass of the whole forward path (router + noisy top-k gate,
capacity and slots, dispatch, both expert layers, combine with residual, and
the balancing losses) over one batch of synthetic input, through the library's
C ABI: `value` times moe_forward over resident inputs; a stage-by-stage pass,
interleaved with it, gives the per-stage breakdown and the GEMM roofline; the
end-to-end leg adds the host copies. Default workload: the top-2 large-expert layer (T=8192, d=4096, E=8,
d_ff=14336, k=2, capacity factor 1.25, noisy gating, bf16), the one the
expert-GEMM share of bf16 peak is quoted on.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

Prints one JSON line (rank 0). With N > 1 (torchrun) every rank runs an
independent replica of the workload on its own GPU (the layer needs no
exchange between replicas); value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparsely_gated_mixture_gb300 import workloads as wl  # noqa: E402

METRIC = "MoE layer fwd tokens/s @1 GB300; expert GEMM % bf16 peak; gate/dispatch HBM %"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
NOMINAL_HBM_GBS = 8000.0  # the part's nominal HBM3e rate, reported beside the measured one
# DRAM bytes (read + write) of the expert FFN stage per step, from one ncu
# capture (profiles/expert_ffn_tc_pair_top2_large_experts.md), valid only for
# the kernel source it was taken on (hash of k_ffn_tc.cu + tc_ptx.cuh). The
# hash was re-keyed once, when the cluster PTX wrappers moved unchanged from
# k_ffn_tc.cu into tc_ptx.cuh (ptxas reports the same registers, spills and
# shared memory for every FFN kernel before and after the move).
FFN_TRAFFIC = {"top2_large_experts": {"bytes": 3855409664, "source": "166bb4bd3ef617ae"}}


class nvtx:
    """A named NVTX range around a library call (a no-op without a profiler
    attached), so ncu --nvtx or nsys can pick out each stage. If the torch
    build has no NVTX, the ranges are skipped."""

    available = None

    def __init__(self, name: str):
        self.name = name

    def __enter__(self):
        import torch
        if nvtx.available is None:
            try:
                torch.cuda.nvtx.range_push("probe")
                torch.cuda.nvtx.range_pop()
                nvtx.available = True
            except Exception:
                nvtx.available = False
        if nvtx.available:
            torch.cuda.nvtx.range_push(self.name)

    def __exit__(self, *exc):
        import torch
        if nvtx.available:
            torch.cuda.nvtx.range_pop()
        return False


def _code_only(src: str) -> str:
    """CUDA source without its comments, blank lines and indentation, so that
    a comment edit keeps a traffic record that the code still matches."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(l.strip() for l in src.splitlines() if l.strip())


def ffn_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in ("k_ffn_tc.cu", "tc_ptx.cuh"):
        with open(os.path.join(ROOT, "sparsely_gated_mixture_gb300", "csrc", f),
                  encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(w) -> int | None:
    rec = FFN_TRAFFIC.get(w.name)
    if rec is None or w != wl.WORKLOADS.get(w.name) or rec["source"] != ffn_source_hash():
        return None
    return rec["bytes"]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def slowest_rank_ms(ms: float, world: int, device) -> float:
    """A per-rank time made the job's: the maximum over all ranks (the job
    ends with its slowest replica). Needs an initialised process group when
    world > 1."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_rank: int, ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms * 1e-3)


def workload_config(w: wl.Workload, extra: dict) -> dict:
    cfg = {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "d_ff": w.d_ff, "k": w.k,
           "capacity_factor": w.cf, "gate": w.mode, "noisy": w.noisy, "capacity": w.capacity,
           "seed": 0}
    cfg.update(extra)
    return cfg


# ----------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        self.proc.wait(timeout=10)
        self.fh.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        hi = sorted(sm)[len(sm) // 2:] or sm  # the loaded half of the samples
        return {"sm_mhz": statistics.median(hi), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- algorithmic traffic


def stage_traffic(w: wl.Workload, accepted: int, experts_used: int) -> dict:
    """What each stage must move (bytes) or compute (flops) per forward."""
    s = 2 if w.dtype == "bf16" else 4
    T, d, E, dff, k = w.T, w.d, w.E, w.d_ff, w.k
    cols = 2 if w.noisy else 1
    gate_bytes = T * d * s + cols * d * E * 4 + (T * E * 4 if w.noisy else 0) + T * k * 8 + T * 8
    dispatch_bytes = T * k * 8 + T * k * 5 + 2 * accepted * d * s + accepted * 8
    ffn_flops = 4 * d * dff * accepted
    ffn_bytes = 2 * experts_used * d * dff * s + accepted * d * s + 2 * accepted * dff * s \
        + accepted * d * 4
    combine_bytes = accepted * d * 4 + 2 * T * d * s + T * k * 9
    return {"gate_bytes": gate_bytes, "dispatch_bytes": dispatch_bytes, "ffn_flops": ffn_flops,
            "ffn_bytes": ffn_bytes, "combine_bytes": combine_bytes,
            "router_flops": w.router_flops()}


# ----------------------------------------------------------------------------- our arm


def run_ours(args, w: wl.Workload):
    import torch
    import torch.distributed as dist

    from sparsely_gated_mixture_gb300 import binding as B

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    inp = wl.generate(w, seed=0)
    act = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def to_dev(a, is_act):
        if a is None:
            return None
        if is_act and w.dtype == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    x = to_dev(inp["x"], True)
    Wg, Wn, noise, bias = (to_dev(inp[k], False) for k in ("Wg", "Wn", "noise", "bias"))
    W1, W2 = to_dev(inp["W1"], True), to_dev(inp["W2"], True)
    b1 = b2 = None
    cfg = B.config_for(w)
    T, k, E, d, dff = w.T, w.k, w.E, w.d, w.d_ff
    A = T * k
    ws = torch.empty(B.moe_workspace_size(cfg), dtype=torch.uint8, device=dev)
    z = dict(device=dev)
    idx = torch.empty((T, k), dtype=torch.int32, **z)
    gate = torch.empty((T, k), dtype=torch.float32, **z)
    thr = torch.empty((T, 2), dtype=torch.float32, **z)
    pos = torch.empty((T, k), dtype=torch.int32, **z)
    keep = torch.empty((T, k), dtype=torch.uint8, **z)
    count = torch.empty(E, dtype=torch.int32, **z)
    offset = torch.empty(E + 1, dtype=torch.int32, **z)
    xbuf = torch.empty((A, d), dtype=act, **z)
    row_token = torch.empty(A, dtype=torch.int32, **z)
    row_gate = torch.empty(A, dtype=torch.float32, **z)
    hbuf = torch.empty((A, dff), dtype=act, **z)
    zbuf = torch.empty((A, d), dtype=torch.float32, **z)
    y = torch.empty((T, d), dtype=act, **z)
    out3 = torch.zeros(3, dtype=torch.float32, **z)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, **z)

    # One step: the five stage entry points, each bracketed by events on the
    # launching stream so the expert GEMMs and the HBM stages are timed live.
    def step(ev=None):
        if ev: ev[0].record(stream)
        with nvtx("moe_gate"):
            B.moe_gate(cfg, x, Wg, Wn, noise, bias, idx, gate, thr, ws, stream)
        if ev: ev[1].record(stream)
        with nvtx("moe_dispatch"):
            B.moe_dispatch(cfg, idx, gate, x, pos, keep, count, offset, xbuf, row_token, row_gate,
                           ws, stream)
        if ev: ev[2].record(stream)
        with nvtx("moe_expert_ffn"):
            B.moe_expert_ffn(cfg, xbuf, offset, row_gate, W1, b1, W2, b2, hbuf, zbuf, ws, stream)
        if ev: ev[3].record(stream)
        with nvtx("moe_combine"):
            B.moe_combine(cfg, x, zbuf, pos, keep, idx, offset, y, ws, stream)
        if ev: ev[4].record(stream)
        with nvtx("moe_aux_loss"):
            B.moe_aux_loss(cfg, ws, out3, None, None, stream)
        if ev: ev[5].record(stream)

    for _ in range(args.warmup):
        step()
    st, det = B.moe_last_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES[st]} ({det}) during warm-up")
    accepted = int(keep.sum().item())
    experts_used = int((torch.minimum(count, torch.tensor(w.capacity, device=dev)) > 0).sum())

    # The step as a user runs it: one moe_forward call over resident inputs.
    def fwd_step():
        with nvtx("moe_forward"):
            B.moe_forward(cfg, x, Wg, Wn, noise, bias, W1, b1, W2, b2, y, out3, ws, idx, gate, pos,
                          keep, stream=stream)

    for _ in range(args.warmup):
        fwd_step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    # Timed region: K forward steps (the value) interleaved with K
    # stage-by-stage steps (the per-stage breakdown), so both see the same
    # clock and power state; the L2 is flushed before each, outside the events.
    for i in range(args.steps):
        flush.zero_()
        fevs[i][0].record(stream)
        fwd_step()
        fevs[i][1].record(stream)
        flush.zero_()
        step(evs[i])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    st, det = B.moe_last_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES[st]} ({det}) in the timed region")
    stages = ["gate", "dispatch", "expert_ffn", "combine", "aux_loss"]
    per = {s: [evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps)]
           for j, s in enumerate(stages)}
    stage_sum_ms = statistics.mean(sum(per[s][i] for s in stages) for i in range(args.steps))
    fwd_times = [fevs[i][0].elapsed_time(fevs[i][1]) for i in range(args.steps)]
    ms = statistics.median(fwd_times)
    ms_mean = statistics.mean(fwd_times)
    ms = slowest_rank_ms(ms, world, dev)
    ms_mean = slowest_rank_ms(ms_mean, world, dev)

    # End to end through the public call moe_forward, as a user streaming
    # batches from the host would run it: every step copies its x and noise in
    # from pinned host memory and reads y and the losses back, inside the timed
    # region. Two device buffer sets and a copy stream let step i+1's inputs
    # arrive and step i-1's result leave while step i computes. (The inputs
    # are larger than L2: 1.88 GB of expert weights stream every step.)
    x_h = torch.empty(x.shape, dtype=x.dtype).pin_memory()
    x_h.copy_(x.cpu())
    noise_h = None
    if noise is not None:
        noise_h = torch.empty(noise.shape, dtype=noise.dtype).pin_memory()
        noise_h.copy_(noise.cpu())
    y_h = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    aux_h = [torch.empty(3, dtype=torch.float32).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    noise_d = [None if noise is None else torch.empty_like(noise) for _ in range(2)]
    y_d = [torch.empty_like(y) for _ in range(2)]
    aux_d = [torch.empty(3, dtype=torch.float32, device=dev) for _ in range(2)]
    # Uploads and downloads on streams of their own, so the two directions
    # overlap each other as well as the compute.
    up_s = torch.cuda.Stream(device=dev)
    down_s = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    h2d_done, fwd_done, d2h_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def h2d(i):
        b = i % 2
        with torch.cuda.stream(up_s):
            if i >= 2:
                up_s.wait_event(fwd_done[b])  # step i-2 has finished reading x_d[b]
            x_d[b].copy_(x_h, non_blocking=True)
            if noise_h is not None:
                noise_d[b].copy_(noise_h, non_blocking=True)
            h2d_done[b].record(up_s)

    def fwd_and_d2h(i):
        b = i % 2
        stream.wait_event(h2d_done[b])
        if i >= 2:
            stream.wait_event(d2h_done[b])  # step i-2's result has left y_d[b]
        B.moe_forward(cfg, x_d[b], Wg, Wn, noise_d[b], bias, W1, b1, W2, b2, y_d[b], aux_d[b],
                      ws, stream=stream)
        fwd_done[b].record(stream)
        with torch.cuda.stream(down_s):
            down_s.wait_event(fwd_done[b])
            y_h[b].copy_(y_d[b], non_blocking=True)
            aux_h[b].copy_(aux_d[b], non_blocking=True)
            d2h_done[b].record(down_s)

    def run_e2e(n):
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d(i + 1)
            fwd_and_d2h(i)

    run_e2e(max(3, args.warmup))
    torch.cuda.synchronize()
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_ev.record(stream)
    up_s.wait_stream(stream)  # the first upload starts after the start mark
    run_e2e(args.steps)
    stream.wait_stream(up_s)
    stream.wait_stream(down_s)  # the last download is inside the timed region
    b_ev.record(stream)
    torch.cuda.synchronize()
    e2e_ms = a_ev.elapsed_time(b_ev) / args.steps
    e2e_ms = slowest_rank_ms(e2e_ms, world, dev)
    st, det = B.moe_last_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES[st]} ({det}) in the e2e region")

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None

    peaks, peak_kind = load_peaks()
    tr = stage_traffic(w, accepted, experts_used)
    mean = {s: statistics.mean(v) for s, v in per.items()}
    ffn_s = mean["expert_ffn"] * 1e-3
    ffn_tflops = tr["ffn_flops"] / ffn_s / 1e12
    bw = lambda b, s: b / (mean[s] * 1e-3) / 1e9
    # The gate's floor: HBM for its algorithmic bytes, or the router's
    # arithmetic -- three bf16 MMAs per product on the tensor cores (the
    # split-weight router, bf16 tokens), else fp32 FMA on the CUDA cores, whose
    # peak is 152 SMs x 128 FMA/clk x 2 FLOP at the sampled SM clock.
    tc_router = w.dtype == "bf16" and w.d % 8 == 0
    ffma_tflops = 152 * 128 * 2 * (clocks.get("sm_mhz") or 2070.0) * 1e6 / 1e12
    gate_hbm_ms = tr["gate_bytes"] / (peaks["hbm_gbs"] * 1e9) * 1e3
    gate_alu_ms = (3 * tr["router_flops"] / (peaks["bf16_tflops"] * 1e12) if tc_router
                   else tr["router_flops"] / (ffma_tflops * 1e12)) * 1e3
    gate_floor_ms = max(gate_hbm_ms, gate_alu_ms)
    stage_rep = {
        "gate": {"ms": mean["gate"], "gbs": bw(tr["gate_bytes"], "gate"),
                 "hbm_frac": bw(tr["gate_bytes"], "gate") / peaks["hbm_gbs"],
                 "hbm_frac_nominal": bw(tr["gate_bytes"], "gate") / NOMINAL_HBM_GBS,
                 "router_tflops": tr["router_flops"] / (mean["gate"] * 1e-3) / 1e12,
                 "floor_ms": gate_floor_ms,
                 "floor_bound": ("hbm" if gate_hbm_ms >= gate_alu_ms else
                                 "tensor (3 bf16 MMAs per product)" if tc_router else
                                 "fp32 FMA (152 SMs x 128 FMA/clk)"),
                 "frac_of_floor": gate_floor_ms / mean["gate"]},
        "dispatch": {"ms": mean["dispatch"], "gbs": bw(tr["dispatch_bytes"], "dispatch"),
                     "hbm_frac": bw(tr["dispatch_bytes"], "dispatch") / peaks["hbm_gbs"],
                     "hbm_frac_nominal": bw(tr["dispatch_bytes"], "dispatch") / NOMINAL_HBM_GBS},
        "expert_ffn": {"ms": mean["expert_ffn"], "tflops": ffn_tflops,
                       "gbs": tr["ffn_bytes"] / ffn_s / 1e9,
                       "hbm_frac": tr["ffn_bytes"] / ffn_s / 1e9 / peaks["hbm_gbs"],
                       "bf16_frac": ffn_tflops / peaks["bf16_tflops"],
                       "bf16_frac_sustained": ffn_tflops / peaks["bf16_tflops_sustained"]},
        "combine": {"ms": mean["combine"], "gbs": bw(tr["combine_bytes"], "combine"),
                    "hbm_frac": bw(tr["combine_bytes"], "combine") / peaks["hbm_gbs"],
                    "hbm_frac_nominal": bw(tr["combine_bytes"], "combine") / NOMINAL_HBM_GBS},
        "aux_loss": {"ms": mean["aux_loss"]},
    }
    tps = job_tokens_per_s(world, T, ms)
    # Router (weight split + tensor-core kernel for bf16), selection (none
    # when the tensor-core router selects in its own epilogue: bf16,
    # d % 8 == 0, every expert in one 64-column block, E % 4 == 0, k <= 8),
    # three slot kernels, gather, two GEMMs, combine, finalize.
    tc_router = w.dtype == "bf16" and w.d % 8 == 0
    fused_sel = (tc_router and (2 * w.E if w.noisy else w.E) <= 64 and w.E % 4 == 0
                 and w.k <= 8)
    launches_per_step = ((2 if tc_router else 1) + (0 if fused_sel else (1 if w.E <= 256 else 2))
                         + 3 + 1 + 2 + 1 + 1)
    # The expert GEMMs' roofline is whichever bound is the tighter for this
    # layer: the bf16 tensor rate, or HBM for the weights and activations they
    # must stream (many small experts).
    t_flops = tr["ffn_flops"] / (peaks["bf16_tflops"] * 1e12)
    t_bytes = tr["ffn_bytes"] / (peaks["hbm_gbs"] * 1e9)
    roof = {"kernel": "moe_expert_ffn (two grouped GEMM launches)"}
    if t_bytes > t_flops:
        ffn_gbs = tr["ffn_bytes"] / ffn_s / 1e9
        roof.update({"bound": "hbm", "achieved": ffn_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ffn_gbs / peaks["hbm_gbs"]})
    else:
        roof.update({"bound": "tensor", "achieved": ffn_tflops, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": ffn_tflops / peaks["bf16_tflops"]})
    roof.update({"peak_source": peak_kind, "algorithmic_flops_per_launch": tr["ffn_flops"],
                 "algorithmic_bytes": tr["ffn_bytes"], "traffic": measured_traffic(w)})
    line = {
        "metric": METRIC,
        "value": tps,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights, N(0,1) gate noise)",
        "config": workload_config(w, {"parallelism": "replicas" if world > 1 else "single",
                                      "l2": "flushed between steps (256 MiB write)",
                                      "accepted_rows": accepted,
                                      "dropped_fraction": 1 - accepted / A}),
        "roofline": roof,
        "stages": stage_rep,
        "stage_sum_ms": stage_sum_ms,
        "ms_per_step_mean": ms_mean,
        "forward_tflops": (tr["ffn_flops"] + tr["router_flops"]) / (ms * 1e-3) / 1e12,
        "forward_frac_of_bf16_peak": (tr["ffn_flops"] + tr["router_flops"]) / (ms * 1e-3) / 1e12
        / peaks["bf16_tflops"],
        "e2e": {"value": job_tokens_per_s(world, T, e2e_ms), "unit": "tokens/s",
                "ms_per_step": e2e_ms,
                "overlap": "uploads of step i+1 and downloads of step i-1, on two copy streams, "
                           "overlap the compute of step i",
                "h2d_bytes_per_step": x.numel() * x.element_size()
                + (0 if noise is None else noise.numel() * 4),
                "d2h_bytes_per_step": y.numel() * y.element_size() + 12},
        "gpu_launches": 2 * launches_per_step * args.steps,  # forward steps + stage steps
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, inp, args.cpu_sample)
    if world > 1:
        dist.destroy_process_group()
    return line


# ----------------------------------------------------------------------------- hierarchical layer


def run_hier(args, w: wl.HierWorkload):
    """The hierarchical layer: the value is moe_forward_hier over resident
    inputs (median of the timed steps, L2 flushed before each); the expert
    GEMMs, dispatch and combine are also timed through the stage calls on the
    layer's own routing (its flat choices over the a*b experts), interleaved."""
    import torch
    import torch.distributed as dist

    from sparsely_gated_mixture_gb300 import binding as B

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    inp = wl.generate_hier(w, seed=0)
    act = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def to_dev(a, is_act=False):
        if a is None:
            return None
        if is_act and w.dtype == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    x = to_dev(inp["x"], True)
    Wp, Wpn, noise_p, Ws, Wsn, noise_s = (to_dev(inp[n]) for n in
                                          ("Wp", "Wpn", "noise_p", "Ws", "Wsn", "noise_s"))
    W1, W2 = to_dev(inp["W1"], True), to_dev(inp["W2"], True)
    hcfg = B.hier_config_for(w)
    fcfg = B.config(w.T, w.d, w.E, w.d_ff, w.k, w.cf, B.MOE_GATE_TOPK_SOFTMAX,
                    B.MOE_BF16 if w.dtype == "bf16" else B.MOE_F32, w.min_cap)
    T, k, E, d, dff = w.T, w.k, w.E, w.d, w.d_ff
    A = T * k
    z = dict(device=dev)
    ws = torch.empty(B.moe_hier_workspace_size(hcfg), dtype=torch.uint8, **z)
    ws_f = torch.empty(B.moe_workspace_size(fcfg), dtype=torch.uint8, **z)
    idx = torch.empty((T, k), dtype=torch.int32, **z)
    gate = torch.empty((T, k), dtype=torch.float32, **z)
    pos = torch.empty((T, k), dtype=torch.int32, **z)
    keep = torch.empty((T, k), dtype=torch.uint8, **z)
    count = torch.empty(E, dtype=torch.int32, **z)
    offset = torch.empty(E + 1, dtype=torch.int32, **z)
    xbuf = torch.empty((A, d), dtype=act, **z)
    row_token = torch.empty(A, dtype=torch.int32, **z)
    row_gate = torch.empty(A, dtype=torch.float32, **z)
    hbuf = torch.empty((A, dff), dtype=act, **z)
    zbuf = torch.empty((A, d), dtype=torch.float32, **z)
    y = torch.empty((T, d), dtype=act, **z)
    y2 = torch.empty_like(y)
    out2 = torch.zeros(2, dtype=torch.float32, **z)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, **z)

    def fwd(xx=x, npp=noise_p, nss=noise_s, yy=y, oo=out2, with_choices=True):
        B.moe_forward_hier(hcfg, xx, Wp, Wpn, npp, Ws, Wsn, nss, W1, None, W2, None, yy, oo, ws,
                           idx if with_choices else None, gate if with_choices else None,
                           stream=stream)

    def stages(ev):
        ev[0].record(stream)
        B.moe_dispatch(fcfg, idx, gate, x, pos, keep, count, offset, xbuf, row_token, row_gate,
                       ws_f, stream)
        ev[1].record(stream)
        B.moe_expert_ffn(fcfg, xbuf, offset, row_gate, W1, None, W2, None, hbuf, zbuf, ws_f,
                         stream)
        ev[2].record(stream)
        B.moe_combine(fcfg, x, zbuf, pos, keep, idx, offset, y2, ws_f, stream)
        ev[3].record(stream)

    for _ in range(args.warmup):
        fwd()
        stages([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    st, det = B.moe_last_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES[st]} ({det}) during warm-up")
    accepted = int(keep.sum().item())
    experts_used = int((torch.minimum(count, torch.tensor(w.capacity, device=dev)) > 0).sum())
    fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    for i in range(args.steps):
        flush.zero_()
        fevs[i][0].record(stream)
        fwd()
        fevs[i][1].record(stream)
        flush.zero_()
        stages(sevs[i])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    st, det = B.moe_last_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES[st]} ({det}) in the timed region")
    ms = slowest_rank_ms(statistics.median(f[0].elapsed_time(f[1]) for f in fevs), world, dev)
    names = ["dispatch", "expert_ffn", "combine"]
    mean = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in sevs)
            for j, n in enumerate(names)}

    # End to end: x and both noise tensors in from pinned host memory, y and
    # the two losses back, every step inside the timed region (copies on
    # their own streams, overlapping the neighbouring steps' compute).
    hosts = [t.cpu().pin_memory() for t in (x, noise_p, noise_s) if t is not None]
    devs = [[torch.empty_like(t) for t in (x, noise_p, noise_s) if t is not None]
            for _ in range(2)]
    y_d = [torch.empty_like(y) for _ in range(2)]
    o_d = [torch.empty(2, dtype=torch.float32, **z) for _ in range(2)]
    y_h = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    o_h = [torch.empty(2, dtype=torch.float32).pin_memory() for _ in range(2)]
    up_s, down_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    fwd_done = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def h2d(i):
        b = i % 2
        with torch.cuda.stream(up_s):
            if i >= 2:
                up_s.wait_event(fwd_done[b])
            for dd, hh in zip(devs[b], hosts):
                dd.copy_(hh, non_blocking=True)
            h2d_done[b].record(up_s)

    def step_e2e(i):
        b = i % 2
        stream.wait_event(h2d_done[b])
        if i >= 2:
            stream.wait_event(d2h_done[b])
        dv = list(devs[b])
        xx = dv.pop(0)
        npp = dv.pop(0) if noise_p is not None else None
        nss = dv.pop(0) if noise_s is not None else None
        fwd(xx, npp, nss, y_d[b], o_d[b], with_choices=False)
        fwd_done[b].record(stream)
        with torch.cuda.stream(down_s):
            down_s.wait_event(fwd_done[b])
            y_h[b].copy_(y_d[b], non_blocking=True)
            o_h[b].copy_(o_d[b], non_blocking=True)
            d2h_done[b].record(down_s)

    def run_e2e(n):
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d(i + 1)
            step_e2e(i)

    run_e2e(max(3, args.warmup))
    torch.cuda.synchronize()
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_ev.record(stream)
    up_s.wait_stream(stream)
    run_e2e(args.steps)
    stream.wait_stream(up_s)
    stream.wait_stream(down_s)
    b_ev.record(stream)
    torch.cuda.synchronize()
    e2e_ms = slowest_rank_ms(a_ev.elapsed_time(b_ev) / args.steps, world, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    peaks, peak_kind = load_peaks()
    s = 2 if w.dtype == "bf16" else 4
    ffn_flops = 4 * d * dff * accepted
    ffn_bytes = (2 * experts_used * d * dff * s + accepted * d * s + 2 * accepted * dff * s
                 + accepted * d * 4)
    ffn_s = mean["expert_ffn"] * 1e-3
    t_flops = ffn_flops / (peaks["bf16_tflops"] * 1e12)
    t_bytes = ffn_bytes / (peaks["hbm_gbs"] * 1e9)
    roof = {"kernel": "moe_expert_ffn (two grouped GEMM launches) on the layer's routing"}
    if t_bytes > t_flops:
        gbs = ffn_bytes / ffn_s / 1e9
        roof.update({"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"]})
    else:
        tf = ffn_flops / ffn_s / 1e12
        roof.update({"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"]})
    roof.update({"peak_source": peak_kind, "algorithmic_flops_per_launch": ffn_flops,
                 "algorithmic_bytes": ffn_bytes, "traffic": None})
    tc = w.dtype == "bf16" and w.d % 8 == 0
    # primary gate (split + router with fused selection, or + selection),
    # primary finalize; the secondary logits: grouped (three slot kernels and
    # a gather packing the pairs by group, split + grouped router) or dense
    # (split + router); two-level selection, finalize, tail; three slot
    # kernels, gather, two GEMMs, combine
    prim_fused = tc and (2 * w.a if w.noisy else w.a) <= 64 and w.a % 4 == 0 and w.kp <= 8
    ncg = (2 if w.noisy else 1) * w.b
    grouped = tc and w.b % 4 == 0 and (ncg in (16, 32) or ncg % 64 == 0)
    launches = ((2 if tc else 1) + (0 if prim_fused else 1) + 1
                + (3 + 1 + 2 if grouped else (2 if tc else 1)) + 1 + 1 + 1 + 3 + 1 + 2 + 1)
    line = {
        "metric": "hierarchical MoE layer fwd tokens/s @1 GB300",
        "value": job_tokens_per_s(world, T, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights, N(0,1) gate noise)",
        "config": {"workload": w.name, "T": T, "d": d, "groups": w.a, "experts_per_group": w.b,
                   "k_primary": w.kp, "k_secondary": w.ks, "d_ff": dff, "capacity_factor": w.cf,
                   "noisy": w.noisy, "capacity": w.capacity, "seed": 0,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between steps (256 MiB write)", "accepted_rows": accepted,
                   "dropped_fraction": 1 - accepted / A},
        "roofline": roof,
        "stages": {n: {"ms": mean[n]} for n in names},
        "e2e": {"value": job_tokens_per_s(world, T, e2e_ms), "unit": "tokens/s",
                "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hosts),
                "d2h_bytes_per_step": y.numel() * y.element_size() + 8},
        "gpu_launches": (launches + 1 + 2 + 1) * args.steps,  # forward + stage calls
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_hier(w, inp, args.cpu_sample)
    if world > 1:
        dist.destroy_process_group()
    return line


def run_balanced(args, w: wl.Workload, threshold: bool = False):
    """Strictly balanced gating: the value is moe_forward_balanced (batchwise
    mask) or, with threshold, moe_forward_threshold (the inference-time
    threshold mask, thresholds from wl.thresholds) over resident inputs
    (median of the timed steps, L2 flushed before each); the expert GEMMs are
    also timed through moe_expert_ffn on the same row layout (m rows for
    every expert; the forward's own rows per expert for the threshold mask),
    interleaved."""
    import torch
    import torch.distributed as dist

    from sparsely_gated_mixture_gb300 import binding as B

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    inp = wl.generate(w, seed=0)
    act = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def to_dev(a, is_act=False):
        if a is None:
            return None
        if is_act and w.dtype == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    x = to_dev(inp["x"], True)
    Wg = to_dev(inp["Wg"])
    W1, W2 = to_dev(inp["W1"], True), to_dev(inp["W2"], True)
    cfg = B.config_for(w)
    T, E, d, dff = w.T, w.E, w.d, w.d_ff
    z = dict(device=dev)
    y = torch.empty((T, d), dtype=act, **z)
    if threshold:
        thr = torch.from_numpy(wl.thresholds(w)).to(dev)
        ws = torch.empty(B.moe_threshold_workspace_size(cfg), dtype=torch.uint8, **z)
        picks = torch.empty((T, w.k), dtype=torch.int32, **z)
        B.moe_forward_threshold(cfg, x, Wg, None, thr, W1, None, W2, None, y, ws, picks, None,
                                None, stream)
        st, det = B.moe_last_device_status(ws, stream)
        if st != 0:
            raise RuntimeError(f"device status {B.STATUS_NAMES[st]} ({det})")
        counts = torch.bincount(picks[picks < E].long(), minlength=E)
        offset = torch.cat([torch.zeros(1, dtype=torch.int64, **z), counts.cumsum(0)]).to(
            torch.int32)
        R = int(counts.sum().item())
        m = R / E  # mean rows per expert (the label)
        # the stage call's buffers: T*k rows, of which the first R are live
        fcfg = cfg
    else:
        m = max(1, min(T, (w.k * T) // E))
        R = E * m
        ws = torch.empty(B.moe_balanced_workspace_size(cfg), dtype=torch.uint8, **z)
        offset = torch.arange(0, (E + 1) * m, m, dtype=torch.int32, **z)
        fcfg = cfg
    ws_f = torch.empty(B.moe_workspace_size(fcfg), dtype=torch.uint8, **z)
    # moe_expert_ffn's row buffers hold T*k rows (its contract: the GEMMs'
    # tensor maps span them, and a ragged last tile reads past the live rows).
    rows_alloc = max(R, T * fcfg.k)
    xbuf = torch.randn((rows_alloc, d), **z).to(act)
    row_gate = torch.ones(rows_alloc, dtype=torch.float32, **z)
    hbuf = torch.empty((rows_alloc, dff), dtype=act, **z)
    zbuf = torch.empty((rows_alloc, d), dtype=torch.float32, **z)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, **z)

    def fwd(xx=x, yy=y):
        if threshold:
            B.moe_forward_threshold(cfg, xx, Wg, None, thr, W1, None, W2, None, yy, ws,
                                    stream=stream)
        else:
            B.moe_forward_balanced(cfg, xx, Wg, None, None, W1, None, W2, None, yy, None, None,
                                   ws, stream)

    def ffn():
        B.moe_expert_ffn(fcfg, xbuf, offset, row_gate, W1, None, W2, None, hbuf, zbuf, ws_f,
                         stream)

    for _ in range(args.warmup):
        fwd()
        ffn()
    st, det = B.moe_last_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES[st]} ({det}) during warm-up")
    fe = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    for i in range(args.steps):
        flush.zero_()
        fe[i][0].record(stream)
        fwd()
        fe[i][1].record(stream)
        flush.zero_()
        fe[i][2].record(stream)
        ffn()
        fe[i][3].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    st, det = B.moe_last_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES[st]} ({det}) in the timed region")
    ms = slowest_rank_ms(statistics.median(e[0].elapsed_time(e[1]) for e in fe), world, dev)
    ffn_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in fe)

    # End to end: x in from pinned host memory and y back, every step.
    x_h = x.cpu().pin_memory()
    x_d = [torch.empty_like(x) for _ in range(2)]
    y_d = [torch.empty_like(y) for _ in range(2)]
    y_h = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    up_s, down_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    fwd_done = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def h2d(i):
        b = i % 2
        with torch.cuda.stream(up_s):
            if i >= 2:
                up_s.wait_event(fwd_done[b])
            x_d[b].copy_(x_h, non_blocking=True)
            h2d_done[b].record(up_s)

    def step_e2e(i):
        b = i % 2
        stream.wait_event(h2d_done[b])
        if i >= 2:
            stream.wait_event(d2h_done[b])
        fwd(x_d[b], y_d[b])
        fwd_done[b].record(stream)
        with torch.cuda.stream(down_s):
            down_s.wait_event(fwd_done[b])
            y_h[b].copy_(y_d[b], non_blocking=True)
            d2h_done[b].record(down_s)

    def run_e2e(n):
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d(i + 1)
            step_e2e(i)

    run_e2e(max(3, args.warmup))
    torch.cuda.synchronize()
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_ev.record(stream)
    up_s.wait_stream(stream)
    run_e2e(args.steps)
    stream.wait_stream(up_s)
    stream.wait_stream(down_s)
    b_ev.record(stream)
    torch.cuda.synchronize()
    e2e_ms = slowest_rank_ms(a_ev.elapsed_time(b_ev) / args.steps, world, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    peaks, peak_kind = load_peaks()
    sb = 2 if w.dtype == "bf16" else 4
    ffn_flops = 4 * d * dff * R
    ffn_bytes = 2 * E * d * dff * sb + R * d * sb + 2 * R * dff * sb + R * d * 4
    ffn_s = ffn_ms * 1e-3
    roof = {"kernel": "moe_expert_ffn (two grouped GEMM launches), m rows per expert"}
    if ffn_bytes / (peaks["hbm_gbs"] * 1e9) > ffn_flops / (peaks["bf16_tflops"] * 1e12):
        gbs = ffn_bytes / ffn_s / 1e9
        roof.update({"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"]})
    else:
        tf = ffn_flops / ffn_s / 1e12
        roof.update({"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"]})
    roof.update({"peak_source": peak_kind, "algorithmic_flops_per_launch": ffn_flops,
                 "algorithmic_bytes": ffn_bytes, "traffic": None})
    tc = w.dtype == "bf16" and w.d % 8 == 0
    if threshold:
        # router (split + tensor-core kernel), threshold gate, three slot
        # kernels, gather, two GEMMs, combine
        launches = (2 if tc else 1) + 1 + 3 + 1 + 2 + 1
    else:
        # router (split + tensor-core kernel), mask memset, softmax, select,
        # token gates, gather, two GEMMs, combine
        launches = (2 if tc else 1) + 3 + 1 + 2 + 1
    line = {
        "metric": ("threshold-mask MoE layer fwd tokens/s @1 GB300" if threshold else
                   "strictly balanced MoE layer fwd tokens/s @1 GB300"),
        "value": job_tokens_per_s(world, T, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) tokens, N(0,1/fan_in) weights)",
        "config": {"workload": w.name, "T": T, "d": d, "E": E, "d_ff": dff, "k": w.k,
                   "rows_per_expert": m,
                   "gate": ("threshold mask, T_i = %g/E" % wl.THR_SCALE if threshold
                            else "batchwise mask"), "seed": 0,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between steps (256 MiB write)"},
        "roofline": roof,
        "stages": {"expert_ffn": {"ms": ffn_ms}},
        "e2e": {"value": job_tokens_per_s(world, T, e2e_ms), "unit": "tokens/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": x.numel() * x.element_size(),
                "d2h_bytes_per_step": y.numel() * y.element_size()},
        "gpu_launches": (launches + 2) * args.steps,  # forward + the timed GEMMs
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_bal(w, inp, args.cpu_sample, threshold)
    if world > 1:
        dist.destroy_process_group()
    return line


def fwd_launches(w: wl.Workload) -> int:
    """Kernels one moe_forward launches (with the balancing losses)."""
    tc_router = w.dtype == "bf16" and w.d % 8 == 0
    fused_sel = (tc_router and (2 * w.E if w.noisy else w.E) <= 64 and w.E % 4 == 0
                 and w.k <= 8)
    return ((2 if tc_router else 1) + (0 if fused_sel else (1 if w.E <= 256 else 2))
            + 3 + 1 + 2 + 1 + 1)


# moe_backward: padded offsets, tail zero, dy gather, four expert GEMMs, two
# bias column sums (two kernels each), dgate, loss coefficients, gate
# backward, router weight gradients (two kernels) and dx share, dx.
BWD_LAUNCHES = 18
# Tokens of the oracle's backward in the CPU baseline: it zeroes and fills
# fp64 weight gradients of the full layer (a fixed cost of seconds at the
# large-expert widths) and spends a fraction of a second to seconds per token
# at those widths, depending on the host.
BWD_CPU_SAMPLE = 16


def run_backward(args, w: wl.Workload):
    """Training step of the layer: moe_forward (with the balancing losses)
    then moe_backward (dy, loss weights 0.01 each), inputs resident, L2
    flushed before each step; the two halves are also timed apart."""
    import torch
    import torch.distributed as dist

    from sparsely_gated_mixture_gb300 import binding as B

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    if w.dtype != "bf16":
        raise SystemExit("bench.py --backward times bf16 layers")
    inp = wl.generate(w, seed=0, biases=True)
    dy_bits = wl.generate_dy(w, 0)

    def to_dev(a, is_act=False):
        if a is None:
            return None
        if is_act:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(a).to(dev)

    x, dy = to_dev(inp["x"], True), to_dev(dy_bits, True)
    Wg, Wn, noise, bias = (to_dev(inp[n]) for n in ("Wg", "Wn", "noise", "bias"))
    W1, b1, W2, b2 = (to_dev(inp[n], True) for n in ("W1", "b1", "W2", "b2"))
    cfg = B.config_for(w)
    T, E, d, dff, k = w.T, w.E, w.d, w.d_ff, w.k
    z = dict(device=dev)
    ws = torch.empty(B.moe_workspace_size(cfg), dtype=torch.uint8, **z)
    bws = torch.empty(B.moe_backward_workspace_size(cfg), dtype=torch.uint8, **z)
    y = torch.empty((T, d), dtype=torch.bfloat16, **z)
    out3 = torch.empty(3, dtype=torch.float32, **z)
    keep = torch.empty((T, k), dtype=torch.uint8, **z)
    f = lambda *sh: torch.empty(sh, dtype=torch.float32, **z)
    grads = [torch.empty((T, d), dtype=torch.bfloat16, **z), f(d, E), f(d, E) if w.noisy else None,
             f(E) if bias is not None else None, f(E, d, dff), f(E, dff), f(E, dff, d), f(E, d),
             None]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, **z)
    wts = (0.01, 0.01, 0.01)

    def fwd(xx=x):
        with nvtx("moe_forward"):
            B.moe_forward(cfg, xx, Wg, Wn, noise, bias, W1, b1, W2, b2, y, out3, ws, None, None,
                          None, keep, stream)

    def bwd(xx=x, dyy=dy, gx=None):
        g = list(grads)
        if gx is not None:
            g[0] = gx
        with nvtx("moe_backward"):
            B.moe_backward(cfg, xx, Wg, Wn, noise, W1, W2, b2, None, None, None, keep, dyy, *wts,
                           *g, ws, bws, stream)

    for _ in range(args.warmup):
        fwd()
        bwd()
    st, det = B.moe_last_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES[st]} ({det}) during warm-up")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        fwd()
        ev[i][1].record(stream)
        bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    st, det = B.moe_last_device_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES[st]} ({det}) in the timed region")
    step = [e[0].elapsed_time(e[2]) for e in ev]
    ms = slowest_rank_ms(statistics.median(step), world, dev)
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    accepted = int(keep.sum().item())

    # End to end through the public calls: x and dy in from pinned host memory
    # and dx back, every step; two buffer sets, uploads of step i+1 and the
    # download of step i-1 on two copy streams beside the compute of step i.
    x_h, dy_h = x.cpu().pin_memory(), dy.cpu().pin_memory()
    dx_h = [torch.empty((T, d), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    dy_d = [torch.empty_like(dy) for _ in range(2)]
    dx_d = [torch.empty_like(grads[0]) for _ in range(2)]
    up_s, down_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    step_done = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def h2d(i):
        b = i % 2
        with torch.cuda.stream(up_s):
            if i >= 2:
                up_s.wait_event(step_done[b])
            x_d[b].copy_(x_h, non_blocking=True)
            dy_d[b].copy_(dy_h, non_blocking=True)
            h2d_done[b].record(up_s)

    def step_e2e(i):
        b = i % 2
        stream.wait_event(h2d_done[b])
        if i >= 2:
            stream.wait_event(d2h_done[b])
        fwd(x_d[b])
        bwd(x_d[b], dy_d[b], dx_d[b])
        step_done[b].record(stream)
        with torch.cuda.stream(down_s):
            down_s.wait_event(step_done[b])
            dx_h[b].copy_(dx_d[b], non_blocking=True)
            d2h_done[b].record(down_s)

    def run_e2e(n):
        h2d(0)
        for i in range(n):
            if i + 1 < n:
                h2d(i + 1)
            step_e2e(i)

    run_e2e(3)
    torch.cuda.synchronize()
    a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_ev.record(stream)
    up_s.wait_stream(stream)
    run_e2e(args.steps)
    stream.wait_stream(up_s)
    stream.wait_stream(down_s)
    b_ev.record(stream)
    torch.cuda.synchronize()
    e2e_ms = slowest_rank_ms(a_ev.elapsed_time(b_ev) / args.steps, world, dev)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return None
    peaks, peak_kind = load_peaks()
    # The backward's four expert GEMMs: dgrad through W2 and W1, wgrad of both,
    # 2 * rows * d * d_ff multiply-adds each over the accepted rows.
    bflops = 8.0 * accepted * d * dff
    tf = bflops / (bwd_ms * 1e-3) / 1e12
    roof = {"kernel": "moe_backward (four grouped GEMM launches plus the gate, router and "
                      "row kernels), timed as one call",
            "bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": tf / peaks["bf16_tflops"], "peak_source": peak_kind,
            "algorithmic_flops_per_launch": bflops, "traffic": None}
    line = {
        "metric": "MoE layer fwd+bwd (training step) tokens/s @1 GB300",
        "value": job_tokens_per_s(world, T, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) tokens and dy, N(0,1/fan_in) weights)",
        "config": {"workload": w.name, "T": T, "d": d, "E": E, "d_ff": dff, "k": k,
                   "loss_weights": list(wts), "seed": 0,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "flushed between steps (256 MiB write)"},
        "roofline": roof,
        "stages": {"forward": {"ms": fwd_ms}, "backward": {"ms": bwd_ms},
                   "accepted_rows": accepted},
        "e2e": {"value": job_tokens_per_s(world, T, e2e_ms), "unit": "tokens/s",
                "ms_per_step": e2e_ms,
                "overlap": "uploads of step i+1 and the download of step i-1, on two copy "
                           "streams, overlap the compute of step i",
                "h2d_bytes_per_step": x.numel() * x.element_size() + dy.numel() * dy.element_size(),
                "d2h_bytes_per_step": T * d * 2},
        "gpu_launches": (fwd_launches(w) + BWD_LAUNCHES) * args.steps,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_bwd(w, inp, dy_bits, wts, BWD_CPU_SAMPLE)
    if world > 1:
        dist.destroy_process_group()
    return line


def cpu_baseline_bwd(w: wl.Workload, inp: dict, dy_bits, wts, n_sample: int) -> dict:
    """The oracle's backward as it stands on the host cores, on the first
    n_sample tokens (a layer of n_sample tokens with the same weights),
    scaled to tokens/s."""
    import oracle

    cores = 1  # orc_backward runs on one thread (its router pass uses OpenMP)
    n = min(n_sample, w.T)
    sub = dict(inp)
    for key in ("x", "noise"):
        if sub.get(key) is not None:
            sub[key] = np.ascontiguousarray(sub[key][:n])
    dy = wl.bf16_bits_to_f32(dy_bits[:n]).astype(np.float64)
    t0 = time.perf_counter()
    oracle.backward(sub, dy, *wts)
    t = time.perf_counter() - t0
    return {"value": n / t, "unit": "tokens/s", "cores": cores, "kind": "oracle", "step_s": t,
            "sample": f"the oracle's forward and backward of the first {n} tokens "
                      f"({t:.2f} s), as a layer of {n} tokens"}


def cpu_baseline_bal(w: wl.Workload, inp: dict, n_sample: int, threshold: bool = False) -> dict:
    """The oracle's balanced layer on the host cores: router, softmax and the
    batchwise mask (or the threshold mask) over every token, then the expert
    loop, timed on its own, for n_sample evenly spaced tokens; the layer's
    tokens/s extrapolates the expert loop to T."""
    import oracle

    if threshold:
        inp = dict(inp, mode_bal=1, thr=wl.thresholds(w), with_loss=False)
    cores = len(os.sched_getaffinity(0))
    n = min(n_sample, w.T)
    tokens = np.linspace(0, w.T - 1, n).astype(np.int32)
    t0 = time.perf_counter()
    ref = oracle.bal_forward(inp, tokens=tokens[:0])
    t_gate = time.perf_counter() - t0
    idx = np.tile(np.arange(w.E, dtype=np.int32), (w.T, 1))
    t0 = time.perf_counter()
    oracle.layer_out(inp["x"], idx, ref["gate"], ref["mask"], inp["W1"], inp["W2"],
                     inp.get("b1"), inp.get("b2"), tokens)
    t_ffn = time.perf_counter() - t0
    full = t_gate + t_ffn * (w.T / n)
    return {"value": w.T / full, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "extrapolated": True, "timed_tokens": n, "step_s": t_gate + t_ffn,
            "sample": f"router, softmax and {'threshold' if threshold else 'batchwise'} mask "
                      f"over all {w.T} tokens ({t_gate:.2f} s) and the expert loop over {n} "
                      f"evenly spaced tokens ({t_ffn:.3f} s), extrapolated to {w.T} tokens"}


def cpu_baseline_hier(w: wl.HierWorkload, inp: dict, n_sample: int) -> dict:
    """The oracle's hierarchical layer on the host cores: both gates, the
    two-level selection, slots and losses over every token, then the expert
    loop, timed on its own, for n_sample evenly spaced tokens; the layer's
    tokens/s extrapolates the expert loop to T."""
    import oracle

    cores = len(os.sched_getaffinity(0))
    n = min(n_sample, w.T)
    tokens = np.linspace(0, w.T - 1, n).astype(np.int32)
    t0 = time.perf_counter()
    ref = oracle.hier_forward(inp, tokens=tokens[:0])
    t_gate = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.layer_out(inp["x"], ref["idx"], ref["gate"], ref["keep"], inp["W1"], inp["W2"],
                     inp.get("b1"), inp.get("b2"), tokens)
    t_ffn = time.perf_counter() - t0
    full = t_gate + t_ffn * (w.T / n)
    return {"value": w.T / full, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "extrapolated": True, "timed_tokens": n, "step_s": t_gate + t_ffn,
            "sample": f"gates, selection, slots and losses over all {w.T} tokens "
                      f"({t_gate:.2f} s) and the expert loop over {n} evenly spaced tokens "
                      f"({t_ffn:.3f} s), extrapolated to {w.T} tokens"}


# ----------------------------------------------------------------------------- oracle timing


def oracle_step(w: wl.Workload, inp: dict, n_sample: int):
    """One timed pass of the fp64 oracle as it stands: the gate, slots and
    balancing sums over every token, then the expert loop for n_sample evenly
    spaced tokens. Returns (gate seconds, expert-loop seconds, tokens looped)."""
    import oracle

    t0 = time.perf_counter()
    c, s, H, _ = oracle.router(inp["x"], inp["Wg"], inp["Wn"], inp["noise"], inp["bias"])
    idx, gate, hk, hk1 = oracle.select(H, w.k, inp["mode"])
    C = oracle.capacity(w.T, w.E, w.k, w.cf, w.min_cap)
    pos, keep, _ = oracle.slots(idx, w.E, C)
    oracle.aux(c, s, H, idx, gate, hk, hk1, w.noisy)
    t_gate = time.perf_counter() - t0
    n = min(n_sample, w.T)
    tokens = np.linspace(0, w.T - 1, n).astype(np.int32)
    t0 = time.perf_counter()
    oracle.layer_out(inp["x"], idx, gate, keep, inp["W1"], inp["W2"], inp["b1"], inp["b2"], tokens)
    return t_gate, time.perf_counter() - t0, n


def _extrapolated(w, t_gate, t_ffn, n):
    """Tokens/s of the whole layer: the gate as timed, the expert loop scaled
    from n tokens to T."""
    return w.T / (t_gate + t_ffn * (w.T / n))


def cpu_baseline(w: wl.Workload, inp: dict, n_sample: int) -> dict:
    """The fp64 oracle on the host cores, all of them and one: each a single
    oracle_step (the gate over all T tokens, the expert loop over n_sample),
    whose layer throughput is extrapolated from the per-token expert cost."""
    import oracle

    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    tg, tf, n = oracle_step(w, inp, n_sample)
    oracle.set_threads(1)
    try:
        tg1, tf1, _ = oracle_step(w, inp, n_sample)
    finally:
        oracle.set_threads(cores)
    return {"value": _extrapolated(w, tg, tf, n), "unit": "tokens/s", "cores": cores,
            "kind": "oracle", "extrapolated": True, "timed_tokens": n,
            "sample": f"gate+slots+aux over all {w.T} tokens ({tg:.2f} s) and the expert "
                      f"loop over {n} evenly spaced tokens ({tf:.2f} s) on {cores} cores; "
                      f"the layer's tokens/s extrapolates the expert loop to {w.T} tokens",
            "single_thread": {"value": _extrapolated(w, tg1, tf1, n), "cores": 1,
                              "sample": f"the same pass on one core: {tg1:.2f} s + {tf1:.2f} s"}}


def run_reference(args, w: wl.Workload):
    """The oracle as the reference arm. Each step is one oracle_step, timed
    as run (ms_per_step is that time); the line's value is the layer
    throughput those steps extrapolate to (the expert loop covers n_sample of
    the T tokens, so each step ends in well under a second)."""
    import oracle

    rank, world, _ = dist_env()
    if rank != 0:
        return None
    inp = wl.generate(w, seed=0)
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    for _ in range(args.warmup):
        oracle_step(w, inp, args.cpu_sample)
    steps = [oracle_step(w, inp, args.cpu_sample) for _ in range(args.steps)]
    step_s = [tg + tf for tg, tf, _ in steps]
    v = statistics.mean(_extrapolated(w, tg, tf, n) for tg, tf, n in steps)
    oracle.set_threads(1)
    try:
        tg1, tf1, n1 = oracle_step(w, inp, args.cpu_sample)
    finally:
        oracle.set_threads(cores)
    n = steps[-1][2]
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": statistics.mean(step_s) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, {"parallelism": "host cores"}),
        "extrapolated": True,
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "extrapolated": True, "timed_tokens": n,
                         "sample": f"each step: gate+slots+aux over all {w.T} tokens and the "
                                   f"expert loop over {n} evenly spaced tokens, timed as run "
                                   f"(ms_per_step); value extrapolates the expert loop to "
                                   f"{w.T} tokens",
                         "single_thread": {"value": _extrapolated(w, tg1, tf1, n1), "cores": 1,
                                           "sample": f"one step on one core: {tg1:.2f} s + "
                                                     f"{tf1:.2f} s"}},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_reference_hier(args, w: wl.HierWorkload):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    inp = wl.generate_hier(w, seed=0)
    cpu_baseline_hier(w, inp, 2)
    samples = [cpu_baseline_hier(w, inp, args.cpu_sample) for _ in range(args.steps)]
    vals, last = [x["value"] for x in samples], samples[-1]
    v = statistics.mean(vals)
    step_ms = statistics.mean(x["step_s"] for x in samples) * 1e3
    return {
        "impl": "reference", "metric": "hierarchical MoE layer fwd tokens/s @1 GB300", "value": v,
        "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "T": w.T, "parallelism": "host cores"},
        "extrapolated": True,
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": last["cores"], "kind": "oracle",
                         "extrapolated": True, "timed_tokens": last["timed_tokens"],
                         "sample": last["sample"] + "; ms_per_step is the time of the steps "
                                                    "as run"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="top2_large_experts",
                    choices=sorted(wl.WORKLOADS) + sorted(wl.HIER_WORKLOADS)
                    + sorted(wl.BAL_WORKLOADS) + sorted(wl.THR_WORKLOADS))
    ap.add_argument("--cpu-sample", type=int, default=16,
                    help="tokens whose expert loop the oracle runs for the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override T (smaller cases for profiler captures)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override E (smaller cases for profiler captures)")
    ap.add_argument("--backward", action="store_true",
                    help="time the training step (moe_forward then moe_backward)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    if args.workload in wl.HIER_WORKLOADS:
        w = wl.HIER_WORKLOADS[args.workload]
        if args.tokens:
            w = w.with_(T=args.tokens)
        line = (run_reference_hier(args, w) if args.impl == "reference" else run_hier(args, w))
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if args.workload in wl.BAL_WORKLOADS or args.workload in wl.THR_WORKLOADS:
        thr_mode = args.workload in wl.THR_WORKLOADS
        w = (wl.THR_WORKLOADS if thr_mode else wl.BAL_WORKLOADS)[args.workload]
        if args.tokens:
            w = w.with_(T=args.tokens)
        if args.impl == "reference":
            rank, world, _ = dist_env()
            if rank == 0:
                inp = wl.generate(w, seed=0)
                vals = [cpu_baseline_bal(w, inp, args.cpu_sample, thr_mode)
                        for _ in range(args.steps)]
                v = statistics.mean(x["value"] for x in vals)
                print(json.dumps({
                    "impl": "reference",
                    "metric": ("threshold-mask MoE layer fwd tokens/s @1 GB300" if thr_mode else
                               "strictly balanced MoE layer fwd tokens/s @1 GB300"),
                    "value": v, "unit": "tokens/s", "n_gpus": world,
                    "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": statistics.mean(x["step_s"] for x in vals) * 1e3,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "dtype": "f64", "data": "synthetic",
                    "config": {"workload": w.name, "T": w.T, "parallelism": "host cores"},
                    "cpu_baseline": dict(vals[-1], value=v),
                    "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}), flush=True)
            return
        line = run_balanced(args, w, thr_mode)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    w = wl.WORKLOADS[args.workload]
    if args.tokens:
        w = w.with_(T=args.tokens)
    if args.experts:
        w = w.with_(E=args.experts)
    if args.backward:
        if args.impl == "reference":
            rank, world, _ = dist_env()
            if rank == 0:
                inp = wl.generate(w, seed=0, biases=True)
                dyb = wl.generate_dy(w, 0)
                # each sample takes tens of seconds at the large-expert widths
                vals = [cpu_baseline_bwd(w, inp, dyb, (0.01, 0.01, 0.01), BWD_CPU_SAMPLE)
                        for _ in range(min(args.steps, 3))]
                v = statistics.mean(x["value"] for x in vals)
                print(json.dumps({
                    "impl": "reference", "metric": "MoE layer fwd+bwd (training step) tokens/s "
                    "@1 GB300", "value": v, "unit": "tokens/s", "n_gpus": world,
                    "steps": len(vals), "warmup": args.warmup,
                    "ms_per_step": statistics.mean(x["step_s"] for x in vals) * 1e3,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "dtype": "f64", "data": "synthetic",
                    "config": {"workload": w.name, "T": w.T, "parallelism": "host cores"},
                    "cpu_baseline": dict(vals[-1], value=v),
                    "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}), flush=True)
            return
        line = run_backward(args, w)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    line = run_reference(args, w) if args.impl == "reference" else run_ours(args, w)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
