"""ctypes binding of libmoe.so: the C-ABI entry points under the same names.

Argument marshalling only. Arrays are torch CUDA tensors (or None where the C
signature allows NULL); they pass as raw device pointers, and every step of
the computation runs in the library's CUDA kernels. A non-zero status raises
MoEError. Loading fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe.so")

MOE_GATE_TOPK_SOFTMAX = 0
MOE_GATE_SWITCH = 1
MOE_F32 = 0
MOE_BF16 = 1

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
                4: "MOE_ERR_NONFINITE", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_BOUNDS"}

# Every symbol include/moe.h declares.
EXPORTS = ("moe_status_string", "moe_capacity", "moe_workspace_size", "moe_gate", "moe_dispatch",
           "moe_expert_ffn", "moe_combine", "moe_aux_loss", "moe_forward",
           "moe_last_device_status", "moe_dispatch_noalloc", "moe_hier_workspace_size",
           "moe_forward_hier", "moe_balanced_workspace_size", "moe_forward_balanced",
           "moe_backward_workspace_size", "moe_backward", "moe_gate_backward",
           "moe_noalloc_last_status", "moe_eval_normal_cdf", "moe_threshold_workspace_size",
           "moe_forward_threshold", "moe_expert_counts", "moe_dispatch_ranked",
           "moe_aux_totals", "moe_aux_from_totals")


class MoEError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class moe_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("d_ff", ctypes.c_int32), ("k", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("min_capacity", ctypes.c_int32),
                ("gate_mode", ctypes.c_int32), ("act_dtype", ctypes.c_int32)]


def config(T, d, E, d_ff, k, capacity_factor, gate_mode=MOE_GATE_TOPK_SOFTMAX,
           act_dtype=MOE_BF16, min_capacity=1) -> moe_config:
    return moe_config(T, d, E, d_ff, k, capacity_factor, min_capacity, gate_mode, act_dtype)


def config_for(w) -> moe_config:
    """moe_config of a workloads.Workload."""
    return config(w.T, w.d, w.E, w.d_ff, w.k, w.cf,
                  MOE_GATE_SWITCH if w.mode == "switch" else MOE_GATE_TOPK_SOFTMAX,
                  MOE_BF16 if w.dtype == "bf16" else MOE_F32, w.min_cap)


class moe_hier_config(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("a", ctypes.c_int32),
                ("b", ctypes.c_int32), ("k_primary", ctypes.c_int32),
                ("k_secondary", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("capacity_factor", ctypes.c_float), ("min_capacity", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32)]


def hier_config_for(w) -> moe_hier_config:
    """moe_hier_config of a workloads.HierWorkload."""
    return moe_hier_config(w.T, w.d, w.a, w.b, w.kp, w.ks, w.d_ff, w.cf, w.min_cap,
                           MOE_BF16 if w.dtype == "bf16" else MOE_F32)


_lock = threading.Lock()
_lib = None


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: run the package build first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            L = ctypes.CDLL(LIB_PATH)
            P, I, CP = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(moe_config)
            L.moe_status_string.argtypes = [I]
            L.moe_status_string.restype = ctypes.c_char_p
            L.moe_capacity.argtypes = [CP, ctypes.POINTER(ctypes.c_int32)]
            L.moe_workspace_size.argtypes = [CP, ctypes.POINTER(ctypes.c_size_t)]
            L.moe_gate.argtypes = [CP] + [P] * 10
            L.moe_dispatch.argtypes = [CP] + [P] * 12
            L.moe_expert_ffn.argtypes = [CP] + [P] * 11
            L.moe_combine.argtypes = [CP] + [P] * 9
            L.moe_aux_loss.argtypes = [CP] + [P] * 5
            L.moe_forward.argtypes = [CP] + [P] * 17
            L.moe_last_device_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int64)]
            L.moe_dispatch_noalloc.argtypes = [CP] + [P] * 11
            L.moe_noalloc_last_status.argtypes = [P, ctypes.POINTER(ctypes.c_int64)]
            L.moe_eval_normal_cdf.argtypes = [P, P, ctypes.c_int64, P]
            L.moe_threshold_workspace_size.argtypes = [CP, ctypes.POINTER(ctypes.c_size_t)]
            L.moe_forward_threshold.argtypes = [CP] + [P] * 14
            I32 = ctypes.c_int32
            L.moe_expert_counts.argtypes = [CP, P, P, P, P]
            L.moe_dispatch_ranked.argtypes = [CP, I32, P, I32, I32] + [P] * 12
            L.moe_aux_totals.argtypes = [CP, P, P, P]
            L.moe_aux_from_totals.argtypes = [CP, ctypes.c_int64, P, P, P, P]
            HP = ctypes.POINTER(moe_hier_config)
            L.moe_hier_workspace_size.argtypes = [HP, ctypes.POINTER(ctypes.c_size_t)]
            L.moe_forward_hier.argtypes = [HP] + [P] * 19
            L.moe_balanced_workspace_size.argtypes = [CP, ctypes.POINTER(ctypes.c_size_t)]
            L.moe_forward_balanced.argtypes = [CP] + [P] * 13
            L.moe_backward_workspace_size.argtypes = [CP, ctypes.POINTER(ctypes.c_size_t)]
            F = ctypes.c_float
            L.moe_backward.argtypes = [CP] + [P] * 12 + [F, F, F] + [P] * 12
            L.moe_gate_backward.argtypes = [CP] + [P] * 7 + [F, F] + [P] * 7
            for name in EXPORTS[1:]:
                getattr(L, name).restype = I
            _lib = L
        return _lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != 0:
        raise MoEError(status, where)


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def moe_capacity(cfg: moe_config) -> int:
    c = ctypes.c_int32()
    _check(lib().moe_capacity(ctypes.byref(cfg), ctypes.byref(c)), "moe_capacity")
    return c.value


def moe_workspace_size(cfg: moe_config) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_gate(cfg, x, Wg, Wnoise, noise, logit_bias, expert_idx, gate, thr, ws, stream=None):
    _check(lib().moe_gate(ctypes.byref(cfg), _p(x), _p(Wg), _p(Wnoise), _p(noise), _p(logit_bias),
                          _p(expert_idx), _p(gate), _p(thr), _p(ws), _stream(stream)), "moe_gate")


def moe_dispatch(cfg, expert_idx, gate, x, pos, keep, expert_count, expert_offset, xbuf,
                 row_token, row_gate, ws, stream=None):
    _check(lib().moe_dispatch(ctypes.byref(cfg), _p(expert_idx), _p(gate), _p(x), _p(pos),
                              _p(keep), _p(expert_count), _p(expert_offset), _p(xbuf),
                              _p(row_token), _p(row_gate), _p(ws), _stream(stream)),
           "moe_dispatch")


def moe_expert_ffn(cfg, xbuf, expert_offset, row_gate, W1, b1, W2, b2, hbuf, zbuf, ws,
                   stream=None):
    _check(lib().moe_expert_ffn(ctypes.byref(cfg), _p(xbuf), _p(expert_offset), _p(row_gate),
                                _p(W1), _p(b1), _p(W2), _p(b2), _p(hbuf), _p(zbuf), _p(ws),
                                _stream(stream)), "moe_expert_ffn")


def moe_combine(cfg, x, zbuf, pos, keep, expert_idx, expert_offset, y, ws, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _p(x), _p(zbuf), _p(pos), _p(keep),
                             _p(expert_idx), _p(expert_offset), _p(y), _p(ws), _stream(stream)),
           "moe_combine")


def moe_aux_loss(cfg, ws, out3, importance=None, load=None, stream=None):
    _check(lib().moe_aux_loss(ctypes.byref(cfg), _p(ws), _p(out3), _p(importance), _p(load),
                              _stream(stream)), "moe_aux_loss")


def moe_forward(cfg, x, Wg, Wnoise, noise, logit_bias, W1, b1, W2, b2, y, aux_out3, ws,
                expert_idx=None, gate=None, pos=None, keep=None, stream=None):
    _check(lib().moe_forward(ctypes.byref(cfg), _p(x), _p(Wg), _p(Wnoise), _p(noise),
                             _p(logit_bias), _p(W1), _p(b1), _p(W2), _p(b2), _p(y), _p(aux_out3),
                             _p(expert_idx), _p(gate), _p(pos), _p(keep), _p(ws),
                             _stream(stream)), "moe_forward")


def moe_hier_workspace_size(cfg: moe_hier_config) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_hier_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_hier_workspace_size")
    return n.value


def moe_forward_hier(cfg, x, Wp, Wp_noise, noise_p, Ws, Ws_noise, noise_s, W1, b1, W2, b2, y,
                     aux_out2, ws, expert_idx=None, gate=None, pos=None, keep=None, stream=None):
    _check(lib().moe_forward_hier(ctypes.byref(cfg), _p(x), _p(Wp), _p(Wp_noise), _p(noise_p),
                                  _p(Ws), _p(Ws_noise), _p(noise_s), _p(W1), _p(b1), _p(W2),
                                  _p(b2), _p(y), _p(aux_out2), _p(expert_idx), _p(gate), _p(pos),
                                  _p(keep), _p(ws), _stream(stream)), "moe_forward_hier")


def moe_balanced_workspace_size(cfg: moe_config) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_balanced_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_balanced_workspace_size")
    return n.value


def moe_forward_balanced(cfg, x, Wg, logit_bias, thresholds, W1, b1, W2, b2, y, loss_out,
                         mask_out, ws, stream=None):
    _check(lib().moe_forward_balanced(ctypes.byref(cfg), _p(x), _p(Wg), _p(logit_bias),
                                      _p(thresholds), _p(W1), _p(b1), _p(W2), _p(b2), _p(y),
                                      _p(loss_out), _p(mask_out), _p(ws), _stream(stream)),
           "moe_forward_balanced")


def moe_backward_workspace_size(cfg: moe_config) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_backward_workspace_size")
    return n.value


def moe_backward(cfg, x, Wg, Wnoise, noise, W1, W2, b2, expert_idx, gate, pos, keep, dy,
                 w_importance, w_load, w_aux, dx, dWg, dWnoise, dlogit_bias, dW1, db1, dW2, db2,
                 dgate, ws, bws, stream=None):
    _check(lib().moe_backward(ctypes.byref(cfg), _p(x), _p(Wg), _p(Wnoise), _p(noise), _p(W1),
                              _p(W2), _p(b2), _p(expert_idx), _p(gate), _p(pos), _p(keep), _p(dy),
                              float(w_importance), float(w_load), float(w_aux), _p(dx), _p(dWg),
                              _p(dWnoise), _p(dlogit_bias), _p(dW1), _p(db1), _p(dW2), _p(db2),
                              _p(dgate), _p(ws), _p(bws), _stream(stream)),
           "moe_backward")


def moe_gate_backward(cfg, x, Wg, Wnoise, noise, expert_idx, gate, dgate, w_load, w_aux, dWg,
                      dWnoise, dlogit_bias, dx_gate, ws, bws, stream=None):
    _check(lib().moe_gate_backward(ctypes.byref(cfg), _p(x), _p(Wg), _p(Wnoise), _p(noise),
                                   _p(expert_idx), _p(gate), _p(dgate), float(w_load),
                                   float(w_aux), _p(dWg), _p(dWnoise), _p(dlogit_bias),
                                   _p(dx_gate), _p(ws), _p(bws), _stream(stream)),
           "moe_gate_backward")


NOALLOC_SCRATCH_BYTES = 4 << 20


def noalloc_scratch_need(cfg) -> int:
    """Bytes of the static scratch array moe_dispatch_noalloc needs for cfg:
    the status word, two [ceil(T*k/512), E] int32 tables and the E+1 tile
    offsets, each rounded up to 256 bytes."""
    r256 = lambda v: (v + 255) // 256 * 256
    chunks = (cfg.T * cfg.k + 511) // 512
    return 256 + 2 * r256(chunks * cfg.E * 4) + r256((cfg.E + 1) * 4)


def moe_dispatch_noalloc(cfg, expert_idx, gate, x, pos, keep, expert_count, expert_offset, xbuf,
                         row_token, row_gate, stream=None):
    """moe_dispatch without a workspace, for callers that cannot allocate
    device memory; its scratch is the library's static 4 MiB device array."""
    st = lib().moe_dispatch_noalloc(ctypes.byref(cfg), _p(expert_idx), _p(gate), _p(x), _p(pos),
                                    _p(keep), _p(expert_count), _p(expert_offset), _p(xbuf),
                                    _p(row_token), _p(row_gate), _stream(stream))
    if st == 2 and noalloc_scratch_need(cfg) > NOALLOC_SCRATCH_BYTES:
        raise MoEError(st, "moe_dispatch_noalloc: these sizes need "
                           f"{noalloc_scratch_need(cfg)} bytes of scratch, more than the "
                           f"library's static {NOALLOC_SCRATCH_BYTES >> 20} MiB array")
    _check(st, "moe_dispatch_noalloc")


def moe_noalloc_last_status(stream=None):
    """Synchronise, return (status, detail) of the last moe_dispatch_noalloc
    on the current device, and clear it."""
    det = ctypes.c_int64()
    st = lib().moe_noalloc_last_status(_stream(stream), ctypes.byref(det))
    return st, det.value


def moe_threshold_workspace_size(cfg) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_threshold_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_threshold_workspace_size")
    return n.value


def moe_forward_threshold(cfg, x, Wg, logit_bias, thresholds, W1, b1, W2, b2, y, ws,
                          expert_idx=None, gate=None, mask_out=None, stream=None):
    """The threshold-mask layer (inference form of strictly balanced gating)."""
    _check(lib().moe_forward_threshold(ctypes.byref(cfg), _p(x), _p(Wg), _p(logit_bias),
                                       _p(thresholds), _p(W1), _p(b1), _p(W2), _p(b2), _p(y),
                                       _p(expert_idx), _p(gate), _p(mask_out), _p(ws),
                                       _stream(stream)),
           "moe_forward_threshold")


def moe_expert_counts(cfg, expert_idx, expert_count, ws, stream=None):
    _check(lib().moe_expert_counts(ctypes.byref(cfg), _p(expert_idx), _p(expert_count), _p(ws),
                                   _stream(stream)), "moe_expert_counts")


def moe_dispatch_ranked(cfg, capacity, counts_all, n_ranks, rank, expert_idx, gate, x, pos, keep,
                        expert_count, expert_offset, xbuf, row_token, row_gate, ws, stream=None):
    _check(lib().moe_dispatch_ranked(ctypes.byref(cfg), int(capacity), _p(counts_all),
                                     int(n_ranks), int(rank), _p(expert_idx), _p(gate), _p(x),
                                     _p(pos), _p(keep), _p(expert_count), _p(expert_offset),
                                     _p(xbuf), _p(row_token), _p(row_gate), _p(ws),
                                     _stream(stream)), "moe_dispatch_ranked")


def moe_aux_totals(cfg, ws, totals, stream=None):
    _check(lib().moe_aux_totals(ctypes.byref(cfg), _p(ws), _p(totals), _stream(stream)),
           "moe_aux_totals")


def moe_aux_from_totals(cfg, T_total, totals, out3, ws, stream=None):
    _check(lib().moe_aux_from_totals(ctypes.byref(cfg), int(T_total), _p(totals), _p(out3),
                                     _p(ws), _stream(stream)), "moe_aux_from_totals")


def moe_eval_normal_cdf(u, out, stream=None):
    """out = Phi(u) as the library's balancing kernels evaluate it (fp32)."""
    _check(lib().moe_eval_normal_cdf(_p(u), _p(out), int(u.numel()), _stream(stream)),
           "moe_eval_normal_cdf")


def moe_last_device_status(ws, stream=None):
    """Synchronise, return (status, detail) recorded on the device, and clear it."""
    det = ctypes.c_int64()
    st = lib().moe_last_device_status(_p(ws), _stream(stream), ctypes.byref(det))
    return st, det.value
