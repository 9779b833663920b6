"""fp64 CPU oracle for the sparsely-gated Mixture-of-Experts layer: the
forward path, its hierarchical and strictly balanced variants, and the flat
layer's backward.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs are the only callers.
The product library never imports this package and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain C, double precision, one loop
per definition); this module only compiles it with gcc, loads it with ctypes
and marshals numpy arrays. Each wrapper names the page passage it follows:

* "Outrageously Large Neural Networks: The Sparsely-Gated Mixture-of-Experts
  Layer" (paper summary), section 3.4: Eq. 4 noisy logits, Eq. 5
  KeepTopK-softmax, Eqs. 6-7 importance and CV^2, Eqs. 8-10 P(x,i) and load.
* "Switch Transformer" (abhik.ai), Implementation steps 1-8: fp32 router,
  argmax gate, capacity, exclusive-cumsum slots, dispatch, ReLU experts,
  combine with residual, auxiliary loss.
* "Mixture-of-Experts: Sparse Computation" (cs8803 lesson), Chapters 1, 2, 5.
* The paper summary's "Hierarchical Mixture-of-Experts" section: the two-level
  gate, y_H, Importance_H and Load_H (``hier_*``).
* Its "Strictly Balanced Gating (Batchwise Mask)" section (and the Lesson's
  Ch. 2 mask form, Ch. 4): the batchwise and threshold masks, the
  renormalised gate and L_batchwise (``bal_*``).

* Its section 3.4 "Training the gating network" and the Switch page's step 8:
  the backward of the layer (``backward``, ``loss``).

Parity status: every function is pinned by ``tests/test_oracle_pins.py``
except the expert FFN's values on random weights, which the pages never print;
those are pinned only through reductions (dense all-experts sum, the Switch
page's dispatch/combine einsum algebra, and the E = 1 dense-MLP special case).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None

TOPK_SOFTMAX = 0
SWITCH = 1
_F32 = 0
_BF16 = 1


def _compile(src: str, out: str) -> None:
    tmp = out + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so with gcc (OpenMP over tokens)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE))
    if force or stale:
        _compile(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return _F32
    if a.dtype in (np.uint16, np.int16):
        return _BF16
    raise TypeError(f"oracle inputs are float32 or bf16 bit patterns, got {a.dtype}")


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


class Oracle:
    """ctypes view of one compiled copy of moe_oracle.c."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.orc_capacity.argtypes = [I, I, I, D, I]
        lib.orc_capacity.restype = I
        lib.orc_router.argtypes = [I, I, I, P, I, P, P, P, P, P, P, P]
        lib.orc_router.restype = I
        lib.orc_select.argtypes = [I, I, I, I, P, P, P, P, P]
        lib.orc_select.restype = None
        lib.orc_gates_given.argtypes = [I, I, I, I, P, P, P]
        lib.orc_gates_given.restype = None
        lib.orc_slots.argtypes = [I, I, I, I, P, P, P, P]
        lib.orc_slots.restype = None
        lib.orc_layer_out.argtypes = [I, I, I, P, I, P, P, P, P, P, P, P, I, P, I, P]
        lib.orc_layer_out.restype = I
        lib.orc_cv2.argtypes = [P, I]
        lib.orc_cv2.restype = D
        lib.orc_aux.argtypes = [I, I, I, P, P, P, P, P, P, P, I, P, P, P, P, P]
        lib.orc_aux.restype = None
        lib.orc_softplus_at.argtypes = [D]
        lib.orc_softplus_at.restype = D
        lib.orc_phi_at.argtypes = [D]
        lib.orc_phi_at.restype = D
        lib.orc_hier_select.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P]
        lib.orc_hier_select.restype = None
        lib.orc_hier_aux.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, I, P, P, P, P, P, P]
        lib.orc_hier_aux.restype = None
        lib.orc_bal_rows.argtypes = [ctypes.c_longlong, I, I]
        lib.orc_bal_rows.restype = I
        lib.orc_softmax_rows.argtypes = [I, I, P, P]
        lib.orc_softmax_rows.restype = None
        lib.orc_bal_gate.argtypes = [I, I, I, I, P, P, P, P]
        lib.orc_bal_gate.restype = None
        lib.orc_bal_loss.argtypes = [I, I, P, P, P]
        lib.orc_bal_loss.restype = D
        lib.orc_backward.argtypes = [I, I, I, I, I, I, D, I, P, I, P, P, P, P, P, P, P, P, I,
                                     P, D, D, D, P, P, P, P, P, P, P, P, P, P, P]
        lib.orc_backward.restype = None
        lib.orc_backward_entries.argtypes = [I, I, I, I, I, I, D, I, P, I, P, P, P, P, P, P, P, I,
                                             P, I, P, P, P, P, P, P]
        lib.orc_backward_entries.restype = None
        lib.orc_hier_backward.argtypes = [I, I, I, I, I, I, I, D, I, P, I, P, P, P, P, P, P, P, P, P,
                                          P, I, P, D, D, P, P, P, P, P, P, P, P, P]
        lib.orc_hier_backward.restype = None
        lib.orc_bal_backward.argtypes = [I, I, I, I, I, I, P, I, P, P, P, P, P, P, P, I, P, D, P, P,
                                         P, P, P, P, P]
        lib.orc_bal_backward.restype = None
        self.lib = lib
        self.path = lib_path

    def capacity(self, T: int, E: int, k: int, cf: float, min_cap: int = 1) -> int:
        """C = max(min_cap, min(T, floor(k*T*cf/E))) (Switch Transformer, step 3)."""
        return int(self.lib.orc_capacity(T, E, k, float(cf), min_cap))

    def softplus(self, z: float) -> float:
        return float(self.lib.orc_softplus_at(float(z)))

    def phi(self, u: float) -> float:
        return float(self.lib.orc_phi_at(float(u)))

    def cv2(self, v) -> float:
        """Squared coefficient of variation, population std (OLNN Eq. 7)."""
        v = np.ascontiguousarray(v, dtype=np.float64)
        return float(self.lib.orc_cv2(_ptr(v), v.size))

    def router(self, x, Wg, Wn=None, noise=None, bias=None):
        """Clean logits c, noise scale sigma and noisy logits H, each [T,E] fp64,
        plus a non-finite flag (OLNN Eq. 4; Switch step 1). x is float32 or
        bf16 bits [T,d]."""
        x = np.ascontiguousarray(x)
        T, d = x.shape
        Wg = _f32(Wg)
        E = Wg.shape[1]
        if (Wn is None) != (noise is None):
            raise ValueError("noise weights and noise come together")
        Wn, noise, bias = _f32(Wn), _f32(noise), _f32(bias)
        c = np.empty((T, E), np.float64)
        s = np.empty((T, E), np.float64)
        H = np.empty((T, E), np.float64)
        bad = self.lib.orc_router(T, d, E, _ptr(x), _dtype_code(x), _ptr(Wg), _ptr(Wn),
                                  _ptr(noise), _ptr(bias), _ptr(c), _ptr(s), _ptr(H))
        return c, s, H, bool(bad)

    def select(self, H, k: int, mode: int):
        """Top-k selection and gates (OLNN Eq. 5, or Switch step 2 for
        mode=SWITCH). Returns idx [T,k] int32, gate [T,k], hk [T] (k-th largest
        H), hk1 [T] ((k+1)-th largest, -inf when k == E)."""
        H = np.ascontiguousarray(H, dtype=np.float64)
        T, E = H.shape
        if mode == SWITCH and k != 1:
            raise ValueError("Switch gating is top-1")
        idx = np.empty((T, k), np.int32)
        gate = np.empty((T, k), np.float64)
        hk = np.empty(T, np.float64)
        hk1 = np.empty(T, np.float64)
        self.lib.orc_select(T, E, k, mode, _ptr(H), _ptr(idx), _ptr(gate), _ptr(hk), _ptr(hk1))
        return idx, gate, hk, hk1

    def gates_given(self, H, idx, mode: int):
        """Gates for a forced expert set idx [T,k] (same formulas as select)."""
        H = np.ascontiguousarray(H, dtype=np.float64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T, E = H.shape
        k = idx.shape[1]
        gate = np.empty((T, k), np.float64)
        self.lib.orc_gates_given(T, E, k, mode, _ptr(H), _ptr(idx), _ptr(gate))
        return gate

    def slots(self, idx, E: int, C: int):
        """Token-order exclusive-cumsum positions, accept mask and pre-capacity
        counts (Switch steps 3-4). Returns pos [T,k] int32, keep [T,k] uint8,
        count [E] int32."""
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T, k = idx.shape
        pos = np.empty((T, k), np.int32)
        keep = np.empty((T, k), np.uint8)
        count = np.empty(E, np.int32)
        self.lib.orc_slots(T, k, E, C, _ptr(idx), _ptr(pos), _ptr(keep), _ptr(count))
        return pos, keep, count

    def layer_out(self, x, idx, gate, keep, W1, W2, b1=None, b2=None, tokens=None):
        """y_t = x_t + sum over accepted choices of gate * E_e(x_t) for the
        listed tokens (OLNN MoE output; Switch steps 6-7; lesson Ch. 1).
        Returns (y [n,d] fp64, any_nonfinite)."""
        x = np.ascontiguousarray(x)
        T, d = x.shape
        W1 = np.ascontiguousarray(W1)
        W2 = np.ascontiguousarray(W2)
        d_ff = W1.shape[2]
        wcode = _dtype_code(W1)
        if _dtype_code(W2) != wcode:
            raise TypeError("W1 and W2 share one element type")
        b1 = None if b1 is None else np.ascontiguousarray(b1)
        b2 = None if b2 is None else np.ascontiguousarray(b2)
        for b in (b1, b2):
            if b is not None and _dtype_code(b) != wcode:
                raise TypeError("biases share the weights' element type")
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        k = idx.shape[1]
        gate = np.ascontiguousarray(gate, dtype=np.float64)
        keep = np.ascontiguousarray(keep, dtype=np.uint8)
        if tokens is None:
            tokens = np.arange(T, dtype=np.int32)
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        y = np.empty((tokens.size, d), np.float64)
        bad = self.lib.orc_layer_out(d, d_ff, k, _ptr(x), _dtype_code(x), _ptr(idx),
                                     _ptr(gate), _ptr(keep), _ptr(W1), _ptr(b1), _ptr(W2),
                                     _ptr(b2), wcode, _ptr(tokens), tokens.size, _ptr(y))
        return y, bool(bad)

    def aux(self, c, sigma, H, idx, gate, hk, hk1, noisy: bool):
        """Importance, load, Switch fractions f and mean probabilities Pbar,
        and out3 = [CV(importance)^2, CV(load)^2, 0.01*E*sum(f*Pbar)]
        (OLNN Eqs. 6-10; Switch step 8)."""
        c = np.ascontiguousarray(c, dtype=np.float64)
        sigma = np.ascontiguousarray(sigma, dtype=np.float64)
        H = np.ascontiguousarray(H, dtype=np.float64)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        gate = np.ascontiguousarray(gate, dtype=np.float64)
        hk = np.ascontiguousarray(hk, dtype=np.float64)
        hk1 = np.ascontiguousarray(hk1, dtype=np.float64)
        T, E = H.shape
        k = idx.shape[1]
        imp = np.empty(E, np.float64)
        load = np.empty(E, np.float64)
        f = np.empty(E, np.float64)
        pbar = np.empty(E, np.float64)
        out3 = np.empty(3, np.float64)
        self.lib.orc_aux(T, E, k, _ptr(c), _ptr(sigma), _ptr(H), _ptr(idx), _ptr(gate),
                         _ptr(hk), _ptr(hk1), int(bool(noisy)), _ptr(imp), _ptr(load),
                         _ptr(f), _ptr(pbar), _ptr(out3))
        return dict(importance=imp, load=load, f=f, pbar=pbar, out3=out3)

    def forward(self, inp: dict, tokens=None) -> dict:
        """The whole forward path on one input set.

        ``inp`` holds numpy arrays and sizes: x, Wg, Wn, noise, bias, W1, b1,
        W2, b2 (optional ones may be None) and k, cf, min_cap, mode.
        ``tokens`` lists the rows of y to compute (all by default); gating,
        slots and the balancing quantities always cover every token, because
        slot positions depend on all earlier tokens.
        """
        x = inp["x"]
        T = x.shape[0]
        E = inp["Wg"].shape[1]
        k = int(inp["k"])
        mode = int(inp["mode"])
        c, s, H, bad_h = self.router(x, inp["Wg"], inp.get("Wn"), inp.get("noise"),
                                     inp.get("bias"))
        idx, gate, hk, hk1 = self.select(H, k, mode)
        C = self.capacity(T, E, k, inp["cf"], inp.get("min_cap", 1))
        pos, keep, count = self.slots(idx, E, C)
        y, bad_y = self.layer_out(x, idx, gate, keep, inp["W1"], inp["W2"], inp.get("b1"),
                                  inp.get("b2"), tokens)
        ax = self.aux(c, s, H, idx, gate, hk, hk1, inp.get("Wn") is not None)
        return dict(c=c, sigma=s, H=H, idx=idx, gate=gate, hk=hk, hk1=hk1, C=C, pos=pos,
                    keep=keep, count=count, y=y, nonfinite=bad_h or bad_y, **ax)

    def loss(self, inp: dict, dy, w_imp: float = 0.0, w_load: float = 0.0,
             w_aux: float = 0.0) -> float:
        """The scalar the backward differentiates: sum <dy, y> + w_imp
        CV(Importance)^2 + w_load CV(Load)^2 + w_aux * (Switch auxiliary loss)."""
        fw = self.forward(inp)
        o3 = fw["out3"]
        return float(np.sum(np.asarray(dy, np.float64) * fw["y"]) + w_imp * o3[0] +
                     w_load * o3[1] + w_aux * o3[2])

    def backward(self, inp: dict, dy, w_imp: float = 0.0, w_load: float = 0.0,
                 w_aux: float = 0.0) -> dict:
        """Gradients of ``loss`` with the forward's discrete choices (top-k,
        capacity, ReLU pattern) held fixed (OLNN section 3.4, "Training the
        gating network"; Switch step 8). Returns fp64 dx, dWg, dWn, dbias, dW1, db1, dW2, db2,
        dgate [T,k] (dL/dgate of each selected gate value), dc and dz [T,E]
        (dL/dc of the clean logits, dL/dz of z = x W_noise);
        dWn and dbias are None without noise weights or router bias, db1 and
        db2 are the gradients at a zero bias when b1 or b2 is None."""
        x = np.ascontiguousarray(inp["x"])
        T, d = x.shape
        Wg = _f32(inp["Wg"])
        E = Wg.shape[1]
        Wn, noise, bias = _f32(inp.get("Wn")), _f32(inp.get("noise")), _f32(inp.get("bias"))
        if (Wn is None) != (noise is None):
            raise ValueError("noise weights and noise come together")
        W1 = np.ascontiguousarray(inp["W1"])
        W2 = np.ascontiguousarray(inp["W2"])
        d_ff = W1.shape[2]
        wcode = _dtype_code(W1)
        b1 = None if inp.get("b1") is None else np.ascontiguousarray(inp["b1"])
        b2 = None if inp.get("b2") is None else np.ascontiguousarray(inp["b2"])
        for a in (W2, b1, b2):
            if a is not None and _dtype_code(a) != wcode:
                raise TypeError("expert weights and biases share one element type")
        k, mode = int(inp["k"]), int(inp["mode"])
        if mode == SWITCH and k != 1:
            raise ValueError("Switch gating is top-1")
        dy = np.ascontiguousarray(dy, dtype=np.float64)
        if dy.shape != (T, d):
            raise ValueError("dy is [T, d]")
        g = dict(dx=np.empty((T, d)), dWg=np.empty((d, E)),
                 dWn=None if Wn is None else np.empty((d, E)),
                 dbias=None if bias is None else np.empty(E),
                 dW1=np.empty((E, d, d_ff)), db1=np.empty((E, d_ff)),
                 dW2=np.empty((E, d_ff, d)), db2=np.empty((E, d)), dgate=np.empty((T, k)),
                 dc=np.empty((T, E)), dz=np.empty((T, E)))
        self.lib.orc_backward(T, d, E, d_ff, k, mode, float(inp["cf"]), int(inp.get("min_cap", 1)),
                              _ptr(x), _dtype_code(x), _ptr(Wg), _ptr(Wn), _ptr(noise),
                              _ptr(bias), _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), wcode,
                              _ptr(dy), float(w_imp), float(w_load), float(w_aux),
                              *[_ptr(g[n]) for n in ("dx", "dWg", "dWn", "dbias", "dW1", "db1",
                                                      "dW2", "db2", "dgate", "dc", "dz")])
        return g

    def backward_entries(self, inp: dict, dy, entries):
        """Chosen expert weight-gradient entries from their definitions, for
        sampling a layer too large for ``backward``. entries: (kind, e, a, b)
        with kind "dW1" (dW1[e][a][b]), "dW2" (dW2[e][a][b]), "db1" (db1[e][a])
        or "db2" (db2[e][a]). Returns (values, sums of |terms|)."""
        kinds = {"dW1": 0, "dW2": 1, "db1": 2, "db2": 3}
        x = np.ascontiguousarray(inp["x"])
        T, d = x.shape
        Wg = _f32(inp["Wg"])
        E = Wg.shape[1]
        Wn, noise, bias = _f32(inp.get("Wn")), _f32(inp.get("noise")), _f32(inp.get("bias"))
        W1 = np.ascontiguousarray(inp["W1"])
        W2 = np.ascontiguousarray(inp["W2"])
        d_ff = W1.shape[2]
        b1 = None if inp.get("b1") is None else np.ascontiguousarray(inp["b1"])
        dy = np.ascontiguousarray(dy, dtype=np.float64)
        n = len(entries)
        kind = np.array([kinds[q[0]] for q in entries], np.int32)
        ex, ea, eb = (np.array([q[i] for q in entries], np.int32) for i in (1, 2, 3))
        out, absum = np.empty(n), np.empty(n)
        self.lib.orc_backward_entries(T, d, E, d_ff, int(inp["k"]), int(inp["mode"]),
                                      float(inp["cf"]), int(inp.get("min_cap", 1)), _ptr(x),
                                      _dtype_code(x), _ptr(Wg), _ptr(Wn), _ptr(noise), _ptr(bias),
                                      _ptr(W1), _ptr(b1), _ptr(W2), _dtype_code(W1), _ptr(dy), n,
                                      _ptr(kind), _ptr(ex), _ptr(ea), _ptr(eb), _ptr(out),
                                      _ptr(absum))
        return out, absum

    # ------------------------------------------------------------ hierarchical
    def hier_select(self, idx_p, g_p, Hs, a: int, b: int, ks: int):
        """Two-level selection (OLNN "Hierarchical Mixture-of-Experts"): for
        each primary pick (group i) the top-ks softmax of the secondary logits
        of group i. Returns flat idx [T, kp*ks] (i*b + j), product gates
        [T, kp*ks], and the in-group thresholds hks, hk1s [T, kp]."""
        idx_p = np.ascontiguousarray(idx_p, dtype=np.int32)
        g_p = np.ascontiguousarray(g_p, dtype=np.float64)
        Hs = np.ascontiguousarray(Hs, dtype=np.float64)
        T, kp = idx_p.shape
        if Hs.shape != (T, a * b):
            raise ValueError("secondary logits are [T, a*b]")
        k = kp * ks
        idx = np.empty((T, k), np.int32)
        gate = np.empty((T, k), np.float64)
        hks = np.empty((T, kp), np.float64)
        hk1s = np.empty((T, kp), np.float64)
        self.lib.orc_hier_select(T, a, b, kp, ks, _ptr(idx_p), _ptr(g_p), _ptr(Hs), _ptr(idx),
                                 _ptr(gate), _ptr(hks), _ptr(hk1s))
        return idx, gate, hks, hk1s

    def hier_aux(self, idx_p, cs, ss, idx, gate, hks, hk1s, load_p, a: int, b: int, ks: int,
                 noisy: bool):
        """Importance_H, |X^(i)|, the in-group secondary loads, Load_H and
        out2 = [CV(Importance_H)^2, CV(Load_H)^2] (OLNN "Hierarchical
        Mixture-of-Experts"; Load_H is 0 for a group no token picked)."""
        idx_p = np.ascontiguousarray(idx_p, dtype=np.int32)
        T, kp = idx_p.shape
        E = a * b
        args = [np.ascontiguousarray(v, dtype=np.float64) for v in (cs, ss)]
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        gate = np.ascontiguousarray(gate, dtype=np.float64)
        hks = np.ascontiguousarray(hks, dtype=np.float64)
        hk1s = np.ascontiguousarray(hk1s, dtype=np.float64)
        load_p = np.ascontiguousarray(load_p, dtype=np.float64)
        imp = np.empty(E, np.float64)
        loadsec = np.empty(E, np.float64)
        count = np.empty(a, np.int32)
        load_H = np.empty(E, np.float64)
        out2 = np.empty(2, np.float64)
        self.lib.orc_hier_aux(T, a, b, kp, ks, _ptr(idx_p), _ptr(args[0]), _ptr(args[1]),
                              _ptr(idx), _ptr(gate), _ptr(hks), _ptr(hk1s), int(bool(noisy)),
                              _ptr(load_p), _ptr(imp), _ptr(loadsec), _ptr(count),
                              _ptr(load_H), _ptr(out2))
        return dict(importance_H=imp, loadsec=loadsec, count=count, load_H=load_H, out2=out2)

    def hier_forward(self, inp: dict, tokens=None) -> dict:
        """The hierarchical layer y_H = x + sum_i sum_j G_p(x)_i G_i(x)_j
        E_ij(x) with the flat path's capacity and slot rules over the a*b
        experts (k = kp*ks choices per token, in primary-then-secondary pick
        order). ``inp``: x, Wp, Wpn, noise_p (primary gate over a groups), Ws,
        Wsn, noise_s (secondary gates, [d, a*b]: group i's columns i*b ..
        i*b+b-1), W1, b1, W2, b2 over the a*b experts, a, b, kp, ks, cf,
        min_cap."""
        x = inp["x"]
        T = x.shape[0]
        a, b, kp, ks = (int(inp[n]) for n in ("a", "b", "kp", "ks"))
        cp, sp, Hp, bad_p = self.router(x, inp["Wp"], inp.get("Wpn"), inp.get("noise_p"))
        idx_p, g_p, hkp, hk1p = self.select(Hp, kp, TOPK_SOFTMAX)
        ax_p = self.aux(cp, sp, Hp, idx_p, g_p, hkp, hk1p, inp.get("Wpn") is not None)
        cs, ss, Hs, bad_s = self.router(x, inp["Ws"], inp.get("Wsn"), inp.get("noise_s"))
        idx, gate, hks, hk1s = self.hier_select(idx_p, g_p, Hs, a, b, ks)
        E, k = a * b, kp * ks
        C = self.capacity(T, E, k, inp["cf"], inp.get("min_cap", 1))
        pos, keep, count = self.slots(idx, E, C)
        y, bad_y = self.layer_out(x, idx, gate, keep, inp["W1"], inp["W2"], inp.get("b1"),
                                  inp.get("b2"), tokens)
        hx = self.hier_aux(idx_p, cs, ss, idx, gate, hks, hk1s, ax_p["load"], a, b, ks,
                           inp.get("Wsn") is not None)
        return dict(cp=cp, sp=sp, Hp=Hp, idx_p=idx_p, g_p=g_p, load_p=ax_p["load"], cs=cs, ss=ss,
                    Hs=Hs, idx=idx, gate=gate, hks=hks, hk1s=hk1s, C=C, pos=pos, keep=keep,
                    expert_count=count, y=y, nonfinite=bad_p or bad_s or bad_y,
                    group_count=hx.pop("count"), **hx)


    def hier_loss(self, inp: dict, dy, w_imp: float = 0.0, w_load: float = 0.0) -> float:
        """sum <dy, y_H> + w_imp CV(Importance_H)^2 + w_load CV(Load_H)^2."""
        fw = self.hier_forward(inp)
        return float(np.sum(np.asarray(dy, np.float64) * fw["y"]) + w_imp * fw["out2"][0] +
                     w_load * fw["out2"][1])

    def hier_backward(self, inp: dict, dy, w_imp: float = 0.0, w_load: float = 0.0) -> dict:
        """Gradients of ``hier_loss`` with the forward's choices fixed (OLNN
        "Hierarchical Mixture-of-Experts"; section 3.4). Returns fp64 dx, dWp,
        dWpn, dWs, dWsn (None without noise weights), dW1, db1, dW2, db2."""
        x = np.ascontiguousarray(inp["x"])
        T, d = x.shape
        a, b, kp, ks = (int(inp[n]) for n in ("a", "b", "kp", "ks"))
        E = a * b
        Wp, Wpn, npn = _f32(inp["Wp"]), _f32(inp.get("Wpn")), _f32(inp.get("noise_p"))
        Ws, Wsn, nsn = _f32(inp["Ws"]), _f32(inp.get("Wsn")), _f32(inp.get("noise_s"))
        W1 = np.ascontiguousarray(inp["W1"])
        W2 = np.ascontiguousarray(inp["W2"])
        d_ff = W1.shape[2]
        b1 = None if inp.get("b1") is None else np.ascontiguousarray(inp["b1"])
        b2 = None if inp.get("b2") is None else np.ascontiguousarray(inp["b2"])
        dy = np.ascontiguousarray(dy, dtype=np.float64)
        g = dict(dx=np.empty((T, d)), dWp=np.empty((d, a)),
                 dWpn=None if Wpn is None else np.empty((d, a)), dWs=np.empty((d, E)),
                 dWsn=None if Wsn is None else np.empty((d, E)), dW1=np.empty((E, d, d_ff)),
                 db1=np.empty((E, d_ff)), dW2=np.empty((E, d_ff, d)), db2=np.empty((E, d)))
        self.lib.orc_hier_backward(T, d, a, b, kp, ks, d_ff, float(inp["cf"]),
                                   int(inp.get("min_cap", 1)), _ptr(x), _dtype_code(x), _ptr(Wp),
                                   _ptr(Wpn), _ptr(npn), _ptr(Ws), _ptr(Wsn), _ptr(nsn), _ptr(W1),
                                   _ptr(b1), _ptr(W2), _ptr(b2), _dtype_code(W1), _ptr(dy),
                                   float(w_imp), float(w_load),
                                   *[_ptr(g[n]) for n in ("dx", "dWp", "dWpn", "dWs", "dWsn", "dW1",
                                                           "db1", "dW2", "db2")])
        return g

    def bal_loss_total(self, inp: dict, dy, w_bal: float = 0.0) -> float:
        """sum <dy, y> + w_bal L_batchwise (the loss term only with thresholds)."""
        return _bal_total(self, inp, dy, w_bal)

    def bal_backward(self, inp: dict, dy, w_bal: float = 0.0) -> dict:
        """Gradients of ``bal_loss_total`` with the masks fixed (OLNN, Strictly
        Balanced Gating; section 3.4). Returns fp64 dx, dWg, dbias (None
        without a router bias), dW1, db1, dW2, db2."""
        x = np.ascontiguousarray(inp["x"])
        T, d = x.shape
        Wg = _f32(inp["Wg"])
        E = Wg.shape[1]
        bias, thr = _f32(inp.get("bias")), _f32(inp.get("thr"))
        W1 = np.ascontiguousarray(inp["W1"])
        W2 = np.ascontiguousarray(inp["W2"])
        d_ff = W1.shape[2]
        b1 = None if inp.get("b1") is None else np.ascontiguousarray(inp["b1"])
        b2 = None if inp.get("b2") is None else np.ascontiguousarray(inp["b2"])
        dy = np.ascontiguousarray(dy, dtype=np.float64)
        g = dict(dx=np.empty((T, d)), dWg=np.empty((d, E)),
                 dbias=None if bias is None else np.empty(E), dW1=np.empty((E, d, d_ff)),
                 db1=np.empty((E, d_ff)), dW2=np.empty((E, d_ff, d)), db2=np.empty((E, d)))
        self.lib.orc_bal_backward(T, d, E, d_ff, int(inp["k"]), int(inp.get("mode_bal", 0)),
                                  _ptr(x), _dtype_code(x), _ptr(Wg), _ptr(bias), _ptr(thr),
                                  _ptr(W1), _ptr(b1), _ptr(W2), _ptr(b2), _dtype_code(W1),
                                  _ptr(dy), float(w_bal),
                                  *[_ptr(g[n]) for n in ("dx", "dWg", "dbias", "dW1", "db1", "dW2",
                                                          "db2")])
        return g

    # ------------------------------------------------------------ strictly balanced
    def softmax_dense(self, H):
        """G_sigma = Softmax(H) over all experts, row by row (OLNN's plain
        softmax gate)."""
        H = np.ascontiguousarray(H, dtype=np.float64)
        T, E = H.shape
        P = np.empty((T, E), np.float64)
        self.lib.orc_softmax_rows(T, E, _ptr(H), _ptr(P))
        return P

    def bal_rows(self, T: int, k: int, E: int) -> int:
        """m = max(1, min(T, floor(k T / E))), the batchwise mask's rows per
        expert (OLNN, Strictly Balanced Gating: m = k|X|/n)."""
        return int(self.lib.orc_bal_rows(int(T), int(k), int(E)))

    def bal_gate(self, P, m: int, thr=None, mode: int = 0):
        """Batchwise (mode 0: top m tokens per expert) or threshold (mode 1:
        P > thr) mask and the renormalised gate (OLNN, Strictly Balanced
        Gating). Returns mask [T,E] uint8, gate [T,E]."""
        P = np.ascontiguousarray(P, dtype=np.float64)
        T, E = P.shape
        thr = None if thr is None else np.ascontiguousarray(thr, dtype=np.float32)
        if mode == 1 and thr is None:
            raise ValueError("the threshold mask needs thresholds")
        mask = np.empty((T, E), np.uint8)
        gate = np.empty((T, E), np.float64)
        self.lib.orc_bal_gate(T, E, int(m), int(mode), _ptr(P), _ptr(thr), _ptr(mask),
                              _ptr(gate))
        return mask, gate

    def bal_loss(self, P, mask_batch, thr) -> float:
        """L_batchwise (OLNN, Strictly Balanced Gating)."""
        P = np.ascontiguousarray(P, dtype=np.float64)
        T, E = P.shape
        mask_batch = np.ascontiguousarray(mask_batch, dtype=np.uint8)
        thr = np.ascontiguousarray(thr, dtype=np.float32)
        return float(self.lib.orc_bal_loss(T, E, _ptr(P), _ptr(mask_batch), _ptr(thr)))

    def bal_forward(self, inp: dict, tokens=None) -> dict:
        """The strictly balanced layer: clean router logits H = x W_g (+ b),
        P = Softmax(H), the batchwise mask with m = max(1, min(T, floor(k*T/E)))
        (or the threshold mask when ``inp['mode_bal'] == 1``), the renormalised
        gates, y = x + sum over picked experts of gate * E_i(x) (no capacity:
        the mask fixes every expert's rows), and L_batchwise when thresholds
        are given (unless ``inp['with_loss']`` is false: the inference-time
        threshold layer has no loss)."""
        x = inp["x"]
        T = x.shape[0]
        E = inp["Wg"].shape[1]
        k = int(inp["k"])
        mode = int(inp.get("mode_bal", 0))
        m = self.bal_rows(T, k, E)
        c, s, H, bad_h = self.router(x, inp["Wg"], None, None, inp.get("bias"))
        P = self.softmax_dense(H)
        thr = inp.get("thr")
        mask, gate = self.bal_gate(P, m, thr, mode)
        idx = np.tile(np.arange(E, dtype=np.int32), (T, 1))
        y, bad_y = self.layer_out(x, idx, gate, mask, inp["W1"], inp["W2"], inp.get("b1"),
                                  inp.get("b2"), tokens)
        out = dict(H=H, P=P, m=m, mask=mask, gate=gate, y=y, nonfinite=bad_h or bad_y)
        if thr is not None and inp.get("with_loss", True):
            mb = mask if mode == 0 else self.bal_gate(P, m, None, 0)[0]
            out["loss"] = self.bal_loss(P, mb, thr)
        return out


def _bal_total(orc, inp, dy, w_bal):
    fw = orc.bal_forward(inp)
    return float(np.sum(np.asarray(dy, np.float64) * fw["y"]) + w_bal * fw.get("loss", 0.0))


def default() -> Oracle:
    """The oracle compiled from moe_oracle.c (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def variant(src_path: str, out_dir: str) -> Oracle:
    """Compile another copy of the oracle source (e.g. one with a planted
    mistake, for the tests that check the pins catch it) and load it."""
    out = os.path.join(out_dir, "liboracle_variant_%d.so" % (abs(hash(src_path)) % 10**8))
    _compile(src_path, out)
    return Oracle(out)


def set_threads(n: int) -> int:
    """Set the number of OpenMP threads the oracle's parallel loops use (its
    arithmetic and results do not depend on it); returns the previous count.
    Used to time the oracle on one host core beside all of them."""
    lib = default().lib
    prev = int(lib.omp_get_max_threads())
    lib.omp_set_num_threads(ctypes.c_int(int(n)))
    return prev


def capacity(*a, **k):
    return default().capacity(*a, **k)


def softplus(z):
    return default().softplus(z)


def phi(u):
    return default().phi(u)


def cv2(v):
    return default().cv2(v)


def router(*a, **k):
    return default().router(*a, **k)


def select(*a, **k):
    return default().select(*a, **k)


def gates_given(*a, **k):
    return default().gates_given(*a, **k)


def slots(*a, **k):
    return default().slots(*a, **k)


def layer_out(*a, **k):
    return default().layer_out(*a, **k)


def aux(*a, **k):
    return default().aux(*a, **k)


def forward(*a, **k):
    return default().forward(*a, **k)


def loss(*a, **k):
    return default().loss(*a, **k)


def backward(*a, **k):
    return default().backward(*a, **k)


def backward_entries(*a, **k):
    return default().backward_entries(*a, **k)


def hier_select(*a, **k):
    return default().hier_select(*a, **k)


def hier_aux(*a, **k):
    return default().hier_aux(*a, **k)


def hier_forward(*a, **k):
    return default().hier_forward(*a, **k)


def hier_loss(*a, **k):
    return default().hier_loss(*a, **k)


def hier_backward(*a, **k):
    return default().hier_backward(*a, **k)


def softmax_dense(*a, **k):
    return default().softmax_dense(*a, **k)


def bal_gate(*a, **k):
    return default().bal_gate(*a, **k)


def bal_loss(*a, **k):
    return default().bal_loss(*a, **k)


def bal_forward(*a, **k):
    return default().bal_forward(*a, **k)


def bal_backward(*a, **k):
    return default().bal_backward(*a, **k)


def bal_loss_total(*a, **k):
    return default().bal_loss_total(*a, **k)


def bal_rows(*a, **k):
    return default().bal_rows(*a, **k)
