"""The expert-parallel layer's bookkeeping (sparsely_gated_mixture_gb300.
expert_parallel.ep_forward) on two gloo ranks on the CPU, against the fp64
oracle's single-process forward over the whole batch ("Outrageously Large
Neural Networks", Distributed Training: Solving the Shrinking Batch Problem:
each expert's batch is every device's tokens for it).

Each rank runs ep_forward on its share of the batch with ``OracleOps``: the
library's steps (gate, counts, ranked dispatch, expert FFN, combine, balancing
totals) restated on the CPU in fp64 from the oracle's functions and the
contracts in include/moe.h. The exchange, the slot offsets across ranks, the
routing of rows to the ranks holding their experts and back, and the
all-reduce of the balancing sums are ep_forward's own. The GPU side of the
same calls is tested on one GPU, ranks emulated in turn, in
test_gpu_expert_parallel.py.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from sparsely_gated_mixture_gb300 import binding as B
from sparsely_gated_mixture_gb300 import expert_parallel as EP
from sparsely_gated_mixture_gb300 import workloads as wl


class OracleOps:
    """ep_forward's steps on the CPU in fp64 (test infrastructure)."""

    z_dtype = torch.float64

    def __init__(self, w, inp_local):
        self.w, self.inp = w, inp_local

    def gate(self, x, Wg, Wn, noise, bias):
        w, inp = self.w, self.inp
        c, s, H, bad = oracle.router(inp["x"], inp["Wg"], inp["Wn"], inp["noise"], inp["bias"])
        assert not bad
        idx, gate, hk, hk1 = oracle.select(H, w.k, inp["mode"])
        ax = oracle.aux(c, s, H, idx, gate, hk, hk1, w.noisy)
        p = np.exp(H - H.max(axis=1, keepdims=True))
        p /= p.sum(axis=1, keepdims=True)
        first = np.bincount(idx[:, 0], minlength=w.E).astype(np.float64)
        self.totals = np.stack([ax["importance"], ax["load"], first, p.sum(axis=0)])
        return torch.from_numpy(idx.astype(np.int32)), torch.from_numpy(gate)

    def counts(self, idx):
        return torch.from_numpy(np.bincount(idx.numpy().ravel(), minlength=self.w.E)
                                .astype(np.int32))

    def dispatch(self, capacity, counts_all, n_ranks, rank, idx, gate, x):
        E, k = self.w.E, self.w.k
        T = idx.shape[0]
        base = counts_all.numpy()[:rank].sum(axis=0)
        iv = idx.numpy()
        pos = np.zeros((T, k), np.int32)
        keep = np.zeros((T, k), np.uint8)
        seen = np.zeros(E, np.int64)
        for t in range(T):  # token order, then choice order
            for j in range(k):
                e = iv[t, j]
                pos[t, j] = seen[e]
                seen[e] += 1
                keep[t, j] = base[e] + pos[t, j] < capacity
        kept = np.zeros(E, np.int64)
        for e in range(E):
            kept[e] = int((keep.ravel() * (iv.ravel() == e)).sum())
        offset = np.concatenate([[0], np.cumsum(kept)]).astype(np.int32)
        xbuf = torch.zeros((T * k, x.shape[1]), dtype=x.dtype)
        row_gate = torch.zeros(T * k, dtype=gate.dtype)
        for t in range(T):
            for j in range(k):
                if keep[t, j]:
                    r = offset[iv[t, j]] + pos[t, j]
                    xbuf[r] = x[t]
                    row_gate[r] = gate[t, j]
        return EP.Dispatch(torch.from_numpy(pos), torch.from_numpy(keep),
                           torch.from_numpy(offset), xbuf, row_gate)

    def ffn(self, rows, offsets, row_gate, W1, b1, W2, b2, zout):
        X = rows.numpy().astype(np.float64)
        for e in range(len(offsets) - 1):
            a, b = offsets[e], offsets[e + 1]
            if a == b:
                continue
            h = np.maximum(X[a:b] @ W1[e] + (0.0 if b1 is None else b1[e]), 0.0)
            o = h @ W2[e] + (0.0 if b2 is None else b2[e])
            zout[a:b] = torch.from_numpy(row_gate.numpy()[a:b, None] * o)

    def combine(self, x, zbuf, d, idx):
        y = x.numpy().astype(np.float64).copy()
        iv, pos, keep, off = idx.numpy(), d.pos.numpy(), d.keep.numpy(), d.offset.numpy()
        Z = zbuf.numpy()
        for t in range(y.shape[0]):
            for j in range(iv.shape[1]):
                if keep[t, j]:
                    y[t] += Z[off[iv[t, j]] + pos[t, j]]
        return torch.from_numpy(y)

    def aux_totals(self):
        return torch.from_numpy(self.totals.copy())

    def aux_from_totals(self, T_total, totals):
        t = totals.numpy()
        E = t.shape[1]
        sw = 0.01 * E * float(np.sum((t[2] / T_total) * (t[3] / T_total)))
        return torch.tensor([oracle.cv2(t[0]), oracle.cv2(t[1]), sw], dtype=torch.float64)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, w, splits, out_dir):
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = wl.generate(w, seed=5, biases=True)
        lo, hi = splits[rank], splits[rank + 1]
        loc = dict(inp)
        loc["x"] = np.ascontiguousarray(inp["x"][lo:hi])
        loc["noise"] = None if inp["noise"] is None else np.ascontiguousarray(inp["noise"][lo:hi])
        mine = EP.owned_experts(w.E, world, rank)
        sl = slice(mine.start, mine.stop)
        f64 = lambda a: None if a is None else np.asarray(a, np.float64)[sl]
        ops = OracleOps(w, loc)
        y, out3, info = EP.ep_forward(
            ops, torch.from_numpy(loc["x"]), None, None, None, None, f64(inp["W1"]),
            f64(inp["b1"]), f64(inp["W2"]), f64(inp["b2"]), E=w.E, k=w.k, cf=w.cf,
            min_cap=w.min_cap, act_dtype=B.MOE_F32)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), y=y.numpy(), out3=out3.numpy(),
                 pos=info["pos"].numpy(), keep=info["keep"].numpy(),
                 counts_all=info["counts_all"].numpy(), capacity=info["capacity"])
    finally:
        dist.destroy_process_group()


CASES = {
    # capacity factor below 1: the whole batch's capacity drops tokens, so a
    # rank's keep depends on the earlier rank's counts
    "drops_even": (wl.Workload("ep_drops", T=96, d=12, E=4, d_ff=16, k=2, cf=0.6,
                               mode=wl.TOPK, dtype="f32", noisy=True), [0, 48, 96]),
    "uneven_split": (wl.Workload("ep_uneven", T=70, d=8, E=6, d_ff=10, k=2, cf=1.0,
                                 mode=wl.TOPK, dtype="f32", noisy=True), [0, 23, 70]),
    "switch": (wl.Workload("ep_switch", T=64, d=8, E=4, d_ff=8, k=1, cf=0.8, mode=wl.SWITCH,
                           dtype="f32", noisy=False), [0, 40, 64]),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_expert_parallel_two_ranks_match_one_process(name, tmp_path):
    w, splits = CASES[name]
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), w, splits, str(tmp_path)),
                       nprocs=world, start_method="spawn")
    got = [np.load(tmp_path / f"rank{r}.npz") for r in range(world)]
    ref = oracle.forward(wl.generate(w, seed=5, biases=True))
    C = oracle.capacity(w.T, w.E, w.k, w.cf, w.min_cap)
    assert int(got[0]["capacity"]) == C
    y = np.concatenate([g["y"] for g in got])
    keep = np.concatenate([g["keep"] for g in got])
    assert np.array_equal(keep, ref["keep"]), "drop masks differ from the whole batch's"
    # positions in the whole batch: this rank's plus the earlier ranks' counts
    counts = got[0]["counts_all"]
    idx = ref["idx"]
    for r in range(world):
        lo, hi = splits[r], splits[r + 1]
        base = counts[:r].sum(axis=0)
        assert np.array_equal(got[r]["pos"] + base[idx[lo:hi]], ref["pos"][lo:hi])
    np.testing.assert_allclose(y, ref["y"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got[0]["out3"], ref["out3"], rtol=1e-10, atol=1e-15)
    np.testing.assert_allclose(got[1]["out3"], ref["out3"], rtol=1e-10, atol=1e-15)


def test_send_counts_and_owned_experts():
    offset = [0, 3, 3, 7, 8, 12, 15]  # six experts' kept rows: 3, 0, 4, 1, 4, 3
    per_dest, per_expert = EP.send_counts(offset, 6, 3)
    assert per_dest == [3, 5, 7]
    assert per_expert == [[3, 0], [4, 1], [4, 3]]
    assert list(EP.owned_experts(6, 3, 1)) == [2, 3]
    with pytest.raises(ValueError):
        EP.owned_experts(7, 2, 0)
