"""Expert parallelism: the experts spread over the ranks of a process group,
each rank gating its own share of the batch ("Outrageously Large Neural
Networks", Distributed Training: Solving the Shrinking Batch Problem: every
token goes to the device holding its expert and its output comes back, so
each expert processes the tokens of all devices together).

The layer's batch is the concatenation, in rank order, of the ranks' batches,
and the layer computes what ``moe_forward`` computes over that whole batch:
the same choices, the same capacity C of the whole batch, the same
token-order slots (rank r's assignments to expert e follow those of ranks
0 .. r-1), the same outputs and balancing losses. Rank q holds experts
q*E/W .. (q+1)*E/W - 1 (E divisible by the world size W).

This module only moves data between ranks and keeps the row bookkeeping
(torch.distributed collectives: NCCL on GPUs, gloo on CPUs). Every step of
the layer's arithmetic is a call on ``ops``; ``LibraryOps`` makes those calls
through the library's C ABI on this rank's GPU (moe_gate, moe_expert_counts,
moe_dispatch_ranked, moe_expert_ffn, moe_combine, moe_aux_totals,
moe_aux_from_totals). The exchange per layer:

1. all_gather of the per-expert choice counts [E] (int32);
2. all_to_all of the kept rows' counts per expert, then of the rows (x) and
   their gates: the kept rows of the experts rank q holds are one contiguous
   range of the sender's packed buffer, so the sends need no reordering;
3. all_to_all of the expert outputs back, into the sender's packed layout;
4. all_reduce of the balancing sums [4, E].
"""
from __future__ import annotations

import dataclasses

import torch
import torch.distributed as dist

from . import binding as B


@dataclasses.dataclass
class Dispatch:
    pos: torch.Tensor       # [T, k] int32, this rank's position per expert
    keep: torch.Tensor      # [T, k] uint8, kept under the whole batch's capacity
    offset: torch.Tensor    # [E+1] int32, packed rows per expert (kept only)
    xbuf: torch.Tensor      # [T*k, d] packed rows
    row_gate: torch.Tensor  # [T*k] fp32, each row's gate


class LibraryOps:
    """The layer's steps on this rank's GPU, through the C ABI. ``cfg`` is
    this rank's moe_config (its T; E = all experts); ``ws`` its workspace
    (moe_workspace_size of cfg, zero-filled once)."""

    z_dtype = torch.float32  # expert outputs and gates travel in fp32

    def __init__(self, cfg, ws: torch.Tensor, stream=None):
        self.cfg, self.ws, self.stream = cfg, ws, stream

    def gate(self, x, Wg, Wn, noise, bias):
        c = self.cfg
        idx = torch.empty((c.T, c.k), dtype=torch.int32, device=x.device)
        gate = torch.empty((c.T, c.k), dtype=torch.float32, device=x.device)
        thr = torch.empty((c.T, 2), dtype=torch.float32, device=x.device)
        B.moe_gate(c, x, Wg, Wn, noise, bias, idx, gate, thr, self.ws, self.stream)
        return idx, gate

    def counts(self, idx):
        out = torch.empty(self.cfg.E, dtype=torch.int32, device=idx.device)
        B.moe_expert_counts(self.cfg, idx, out, self.ws, self.stream)
        return out

    def dispatch(self, capacity, counts_all, n_ranks, rank, idx, gate, x) -> Dispatch:
        c = self.cfg
        dev = x.device
        A = c.T * c.k
        pos = torch.empty((c.T, c.k), dtype=torch.int32, device=dev)
        keep = torch.empty((c.T, c.k), dtype=torch.uint8, device=dev)
        count = torch.empty(c.E, dtype=torch.int32, device=dev)
        offset = torch.empty(c.E + 1, dtype=torch.int32, device=dev)
        xbuf = torch.empty((A, c.d), dtype=x.dtype, device=dev)
        row_token = torch.empty(A, dtype=torch.int32, device=dev)
        row_gate = torch.empty(A, dtype=torch.float32, device=dev)
        B.moe_dispatch_ranked(c, capacity, counts_all, n_ranks, rank, idx, gate, x, pos, keep,
                              count, offset, xbuf, row_token, row_gate, self.ws, self.stream)
        return Dispatch(pos, keep, offset, xbuf, row_gate)

    def ffn(self, rows, offsets, row_gate, W1, b1, W2, b2, zout):
        """Expert outputs for ``rows`` [n, d] of the local experts (offsets
        [E_local+1] int32, host list) into zout [n, d] fp32."""
        n = rows.shape[0]
        if n == 0:
            return
        E_loc = len(offsets) - 1
        c = self.cfg
        lc = B.config(n, c.d, E_loc, c.d_ff, 1, float(E_loc), act_dtype=c.act_dtype)
        dev = rows.device
        off = torch.tensor(offsets, dtype=torch.int32, device=dev)
        hbuf = torch.empty((n, c.d_ff), dtype=rows.dtype, device=dev)
        ws = torch.zeros(B.moe_workspace_size(lc), dtype=torch.uint8, device=dev)
        B.moe_expert_ffn(lc, rows, off, row_gate, W1, b1, W2, b2, hbuf, zout, ws, self.stream)

    def combine(self, x, zbuf, d: Dispatch, idx):
        y = torch.empty_like(x)
        B.moe_combine(self.cfg, x, zbuf, d.pos, d.keep, idx, d.offset, y, self.ws, self.stream)
        return y

    def aux_totals(self):
        out = torch.empty((4, self.cfg.E), dtype=torch.float32, device=self.ws.device)
        B.moe_aux_totals(self.cfg, self.ws, out, self.stream)
        return out

    def aux_from_totals(self, T_total, totals):
        out3 = torch.empty(3, dtype=torch.float32, device=totals.device)
        B.moe_aux_from_totals(self.cfg, T_total, totals, out3, self.ws, self.stream)
        return out3


def owned_experts(E: int, world: int, rank: int) -> range:
    """The experts rank ``rank`` holds: a contiguous block of E / world."""
    if E % world:
        raise ValueError(f"{E} experts do not divide over {world} ranks")
    n = E // world
    return range(rank * n, (rank + 1) * n)


def send_counts(offset: list[int], E: int, world: int) -> tuple[list[int], list[list[int]]]:
    """From this rank's packed offsets [E+1]: the rows it sends to each rank
    (one contiguous range per destination) and the kept rows per expert of
    each destination's experts."""
    n = E // world
    per_dest, per_expert = [], []
    for q in range(world):
        lo, hi = q * n, (q + 1) * n
        per_dest.append(offset[hi] - offset[lo])
        per_expert.append([offset[e + 1] - offset[e] for e in range(lo, hi)])
    return per_dest, per_expert


def layer_capacity(T_total: int, E: int, k: int, cf: float, min_cap: int, act_dtype: int) -> int:
    """The whole batch's capacity, by the library's rule (moe_capacity)."""
    return B.moe_capacity(B.config(T_total, 8, E, 8, k, cf, act_dtype=act_dtype,
                                   min_capacity=min_cap))


def ep_forward(ops, x, Wg, Wn, noise, bias, W1_local, b1_local, W2_local, b2_local, *, E: int,
               k: int, cf: float, min_cap: int = 1, act_dtype: int = B.MOE_BF16, group=None):
    """One forward of the expert-parallel layer on this rank: x [T, d] this
    rank's tokens (their gate inputs Wg, Wn, noise [T, E], bias as for
    moe_gate); W1_local, b1_local, W2_local, b2_local the weights of the
    experts this rank holds (owned_experts). Returns (y [T, d], out3 [3]: the
    whole batch's CV^2 of importance and load and its Switch loss, and a dict
    of the bookkeeping, for inspection)."""
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    T = x.shape[0]
    dev = x.device
    # The whole batch's size, hence its capacity.
    tt = torch.tensor([T], dtype=torch.int64, device=dev)
    dist.all_reduce(tt, group=group)
    T_total = int(tt.item())
    C = layer_capacity(T_total, E, k, cf, min_cap, act_dtype)
    # 1. Gate this rank's tokens; gather every rank's counts per expert.
    idx, gate = ops.gate(x, Wg, Wn, noise, bias)
    counts = ops.counts(idx)
    gathered = [torch.empty_like(counts) for _ in range(world)]
    dist.all_gather(gathered, counts, group=group)
    counts_all = torch.stack(gathered).contiguous()
    # 2. Slots after the earlier ranks' and the packed kept rows.
    dsp = ops.dispatch(C, counts_all, world, rank, idx, gate, x)
    offset = dsp.offset.tolist()
    send_rows, send_per_expert = send_counts(offset, E, world)
    # 3. Each destination's rows per expert, then the rows and their gates.
    n_loc = E // world
    sc = torch.tensor(send_per_expert, dtype=torch.int32, device=dev).reshape(-1)
    rc = torch.empty_like(sc)
    dist.all_to_all_single(rc, sc, group=group)
    recv_per_expert = rc.reshape(world, n_loc).tolist()
    recv_rows = [sum(r) for r in recv_per_expert]
    n_send, n_recv = sum(send_rows), sum(recv_rows)
    zt = getattr(ops, "z_dtype", torch.float32)
    xrecv = torch.empty((n_recv, x.shape[1]), dtype=x.dtype, device=dev)
    grecv = torch.empty(n_recv, dtype=dsp.row_gate.dtype, device=dev)
    dist.all_to_all_single(xrecv, dsp.xbuf[:n_send], output_split_sizes=recv_rows,
                           input_split_sizes=send_rows, group=group)
    dist.all_to_all_single(grecv, dsp.row_gate[:n_send], output_split_sizes=recv_rows,
                           input_split_sizes=send_rows, group=group)
    # 4. The local experts on each source rank's block (rows per expert in
    #    that rank's token order; the blocks in rank order).
    zrecv = torch.empty((n_recv, x.shape[1]), dtype=zt, device=dev)
    r0 = 0
    for q in range(world):
        n = recv_rows[q]
        offs = [0]
        for v in recv_per_expert[q]:
            offs.append(offs[-1] + v)
        # A block's rows start on a 16-byte boundary when d*2 is a multiple
        # of 16; its gates (4 bytes each) get a buffer of their own.
        ops.ffn(xrecv[r0:r0 + n], offs, grecv[r0:r0 + n].clone(), W1_local, b1_local, W2_local,
                b2_local, zrecv[r0:r0 + n])
        r0 += n
    # 5. The outputs back into this rank's packed layout, then the combine.
    zbuf = torch.zeros((T * k, x.shape[1]), dtype=zt, device=dev)
    dist.all_to_all_single(zbuf[:n_send], zrecv, output_split_sizes=send_rows,
                           input_split_sizes=recv_rows, group=group)
    y = ops.combine(x, zbuf, dsp, idx)
    # 6. The balancing losses of the whole batch.
    totals = ops.aux_totals()
    dist.all_reduce(totals, group=group)
    out3 = ops.aux_from_totals(T_total, totals)
    info = dict(idx=idx, gate=gate, pos=dsp.pos, keep=dsp.keep, counts_all=counts_all,
                capacity=C, send_rows=send_rows, recv_rows=recv_rows, T_total=T_total)
    return y, out3, info
