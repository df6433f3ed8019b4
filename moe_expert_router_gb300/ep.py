"""Expert parallelism across devices (EP > 1), with the exchange staged locally.

The MegaMoE guide (opening section) fuses the expert-parallel all-to-all into
its two grouped GEMMs: dispatch_grouped_gemm sends each routed token row to the
rank that owns its expert, grouped_gemm_combine sends the expert outputs back
and forms the weighted sum. Here the exchange is a plain collective into local
receive buffers, between device steps of this library:

    rank p, experts [p E/P, (p+1) E/P) of E; its own T tokens and their routing
    1. routing metadata of its T*k slots (moe_routing_metadata). Routed rows are
       expert-major, so the rows bound for rank q are one contiguous range.
    2. send buffer: x rows in routed order and each row's routing weight
       (moe_dispatch_rows).
    3. all-to-all of the per-(rank, local expert) row counts, then of the rows
       and the weights (variable splits).
    4. the received rows are tokens with k = 1 for the local experts (their
       expert index follows from the counts): the single-device expert path
       (moe_forward) gives each received row's weighted output.
    5. all-to-all back (the reverse splits): every row returns to its source
       rank in that rank's routed order.
    6. combine: y[t] = sum of the token's returned rows (moe_combine_rows).

The split sizes are needed on the host by the collective, so step 3 reads the
counts back once per step (the guide's fused kernels avoid that with a symmetric
buffer and a cross-rank handshake).

``ExpertParallel`` holds only this bookkeeping and calls the device work through
an ``ops`` object: ``LibmoeOps`` (the CUDA kernels of libmoe) by default. There is
no CPU fallback; tests of the exchange logic on CPU ranks pass their own ops.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist

from . import binding as B


class LibmoeOps:
    """The device steps of one rank, through libmoe (CUDA tensors only)."""

    def __init__(self, device):
        B.load()
        self.device = torch.device(device)

    def route(self, x, topk_idx, topk_w, E):
        """Metadata, send rows and row weights of this rank's slots; returns
        (per-expert counts as a host array, rows, row weights, state)."""
        T, H = x.shape
        k = topk_idx.shape[1]
        shp = B.shape(T, H, 8, E, k)
        ws = B.new_workspace(shp, self.device)
        B.moe_routing_metadata(topk_idx, shp, ws)
        rows = torch.empty((T * k, H), dtype=torch.bfloat16, device=self.device)
        row_w = torch.empty((T * k,), dtype=torch.float32, device=self.device)
        B.moe_dispatch_rows(x, shp, rows, ws, topk_w=topk_w, row_weight=row_w)
        L = B.moe_workspace_layout(shp)
        counts = ws[L.counts:L.counts + 4 * E].view(torch.int32).cpu().numpy()
        return counts, rows, row_w, (shp, ws)

    def expert_forward(self, rows, expert, weight, w1, w2):
        """Weighted outputs of received rows (k = 1) on the local experts."""
        R, H = rows.shape
        E_loc, twoI, _ = w1.shape
        out = torch.empty((R, H), dtype=torch.bfloat16, device=self.device)
        if R == 0:
            return out
        shp = B.shape(R, H, twoI // 2, E_loc, 1)
        ws = B.new_workspace(shp, self.device)
        B.moe_forward(rows, expert.view(R, 1), weight.view(R, 1), w1, w2, shp, out, ws)
        return out

    def combine(self, rows_back, state, T, H):
        shp, ws = state
        y = torch.empty((T, H), dtype=torch.bfloat16, device=self.device)
        B.moe_combine_rows(rows_back, shp, y, ws)
        return y

    def to_device(self, array, dtype):
        return torch.as_tensor(array, dtype=dtype).to(self.device)


def plan_splits(counts_all: np.ndarray, P: int) -> tuple[np.ndarray, np.ndarray]:
    """Rows this rank sends to each rank, from its per-expert counts [E] (experts of
    rank q are [q E/P, (q+1) E/P)): (send counts [P], per-(rank, local expert) counts [P, E/P])."""
    E = counts_all.shape[0]
    per = counts_all.reshape(P, E // P)
    return per.sum(axis=1), per


def local_expert_index(recv_per: np.ndarray) -> np.ndarray:
    """Local expert of every received row: source segments in rank order, each
    grouped by local expert (the sender's routed order). recv_per [P, E/P]."""
    P, E_loc = recv_per.shape
    return np.concatenate([np.repeat(np.arange(E_loc, dtype=np.int32), recv_per[p]) for p in range(P)]
                          ) if recv_per.sum() else np.zeros((0,), np.int32)


class ExpertParallel:
    """The expert path with experts sharded over the ranks of ``group``."""

    def __init__(self, E: int, group=None, ops=None, device=None):
        self.group = group
        self.P = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if E % self.P:
            raise ValueError("E must be a multiple of the number of ranks")
        self.E = E
        self.E_loc = E // self.P
        self.ops = ops if ops is not None else LibmoeOps(device)

    def _all_to_all(self, send, send_counts, recv_counts, row_shape, dtype, device):
        recv = torch.empty((int(recv_counts.sum()),) + row_shape, dtype=dtype, device=device)
        dist.all_to_all_single(recv, send[: int(send_counts.sum())].contiguous(),
                               output_split_sizes=[int(c) for c in recv_counts],
                               input_split_sizes=[int(c) for c in send_counts], group=self.group)
        return recv

    def forward(self, x, topk_idx, topk_w, w1_local, w2_local):
        """y [T, H] for this rank's tokens; w1_local / w2_local hold this rank's experts."""
        T, H = x.shape
        counts, rows, row_w, state = self.ops.route(x, topk_idx, topk_w, self.E)
        send_counts, send_per = plan_splits(counts, self.P)
        # exchange the per-(rank, local expert) counts: row q of send_per goes to rank q
        per_t = torch.as_tensor(send_per.astype(np.int64))
        recv_per_t = torch.empty_like(per_t)
        if x.is_cuda:
            per_t, recv_per_t = per_t.to(x.device), recv_per_t.to(x.device)
        dist.all_to_all_single(recv_per_t, per_t, group=self.group)
        recv_per = recv_per_t.cpu().numpy()
        recv_counts = recv_per.sum(axis=1)
        # the rows and their weights
        rows_recv = self._all_to_all(rows, send_counts, recv_counts, (H,), rows.dtype, rows.device)
        w_recv = self._all_to_all(row_w, send_counts, recv_counts, (), row_w.dtype, row_w.device)
        expert = self.ops.to_device(local_expert_index(recv_per), torch.int32)
        out = self.ops.expert_forward(rows_recv, expert, w_recv, w1_local, w2_local)
        # back to the sources, in their routed order
        rows_back = self._all_to_all(out, recv_counts, send_counts, (H,), out.dtype, out.device)
        return self.ops.combine(rows_back, state, T, H)
