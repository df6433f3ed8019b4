"""Expert parallelism across devices (EP > 1) without host synchronisation.

The MegaMoE guide (opening section) fuses the expert-parallel all-to-all into
its two grouped GEMMs: dispatch_grouped_gemm sends each routed token row to the
rank that owns its expert, grouped_gemm_combine sends the expert outputs back
and forms the weighted sum; its "Example 2" runs the whole layer under one CUDA
graph, so no step may wait for the host. Here the exchange is a plain
collective into local receive buffers, between device steps of this library,
with every buffer of a fixed size so that the collectives need no split sizes
and the per-expert counts never leave the device:

    rank p of P, experts [p E/P, (p+1) E/P); its own T tokens and their routing;
    C = capacity rows per (sender, receiver) block, the same on every rank
        (default: the largest T k of the group, so nothing drops)
    1. routing metadata of its T k slots, then the send buffer (moe_ep_pack):
       block q holds the rows of rank q's experts in routed order from place 0,
       with each row's routing weight, and the per-(rank, local expert) counts.
    2. all-to-all (equal splits) of the counts, the rows and the weights.
    3. the receiver's routing metadata from the received counts alone
       (moe_ep_receive_metadata), then the single-device expert path on the
       P C received rows as tokens with k = 1: each received row's weighted
       output at the place it arrived.
    4. all-to-all back (equal splits), and the sum of each token's returned
       rows (moe_ep_combine).

Buffers and workspaces are allocated once, when the ``ExpertParallel`` is built;
a forward allocates nothing and reads nothing back to the host.

``ExpertParallel`` holds only this bookkeeping and calls the device work through
an ``ops`` object: ``LibmoeOps`` (the CUDA kernels of libmoe) by default. There is
no CPU fallback; tests of the exchange logic on CPU ranks pass their own ops.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding as B


class LibmoeOps:
    """The device steps of one rank, through libmoe (CUDA tensors only). setup()
    allocates every buffer once; the steps only enqueue kernels."""

    def __init__(self, device):
        B.load()
        self.device = torch.device(device)

    def setup(self, T, H, I, E, k, P, C):
        dev = self.device
        self.P, self.C, self.E_loc = P, C, E // P
        self.shp = B.shape(T, H, I, E, k)
        self.ws = B.new_workspace(self.shp, dev)
        self.rshp = B.shape(P * C, H, I, E // P, 1)
        self.rws = B.new_workspace(self.rshp, dev)
        self.send_rows = torch.empty((P * C, H), dtype=torch.bfloat16, device=dev)
        self.send_w = torch.empty((P * C,), dtype=torch.float32, device=dev)
        self.send_counts = torch.empty((P, E // P), dtype=torch.int32, device=dev)
        self.a = torch.empty((P * C, I), dtype=torch.bfloat16, device=dev)
        self.y_recv = torch.empty((P * C, H), dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)

    def receive_buffers(self):
        """(rows, weights, counts, returned rows): the receiving ends of the collectives."""
        return (torch.empty_like(self.send_rows), torch.empty_like(self.send_w),
                torch.empty_like(self.send_counts), torch.empty_like(self.send_rows))

    def pack(self, x, topk_idx, topk_w):
        B.moe_routing_metadata(topk_idx, self.shp, self.ws)
        B.moe_ep_pack(x, topk_w, self.shp, self.P, self.C, self.send_rows, self.send_w, self.send_counts, self.ws)
        return self.send_rows, self.send_w, self.send_counts

    def expert_forward(self, recv_counts, recv_rows, recv_w, w1, w2):
        B.moe_ep_receive_metadata(recv_counts, self.P, self.C, self.rshp, self.rws)
        B.moe_dispatch_gemm1(recv_rows, w1, self.rshp, self.a, self.rws)
        B.moe_swiglu_gemm2_combine(self.a, recv_w.view(-1, 1), w2, self.rshp, self.y_recv, self.rws)
        return self.y_recv

    def combine(self, back_rows):
        B.moe_ep_combine(back_rows, self.shp, self.P, self.C, self.y, self.ws)
        return self.y

    def device_errors(self):
        """The two workspaces' error words (a host sync; not for the step itself)."""
        return B.moe_get_device_error(self.ws) | B.moe_get_device_error(self.rws)


class ExpertParallel:
    """The expert path with experts sharded over the ranks of ``group``, for T
    tokens of hidden size H per rank (intermediate size I, k experts per token)."""

    def __init__(self, E: int, T: int, H: int, I: int, k: int, group=None, ops=None, device=None,
                 capacity: int | None = None):
        self.group = group
        self.P = dist.get_world_size(group)
        self.rank = dist.get_rank(group)
        if E % self.P:
            raise ValueError("E must be a multiple of the number of ranks")
        self.E, self.T, self.k = E, T, k
        self.E_loc = E // self.P
        if capacity is None:
            # every rank's blocks must have one size: the largest T k of the group
            # (agreed once, here; a forward never talks to the host)
            sizes = [None] * self.P
            dist.all_gather_object(sizes, int(T) * int(k), group=group)
            capacity = max(1, max(sizes))
        self.C = int(capacity)
        self.ops = ops if ops is not None else LibmoeOps(device)
        self.ops.setup(T, H, I, E, k, self.P, self.C)
        self.recv_rows, self.recv_w, self.recv_counts, self.back = self.ops.receive_buffers()

    def forward(self, x, topk_idx, topk_w, w1_local, w2_local):
        """y [T, H] for this rank's tokens; w1_local / w2_local hold this rank's experts."""
        if x.shape[0] != self.T:
            raise ValueError("x must have the T rows the ExpertParallel was built for")
        send_rows, send_w, send_counts = self.ops.pack(x, topk_idx, topk_w)
        dist.all_to_all_single(self.recv_counts, send_counts, group=self.group)
        dist.all_to_all_single(self.recv_rows, send_rows, group=self.group)
        dist.all_to_all_single(self.recv_w, send_w, group=self.group)
        y_recv = self.ops.expert_forward(self.recv_counts, self.recv_rows, self.recv_w, w1_local, w2_local)
        dist.all_to_all_single(self.back, y_recv, group=self.group)
        return self.ops.combine(self.back)
