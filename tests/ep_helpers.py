"""Test-only device steps for ExpertParallel on CPU ranks: the oracle does the
routing metadata and the expert math, numpy the row moves. Used to check the
exchange logic (splits, counts, ordering, the return trip) without a GPU."""
import numpy as np
import torch

import oracle


class OracleOps:
    def route(self, x, topk_idx, topk_w, E):
        md = oracle.routing_metadata(topk_idx, E)
        k = topk_idx.shape[1]
        perm = torch.as_tensor(md.perm_slot, dtype=torch.long)
        rows = x[perm // k].contiguous()
        row_w = topk_w.reshape(-1)[perm].to(torch.float64).contiguous()
        return md.counts, rows, row_w, md

    def expert_forward(self, rows, expert, weight, w1, w2):
        if rows.shape[0] == 0:
            return torch.zeros((0, rows.shape[1]), dtype=torch.float64)
        y = oracle.expert_forward(rows, expert.view(-1, 1), weight.view(-1, 1), w1, w2)
        return torch.as_tensor(y)

    def combine(self, rows_back, md, T, H):
        k = md.row_of.shape[0] // T if T else 1
        y = np.zeros((T, H))
        rb = rows_back.numpy()
        for s, r in enumerate(md.row_of):
            if r >= 0:
                y[s // k] += rb[r]
        return torch.as_tensor(y)

    def to_device(self, array, dtype):
        return torch.as_tensor(array, dtype=dtype)
