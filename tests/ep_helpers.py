"""Test-only device steps for ExpertParallel on CPU ranks: the oracle does the
routing metadata and the expert math, numpy the row moves into the fixed-size
blocks. Used to check the exchange logic (block places, counts, the receiver's
expert order, the return trip, the capacity) without a GPU. Written from the
layout the library documents, independently of its kernels."""
import numpy as np
import torch

import oracle


class OracleOps:
    def setup(self, T, H, I, E, k, P, C):
        self.T, self.H, self.E, self.k, self.P, self.C, self.E_loc = T, H, E, k, P, C, E // P
        self.send_rows = torch.zeros((P * C, H), dtype=torch.bfloat16)
        self.send_w = torch.zeros((P * C,), dtype=torch.float64)
        self.send_counts = torch.zeros((P, E // P), dtype=torch.int32)

    def receive_buffers(self):
        return (torch.empty_like(self.send_rows), torch.empty_like(self.send_w),
                torch.empty_like(self.send_counts), torch.empty((self.P * self.C, self.H), dtype=torch.float64))

    def _place(self, r):
        """(block place of routed row r, or -1 past the capacity)."""
        off = self.md.offsets
        e = int(np.searchsorted(off, r, side="right")) - 1
        q = e // self.E_loc
        pos = r - int(off[q * self.E_loc])
        return q * self.C + pos if pos < self.C else -1

    def pack(self, x, topk_idx, topk_w):
        self.md = md = oracle.routing_metadata(topk_idx, self.E)
        k = self.k
        self.send_rows.zero_()
        self.send_w.zero_()
        wflat = topk_w.reshape(-1).to(torch.float64)
        for r, slot in enumerate(md.perm_slot.tolist()):
            pl = self._place(r)
            if pl >= 0:
                self.send_rows[pl] = x[slot // k]
                self.send_w[pl] = wflat[slot]
        sent = np.zeros((self.E,), np.int32)
        for r in range(len(md.perm_slot)):
            if self._place(r) >= 0:
                sent[int(np.searchsorted(md.offsets, r, side="right")) - 1] += 1
        self.send_counts.copy_(torch.as_tensor(sent.reshape(self.P, self.E_loc)))
        return self.send_rows, self.send_w, self.send_counts

    def expert_forward(self, recv_counts, recv_rows, recv_w, w1, w2):
        """Received block p: its rows in place order, grouped by local expert."""
        y = torch.zeros((self.P * self.C, self.H), dtype=torch.float64)
        cnt = recv_counts.numpy()
        for p in range(self.P):
            n = int(cnt[p].sum())
            if n == 0:
                continue
            experts = np.repeat(np.arange(self.E_loc, dtype=np.int32), cnt[p])
            rows = slice(p * self.C, p * self.C + n)
            out = oracle.expert_forward(recv_rows[rows], torch.as_tensor(experts).view(-1, 1),
                                        recv_w[rows].view(-1, 1), w1, w2)
            y[rows] = torch.as_tensor(out)
        return y

    def combine(self, back_rows):
        y = np.zeros((self.T, self.H))
        b = back_rows.numpy()
        for s, r in enumerate(self.md.row_of.tolist()):
            if r >= 0:
                pl = self._place(r)
                if pl >= 0:
                    y[s // self.k] += b[pl]
        return torch.as_tensor(y)
