"""MXFP8 weight-quant cache (MegaMoE guide, section "Expert precision").

The guide's mxfp8 path keeps the expert parameters in bf16 and holds their
MXFP8 quantization in a cache keyed on the weight tensor's version counter;
once per optimizer step the cache is dropped as well, because an optimizer can
update the weights in place without bumping that counter. This module is the
same bookkeeping on the host: it calls the library's quantizer
(``moe_mx_quantize``) and does no arithmetic of its own.
"""
from __future__ import annotations

import weakref

import torch

from . import binding as B


def _gpu_quantize(w: torch.Tensor):
    """codes, scales of a bf16 [E, rows, K] weight, quantized along K by libmoe
    (scales k-block-major: [K / 128, E, rows, 4])."""
    codes = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    scales = B.mx_scales_empty(w.shape, w.device)
    B.moe_mx_quantize(w, codes, scales)
    return codes, scales


class MxWeightCache:
    """MXFP8 copies of bf16 expert weights, kept while the weights are unchanged.

    ``get(w)`` returns ``(codes, scales)`` for ``w`` and quantizes again when the
    tensor's version counter moved since the cached copy was made (an in-place
    update through autograd-visible ops), or when ``w`` is not the tensor object
    the entry was made for (a weight freed and another allocated at its address
    starts again at version 0; a detached view is another object and is quantized
    on its own). An entry is dropped when its weight is freed. ``invalidate()``
    drops every entry: call it once per optimizer step.
    """

    def __init__(self, quantize=None):
        self._quantize = quantize or _gpu_quantize
        self._store = {}
        self.quantizations = 0

    @staticmethod
    def _key(w: torch.Tensor):
        return (w.device, w.data_ptr(), tuple(w.shape), w.dtype)

    def get(self, w: torch.Tensor):
        if w.dtype != torch.bfloat16 or w.shape[-1] % 32:
            raise ValueError("MXFP8 weights are quantized from bf16 along a last dimension of 32k")
        key = self._key(w)
        hit = self._store.get(key)
        if hit is not None and hit[0]() is w and hit[1] == w._version:
            return hit[2]
        q = self._quantize(w)
        self.quantizations += 1
        self._store[key] = (weakref.ref(w, self._dropper(key)), w._version, q)
        return q

    def _dropper(self, key):
        # when the weight is freed its entry (and the device memory of its copy) goes
        # too, unless the key already holds a newer entry
        store = self._store

        def drop(ref):
            entry = store.get(key)
            if entry is not None and entry[0] is ref:
                del store[key]
        return drop

    def invalidate(self):
        """Drop every cached quantization (once per optimizer step)."""
        self._store.clear()

    def __len__(self):
        return len(self._store)
