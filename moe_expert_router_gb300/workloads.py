"""Workload shapes and seeded synthetic inputs.

This module only draws random inputs; it holds none of the router or expert
arithmetic, so both the CUDA path and the oracle can be fed from it.

Recipe (every config, one ``torch.Generator`` seeded with ``seed``), draws in
this order, each in fp32 and cast afterwards where the config says bf16:

1. x       [T, H]      ~ N(0, 1)                       -> bf16
2. W_r     [E, H]      ~ N(0, 0.02^2)                  fp32
3. bias    [E]         ~ N(0, 0.01^2)  (selection-bias configs only)  fp32
4. w1      [E, 2I, H]  ~ N(0, 1/H), one expert at a time -> bf16
5. w2      [E, H, I]   ~ N(0, 1/I), one expert at a time -> bf16
6. Zipf    randperm(E) -> rank r_e = 1 + perm[e]; offset_e = ln(p_e) with
           p_e = r_e^-s / sum_f r_f^-s (skewed configs only)   fp32
7. dY      [T, H]      ~ N(0, 1)  (training config only)   -> bf16

Generation on a CUDA device uses a CUDA generator, whose stream differs from
the CPU one; every comparison reads the very tensors it was given, so this
only changes which random inputs are seen, never what is compared.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int          # tokens
    H: int          # hidden size
    I: int          # expert intermediate size
    E: int          # experts (all local: expert parallelism 1)
    k: int          # experts per token
    score: str = "softmax"      # "softmax" | "sigmoid"
    normalize: bool = True      # divide top-k weights by their score sum
    scale: float = 1.0          # multiply top-k weights
    n_group: int = 1            # 1 = no group limit
    topk_group: int = 1
    group_topn: int = 2
    sel_bias: bool = False      # per-expert bias used only for selection
    zipf_s: float | None = None
    backward: bool = False
    description: str = ""

    @property
    def R(self) -> int:
        return self.T * self.k

    def with_tokens(self, T: int) -> "MoEConfig":
        return replace(self, T=T)

    def expert_flops(self) -> float:
        """6 R H I: GEMM1 (2 R H 2I) + GEMM2 (2 R H I); SwiGLU and combine not counted."""
        return 6.0 * self.R * self.H * self.I


CONFIGS: dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", T=256, H=128, I=64, E=8, k=2,
                      description="tiny forward, softmax, normalised top-2"),
    "mid": MoEConfig("mid", T=4096, H=2048, I=1408, E=64, k=6,
                     description="mid forward, softmax top-6, aux reported"),
    "large_group": MoEConfig("large_group", T=8192, H=7168, I=2048, E=256, k=8,
                             score="sigmoid", scale=2.5, n_group=8, topk_group=4,
                             group_topn=2, sel_bias=True,
                             description="large forward, sigmoid + selection bias, "
                                         "8 groups keep 4, weights x2.5"),
    "zipf_prefill": MoEConfig("zipf_prefill", T=16384, H=4096, I=1536, E=128, k=8, zipf_s=1.2,
                              description="Zipf(1.2)-skewed routing, T=16384"),
    "zipf_decode": MoEConfig("zipf_decode", T=64, H=4096, I=1536, E=128, k=8, zipf_s=1.2,
                             description="Zipf(1.2)-skewed routing, decode-like T=64"),
    "train": MoEConfig("train", T=8192, H=4096, I=1536, E=64, k=6, backward=True,
                       description="training step: forward and backward (dX, dW1, dW2, router gradient)"),
    # profiling size: the large_group geometry per expert (H, I, k, groups, about
    # 256 routed rows per expert) with 32 experts, so that a full ncu capture
    # holds about 3 GB on the device
    "large_group_slice": MoEConfig("large_group_slice", T=1024, H=7168, I=2048, E=32, k=8,
                                   score="sigmoid", scale=2.5, n_group=8, topk_group=4,
                                   group_topn=2, sel_bias=True,
                                   description="large_group per-expert geometry, 32 experts "
                                               "(profiling size)"),
    # profiling size of zipf_prefill: its shapes and Zipf(1.2) expert popularity at a
    # quarter of the tokens, so that a full ncu capture holds about 5 GB on the device
    "zipf_prefill_slice": MoEConfig("zipf_prefill_slice", T=4096, H=4096, I=1536, E=128, k=8,
                                    zipf_s=1.2,
                                    description="zipf_prefill shapes at T=4096 (profiling size)"),
    # profiling size of large_group's router: its tokens, hidden size, 256 experts and
    # group-limited sigmoid routing (the same router kernels and split) with I = 128, so
    # that a full ncu capture holds about 3 GB on the device
    "large_group_router": MoEConfig("large_group_router", T=8192, H=7168, I=128, E=256, k=8,
                                    score="sigmoid", scale=2.5, n_group=8, topk_group=4,
                                    group_topn=2, sel_bias=True,
                                    description="large_group router geometry, I = 128 (profiling size)"),
    # profiling size of the training step: the train geometry per expert (H, I, k,
    # about 768 routed rows per expert) with 16 experts, about 1 GB on the device
    "train_slice": MoEConfig("train_slice", T=2048, H=4096, I=1536, E=16, k=6, backward=True,
                             description="train per-expert geometry, 16 experts (profiling size)"),
}


def _randn(gen, shape, std, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32) * std


def generate(cfg: MoEConfig, seed: int = 0, device="cpu") -> dict:
    """Seeded synthetic inputs of ``cfg`` on ``device`` (see module docstring)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    T, H, I, E = cfg.T, cfg.H, cfg.I, cfg.E
    out = {}
    out["x"] = _randn(gen, (T, H), 1.0, device).to(torch.bfloat16)
    out["w_r"] = _randn(gen, (E, H), 0.02, device)
    out["sel_bias"] = _randn(gen, (E,), 0.01, device) if cfg.sel_bias else None
    w1 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=device)
    for e in range(E):
        w1[e] = _randn(gen, (2 * I, H), 1.0 / math.sqrt(H), device).to(torch.bfloat16)
    out["w1"] = w1
    w2 = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
    for e in range(E):
        w2[e] = _randn(gen, (H, I), 1.0 / math.sqrt(I), device).to(torch.bfloat16)
    out["w2"] = w2
    if cfg.zipf_s is not None:
        perm = torch.randperm(E, generator=gen, device=device).cpu()
        ranks = (perm + 1).to(torch.float64)
        p = ranks.pow(-cfg.zipf_s)
        p = p / p.sum()
        out["logit_offset"] = p.log().to(torch.float32).to(device)
    else:
        out["logit_offset"] = None
    out["dy"] = _randn(gen, (T, H), 1.0, device).to(torch.bfloat16) if cfg.backward else None
    return out


def even_routing(T: int, k: int, E: int, device="cpu"):
    """Round-robin routing topk_idx[t, j] = (t*k + j) % E.

    This is the deterministic ``even`` force-load-balancing mode of the MegaMoE
    guide (section "Router force load balancing"); weights are 1/k each.
    """
    slots = torch.arange(T * k, device=device, dtype=torch.int64)
    idx = (slots % E).to(torch.int32).view(T, k)
    w = torch.full((T, k), 1.0 / k, dtype=torch.float32, device=device)
    return idx, w


def routing_with_counts(counts, T: int, k: int, seed: int = 0, device="cpu"):
    """A random routing whose per-expert row counts are exactly ``counts``.

    ``sum(counts)`` must equal T*k. Experts of one token need not be distinct;
    the expert path gives each (token, choice) its own contribution either way.
    Weights are uniform in [0.1, 1).
    """
    counts = [int(c) for c in counts]
    assert sum(counts) == T * k, "counts must add up to T*k"
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    ids = torch.cat([torch.full((c,), e, dtype=torch.int32) for e, c in enumerate(counts)])
    ids = ids[torch.randperm(T * k, generator=gen)]
    w = torch.rand((T, k), generator=gen, dtype=torch.float32) * 0.9 + 0.1
    return ids.view(T, k).to(device), w.to(device)
