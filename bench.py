"""Benchmark of the MoE expert path (router -> routing metadata -> stage 1 ->
stage 2, and for the training workload the backward: stage 2 data / weight,
router, stage 1 data / weight) through the C ABI of libmoe on one or more GPUs
of one node.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference] [--no-cpu-baseline]

The default workload is large_group (T=8192, H=7168, I=2048, E=256, k=8,
sigmoid scores with a selection bias, 8 groups keep 4, weights x2.5): the
largest configuration that fits one GPU.

A step is one pass of the whole path over one batch of seeded synthetic
inputs already resident in HBM. Each rank runs its own independent replica
(the path has no exchange step at expert parallelism 1), so scaling is weak.
Rank 0 prints one JSON line.

--impl reference times the fp64 CPU oracle on the host cores instead (each
step a bounded sample of the same workload); under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from moe_expert_router_gb300.workloads import CONFIGS, generate  # noqa: E402

METRIC = "MoE expert-path TFLOP/s and tokens/s (1 GB300) and fraction of bf16/HBM roofline"
L2_FLUSH_BYTES = 256 << 20

# DRAM bytes (read + write) per launch of stage 1 -- the dispatch copy plus the
# stage-1 GEMM, the two kernels its CUDA-event time covers -- from ncu captures
# of `bench.py --workload <name> --steps 2 --warmup 1 --no-cpu-baseline`
# (summaries under profiles/). Reported only while the kernel sources still
# hash to the value recorded with the capture; otherwise traffic is null.
KERNEL_SOURCES = ("moe_expert_router_gb300/csrc/gemm_kernel.cuh", "moe_expert_router_gb300/csrc/grouped_gemm.cu",
                  "moe_expert_router_gb300/csrc/ptx.cuh", "moe_expert_router_gb300/csrc/internal.cuh")
STAGE1_TRAFFIC = {
    # profiles/tc_gemm_large_group_ncu.md, one step at full size: dispatch copy
    # 117.76 MB read + 875.45 MB written, tc_gemm_kernel<0> 16.274 GB + 263.98 MB
    "large_group": {"src": "76bbf096a270446f", "bytes": 117.76e6 + 875.45e6 + 16.274e9 + 263.98e6},
}


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.06 <= r[0] <= self.t1 + 0.06]
        use = inside if inside else rows[-3:]
        sm = [float(p[2]) for _, p in use if p[2].replace(".", "").isdigit()]
        mx = [float(p[3]) for _, p in use if p[3].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in use:
            for name, v in zip(names, p[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside),
                "window": "timed region" if inside else "nearest samples (timed region shorter than the sampling period)"}


# ---------------------------------------------------------------- our arm

def bytes_and_flops(cfg, counts, precision="bf16"):
    """Algorithmic flops and bytes of each GEMM stage (bytes the kernels could avoid
    are not counted), keyed by the stage name used for the step's events."""
    R, H, I, T, E = cfg.R, cfg.H, cfg.I, cfg.T, cfg.E
    active = int((counts > 0).sum())
    if precision == "mxfp8":
        q = 1.0 + 1.0 / 32           # E4M3 byte + one E8M0 byte per 32 elements
        st = {
            "gemm1": {"flops": 4.0 * R * H * I,
                      "bytes": 2.0 * H * I * q * active + R * H * q + R * I * q + (4.0 * R * I if cfg.backward else 0),
                      "kernel": "tc_gemm_kernel<kStage1Mx> (stage 1 in MXFP8: dispatched E4M3 x rows, "
                                "block-scaled MMA, SwiGLU + MXFP8 quantization of a%s)"
                                % (", h saved in bf16" if cfg.backward else ""), "precision": "mxfp8"},
            "gemm2_combine": {"flops": 2.0 * R * H * I,
                              "bytes": H * I * q * active + R * I * q + 2.0 * T * H,
                              "kernel": "tc_gemm_kernel<kStage2Mx> + combine_kernel (stage 2 in MXFP8)",
                              "precision": "mxfp8"},
        }
        if cfg.backward:
            bf = bytes_and_flops(cfg, counts, "bf16")["stages"]
            st["bwd_stage2_data"] = bf["bwd_stage2_data"]
            st["bwd_stage1_data"] = bf["bwd_stage1_data"]
            # quantization of dY and w a (read 2 R (H + I), write (R + 128 E)(H + I) q), then the GEMM
            ld = R + 128 * E
            st["bwd_stage2_weight"] = {
                "flops": 2.0 * R * H * I,
                "bytes": 2.0 * R * (H + I) + 2.0 * ld * (H + I) * q + 2.0 * E * H * I,
                "kernel": "mx_quantize_rows_t_kernel x2 + tc_gemm_kernel<kWgradMx>: dW2 in MXFP8",
                "precision": "mxfp8"}
            st["bwd_stage1_weight"] = {
                "flops": 4.0 * R * H * I,
                "bytes": 2.0 * R * (2 * I) + 2.0 * T * H + 2.0 * ld * (2 * I + H) * q + 4.0 * E * H * I,
                "kernel": "mx_quantize_rows_t_kernel x2 + tc_gemm_kernel<kWgradMx>: dW1 in MXFP8",
                "precision": "mxfp8"}
        return {"stages": st, "active_experts": active}
    st = {
        "gemm1": {"flops": 4.0 * R * H * I,
                  "bytes": 4.0 * H * I * active + 2.0 * T * H + 2.0 * R * I * (3 if cfg.backward else 1),
                  "kernel": "tc_gemm_kernel<kStage1%s> (stage 1: dispatch copy of x + GEMM1 + SwiGLU)"
                            % ("SaveH" if cfg.backward else "")},
        "gemm2_combine": {"flops": 2.0 * R * H * I,
                          "bytes": 2.0 * H * I * active + 2.0 * R * I + 2.0 * T * H,
                          "kernel": "tc_gemm_kernel<kStage2> + combine_kernel (stage 2)"},
    }
    if cfg.backward:
        st["bwd_stage2_data"] = {
            "flops": 2.0 * R * H * I,
            "bytes": 2.0 * H * I * active + 2.0 * T * H + 4.0 * R * I + 4.0 * R * I + 2.0 * R * I,
            "kernel": "tc_gemm_kernel<kBwdDA> (+ zero_tail_rows, dtw_reduce): dA + SwiGLU backward"}
        st["bwd_stage2_weight"] = {
            "flops": 2.0 * R * H * I,
            "bytes": 2.0 * T * H + 2.0 * R * I + 2.0 * E * H * I,
            "kernel": "tc_gemm_kernel<kBwdDW2>: dW2"}
        st["bwd_stage1_data"] = {
            "flops": 4.0 * R * H * I,
            "bytes": 4.0 * R * I + 4.0 * H * I * active + 4.0 * R * H + 2.0 * T * H,
            "kernel": "tc_gemm_kernel<kBwdDX> + combine_bwd_kernel: dX"}
        st["bwd_stage1_weight"] = {
            "flops": 4.0 * R * H * I,
            "bytes": 4.0 * R * I + 2.0 * T * H + 4.0 * E * H * I,
            "kernel": "tc_gemm_kernel<kBwdDW1>: dW1"}
    return {"stages": st, "active_experts": active}


def step_flops(cfg):
    """Expert-path flops of one step: 6 R H I forward, + 12 R H I with the backward."""
    return cfg.expert_flops() * (3.0 if cfg.backward else 1.0)


def run_ours(args, cfg, rank, world, local_rank):
    from moe_expert_router_gb300 import binding as B
    from moe_expert_router_gb300 import build as moe_build

    moe_build.build()
    B.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp = generate(cfg, seed=rank, device=dev)
    train = cfg.backward
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, training=train)
    ws = B.new_workspace(shp, dev)
    rcfg = B.router_cfg(cfg.score, cfg.normalize, cfg.scale, cfg.n_group, cfg.topk_group,
                        cfg.group_topn)
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=dev)
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)
    aux = torch.zeros((1,), dtype=torch.float32, device=dev)
    a = torch.empty((cfg.R, cfg.I), dtype=torch.bfloat16, device=dev)
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    x_dev = inp["x"]
    if train:
        logits = torch.empty((cfg.T, cfg.E), dtype=torch.float32, device=dev)
        h = torch.empty((cfg.R, 2 * cfg.I), dtype=torch.bfloat16, device=dev)
        dy_dev = inp["dy"]
        dx = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)
        dw1 = torch.empty_like(inp["w1"])
        dw2 = torch.empty_like(inp["w2"])
        dwr = torch.empty_like(inp["w_r"])
        dtw = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=dev)

    uniform = args.routing == "uniform"
    mx = args.precision == "mxfp8"
    w1_f, w2_f = inp["w1"], inp["w2"]      # the forward's weight operands
    if args.weights == "packed":
        if train or mx:
            raise SystemExit("--weights packed covers the bf16 forward workloads")
        shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, packed=True)
        ws = B.new_workspace(shp, dev)
        # packed once, outside the timed region (a weight-layout cache, like the MXFP8 one)
        w1_f, w2_f = B.moe_pack_weights(inp["w1"], inp["w2"], shp)
        torch.cuda.synchronize(dev)
    if mx:
        from moe_expert_router_gb300.mx_cache import MxWeightCache
        shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, training=train, mxfp8=True)
        ws = B.new_workspace(shp, dev)
        cache = MxWeightCache()           # weights quantized once, outside the timed region
        w1q, w1s = cache.get(inp["w1"])
        w2q, w2s = cache.get(inp["w2"])
        aq = torch.empty((cfg.R, cfg.I), dtype=torch.uint8, device=dev)
        as_ = B.mx_scales_empty((cfg.R, cfg.I), dev)
    if uniform:
        # the guide's `uniform` force-balance mode: each step routes fresh N(0,1)
        # logits (drawn before the timed region; a pool of 8 steps' worth is cycled)
        gen = torch.Generator(device=dev)
        gen.manual_seed(1000 + rank)
        logit_pool = [torch.randn((cfg.T, cfg.E), generator=gen, device=dev) for _ in range(8)]
    step_no = [0]

    names = ["router", "metadata", "gemm1", "gemm2_combine"]
    if mx:
        names = ["router", "metadata", "mx_dispatch", "gemm1", "gemm2_combine"]
    if train:
        names += ["bwd_stage2_data", "bwd_stage2_weight", "router_bwd", "bwd_stage1_data",
                  "bwd_stage1_weight"]

    def calls(x_in, dy_in, y=y, aux=aux, dx=dx if train else None):
        """The step's C-ABI calls in order (one per event interval); y, aux and dx are
        the step's outputs (double-buffered by the end-to-end loop)."""
        if uniform:
            lg = logit_pool[step_no[0] % len(logit_pool)]
            step_no[0] += 1
            yield lambda: B.moe_route_logits(lg, shp, rcfg, idx, w, ws, aux=aux,
                                             logit_offset=inp["logit_offset"], sel_bias=inp["sel_bias"])
        elif train:
            yield lambda: B.moe_router_train(x_in, inp["w_r"], shp, rcfg, idx, w, logits, ws, aux=aux,
                                             logit_offset=inp["logit_offset"], sel_bias=inp["sel_bias"])
        else:
            yield lambda: B.moe_router(x_in, inp["w_r"], shp, rcfg, idx, w, ws, aux=aux,
                                       logit_offset=inp["logit_offset"], sel_bias=inp["sel_bias"])
        yield lambda: B.moe_routing_metadata(idx, shp, ws)
        if mx:
            yield lambda: B.moe_mx_quantize_dispatch(x_in, shp, ws)
            if train:
                yield lambda: B.moe_dispatch_gemm1_mx_train(w1q, w1s, shp, aq, as_, h, ws)
            else:
                yield lambda: B.moe_dispatch_gemm1_mx(w1q, w1s, shp, aq, as_, ws)
            yield lambda: B.moe_swiglu_gemm2_combine_mx(aq, as_, w, w2q, w2s, shp, y, ws)
            if not train:
                return
            # the guide's mxfp8 training: bf16 data gradients, MXFP8 weight gradients
            yield lambda: B.moe_backward_stage2_data(dy_in, w, inp["w2"], h, shp, ws, dtopk_w=dtw)
            yield lambda: B.moe_backward_stage2_weight_mx(dy_in, shp, dw2, ws)
            if uniform:
                yield lambda: None
                yield lambda: B.moe_backward_stage1_data(inp["w1"], shp, dx, ws)
            else:
                yield lambda: B.moe_router_backward(x_in, logits, idx, w, dtw, shp, rcfg, dwr, ws)
                yield lambda: B.moe_backward_stage1_data(inp["w1"], shp, dx, ws, w_r=inp["w_r"],
                                                         topk_idx=idx, cfg=rcfg)
            yield lambda: B.moe_backward_stage1_weight_mx(x_in, shp, dw1, ws)
            return
        if train:
            yield lambda: B.moe_dispatch_gemm1_train(x_in, inp["w1"], shp, a, h, ws)
        else:
            yield lambda: B.moe_dispatch_gemm1(x_in, w1_f, shp, a, ws)
        yield lambda: B.moe_swiglu_gemm2_combine(a, w, w2_f, shp, y, ws)
        if train:
            yield lambda: B.moe_backward_stage2_data(dy_in, w, inp["w2"], h, shp, ws, dtopk_w=dtw)
            yield lambda: B.moe_backward_stage2_weight(dy_in, shp, dw2, ws)
            if uniform:         # random logits: no gradient reaches the router
                yield lambda: None
                yield lambda: B.moe_backward_stage1_data(inp["w1"], shp, dx, ws)
            else:
                yield lambda: B.moe_router_backward(x_in, logits, idx, w, dtw, shp, rcfg, dwr, ws)
                yield lambda: B.moe_backward_stage1_data(inp["w1"], shp, dx, ws, w_r=inp["w_r"],
                                                         topk_idx=idx, cfg=rcfg)
            yield lambda: B.moe_backward_stage1_weight(x_in, shp, dw1, ws)

    def step(ev=None, per_stage=False):
        """One step. ev: [start, end] events, or with per_stage one event before every
        call and one after the last (the breakdown pass: an event between two calls
        keeps their kernels from overlapping, so the timed steps record only the two
        ends)."""
        for j, call in enumerate(calls(x_dev, inp["dy"] if train else None)):
            if ev is not None and (per_stage or j == 0):
                ev[j].record(stream)
            call()
        if ev is not None:
            ev[-1].record(stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize(dev)
    err = B.moe_get_device_error(ws)
    if err:
        raise RuntimeError(f"device error word {err:#x} after warm-up")

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    launches0 = B.moe_kernel_launch_count()
    if sampler:
        sampler.mark_begin()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)           # evict L2 between steps (outside the step's events)
        step(events[i])
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall0
    if sampler:
        sampler.mark_end()
    if world > 1:
        torch.distributed.barrier()
    launches = B.moe_kernel_launch_count() - launches0
    clocks = sampler.stop() if sampler else None
    step_ms = [ev[0].elapsed_time(ev[1]) for ev in events]
    total_ms = sum(step_ms)

    # per-stage breakdown (not part of the timed region): events between the calls
    n_bd = min(args.steps, 10)
    bd_events = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(n_bd)]
    for i in range(n_bd):
        flush.fill_(i & 0xFF)
        step(bd_events[i], per_stage=True)
    torch.cuda.synchronize(dev)
    stage_ms = {n: [] for n in names}
    for ev in bd_events:
        for j, n in enumerate(names):
            stage_ms[n].append(ev[j].elapsed_time(ev[j + 1]))

    # metadata for the algorithmic byte counts
    L = B.moe_workspace_layout(shp)
    counts = ws[L.counts:L.counts + 4 * cfg.E].view(torch.int32).cpu()
    bf = bytes_and_flops(cfg, counts, args.precision)

    # end to end, as a serving loop runs it: every step uploads its x (and dY) from
    # pinned host memory and downloads y + aux (and dX); weight gradients stay on the
    # device for the optimizer. Inputs and outputs are double-buffered and the copies
    # run on two copy streams, so step i's download and step i + 1's upload overlap
    # the neighbouring steps' compute; the timed interval runs from before the first
    # upload to after the last download.
    x_host = inp["x"].cpu().pin_memory()
    y_host = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    aux_host = [torch.empty((1,), dtype=torch.float32).pin_memory() for _ in range(2)]
    x_buf = [torch.empty_like(x_dev) for _ in range(2)]
    y_buf = [y, torch.empty_like(y)]
    aux_buf = [aux, torch.empty_like(aux)]
    if train:
        dy_host = inp["dy"].cpu().pin_memory()
        dy_buf = [torch.empty_like(inp["dy"]) for _ in range(2)]
        dx_host = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        dx_buf = [dx, torch.empty_like(dx)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(n):
        """n pipelined end-to-end steps; returns the milliseconds from the first upload's
        start to the last download's end."""
        uploaded = [torch.cuda.Event() for _ in range(2)]
        computed = [torch.cuda.Event() for _ in range(2)]
        downloaded = [torch.cuda.Event() for _ in range(2)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def upload(j):
            with torch.cuda.stream(up):
                x_buf[j].copy_(x_host, non_blocking=True)
                if train:
                    dy_buf[j].copy_(dy_host, non_blocking=True)
            uploaded[j].record(up)

        t0.record(up)
        upload(0)
        for i in range(n):
            cur, nxt = i % 2, (i + 1) % 2
            stream.wait_event(uploaded[cur])
            if i >= 2:
                stream.wait_event(downloaded[cur])   # step i - 2's outputs have reached the host
            for call in calls(x_buf[cur], dy_buf[cur] if train else None, y=y_buf[cur], aux=aux_buf[cur],
                              dx=dx_buf[cur] if train else None):
                call()
            computed[cur].record(stream)
            if i + 1 < n:
                if i >= 1:
                    up.wait_event(computed[nxt])     # step i - 1 is done with those buffers
                upload(nxt)
            down.wait_event(computed[cur])
            with torch.cuda.stream(down):
                y_host[cur].copy_(y_buf[cur], non_blocking=True)
                aux_host[cur].copy_(aux_buf[cur], non_blocking=True)
                if train:
                    dx_host[cur].copy_(dx_buf[cur], non_blocking=True)
            downloaded[cur].record(down)
        up.wait_stream(down)
        t1.record(up)
        t1.synchronize()                     # the host holds every step's result
        return t0.elapsed_time(t1)

    e2e_run(max(2, args.warmup))
    torch.cuda.synchronize(dev)
    e2e_total = e2e_run(args.steps)
    e2e_ms = [e2e_total]
    h2d = x_host.numel() * x_host.element_size() * (2 if train else 1)
    d2h = y_host[0].numel() * y_host[0].element_size() * (2 if train else 1) + 4
    err = B.moe_get_device_error(ws)
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed region")

    return {"total_ms": total_ms, "step_ms": step_ms, "stage_ms": stage_ms, "bf": bf,
            "clocks": clocks, "launches": launches, "e2e_ms": sum(e2e_ms), "h2d": h2d, "d2h": d2h,
            "wall_s": t_wall}


# ---------------------------------------------------------------- oracle (CPU) arm

_MX_WEIGHTS = {}


def oracle_sample(cfg, n_tokens, seed=0, inputs=None, routing="router", precision="bf16"):
    """Run the oracle's step (router + expert path, and for a training workload the
    expert and router backward) on the first n_tokens tokens; return seconds. With
    uniform routing the oracle routes N(0,1) logits (its router on x = identity and
    W_r = the logits transposed) and the router backward is skipped."""
    import oracle
    inp = inputs if inputs is not None else cpu_inputs(cfg, seed)
    x = inp["x"][:n_tokens]
    if routing == "uniform":
        g = torch.Generator().manual_seed(1000 + seed)
        rx = torch.eye(n_tokens, dtype=torch.float32).to(torch.bfloat16)
        rw = torch.randn((cfg.E, n_tokens), generator=g, dtype=torch.float32)
    else:
        rx, rw = x, inp["w_r"]
    t0 = time.perf_counter()
    r = oracle.router(rx, rw, cfg.k, score=cfg.score, normalize=cfg.normalize,
                      scale=cfg.scale, n_group=cfg.n_group, topk_group=cfg.topk_group,
                      group_topn=cfg.group_topn, logit_offset=inp["logit_offset"],
                      sel_bias=inp["sel_bias"])
    if precision == "mxfp8":
        # weights quantized once per workload (the cache), x per sample
        if cfg.name not in _MX_WEIGHTS:
            t1 = time.perf_counter()
            _MX_WEIGHTS[cfg.name] = oracle.mx_quantize(inp["w1"]) + oracle.mx_quantize(inp["w2"])
            t0 += time.perf_counter() - t1
        w1q, w1s, w2q, w2s = _MX_WEIGHTS[cfg.name]
        xq, xs = oracle.mx_quantize(x)
        oracle.expert_forward_mx(xq, xs, r.topk_idx, r.topk_w, w1q, w1s, w2q, w2s)
        if cfg.backward:
            b = oracle.expert_backward_mx(x, xq, xs, r.topk_idx, r.topk_w, inp["w1"], w1q, w1s, inp["w2"],
                                          inp["dy"][:n_tokens])
            if routing != "uniform":
                oracle.router_backward(x, inp["w_r"], r.topk_idx, r.topk_w, b.dtopk_w, score=cfg.score,
                                       normalize=cfg.normalize, scale=cfg.scale, logit_offset=inp["logit_offset"])
        return time.perf_counter() - t0
    oracle.expert_forward(x, r.topk_idx, r.topk_w, inp["w1"], inp["w2"])
    if cfg.backward and routing == "uniform":
        oracle.expert_backward(x, r.topk_idx, r.topk_w, inp["w1"], inp["w2"], inp["dy"][:n_tokens])
    elif cfg.backward:
        b = oracle.expert_backward(x, r.topk_idx, r.topk_w, inp["w1"], inp["w2"], inp["dy"][:n_tokens])
        oracle.router_backward(x, inp["w_r"], r.topk_idx, r.topk_w, b.dtopk_w, score=cfg.score,
                               normalize=cfg.normalize, scale=cfg.scale, logit_offset=inp["logit_offset"])
    return time.perf_counter() - t0


def sample_flops(cfg, n_tokens):
    return step_flops(cfg) * n_tokens / cfg.T


_CPU_INPUTS = {}


def cpu_inputs(cfg, seed=0):
    key = (cfg.name, seed)
    if key not in _CPU_INPUTS:
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        inp = generate(cfg, seed=seed, device=dev)
        _CPU_INPUTS[key] = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    return _CPU_INPUTS[key]


def cpu_baseline(cfg, budget_s=15.0, routing="router", precision="bf16"):
    """Oracle timed on the host cores on a bounded token sample (~budget_s of work)."""
    import oracle
    oracle.build()
    inp = cpu_inputs(cfg)
    n_cal = min(cfg.T, 8)
    t_cal = oracle_sample(cfg, n_cal, inputs=inp, routing=routing, precision=precision)
    n = int(max(1, min(cfg.T, n_cal * budget_s / max(t_cal, 1e-6))))
    t = oracle_sample(cfg, n, inputs=inp, routing=routing, precision=precision) if n != n_cal else t_cal
    flops = sample_flops(cfg, n)
    what = "forward and backward" if cfg.backward else "router + expert path"
    if precision == "mxfp8":
        what += " in MXFP8 (weights quantized once, outside the timing)"
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "tokens_per_s": n / t,
            "sample": f"first {n} of {cfg.T} tokens of the '{cfg.name}' workload: fp64 {what}, {t:.2f} s"}


def run_reference(args, cfg):
    import oracle
    oracle.build()
    inp = cpu_inputs(cfg)
    n_cal = min(cfg.T, 8)
    kw = dict(inputs=inp, routing=args.routing, precision=args.precision)
    t_cal = oracle_sample(cfg, n_cal, **kw)
    per_step_budget = min(20.0, 150.0 / max(1, args.steps + args.warmup))
    n = int(max(1, min(cfg.T, n_cal * per_step_budget / max(t_cal, 1e-6))))
    for _ in range(args.warmup):
        oracle_sample(cfg, n, **kw)
    times = [oracle_sample(cfg, n, **kw) for _ in range(args.steps)]
    tot = sum(times)
    flops = sample_flops(cfg, n) * args.steps
    value = flops / tot / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "tokens_per_s": n * args.steps / tot,
        "config": config_dict(cfg, args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"each step: first {n} of {cfg.T} tokens, fp64 "
                                   f"{'forward and backward' if cfg.backward else 'router + expert path'}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def max_over_ranks(values, world, device="cpu"):
    """Element-wise maximum over the ranks of the job (the job is as slow as its
    slowest replica); identity for a single process."""
    if world <= 1:
        return [float(v) for v in values]
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_throughput(units_per_rank_step, steps, world, total_ms):
    """Units processed by all ranks per second over the slowest rank's time."""
    return units_per_rank_step * steps * world / (total_ms / 1e3)


def config_dict(cfg, args):
    return {"workload": cfg.name, "description": cfg.description, "routing": args.routing,
            "precision": args.precision, "weights": getattr(args, "weights", "rowmajor"),
            "T": cfg.T, "H": cfg.H,
            "I": cfg.I, "E": cfg.E, "k": cfg.k, "score": cfg.score, "n_group": cfg.n_group,
            "topk_group": cfg.topk_group, "zipf_s": cfg.zipf_s, "parallelism": f"replicas x{args.gpus}",
            "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write outside the step events); "
                  "weights exceed L2"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    # default: the largest single-GPU configuration (DeepSeek-V3 geometry, group-limited routing)
    ap.add_argument("--workload", default="large_group", choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--precision", default="bf16", choices=["bf16", "mxfp8"],
                    help="expert-path precision: bf16, or the guide's mxfp8 (E4M3 + E8M0 block scales)")
    ap.add_argument("--weights", default="rowmajor", choices=["rowmajor", "packed"],
                    help="rowmajor: w1 / w2 as given; packed: tile-packed once by moe_pack_weights "
                         "before the timed region (bf16 forward workloads)")
    ap.add_argument("--routing", default="router", choices=["router", "uniform"],
                    help="router: the fused router on x; uniform: the guide's force-balance mode "
                         "(fresh N(0,1) logits each step, routed by moe_route_logits)")
    args = ap.parse_args()
    cfg = CONFIGS[args.workload]

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, cfg)), flush=True)
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, cfg, rank, world, local_rank)
    total_ms, e2e_ms = max_over_ranks([res["total_ms"], res["e2e_ms"]], world,
                                      device=torch.device("cuda", local_rank))

    if rank == 0:
        peaks = measured_peaks()
        flops_step = step_flops(cfg)
        value = whole_job_throughput(flops_step, args.steps, world, total_ms) / 1e12
        tokens_per_s = whole_job_throughput(cfg.T, args.steps, world, total_ms)
        # dominant GEMM stage of the step and its roofline
        stage_avg = {n: sum(v) / len(v) for n, v in res["stage_ms"].items()}
        bf = res["bf"]
        dom = max(bf["stages"], key=lambda n: stage_avg[n])
        dom_ms = stage_avg[dom]
        f, b = bf["stages"][dom]["flops"], bf["stages"][dom]["bytes"]
        # an MXFP8 contraction takes the fp8 peak: the measured bf16 peak times the
        # nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s dense); the MXFP8 training
        # step's data gradients stay bf16
        dom_mx = bf["stages"][dom].get("precision", args.precision) == "mxfp8"
        tc_peak = peaks["bf16_tflops"] * (2.0 if dom_mx else 1.0)
        t_tc = f / (tc_peak * 1e12)
        t_hbm = b / (peaks["hbm_gbs"] * 1e9)
        if t_tc >= t_hbm:
            roof = {"bound": "tensor", "achieved": f / (dom_ms / 1e3) / 1e12,
                    "peak": tc_peak, "unit": "TFLOP/s"}
        else:
            roof = {"bound": "hbm", "achieved": b / (dom_ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                    "unit": "GB/s"}
        roof["frac"] = roof["achieved"] / roof["peak"]
        # the capture is of the bf16 stage-1 kernel on row-major weights under the router's routing
        rec = STAGE1_TRAFFIC.get(cfg.name)
        same_path = (args.precision == "bf16" and args.routing == "router" and
                     getattr(args, "weights", "rowmajor") == "rowmajor")
        roof["traffic"] = (rec["bytes"] if (dom == "gemm1" and same_path and rec and rec["src"] == kernel_source_hash())
                           else None)
        roof["algorithmic_bytes"] = b
        roof["kernel"] = bf["stages"][dom]["kernel"]
        roof["stage"] = dom
        roof["peak_kind"] = (f"{peaks['source']} bf16 burst x 2 (nominal fp8/bf16 ratio)"
                             if dom_mx and roof["bound"] == "tensor"
                             else f"{peaks['source']} burst")
        roof["kernel_ms"] = dom_ms
        out = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("bf16" if args.precision != "mxfp8" else
                      "mxfp8 (e4m3 + e8m0 scales, fp32 accumulate)" if not cfg.backward else
                      "mxfp8 expert stages and weight gradients (e4m3 + e8m0, fp32 accumulate), bf16 data gradients"),
            "data": "synthetic", "config": config_dict(cfg, args),
            "tokens_per_s": tokens_per_s,
            "stage_ms": {n: round(v, 5) for n, v in stage_avg.items()},
            "active_experts": bf["active_experts"],
            "roofline": roof,
            "e2e": {"value": flops_step * args.steps * world / (e2e_ms / 1e3) / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                    "ms_per_step": e2e_ms / args.steps,
                    "copies": "pinned host buffers, double-buffered; uploads and downloads on two copy "
                              "streams overlap the neighbouring steps' compute"},
            "gpu_launches": res["launches"],
            "clocks": res["clocks"],
        }
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(cfg, routing=args.routing, precision=args.precision)
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
