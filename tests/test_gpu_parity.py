"""CUDA path (through the C ABI) against the fp64 oracle, element by element.

Bars: routing indices and counts bit-exact (tokens with an oracle selection gap
below 1e-6 excluded); metadata bit-exact; `a` and y within relative Frobenius
error 1e-2 and max abs error 3e-2 * max|ref|.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (A_REL_FRO, assert_close_y, check_router_against_oracle, oracle_router, oracle_y_for_tokens,
                         order_mismatches, read_metadata, routing_mismatches, run_forward, run_router,
                         tile_sample_tokens)
from moe_expert_router_gb300 import binding as B
from moe_expert_router_gb300.workloads import (CONFIGS, MoEConfig, even_routing, generate,
                                               routing_with_counts)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()   # raises when libmoe.so is missing: there is no fallback
    torch.manual_seed(0)


def _cfg(T, H, I, E, k, **kw):
    return MoEConfig("case", T=T, H=H, I=I, E=E, k=k, **kw)


def _check_metadata(ws, shp, idx):
    counts, offsets, mt, perm, row_of = read_metadata(ws, shp)
    ref = oracle.routing_metadata(idx.cpu(), shp.E)
    np.testing.assert_array_equal(counts, ref.counts)
    np.testing.assert_array_equal(offsets, ref.offsets)
    np.testing.assert_array_equal(perm, ref.perm_slot)
    np.testing.assert_array_equal(row_of, ref.row_of)
    want_mt = np.concatenate([[0], np.cumsum((ref.counts + 255) // 256)])
    np.testing.assert_array_equal(mt, want_mt)
    return ref


# ------------------------------------------------------------------ routing metadata

def test_metadata_even_round_robin():
    T, k, E = 256, 2, 8
    idx, _ = even_routing(T, k, E, device=DEV)
    shp = B.shape(T, 128, 64, E, k)
    ws = B.new_workspace(shp)
    B.moe_routing_metadata(idx, shp, ws)
    ref = _check_metadata(ws, shp, idx)
    assert (ref.counts == T * k // E).all()
    assert B.moe_get_device_error(ws) == 0


@pytest.mark.parametrize("counts", [
    [0, 1, 127, 128, 129, 255, 256, 257, 0, 3],
    [512] + [0] * 7,
    [1] * 64,
])
def test_metadata_ragged_counts(counts):
    k = 1
    T = sum(counts)
    idx, _ = routing_with_counts(counts, T, k, seed=len(counts), device=DEV)
    shp = B.shape(T, 64, 64, len(counts), k)
    ws = B.new_workspace(shp)
    B.moe_routing_metadata(idx, shp, ws)
    _check_metadata(ws, shp, idx)


def test_metadata_large_zipf_like():
    T, k, E = 16384, 8, 128
    g = torch.Generator().manual_seed(1)
    p = torch.arange(1, E + 1, dtype=torch.float64) ** -1.2
    idx = torch.multinomial(p / p.sum(), T * k, replacement=True, generator=g).to(torch.int32)
    idx = idx.view(T, k).to(DEV)
    shp = B.shape(T, 64, 64, E, k)
    ws = B.new_workspace(shp)
    B.moe_routing_metadata(idx, shp, ws)
    _check_metadata(ws, shp, idx)


@pytest.mark.parametrize("T,k,E", [
    (8192, 8, 1024),    # 65,536 slots at the largest E
    (8193, 8, 256),     # a partial last chunk of slots
    (65536, 1, 3),      # few experts, 21,845 or more rows each
])
def test_metadata_many_slots(T, k, E):
    g = torch.Generator().manual_seed(T + E)
    idx = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32).to(DEV)
    shp = B.shape(T, 64, 64, E, k)
    ws = B.new_workspace(shp)
    B.moe_routing_metadata(idx, shp, ws)
    _check_metadata(ws, shp, idx)
    assert B.moe_get_device_error(ws) == 0


def test_metadata_bad_index_flags_and_drops():
    T, k, E = 100, 3, 7
    g = torch.Generator().manual_seed(2)
    idx = torch.randint(0, E, (T, k), generator=g, dtype=torch.int32)
    idx[3, 1] = -1
    idx[50, 0] = E
    idx[99, 2] = 1 << 20
    idx = idx.to(DEV)
    shp = B.shape(T, 64, 64, E, k)
    ws = B.new_workspace(shp)
    B.moe_routing_metadata(idx, shp, ws)
    ref = _check_metadata(ws, shp, idx)
    assert ref.dropped == 3
    assert B.moe_get_device_error(ws) & B.DEVERR_BAD_EXPERT_INDEX
    assert B.moe_get_device_error(ws) == 0   # reading clears the word


# ------------------------------------------------------------------ expert path

def _random_problem(cfg, seed, routing="random"):
    inp = generate(cfg, seed=seed, device=DEV)
    if routing == "random":
        g = torch.Generator().manual_seed(seed)
        idx = torch.randint(0, cfg.E, (cfg.T, cfg.k), generator=g, dtype=torch.int32).to(DEV)
        w = (torch.rand((cfg.T, cfg.k), generator=g) * 0.9 + 0.1).to(DEV)
    else:
        idx, w = routing
    return inp, idx, w


SHAPES = [
    # (T, H, I, E, k)
    (256, 128, 64, 8, 2),      # the tiny forward configuration
    (1, 64, 64, 4, 2),         # one token
    (37, 200, 136, 6, 3),      # K and N tails (H % 64 != 0, I % 128 != 0)
    (300, 328, 200, 5, 3),     # several row tiles per expert plus a ragged tail
    (1000, 512, 256, 16, 4),   # many units per CTA
    (550, 1000, 328, 4, 2),    # 257-320 rows per expert: a short last row tile, partial n-tiles
    (700, 520, 200, 4, 3),     # a full row tile before a short one, and experts without one
    (64, 64, 64, 1024, 32),    # the largest E and k: 2048 slots over 1024 experts
    (300, 256, 192, 1, 1),     # one expert, k = 1: a dense SwiGLU MLP over two row tiles
    (64, 256, 128, 128, 8),    # more experts than rows: many empty experts
    (33, 8, 8, 3, 2),          # smallest dimensions
]



@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_stage1_a_rows(shape):
    T, H, I, E, k = shape
    cfg = _cfg(T, H, I, E, k)
    inp, idx, w = _random_problem(cfg, seed=T + H)
    y, ws, a = run_forward(inp, idx, w, cfg, staged=True)
    shp = B.shape(T, H, I, E, k)
    ref_md = _check_metadata(ws, shp, idx)
    _, a_ref, _ = oracle.expert_forward(inp["x"].cpu(), idx.cpu(), w.cpu().double(),
                                        inp["w1"].cpu(), inp["w2"].cpu(), want_a=True)
    n = int(ref_md.offsets[-1])
    rel, _ = assert_close_y(a[:n], a_ref[ref_md.perm_slot], what="a (routed order)")
    # a is one bf16 rounding (relative Frobenius ~1e-3) plus the SiLU's tanh
    # approximation away from the fp64 value: a tighter bound than the outputs'
    assert rel <= A_REL_FRO, f"a: relative Frobenius error {rel:.3e} > {A_REL_FRO}"
    assert B.moe_get_device_error(ws) == 0


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("staged", [False, True], ids=["one_shot", "staged"])
def test_expert_path_y(shape, staged):
    T, H, I, E, k = shape
    cfg = _cfg(T, H, I, E, k)
    inp, idx, w = _random_problem(cfg, seed=7 * T + E)
    y, ws, _ = run_forward(inp, idx, w, cfg, staged=staged)
    y_ref = oracle.expert_forward(inp["x"].cpu(), idx.cpu(), w.cpu().double(), inp["w1"].cpu(),
                                  inp["w2"].cpu())
    assert_close_y(y, y_ref)
    assert B.moe_get_device_error(ws) == 0


def test_even_routing_forward():
    cfg = CONFIGS["tiny"]
    idx, w = even_routing(cfg.T, cfg.k, cfg.E, device=DEV)
    inp, idx, w = _random_problem(cfg, seed=3, routing=(idx, w))
    y, ws, _ = run_forward(inp, idx, w, cfg)
    y_ref = oracle.expert_forward(inp["x"].cpu(), idx.cpu(), w.cpu().double(), inp["w1"].cpu(),
                                  inp["w2"].cpu())
    assert_close_y(y, y_ref)


def test_unused_experts_poisoned_with_nan():
    cfg = _cfg(200, 256, 128, 12, 2)
    inp, idx, w = _random_problem(cfg, seed=5)
    idx = idx % 7                                    # experts 7..11 get no rows
    y_ref = oracle.expert_forward(inp["x"].cpu(), idx.cpu(), w.cpu().double(), inp["w1"].cpu(),
                                  inp["w2"].cpu())
    inp["w1"][7:] = float("nan")
    inp["w2"][7:] = float("nan")
    y, ws, _ = run_forward(inp, idx, w, cfg)
    assert torch.isfinite(y.float()).all()
    assert_close_y(y, y_ref)


def test_dropped_slots_contribute_nothing():
    cfg = _cfg(64, 128, 64, 4, 2)
    inp, idx, w = _random_problem(cfg, seed=9)
    bad = idx.clone()
    bad[0, 0] = -1
    bad[5, 1] = cfg.E
    bad[7] = -3                                     # a token with every slot dropped
    y, ws, _ = run_forward(inp, bad, w, cfg)
    assert B.moe_get_device_error(ws) & B.DEVERR_BAD_EXPERT_INDEX
    y_ref = oracle.expert_forward(inp["x"].cpu(), bad.cpu(), w.cpu().double(), inp["w1"].cpu(),
                                  inp["w2"].cpu())
    assert_close_y(y, y_ref)
    assert (y[7] == 0).all()


def test_zero_tokens_is_a_no_op():
    shp = B.shape(0, 64, 64, 4, 2)
    ws = B.new_workspace(shp)
    x = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    w1 = torch.zeros((4, 128, 64), dtype=torch.bfloat16, device=DEV)
    w2 = torch.zeros((4, 64, 64), dtype=torch.bfloat16, device=DEV)
    idx = torch.empty((0, 2), dtype=torch.int32, device=DEV)
    w = torch.empty((0, 2), dtype=torch.float32, device=DEV)
    y = torch.empty((0, 64), dtype=torch.bfloat16, device=DEV)
    n0 = B.moe_kernel_launch_count()
    B.moe_forward(x, idx, w, w1, w2, shp, y, ws)
    B.moe_router(x, torch.zeros((4, 64), device=DEV), shp, B.router_cfg(), idx, w, ws)
    torch.cuda.synchronize()
    assert B.moe_kernel_launch_count() == n0


def test_argument_errors_are_synchronous():
    cfg = _cfg(16, 64, 64, 4, 2)
    inp, idx, w = _random_problem(cfg, seed=1)
    shp = B.shape(16, 64, 64, 4, 2)
    ws = B.new_workspace(shp)
    y = torch.empty((16, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(B.MoEError) as e:
        B.moe_forward(inp["x"], idx, w, inp["w1"], inp["w2"], shp, y, ws[:1024])
    assert e.value.status == 4
    bad = B.shape(16, 60, 64, 4, 2)       # H not a multiple of 8
    with pytest.raises(B.MoEError) as e:
        B.moe_forward(inp["x"], idx, w, inp["w1"], inp["w2"], bad, y, ws)
    assert e.value.status == 2


def test_graph_capture_replays():
    """The path is sync-free: capture router + expert path in a CUDA graph and replay."""
    cfg = CONFIGS["tiny"]
    inp = generate(cfg, seed=4, device=DEV)
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    ws = B.new_workspace(shp)
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
    rcfg = B.router_cfg()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # warm-up outside capture (per-device set-up)
        B.moe_router(inp["x"], inp["w_r"], shp, rcfg, idx, w, ws)
        B.moe_forward(inp["x"], idx, w, inp["w1"], inp["w2"], shp, y, ws)
    torch.cuda.current_stream().wait_stream(s)
    y_eager = y.clone()
    y.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.moe_router(inp["x"], inp["w_r"], shp, rcfg, idx, w, ws)
        B.moe_forward(inp["x"], idx, w, inp["w1"], inp["w2"], shp, y, ws)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, y_eager)


# ------------------------------------------------------------------ router

ROUTER_CASES = {
    "tiny_softmax": CONFIGS["tiny"],
    "softmax_e64_k6": _cfg(1024, 512, 64, 64, 6),
    "sigmoid_groups_bias": _cfg(1024, 512, 64, 64, 8, score="sigmoid", scale=2.5, n_group=8,
                                topk_group=4, group_topn=2, sel_bias=True),
    "sigmoid_groups_e256": _cfg(512, 256, 64, 256, 8, score="sigmoid", scale=2.5, n_group=8,
                                topk_group=4, group_topn=2, sel_bias=True),
    "zipf_offset_e128": _cfg(2048, 256, 64, 128, 8, zipf_s=1.2),
    # groups of exactly 32 experts (the warp-wide group sums): the best one per group,
    # and 16 groups of E = 512
    "softmax_groups_e128_top1": _cfg(700, 256, 64, 128, 6, n_group=4, topk_group=2, group_topn=1),
    "sigmoid_groups_e512": _cfg(300, 256, 64, 512, 8, score="sigmoid", scale=2.5, n_group=16,
                                topk_group=4, group_topn=2, sel_bias=True),
    "e1024_k32": _cfg(64, 128, 64, 1024, 32),
    "e3_k3": _cfg(50, 64, 64, 3, 3),
    # E between 32 and 64 (each weight part padded to 64 accumulator columns), a K tail
    # (H = 200) and a partial 256-token tile
    "e40_k4_ktail": _cfg(300, 200, 64, 40, 4),
}


@pytest.mark.parametrize("name", sorted(ROUTER_CASES))
def test_router_vs_oracle(name):
    cfg = ROUTER_CASES[name]
    inp = generate(cfg, seed=11, device=DEV)
    check_router_against_oracle(inp, cfg)


# ------------------------------------------------------------------ full sizes

FULL = ["mid", "large_group", "zipf_prefill", "zipf_decode", "train"]
# workloads whose every token is compared with the oracle (the others: a sample
# that reaches every (expert, 256-row tile) work unit)
ALL_TOKENS = {"mid", "zipf_decode"}


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_full_size_config(name):
    """Full-size workload in the bench's launch configuration (staged C-ABI calls):
    routing of every token against the oracle (sets, and the best-first order of
    tokens without near-ties); y of every token (mid, zipf_decode) or of the tokens
    of the first, middle and last rows of every 256-row tile of every expert, plus
    the first, last and middle tokens and tokens of the most and least loaded
    experts; stage 1's a rows of the sampled tokens' slots."""
    cfg = CONFIGS[name]
    inp = generate(cfg, seed=0, device=DEV)
    idx, w, aux, ws = run_router(inp, cfg)
    ref = oracle_router(inp, cfg)
    n, bad, excluded = routing_mismatches(idx, ref, cfg)
    assert not bad, f"{len(bad)} of {n} tokens routed differently, e.g. {bad[:5]}"
    n_ord, bad_ord = order_mismatches(idx, ref, excluded, inp.get("sel_bias"))
    assert n_ord > 0 and not bad_ord, f"{len(bad_ord)} of {n_ord} tokens not best first, e.g. {bad_ord[:5]}"
    y, ws, a = run_forward(inp, idx, w, cfg, ws=ws, staged=True)
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    counts, offsets, _, perm, row_of = read_metadata(ws, shp)
    ref_counts = np.bincount(ref.topk_idx.reshape(-1), minlength=cfg.E)
    if not excluded.any():
        np.testing.assert_array_equal(counts, ref_counts)
    else:
        # an excluded (near-tie) token may move one row between the expert the
        # oracle chose and the one the GPU chose: credit both
        gx = idx.cpu().numpy()[excluded]
        touched = (np.bincount(ref.topk_idx[excluded].reshape(-1), minlength=cfg.E) +
                   np.bincount(gx.reshape(-1), minlength=cfg.E))
        assert (np.abs(counts - ref_counts) <= touched).all()
    assert int(offsets[-1]) == cfg.T * cfg.k
    if cfg.score == "softmax":
        assert abs(aux.item() - ref.aux) <= 1e-4 * abs(ref.aux) + excluded.sum() * 4.0 / cfg.T
    g = idx.cpu().numpy()
    big = int(np.argmax(counts))
    small = int(np.argmin(np.where(counts > 0, counts, np.iinfo(np.int32).max)))
    t_big = int(np.nonzero((g == big).any(1))[0][-1])
    t_small = int(np.nonzero((g == small).any(1))[0][0])
    extra = {0, 1, cfg.T // 2, cfg.T - 1, t_big, t_small}
    if name in ALL_TOKENS:
        tokens = list(range(cfg.T))
    else:
        tokens = tile_sample_tokens(counts, offsets, perm, cfg.k, extra)
    y_ref, a_ref = oracle_y_for_tokens(inp, idx, w, tokens, want_a=True)
    assert_close_y(y[tokens], y_ref, what=f"{name} y[{len(tokens)} tokens]")
    # stage 1 alone: the a rows of those tokens' slots, in routed order on the GPU
    slots = (np.asarray(tokens)[:, None] * cfg.k + np.arange(cfg.k)[None, :]).reshape(-1)
    rows = torch.as_tensor(row_of[slots], dtype=torch.long)
    rel, _ = assert_close_y(a[rows.to(DEV)], a_ref, what=f"{name} a[{len(slots)} slots]")
    assert rel <= A_REL_FRO, f"a: relative Frobenius error {rel:.3e} > {A_REL_FRO}"
    assert torch.isfinite(y.float()).all()
    assert B.moe_get_device_error(ws) == 0


# ------------------------------------------------------------------ routing from given logits

@pytest.mark.parametrize("case", [
    dict(T=512, E=64, k=6),
    dict(T=300, E=256, k=8, score="sigmoid", scale=2.5, n_group=8, topk_group=4, group_topn=2,
         sel_bias=True),
    dict(T=64, E=128, k=8, zipf_s=1.2),
    dict(T=40, E=1024, k=32, normalize=False),
])
def test_route_logits_uniform_mode(case):
    """The `uniform` force-balance mode: N(0,1) logits routed like the router's own
    logits. Oracle: its router with x = identity (bf16) and W_r = logits^T, which
    gives exactly those logits."""
    case = dict(case)
    T, E, k = case.pop("T"), case.pop("E"), case.pop("k")
    zipf = case.pop("zipf_s", None)
    cfg = _cfg(T, 64, 64, E, k, zipf_s=zipf, **case)
    g = torch.Generator().manual_seed(T + E)
    logits = torch.randn((T, E), generator=g, dtype=torch.float32)
    inp = generate(cfg, seed=1)                        # selection bias / Zipf offsets only
    shp = B.shape(T, 64, 64, E, k)
    ws = B.new_workspace(shp)
    idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    aux = torch.zeros((1,), dtype=torch.float32, device=DEV)
    off = inp["logit_offset"].to(DEV) if inp["logit_offset"] is not None else None
    bias = inp["sel_bias"].to(DEV) if inp["sel_bias"] is not None else None
    B.moe_route_logits(logits.to(DEV), shp, B.router_cfg(cfg.score, cfg.normalize, cfg.scale, cfg.n_group,
                                                          cfg.topk_group, cfg.group_topn),
                       idx, w, ws, aux=aux, logit_offset=off, sel_bias=bias)
    assert B.moe_get_device_error(ws) == 0
    eye = torch.eye(T, dtype=torch.float32).to(torch.bfloat16)
    ref = oracle.router(eye, logits.T.contiguous(), k, score=cfg.score, normalize=cfg.normalize,
                        scale=cfg.scale, n_group=cfg.n_group, topk_group=cfg.topk_group,
                        group_topn=cfg.group_topn, logit_offset=inp["logit_offset"],
                        sel_bias=inp["sel_bias"])
    n, bad, excluded = routing_mismatches(idx, ref, cfg)
    assert not bad, f"{len(bad)} of {n} tokens routed differently"
    keep = ~excluded
    gi, gw = idx.cpu().numpy(), w.cpu().double().numpy()
    for t in np.nonzero(keep)[0]:
        order = np.argsort(gi[t])
        ro = np.argsort(ref.topk_idx[t])
        np.testing.assert_allclose(gw[t][order], ref.topk_w[t][ro], rtol=2e-5, atol=1e-7)
    if keep.all():
        assert abs(aux.item() - ref.aux) <= 1e-4 * max(1.0, abs(ref.aux))
