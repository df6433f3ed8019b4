"""Pins of the fp64 oracle to facts outside itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError if
the oracle disagrees with something the pages or mathematics fix:

* hand-worked examples whose expected values are closed forms (tests/golden);
* the 'even' round-robin routing of the MegaMoE guide (section "Router force
  load balancing"), whose metadata has a closed form;
* a dense SwiGLU MLP written with torch fp64 library ops (E = 1, k = 1);
* brute force by sorting (top-k, group-limited top-k, stable permutation);
* a grouped (per-expert batched) re-formulation of the expert path;
* invariants: weight sums, count sums, NaN-poisoned unused experts,
  token-permutation equivariance, linearity in w2, dropped slots, aux limits;
* for the backward: torch fp64 autograd through a forward written here with
  library ops, the forward oracle's own o rows, exact scaling in dY, zero
  gradients for unused experts and dropped slots;
* for MXFP8: torch's float8_e4m3fn conversion (round to nearest even), the
  round trip of every finite E4M3 code under several block scales, the
  shared-exponent rule on chosen maxima, and the MX forward as a composition
  of the bf16 oracle (on dequantized inputs), the quantizer and torch fp64
  matmuls; the MX backward against the bf16 backward where MXFP8 holds the
  forward's inputs exactly, against the MX forward's a, and its weight
  gradients as a composition of the quantizer (along the expert's rows) and
  fp64 matmuls.

tests/test_oracle_mutants.py compiles deliberately broken copies of the oracle
and checks that every one of them fails at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _sigmoid(z):
    return 1.0 / (1.0 + math.exp(-z))


def _silu(z):
    return z * _sigmoid(z)


_CLOSED_FORM_NS = {"sigmoid": _sigmoid, "silu": _silu, "exp": math.exp, "log": math.log}


def _closed(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, dict(_CLOSED_FORM_NS)))


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(a):
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _rand_bf16(gen, shape, std=1.0):
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)


# --------------------------------------------------------------------------- worked examples

def pin_worked_example_softmax(orc):
    g = _golden("worked_example_softmax.json")
    sh = g["shape"]
    T, H, I, E, k = sh["T"], sh["H"], sh["I"], sh["E"], sh["k"]
    x = _bf16(g["x"])
    w_r = np.eye(E, H, dtype=np.float32)
    w1 = np.zeros((E, 2 * I, H), np.float32)
    w2 = np.zeros((E, H, I), np.float32)
    for e in range(E):
        w1[e, 0, e] = 1.0      # gate row = onehot(e)
        w1[e, 1, :] = 1.0      # up row = ones
        w2[e, e, 0] = 1.0      # down column = onehot(e)
    r = orc.router(x, w_r, k, score="softmax", normalize=True)
    ex = g["expected"]
    assert r.topk_idx.tolist() == ex["topk_idx"], r.topk_idx
    want_w = np.array([[_closed(v) for v in row] for row in ex["topk_w"]])
    np.testing.assert_allclose(r.topk_w, want_w, rtol=1e-12, atol=1e-14)
    y = orc.expert_forward(x, r.topk_idx, r.topk_w, _bf16(w1), _bf16(w2))
    want_y = np.array([[_closed(v) for v in row] for row in ex["y"]])
    np.testing.assert_allclose(y, want_y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y[0], ex["y_numeric_t0"], rtol=1e-9, atol=1e-9)
    md = orc.routing_metadata(r.topk_idx, E)
    assert md.counts.tolist() == ex["counts"]
    # aux from its closed form: E * sum_e (c_e / (T k)) * mean_t softmax(x_t)_e
    xs = np.asarray(g["x"], dtype=np.float64)
    P = [sum(math.exp(xs[t, e]) / sum(math.exp(v) for v in xs[t]) for t in range(T)) / T
         for e in range(E)]
    want_aux = E * sum(c / (T * k) * P[e] for e, c in enumerate(ex["counts"]))
    assert abs(r.aux - want_aux) < 1e-12, (r.aux, want_aux)
    assert abs(r.aux - 1.1847241832) < 1e-9, r.aux


def pin_worked_example_group(orc):
    g = _golden("worked_example_group.json")
    sh = g["shape"]
    E, H, k = sh["E"], sh["H"], sh["k"]
    x = _bf16(g["x"])
    w_r = np.eye(E, H, dtype=np.float32)
    bias = np.asarray(g["bias"], np.float32)
    r = orc.router(x, w_r, k, score="sigmoid", normalize=True, scale=sh["scale"],
                   n_group=sh["n_group"], topk_group=sh["topk_group"],
                   group_topn=sh["group_topn"], sel_bias=bias)
    ex = g["expected"]
    assert r.topk_idx.tolist() == ex["topk_idx"], r.topk_idx
    want_w = np.array([[_closed(v) for v in row] for row in ex["topk_w"]])
    np.testing.assert_allclose(r.topk_w, want_w, rtol=1e-12)
    np.testing.assert_allclose(r.topk_w.sum(), 2.5, rtol=1e-12)
    np.testing.assert_allclose(r.group_gap[0], _closed(ex["group_gap"]), rtol=1e-12)
    np.testing.assert_allclose(r.sel_gap[0], _closed(ex["sel_gap"]), rtol=1e-12)


# --------------------------------------------------------------------------- special cases

def pin_dense_swiglu(orc):
    """E = 1, k = 1: the layer is a dense SwiGLU MLP; compare with torch fp64 ops."""
    gen = torch.Generator().manual_seed(11)
    T, H, I = 16, 48, 24
    x = _rand_bf16(gen, (T, H))
    w1 = _rand_bf16(gen, (1, 2 * I, H), H ** -0.5)
    w2 = _rand_bf16(gen, (1, H, I), I ** -0.5)
    idx = torch.zeros((T, 1), dtype=torch.int32)
    w = torch.ones((T, 1), dtype=torch.float64)
    y = orc.expert_forward(x, idx, w, w1, w2)
    X = x.double()
    G, U = w1[0, :I].double(), w1[0, I:].double()
    ref = (torch.nn.functional.silu(X @ G.T) * (X @ U.T)) @ w2[0].double().T
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-10, atol=1e-10)
    # the router with one expert: the weight is exactly 1 (normalised), 0.5 (sigmoid(0) unnormalised)
    r = orc.router(x, np.zeros((1, H), np.float32), 1)
    assert (r.topk_idx == 0).all() and np.allclose(r.topk_w, 1.0)
    r = orc.router(x, np.zeros((1, H), np.float32), 1, score="sigmoid", normalize=False)
    assert np.allclose(r.topk_w, 0.5)


def pin_logit_offset(orc):
    """W_r = 0 and offset = ln p: softmax scores equal p exactly."""
    E = 16
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.2
    p /= p.sum()
    off = np.log(p).astype(np.float32)
    x = _bf16(np.ones((3, 8)))
    r = orc.router(x, np.zeros((E, 8), np.float32), 4, logit_offset=off)
    pe = np.exp(off.astype(np.float64))
    pe /= pe.sum()
    np.testing.assert_allclose(r.scores, np.tile(pe, (3, 1)), rtol=1e-12)
    assert r.topk_idx.tolist() == [[0, 1, 2, 3]] * 3


# --------------------------------------------------------------------------- metadata

def pin_even_metadata(orc):
    for case in _golden("even_routing.json")["cases"]:
        T, k, E = case["T"], case["k"], case["E"]
        idx = np.array([[(t * k + j) % E for j in range(k)] for t in range(T)], np.int32)
        assert idx.tolist() == case["topk_idx"]
        md = orc.routing_metadata(idx, E)
        assert md.counts.tolist() == case["counts"]
        assert md.offsets.tolist() == case["offsets"]
        assert md.perm_slot.tolist() == case["perm_slot"]
    # closed form at a larger size: E | T k, so c_e = T k / E and row i of e is slot e + i E
    T, k, E = 96, 6, 16
    idx = np.array([[(t * k + j) % E for j in range(k)] for t in range(T)], np.int32)
    md = orc.routing_metadata(idx, E)
    c = T * k // E
    assert (md.counts == c).all()
    assert md.offsets.tolist() == [e * c for e in range(E + 1)]
    want = [e + i * E for e in range(E) for i in range(c)]
    assert md.perm_slot.tolist() == want
    s = np.arange(T * k)
    assert (md.row_of == (s % E) * c + s // E).all()


def pin_metadata_sort(orc):
    """Stable permutation = sort of (expert, slot); invalid indices dropped."""
    rng = np.random.default_rng(5)
    T, k, E = 77, 3, 9
    idx = rng.integers(-1, E + 1, size=(T, k)).astype(np.int32)
    md = orc.routing_metadata(idx, E)
    flat = idx.reshape(-1)
    valid = [(int(e), s) for s, e in enumerate(flat) if 0 <= e < E]
    want = [s for _, s in sorted(valid)]
    assert md.perm_slot.tolist() == want
    assert md.dropped == T * k - len(valid)
    assert md.counts.sum() == len(valid)
    assert md.counts.tolist() == [int((flat == e).sum()) for e in range(E)]
    for r, s in enumerate(want):
        assert md.row_of[s] == r
    assert all(md.row_of[s] == -1 for s, e in enumerate(flat) if not 0 <= e < E)


# --------------------------------------------------------------------------- router

def pin_topk_sort(orc):
    """Scores equal torch softmax / sigmoid of fp64 logits; top-k equals a sort."""
    gen = torch.Generator().manual_seed(3)
    T, H, E, k = 40, 32, 12, 3
    x = _rand_bf16(gen, (T, H))
    w_r = torch.randn((E, H), generator=gen) * 0.3
    logits = x.double() @ w_r.double().T
    for score in ("softmax", "sigmoid"):
        r = orc.router(x, w_r, k, score=score, normalize=(score == "softmax"))
        ref = torch.softmax(logits, dim=-1) if score == "softmax" else torch.sigmoid(logits)
        np.testing.assert_allclose(r.scores, ref.numpy(), rtol=1e-12, atol=1e-15)
        for t in range(T):
            order = sorted(range(E), key=lambda e: (-r.scores[t, e], e))
            assert r.topk_idx[t].tolist() == order[:k]
            sw = r.scores[t, order[:k]]
            want = sw / sw.sum() if score == "softmax" else sw
            np.testing.assert_allclose(r.topk_w[t], want, rtol=1e-12)
            np.testing.assert_allclose(r.sel_gap[t], r.scores[t, order[k - 1]] - r.scores[t, order[k]],
                                       rtol=1e-12, atol=1e-15)
    # exact ties: all scores equal -> the lowest indices, in order
    r = orc.router(x[:2], np.zeros((E, H), np.float32), k)
    assert r.topk_idx.tolist() == [list(range(k))] * 2


def pin_group_sort(orc):
    """Group-limited selection equals sorting groups, then eligible experts."""
    gen = torch.Generator().manual_seed(4)
    T, H, E, k, G, KG, N = 30, 16, 16, 3, 4, 2, 2
    x = _rand_bf16(gen, (T, H))
    w_r = torch.randn((E, H), generator=gen) * 0.5
    bias = torch.randn((E,), generator=gen) * 0.1
    r = orc.router(x, w_r, k, score="sigmoid", normalize=True, scale=2.5, n_group=G,
                   topk_group=KG, group_topn=N, sel_bias=bias)
    s = torch.sigmoid(x.double() @ w_r.double().T).numpy()
    np.testing.assert_allclose(r.scores, s, rtol=1e-12)
    sel = s + bias.double().numpy()[None, :]
    gs = E // G
    for t in range(T):
        gsc = [sum(sorted(sel[t, g * gs:(g + 1) * gs])[-N:]) for g in range(G)]
        gorder = sorted(range(G), key=lambda g: (-gsc[g], g))
        kept = set(gorder[:KG])
        elig = [e for e in range(E) if e // gs in kept]
        order = sorted(elig, key=lambda e: (-sel[t, e], e))
        assert r.topk_idx[t].tolist() == order[:k], (t, r.topk_idx[t], order[:k])
        sw = s[t, order[:k]]
        np.testing.assert_allclose(r.topk_w[t], 2.5 * sw / sw.sum(), rtol=1e-12)
        np.testing.assert_allclose(r.group_gap[t], gsc[gorder[KG - 1]] - gsc[gorder[KG]], rtol=1e-9,
                                   atol=1e-15)


def pin_weights_sum(orc):
    gen = torch.Generator().manual_seed(6)
    x = _rand_bf16(gen, (50, 24))
    w_r = torch.randn((32, 24), generator=gen) * 0.2
    r = orc.router(x, w_r, 4)
    np.testing.assert_allclose(r.topk_w.sum(1), 1.0, rtol=1e-12)
    r = orc.router(x, w_r, 4, score="sigmoid", scale=2.5, n_group=8, topk_group=3,
                   sel_bias=torch.randn((32,), generator=gen) * 0.01)
    np.testing.assert_allclose(r.topk_w.sum(1), 2.5, rtol=1e-12)
    for t in range(50):
        assert len(set(r.topk_idx[t].tolist())) == 4   # distinct experts


def pin_aux_limits(orc):
    """Uniform scores give aux = 1 whatever the counts; all mass on one expert gives E."""
    E, H, T = 8, 16, 20
    x = _bf16(np.ones((T, H)))
    r = orc.router(x, np.zeros((E, H), np.float32), 2)
    assert abs(r.aux - 1.0) < 1e-12, r.aux
    w_r = np.zeros((E, H), np.float32)
    w_r[5, :] = 4.0                      # logit 64 for expert 5: softmax ~ onehot(5)
    r = orc.router(x, w_r, 1)
    assert (r.topk_idx == 5).all()
    assert abs(r.aux - E) < 1e-12 * E, r.aux
    # balanced one-hot routing: token t -> expert t % E with dominant logits
    xs = np.zeros((16, E), np.float32)
    for t in range(16):
        xs[t, t % E] = 1.0
    r = orc.router(_bf16(xs), np.eye(E, dtype=np.float32) * 64.0, 1)
    assert r.topk_idx[:, 0].tolist() == [t % E for t in range(16)]
    assert abs(r.aux - 1.0) < 1e-9, r.aux


# --------------------------------------------------------------------------- expert path

def _problem(seed, T=24, H=40, I=16, E=6, k=3, std=1.0):
    gen = torch.Generator().manual_seed(seed)
    x = _rand_bf16(gen, (T, H), std)
    w1 = _rand_bf16(gen, (E, 2 * I, H), H ** -0.5)
    w2 = _rand_bf16(gen, (E, H, I), I ** -0.5)
    idx = torch.randint(0, E, (T, k), generator=gen, dtype=torch.int32)
    w = torch.rand((T, k), generator=gen, dtype=torch.float64)
    return x, w1, w2, idx, w


def pin_grouped_formulation(orc):
    """Per-expert batched formulation (gather rows, two matmuls, scatter-add) agrees."""
    x, w1, w2, idx, w = _problem(7)
    T, H = x.shape
    E, twoI, _ = w1.shape
    I = twoI // 2
    y, a, o = orc.expert_forward(x, idx, w, w1, w2, want_a=True, want_o=True)
    ref = torch.zeros((T, H), dtype=torch.float64)
    flat = idx.reshape(-1).long()
    for e in range(E):
        slots = torch.nonzero(flat == e).flatten()
        if slots.numel() == 0:
            continue
        toks = slots // idx.shape[1]
        Xe = x[toks].double()
        He = Xe @ w1[e].double().T
        Ae = torch.nn.functional.silu(He[:, :I]) * He[:, I:]
        Oe = Ae @ w2[e].double().T
        np.testing.assert_allclose(a[slots.numpy()], Ae.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(o[slots.numpy()], Oe.numpy(), rtol=1e-10, atol=1e-12)
        ref.index_add_(0, toks, Oe * w.reshape(-1)[slots].unsqueeze(1))
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-10, atol=1e-12)


def pin_nan_unused_experts(orc):
    x, w1, w2, idx, w = _problem(8, E=8)
    idx = idx % 5                                   # experts 5..7 never used
    y = orc.expert_forward(x, idx, w, w1, w2)
    w1p, w2p = w1.clone(), w2.clone()
    w1p[5:] = float("nan")
    w2p[5:] = float("nan")
    yp = orc.expert_forward(x, idx, w, w1p, w2p)
    assert np.isfinite(yp).all()
    np.testing.assert_array_equal(y, yp)


def pin_token_permutation(orc):
    x, w1, w2, idx, w = _problem(9)
    y = orc.expert_forward(x, idx, w, w1, w2)
    p = torch.randperm(x.shape[0], generator=torch.Generator().manual_seed(1))
    yp = orc.expert_forward(x[p], idx[p], w[p], w1, w2)
    np.testing.assert_allclose(yp, y[p.numpy()], rtol=1e-13, atol=1e-13)


def pin_linear_in_w2(orc):
    x, w1, w2, idx, w = _problem(10)
    y = orc.expert_forward(x, idx, w, w1, w2)
    y2 = orc.expert_forward(x, idx, w, w1, w2 * 2)       # exact in bf16
    yn = orc.expert_forward(x, idx, w, w1, -w2)
    np.testing.assert_allclose(y2, 2 * y, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(yn, -y, rtol=1e-13, atol=1e-13)
    # linear in the routing weights too, and a zero weight removes the contribution
    yw = orc.expert_forward(x, idx, 3 * w, w1, w2)
    np.testing.assert_allclose(yw, 3 * y, rtol=1e-12, atol=1e-12)


def pin_dropped_slots(orc):
    x, w1, w2, idx, w = _problem(12)
    bad = idx.clone()
    bad[0, 0] = -1
    bad[3, 1] = w1.shape[0]
    y = orc.expert_forward(x, bad, w, w1, w2)
    w0 = w.clone()
    w0[0, 0] = 0.0
    w0[3, 1] = 0.0
    ref = orc.expert_forward(x, idx, w0, w1, w2)
    np.testing.assert_allclose(y, ref, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------- backward

def _torch_expert_forward(x, idx, w, w1, w2):
    """Grouped expert forward in torch fp64, differentiable in x, w, w1 and w2."""
    T, H = x.shape
    E, twoI, _ = w1.shape
    I = twoI // 2
    k = idx.shape[1]
    flat = idx.reshape(-1).long()
    y = torch.zeros((T, H), dtype=torch.float64)
    for e in range(E):
        slots = torch.nonzero(flat == e).flatten()
        if slots.numel() == 0:
            continue
        toks = slots // k
        he = x[toks] @ w1[e].T
        ae = torch.nn.functional.silu(he[:, :I]) * he[:, I:]
        oe = ae @ w2[e].T
        y = y.index_add(0, toks, oe * w.reshape(-1)[slots].unsqueeze(1))
    return y


def _leaf(t):
    return t.detach().double().clone().requires_grad_(True)


def pin_backward_autograd_expert(orc):
    """dX, dW1, dW2 and d(routing weight) equal torch autograd of <dY, y>."""
    x, w1, w2, idx, w = _problem(20, E=7)
    idx = idx % 6                                   # expert 6 unused
    gen = torch.Generator().manual_seed(21)
    dy = _rand_bf16(gen, x.shape)
    xd, w1d, w2d, wd = _leaf(x), _leaf(w1), _leaf(w2), _leaf(w)
    y = _torch_expert_forward(xd, idx, wd, w1d, w2d)
    (y * dy.double()).sum().backward()
    b = orc.expert_backward(x, idx, w, w1, w2, dy)
    np.testing.assert_allclose(b.dx, xd.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(b.dw1, w1d.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(b.dw2, w2d.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(b.dtopk_w, wd.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert not b.dw1[6].any() and not b.dw2[6].any()


def pin_backward_routing_weight_is_o_dot_dy(orc):
    """y is linear in each routing weight: its gradient is <dY_t, o_slot> of the forward."""
    x, w1, w2, idx, w = _problem(22)
    dy = _rand_bf16(torch.Generator().manual_seed(23), x.shape)
    _, _, o = orc.expert_forward(x, idx, w, w1, w2, want_o=True)
    b = orc.expert_backward(x, idx, w, w1, w2, dy, want_dw=False)
    T, k = idx.shape
    want = np.einsum("tkh,th->tk", o.reshape(T, k, -1), dy.double().numpy())
    np.testing.assert_allclose(b.dtopk_w, want, rtol=1e-10, atol=1e-12)


def pin_backward_scaling_and_drops(orc):
    """Doubling dY doubles every gradient exactly; dropped slots give nothing."""
    x, w1, w2, idx, w = _problem(24)
    dy = _rand_bf16(torch.Generator().manual_seed(25), x.shape)
    b1 = orc.expert_backward(x, idx, w, w1, w2, dy)
    b2 = orc.expert_backward(x, idx, w, w1, w2, dy * 2)
    for f in ("dx", "dw1", "dw2", "dtopk_w"):
        np.testing.assert_array_equal(getattr(b2, f), 2 * getattr(b1, f))
    bad = idx.clone()
    bad[1, 0] = -1
    bad[5, 2] = w1.shape[0]
    w0 = w.clone()
    w0[1, 0] = 0.0
    w0[5, 2] = 0.0
    bd = orc.expert_backward(x, bad, w, w1, w2, dy)
    b0 = orc.expert_backward(x, idx, w0, w1, w2, dy)
    assert bd.dtopk_w[1, 0] == 0.0 and bd.dtopk_w[5, 2] == 0.0
    for f in ("dx", "dw1", "dw2"):
        np.testing.assert_allclose(getattr(bd, f), getattr(b0, f), rtol=1e-13, atol=1e-13)


def _torch_router_weights(xd, wrd, off, idx, score, normalize, scale):
    logits = xd @ wrd.T
    if off is not None:
        logits = logits + torch.as_tensor(off, dtype=torch.float64)
    logits.retain_grad()
    s = torch.softmax(logits, dim=1) if score == "softmax" else torch.sigmoid(logits)
    chosen = torch.gather(s, 1, idx.long())
    if normalize:
        chosen = chosen / chosen.sum(dim=1, keepdim=True)
    return logits, chosen * scale


def pin_backward_autograd_router(orc):
    """Logit, dX and dW_r gradients of the routing weights equal torch autograd.

    The selection is held fixed (it is piecewise constant); the selection bias
    and the group limit steer it but must not enter the gradient.
    """
    gen = torch.Generator().manual_seed(26)
    T, H, E, k = 20, 24, 16, 4
    x = _rand_bf16(gen, (T, H))
    w_r = torch.randn((E, H), generator=gen, dtype=torch.float32) * 0.3
    off = (torch.randn((E,), generator=gen, dtype=torch.float32) * 0.5).numpy()
    bias = (torch.randn((E,), generator=gen, dtype=torch.float32) * 0.05).numpy()
    for score, normalize, scale in (("softmax", True, 2.5), ("softmax", False, 1.75),
                                    ("sigmoid", True, 2.5), ("sigmoid", False, 1.75)):
        r = orc.router(x, w_r, k, score=score, normalize=normalize, scale=scale, n_group=4,
                       topk_group=2, group_topn=2, logit_offset=off, sel_bias=bias)
        idx = torch.as_tensor(r.topk_idx)
        dtw = torch.randn((T, k), generator=gen, dtype=torch.float64)
        xd, wrd = _leaf(x), _leaf(w_r)
        logits, wt = _torch_router_weights(xd, wrd, off, idx, score, normalize, scale)
        np.testing.assert_allclose(r.topk_w, wt.detach().numpy(), rtol=1e-12, atol=1e-14)
        (wt * dtw).sum().backward()
        b = orc.router_backward(x, w_r, r.topk_idx, r.topk_w, dtw.numpy(), score=score,
                                normalize=normalize, scale=scale, logit_offset=off)
        np.testing.assert_allclose(b.dlogits, logits.grad.numpy(), rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(b.dx_add, xd.grad.numpy(), rtol=1e-10, atol=1e-13)
        np.testing.assert_allclose(b.dw_r, wrd.grad.numpy(), rtol=1e-10, atol=1e-13)


def _grid_bf16(gen, shape, step=1.0 / 64, lim=1.5):
    """bf16 values on a grid of ``step`` (exact in bf16, so v +- step is too)."""
    v = torch.round(torch.randn(shape, generator=gen, dtype=torch.float64) * 0.6 / step) * step
    return v.clamp(-lim, lim).to(torch.bfloat16)


def pin_backward_finite_difference(orc):
    """Central differences of the forward oracle match the backward's gradients.

    Perturbations stay on the bf16 grid, so the forward sees them exactly; y is
    linear in w2 and in the routing weights, quadratic-plus in x and w1.
    """
    gen = torch.Generator().manual_seed(27)
    T, H, I, E, k = 3, 8, 4, 2, 2
    x = _grid_bf16(gen, (T, H))
    w1 = _grid_bf16(gen, (E, 2 * I, H))
    w2 = _grid_bf16(gen, (E, H, I))
    idx = torch.tensor([[0, 1], [1, 0], [1, 1]], dtype=torch.int32)
    w = torch.rand((T, k), generator=gen, dtype=torch.float64) + 0.2
    dy = _grid_bf16(gen, (T, H))
    dyd = dy.double().numpy()
    b = orc.expert_backward(x, idx, w, w1, w2, dy)
    d = 1.0 / 64

    def loss(xx=x, ww1=w1, ww2=w2, ww=w):
        return float((orc.expert_forward(xx, idx, ww, ww1, ww2) * dyd).sum())

    def central(name, tensor, pos, grad):
        plus, minus = tensor.clone(), tensor.clone()
        plus[pos] = float(tensor[pos]) + d
        minus[pos] = float(tensor[pos]) - d
        fd = (loss(**{name: plus}) - loss(**{name: minus})) / (2 * d)
        assert abs(fd - grad) <= 2e-3 * max(1.0, abs(grad)), (name, pos, fd, grad)

    for pos in [(0, 0), (1, 5), (2, 7)]:
        central("xx", x, pos, b.dx[pos])
    for pos in [(0, 0, 3), (1, 2, 0), (0, 5, 6), (1, 7, 7)]:
        central("ww1", w1, pos, b.dw1[pos])
    for pos in [(0, 0, 0), (1, 6, 3)]:
        central("ww2", w2, pos, b.dw2[pos])
    for pos in [(0, 1), (2, 0)]:
        central("ww", w, pos, b.dtopk_w[pos])


def pin_router_backward_finite_difference(orc):
    """Central differences of the forward router in W_r and in the logit offsets.

    fp32 steps of 2^-12 are exact on these inputs; the selection is checked to
    stay the same on both sides of every step.
    """
    gen = torch.Generator().manual_seed(28)
    T, H, E, k = 6, 8, 8, 3
    x = _grid_bf16(gen, (T, H))
    w_r = (torch.randn((E, H), generator=gen, dtype=torch.float32) * 0.5).numpy()
    off = (torch.randn((E,), generator=gen, dtype=torch.float32) * 0.5).numpy()
    dtw = torch.randn((T, k), generator=gen, dtype=torch.float64).numpy()
    d = 2.0 ** -12
    for score, normalize, scale in (("softmax", True, 2.0), ("sigmoid", True, 2.5),
                                    ("softmax", False, 1.0), ("sigmoid", False, 1.5)):
        kw = dict(score=score, normalize=normalize, scale=scale)
        r = orc.router(x, w_r, k, logit_offset=off, **kw)
        b = orc.router_backward(x, w_r, r.topk_idx, r.topk_w, dtw, logit_offset=off, **kw)

        def loss(wr, of):
            rr = orc.router(x, wr, k, logit_offset=of, **kw)
            assert (rr.topk_idx == r.topk_idx).all(), "selection moved under the step"
            return float((rr.topk_w * dtw).sum())

        for e in range(E):
            op, om = off.copy(), off.copy()
            op[e] += d
            om[e] -= d
            fd = (loss(w_r, op) - loss(w_r, om)) / (2 * d)
            want = b.dlogits[:, e].sum()
            assert abs(fd - want) <= 1e-5 * max(1.0, abs(want)), (score, normalize, e, fd, want)
        for e, h in [(0, 0), (3, 5), (7, 7)]:
            wp, wm = w_r.copy(), w_r.copy()
            wp[e, h] += d
            wm[e, h] -= d
            fd = (loss(wp, off) - loss(wm, off)) / (2 * d)
            assert abs(fd - b.dw_r[e, h]) <= 1e-5 * max(1.0, abs(b.dw_r[e, h])), (e, h, fd)


# --------------------------------------------------------------------------- MXFP8

def pin_mx_elements_match_torch_fp8(orc):
    """With the block maximum in [256, 512) the scale is 2^0, so the codes are plain E4M3
    conversions: they match torch's float8_e4m3fn cast (after clamping to +-448)."""
    g = torch.Generator().manual_seed(30)
    rows = 64
    v = (torch.rand((rows, 32), generator=g, dtype=torch.float64) * 2 - 1) * 470.0
    v[:, 0] = 300.0 + torch.rand((rows,), generator=g, dtype=torch.float64) * 150   # amax in [256, 512)
    v[1] = torch.linspace(-0.03, 0.03, 32, dtype=torch.float64)                  # subnormal range
    v[1, 0] = 260.0
    vals = torch.tensor([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 8.0, 16.0, 240.0, 416.0, 448.0], dtype=torch.float64)
    mids = (vals[:-1] + vals[1:]) / 2
    v[2, 1:1 + len(mids)] = mids                                                   # not all exact ties
    v[3, 1:4] = torch.tensor([1.0625, 1.1875, 17.0], dtype=torch.float64)         # exact ties: to even
    v[4, 1:4] = torch.tensor([460.0, 479.0, -500.0], dtype=torch.float64)         # saturation
    codes, scales = orc.mx_quantize(v.numpy())
    assert (scales == 127).all(), scales
    want = v.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(codes, want)


def pin_mx_roundtrip_every_code(orc):
    """A block holding code c's value times 2^s and an anchor 256 * 2^s quantizes back to
    c with scale code s + 127, for every finite E4M3 code."""
    import oracle as oracle_pkg
    vals = oracle_pkg.e4m3_values()
    finite = [c for c in range(256) if np.isfinite(vals[c])]
    for sh in (-20, -3, 0, 5):
        blk = np.zeros((len(finite), 32))
        blk[:, 0] = [-0.0 if c == 0x80 else vals[c] * 2.0 ** sh for c in finite]
        blk[:, 1] = 256.0 * 2.0 ** sh
        codes, scales = orc.mx_quantize(blk)
        assert (scales == sh + 127).all(), (sh, scales[:4])
        assert codes[:, 0].tolist() == finite, sh


def pin_mx_shared_exponent_rule(orc):
    """Scale code = floor(log2 amax) - 8 + 127 (clamped at 0), zero blocks get code 0."""
    amax = [2.0 ** -133, 2.0 ** -120, 0.75, 1.0, 1.999, 3.0, 2.0 ** 20 * 1.5, 2.0 ** 127]
    blk = np.zeros((len(amax) + 1, 32))
    for i, a in enumerate(amax):
        blk[i, 5] = -a
        blk[i, 6] = a / 3
    codes, scales = orc.mx_quantize(blk)
    for i, a in enumerate(amax):
        e = int(np.floor(np.log2(a)))
        assert scales[i, 0] == max(0, e - 8 + 127), (a, scales[i, 0])
        assert codes[i, 5] & 0x80                      # sign kept
    assert scales[-1, 0] == 0 and not codes[-1].any()


def pin_mx_forward_composition(orc):
    """MX forward = bf16 forward on dequantized inputs up to a, then the quantizer on a,
    then a torch fp64 matmul per expert and the weighted sum."""
    import oracle as oracle_pkg
    T, H, I, E, k = 12, 64, 64, 4, 2
    x, w1, w2, idx, w = _problem(31, T=T, H=H, I=I, E=E, k=k)
    xq, xs = orc.mx_quantize(x)
    w1q, w1s = orc.mx_quantize(w1)
    w2q, w2s = orc.mx_quantize(w2)
    y, a_pre, ac, asc = orc.expert_forward_mx(xq, xs, idx, w, w1q, w1s, w2q, w2s, want_a=True)
    xd = oracle_pkg.mx_dequantize(xq, xs)
    w1d = oracle_pkg.mx_dequantize(w1q, w1s)
    w2d = oracle_pkg.mx_dequantize(w2q, w2s)
    # dequantized values are exact in bf16 at these scales
    bf = lambda a: torch.as_tensor(a).to(torch.bfloat16)
    assert np.array_equal(bf(xd).double().numpy(), xd)
    _, a_ref, _ = orc.expert_forward(bf(xd), idx, w, bf(w1d), bf(w2d), want_a=True)
    np.testing.assert_allclose(a_pre, a_ref, rtol=1e-12, atol=1e-14)
    c2, s2 = orc.mx_quantize(a_pre)
    np.testing.assert_array_equal(ac, c2)
    np.testing.assert_array_equal(asc, s2)
    aq = torch.as_tensor(oracle_pkg.mx_dequantize(ac, asc))
    y_ref = torch.zeros((T, H), dtype=torch.float64)
    flat = idx.reshape(-1).long()
    for slot in range(T * k):
        e = int(flat[slot])
        o = torch.as_tensor(w2d[e]) @ aq[slot]
        y_ref[slot // k] += float(w.reshape(-1)[slot]) * o
    np.testing.assert_allclose(y, y_ref.numpy(), rtol=1e-11, atol=1e-12)


def _mx_exact_bf16(gen, shape, scale=1.0):
    """bf16 values that MXFP8 holds exactly in any block: each is in
    {0, +-1/4, +-1/2, +-3/4, +-1, +-3/2} times `scale` (a power of two), so with
    the block's scale 2^(floor(log2 amax) - 8) every value maps to an E4M3 code
    (at most 1.5 * 2^8 = 384) without rounding."""
    vals = torch.tensor([0.0, 0.25, 0.5, 0.75, 1.0, 1.5, -0.25, -0.5, -0.75, -1.0, -1.5], dtype=torch.float64)
    pick = torch.randint(0, len(vals), shape, generator=gen)
    return (vals[pick] * scale).to(torch.bfloat16)


def _mx_backward_problem(seed, T=40, H=64, I=64, E=4, k=2, exact=False):
    gen = torch.Generator().manual_seed(seed)
    if exact:
        x = _mx_exact_bf16(gen, (T, H))
        w1 = _mx_exact_bf16(gen, (E, 2 * I, H), 0.125)
    else:
        x = _rand_bf16(gen, (T, H))
        w1 = _rand_bf16(gen, (E, 2 * I, H), H ** -0.5)
    w2 = _rand_bf16(gen, (E, H, I), I ** -0.5)
    dy = _rand_bf16(gen, (T, H))
    idx = torch.randint(0, E - 1, (T, k), generator=gen, dtype=torch.int32)   # expert E-1 gets no row
    w = torch.rand((T, k), generator=gen, dtype=torch.float64) + 0.1
    return x, w1, w2, dy, idx, w


def pin_mx_backward_exact_forward_is_bf16(orc):
    """When MXFP8 holds x and w1 exactly, the MX forward's g, u are the bf16 forward's,
    so the MX backward's data-gradient path (dX, the routing-weight gradient, w a)
    must be the bf16 backward oracle's (itself pinned by autograd and finite
    differences) and the bf16 forward's a times the weight."""
    import oracle as oracle_pkg
    x, w1, w2, dy, idx, w = _mx_backward_problem(41, exact=True)
    xq, xs = orc.mx_quantize(x)
    w1q, w1s = orc.mx_quantize(w1)
    assert np.array_equal(oracle_pkg.mx_dequantize(xq, xs), x.double().numpy())
    assert np.array_equal(oracle_pkg.mx_dequantize(w1q, w1s), w1.double().numpy())
    b_mx, dh, wa = orc.expert_backward_mx(x, xq, xs, idx, w, w1, w1q, w1s, w2, dy, want_slots=True)
    b = orc.expert_backward(x, idx, w, w1, w2, dy, want_dw=False)
    np.testing.assert_allclose(b_mx.dx, b.dx, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(b_mx.dtopk_w, b.dtopk_w, rtol=1e-11, atol=1e-12)
    _, a_ref, _ = orc.expert_forward(x, idx, w, w1, w2, want_a=True)
    np.testing.assert_allclose(wa, w.numpy().reshape(-1, 1) * a_ref, rtol=1e-12, atol=1e-14)
    assert not b_mx.dw1[-1].any() and not b_mx.dw2[-1].any()          # the expert without rows


def pin_mx_backward_forward_is_the_mx_forward(orc):
    """With inputs MXFP8 rounds, w a per slot is the routing weight times the MX
    forward oracle's a before its quantization (x and w1 quantized along H)."""
    x, w1, w2, dy, idx, w = _mx_backward_problem(43)
    xq, xs = orc.mx_quantize(x)
    w1q, w1s = orc.mx_quantize(w1)
    w2q, w2s = orc.mx_quantize(w2)
    _, dh, wa = orc.expert_backward_mx(x, xq, xs, idx, w, w1, w1q, w1s, w2, dy, want_dw=False, want_slots=True)
    _, a_pre, _, _ = orc.expert_forward_mx(xq, xs, idx, w, w1q, w1s, w2q, w2s, want_a=True)
    np.testing.assert_allclose(wa, w.numpy().reshape(-1, 1) * a_pre, rtol=1e-12, atol=1e-14)
    # x really is rounded here: the unquantized x would give other values of a
    _, a_bf, _ = orc.expert_forward(x, idx, w, w1, w2, want_a=True)
    assert np.abs(a_bf - a_pre).max() > 1e-3


def pin_mx_backward_wgrad_composition(orc):
    """dW1 and dW2 of the MX backward = per expert, the rows of its slots in
    increasing slot order, zero-padded to whole blocks of 32 rows, each column
    quantized by the (separately pinned) MXFP8 quantizer along the rows, then one
    fp64 matmul of the dequantized operands: dW2_e = Q(dY)^T Q(w a),
    dW1_e = Q(dH)^T Q(x)."""
    import oracle as oracle_pkg
    T, k = 70, 2
    x, w1, w2, dy, idx, w = _mx_backward_problem(47, T=T, k=k)
    xq, xs = orc.mx_quantize(x)
    w1q, w1s = orc.mx_quantize(w1)
    b, dh, wa = orc.expert_backward_mx(x, xq, xs, idx, w, w1, w1q, w1s, w2, dy, want_slots=True)
    xd, dyd = x.double().numpy(), dy.double().numpy()
    flat = idx.numpy().reshape(-1)

    def q_rows(m):
        n = m.shape[0]
        pad = np.zeros((-(-n // 32) * 32, m.shape[1]))
        pad[:n] = m
        c, sc = orc.mx_quantize(np.ascontiguousarray(pad.T))
        return oracle_pkg.mx_dequantize(c, sc).T

    sizes = []
    for e in range(w1.shape[0]):
        slots = np.nonzero(flat == e)[0]
        sizes.append(len(slots))
        if len(slots) == 0:
            assert not b.dw1[e].any() and not b.dw2[e].any()
            continue
        tok = slots // k
        np.testing.assert_allclose(b.dw2[e], q_rows(dyd[tok]).T @ q_rows(wa[slots]), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(b.dw1[e], q_rows(dh[slots]).T @ q_rows(xd[tok]), rtol=1e-12, atol=1e-12)
    assert any(s % 32 for s in sizes) and max(sizes) > 32        # partial blocks and several blocks


ALL_PINS = [v for n, v in sorted(globals().items()) if n.startswith("pin_") and callable(v)]
