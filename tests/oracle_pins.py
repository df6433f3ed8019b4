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
  token-permutation equivariance, linearity in w2, dropped slots, aux limits.

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


ALL_PINS = [v for n, v in sorted(globals().items()) if n.startswith("pin_") and callable(v)]
