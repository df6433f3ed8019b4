"""The torch.library operators (moe_expert_router_gb300/torch_ops.py): schemas and
shape functions on the host (fake tensors, no device call)."""
import torch
from torch._subclasses.fake_tensor import FakeTensorMode

from moe_expert_router_gb300 import torch_ops  # noqa: F401  (registers the operators)


def test_operators_are_registered():
    for name in ("router", "forward", "forward_mx", "layer_train", "layer_backward", "layer_train_mx",
                 "layer_backward_mx"):
        assert hasattr(torch.ops.moe_gb300, name)


def test_fake_shapes():
    T, H, I, E, k = 24, 256, 128, 8, 3
    with FakeTensorMode():
        x = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        w_r = torch.empty((E, H), dtype=torch.float32, device="cuda")
        idx, w, aux = torch.ops.moe_gb300.router(x, w_r, k, "sigmoid", True, 2.5, 4, 2, 2)
        assert idx.shape == (T, k) and idx.dtype == torch.int32
        assert w.shape == (T, k) and w.dtype == torch.float32 and aux.shape == (1,)
        w1 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device="cuda")
        w2 = torch.empty((E, H, I), dtype=torch.bfloat16, device="cuda")
        y = torch.ops.moe_gb300.forward(x, idx, w, w1, w2)
        assert y.shape == (T, H) and y.dtype == torch.bfloat16
        c1 = torch.empty((E, 2 * I, H), dtype=torch.uint8, device="cuda")
        s1 = torch.empty((H // 128, E, 2 * I, 4), dtype=torch.uint8, device="cuda")
        c2 = torch.empty((E, H, I), dtype=torch.uint8, device="cuda")
        s2 = torch.empty((I // 128, E, H, 4), dtype=torch.uint8, device="cuda")
        y = torch.ops.moe_gb300.forward_mx(x, idx, w, c1, s1, c2, s2)
        assert y.shape == (T, H) and y.dtype == torch.bfloat16


def test_layer_autograd_shapes():
    """moe_layer's forward and its registered backward on shape-only tensors: output
    and gradient shapes and dtypes, the routing outputs without a gradient."""
    T, H, I, E, k = 40, 256, 128, 8, 2
    # meta tensors: the operators' shape functions run, and the autograd engine needs no device
    x = torch.empty((T, H), dtype=torch.bfloat16, device="meta", requires_grad=True)
    w_r = torch.empty((E, H), dtype=torch.float32, device="meta", requires_grad=True)
    w1 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device="meta", requires_grad=True)
    w2 = torch.empty((E, H, I), dtype=torch.bfloat16, device="meta", requires_grad=True)
    y, idx, w, aux = torch_ops.moe_layer(x, w_r, w1, w2, k, "sigmoid", True, 2.5, 4, 2, 2)
    assert y.shape == (T, H) and y.dtype == torch.bfloat16 and y.requires_grad
    assert idx.shape == (T, k) and not w.requires_grad and not aux.requires_grad
    y.backward(torch.empty_like(y))
    assert x.grad.shape == x.shape and x.grad.dtype == torch.bfloat16
    assert w_r.grad.shape == w_r.shape and w_r.grad.dtype == torch.float32
    assert w1.grad.shape == w1.shape and w2.grad.shape == w2.shape


def test_mx_layer_autograd_shapes():
    """moe_layer(precision="mxfp8") on meta tensors, with a cache whose quantizer only
    allocates: the MXFP8 operators' shapes and the registered backward's gradients."""
    from moe_expert_router_gb300 import binding as B
    from moe_expert_router_gb300.mx_cache import MxWeightCache

    def shapes_only(w):
        return torch.empty(w.shape, dtype=torch.uint8, device=w.device), B.mx_scales_empty(w.shape, w.device)

    T, H, I, E, k = 40, 256, 128, 8, 2
    x = torch.empty((T, H), dtype=torch.bfloat16, device="meta", requires_grad=True)
    w_r = torch.empty((E, H), dtype=torch.float32, device="meta", requires_grad=True)
    w1 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device="meta", requires_grad=True)
    w2 = torch.empty((E, H, I), dtype=torch.bfloat16, device="meta", requires_grad=True)
    cache = MxWeightCache(quantize=shapes_only)
    y, idx, w, aux = torch_ops.moe_layer(x, w_r, w1, w2, k, precision="mxfp8", weight_cache=cache)
    assert y.shape == (T, H) and y.requires_grad and len(cache) == 2
    y.backward(torch.empty_like(y))
    assert x.grad.shape == x.shape and w_r.grad.shape == w_r.shape
    assert w1.grad.shape == w1.shape and w2.grad.shape == w2.shape


def test_operators_refuse_wrong_types_and_shapes():
    """The library reads raw pointers, so the operators check every argument's type and
    shape first (in their shape functions too, which run here on meta tensors)."""
    import pytest
    T, H, I, E, k = 16, 256, 128, 8, 2
    m = dict(device="meta")
    x = torch.empty((T, H), dtype=torch.bfloat16, **m)
    w_r = torch.empty((E, H), dtype=torch.float32, **m)
    w1 = torch.empty((E, 2 * I, H), dtype=torch.bfloat16, **m)
    w2 = torch.empty((E, H, I), dtype=torch.bfloat16, **m)
    idx = torch.empty((T, k), dtype=torch.int32, **m)
    w = torch.empty((T, k), dtype=torch.float32, **m)
    with pytest.raises(TypeError):
        torch.ops.moe_gb300.router(x.float(), w_r, k)
    with pytest.raises(TypeError):
        torch.ops.moe_gb300.router(x, w_r.bfloat16(), k)
    with pytest.raises(ValueError):
        torch.ops.moe_gb300.router(x, w_r, E + 1)
    with pytest.raises(ValueError):
        torch.ops.moe_gb300.router(x, w_r, k, sel_bias=torch.empty((E + 1,), **m))
    with pytest.raises(TypeError):
        torch.ops.moe_gb300.forward(x, idx.long(), w, w1, w2)
    with pytest.raises(ValueError):
        torch.ops.moe_gb300.forward(x, idx, w, w1, torch.empty((E, H, I + 8), dtype=torch.bfloat16, **m))
    with pytest.raises(ValueError):
        torch.ops.moe_gb300.forward(x[:, :128], idx, w, w1, w2)
    c1 = torch.empty((E, 2 * I, H), dtype=torch.uint8, **m)
    s1 = torch.empty((H // 128, E, 2 * I, 4), dtype=torch.uint8, **m)
    c2 = torch.empty((E, H, I), dtype=torch.uint8, **m)
    with pytest.raises(ValueError):
        torch.ops.moe_gb300.forward_mx(x, idx, w, c1, s1, c2, torch.empty((I // 128, E, H, 3), dtype=torch.uint8, **m))
    with pytest.raises(TypeError):
        torch_ops.moe_layer(x, w_r, w1.float(), w2, k)
    with pytest.raises(ValueError):
        torch_ops.moe_layer(x, w_r, w1, w2, k, precision="fp4")
