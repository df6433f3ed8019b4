"""The MXFP8 weight-quant cache's bookkeeping (host only; the quantizer is a fake)."""
import torch

from moe_expert_router_gb300.mx_cache import MxWeightCache


def _fake_quantize(w):
    return ("codes", w.clone()), ("scales", w.shape)


def test_cache_hits_until_the_weight_changes():
    c = MxWeightCache(quantize=_fake_quantize)
    w = torch.zeros((2, 4, 64), dtype=torch.bfloat16)
    q1 = c.get(w)
    assert c.get(w) is q1 and c.quantizations == 1
    w.add_(1.0)                              # in-place update bumps the version counter
    q2 = c.get(w)
    assert q2 is not q1 and c.quantizations == 2
    assert torch.equal(q2[0][1], w)


def test_invalidate_drops_entries_the_version_cannot_see():
    c = MxWeightCache(quantize=_fake_quantize)
    w = torch.zeros((2, 4, 64), dtype=torch.bfloat16)
    c.get(w)
    with torch.no_grad():
        w.data.fill_(3.0)                    # a write through .data does not bump the version
    assert c.get(w)[0][1].max().item() == 0.0     # stale, as in the guide's optimizer case
    c.invalidate()
    assert len(c) == 0
    assert c.get(w)[0][1].max().item() == 3.0 and c.quantizations == 2


def test_separate_tensors_have_separate_entries():
    c = MxWeightCache(quantize=_fake_quantize)
    w1 = torch.zeros((2, 4, 64), dtype=torch.bfloat16)
    w2 = torch.ones((2, 8, 32), dtype=torch.bfloat16)
    c.get(w1)
    c.get(w2)
    assert len(c) == 2 and c.quantizations == 2
    try:
        c.get(torch.zeros((2, 4, 48), dtype=torch.bfloat16))
    except ValueError:
        pass
    else:
        raise AssertionError("a last dimension that is not a multiple of 32 must be rejected")


def test_another_tensor_at_the_same_address_is_not_a_hit():
    """An entry belongs to one tensor object: a detached view (same storage, shape,
    dtype and version) is quantized on its own, and so would be a new weight that
    the allocator placed where a freed one was."""
    c = MxWeightCache(quantize=_fake_quantize)
    w = torch.zeros((2, 4, 64), dtype=torch.bfloat16)
    c.get(w)
    v = w.detach()
    assert v.data_ptr() == w.data_ptr() and v._version == w._version
    c.get(v)
    assert c.quantizations == 2
    c.get(v)
    assert c.quantizations == 2


def test_a_freed_weight_drops_its_entry():
    import gc
    c = MxWeightCache(quantize=_fake_quantize)
    w = torch.zeros((2, 4, 64), dtype=torch.bfloat16)
    keep = torch.ones((2, 4, 64), dtype=torch.bfloat16)
    c.get(w)
    c.get(keep)
    assert len(c) == 2
    del w
    gc.collect()
    assert len(c) == 1 and c.get(keep) is not None and c.quantizations == 2
