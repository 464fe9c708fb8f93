"""Host-side structure of the lazy graph (CPU, nothing realized): the
rewrites the graph builder makes must leave every value unchanged.
"""
import numpy as np
import torch

from primitive_sm_graph_gb300 import graph as G


def _nodes(root):
    seen, stack, out = set(), [root], []
    while stack:
        t = stack.pop()
        if id(t) in seen:
            continue
        seen.add(id(t))
        out.append(t)
        stack.extend(t.src)
    return out


def test_relu_backward_takes_its_mask_from_the_output():
    """The gradient of relu(x) = WHERE(CMPLT(0, x), x, 0) is WHERE(mask, g, 0);
    the mask is built from the ReLU's output, so x is read by the ReLU
    alone (and a contraction producing x can run the ReLU in its epilogue)."""
    x = G.Tensor.from_torch(torch.randn(4, 6), requires_grad=True)
    y = x.relu()
    assert G._is_relu(y)
    loss = y.reshape(1, -1).sum(-1, keepdim=False)
    G.backward(loss)
    wheres = [t for t in _nodes(x.grad) if t.op == "WHERE" and t is not y]
    assert wheres
    for t in wheres:
        c = t.src[0]
        assert c.op == "CMPLT" and c.src[1] is y and c.src[0].op == "CONST" and c.src[0].arg == 0.0
    # x's users in the whole graph: the ReLU's CMPLT and WHERE only
    users = [t for t in _nodes(x.grad) if any(s is x for s in t.src)]
    assert {t.op for t in users} <= {"CMPLT", "WHERE"} and all(t is y or t is y.src[0] for t in users)


def test_relu_masks_agree_on_every_special_value():
    """0 < x and 0 < relu(x) are the same bit for every float: NaN, both
    zeros, both infinities, subnormals and ordinary values."""
    specials = np.array([np.nan, -np.nan, 0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 1e-38, -1e-38,
                         1.0, -1.0, 3.4e38, -3.4e38], np.float32)
    rnd = np.random.default_rng(0).standard_normal(4096).astype(np.float32)
    bits = np.random.default_rng(1).integers(0, 2 ** 32, 4096, dtype=np.uint64).astype(np.uint32).view(np.float32)
    for x in (specials, rnd, bits):
        with np.errstate(invalid="ignore"):
            relu = np.where(np.float32(0) < x, x, np.float32(0))
            assert np.array_equal(np.float32(0) < relu, np.float32(0) < x)


def test_a_scalar_constant_broadcasts_as_one_constant_node():
    """x + 2 builds ADD(x, CONST 2 at x's shape): the same value in every
    cell, no movement nodes between."""
    x = G.Tensor.from_torch(torch.zeros(3, 5))
    y = x + 2.0
    assert y.op == "ADD"
    c = y.src[1]
    assert c.op == "CONST" and c.shape == (3, 5) and c.arg == 2.0 and not c.src
