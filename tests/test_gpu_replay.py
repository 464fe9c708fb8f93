"""GPU tests of capture/replay (graph.Replay): a recorded step relaunches the
same kernels in the same order, and every kernel of the library is
deterministic, so a replay must give the eager result bit for bit, on the
recorded inputs and on new ones copied in.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def G():
    from primitive_sm_graph_gb300 import graph
    return graph


def _same(a, b):
    return np.array_equal(a.detach().cpu().view(torch.int16 if a.element_size() == 2 else torch.int32).numpy(),
                          b.detach().cpu().view(torch.int16 if b.element_size() == 2 else torch.int32).numpy())


def test_tiny_graph_replay_is_bit_exact(G):
    from primitive_sm_graph_gb300.workloads import tiny_graph

    def step(a, b):
        return tiny_graph(G.Tensor.from_torch(a), G.Tensor.from_torch(b)).realize()

    a, b = (t.cuda() for t in SI.tiny_graph(0))
    rep = G.Replay(step, a, b)
    assert _same(rep(a, b), step(a, b))
    a2, b2 = (t.cuda() for t in SI.tiny_graph(1))
    eager = step(a2, b2).clone()
    assert _same(rep(a2, b2), eager)


def test_gpt_block_step_replay_is_bit_exact(G):
    from primitive_sm_graph_gb300.workloads import GPT_WEIGHTS, gpt_step
    shapes = dict(B=2, T=16, V=64, D=64, H=2, F=128)
    H = shapes["H"]

    def step(tok, *ws):
        loss, grads = gpt_step(tok, dict(zip(GPT_WEIGHTS, ws)), H)
        return (loss,) + tuple(grads[k] for k in GPT_WEIGHTS)

    tok, w = SI.gpt_block(3, **shapes)
    ins = [tok.cuda()] + [w[k].cuda() for k in GPT_WEIGHTS]
    rep = G.Replay(step, *ins)
    got = [t.clone() for t in rep(*ins)]
    ref = step(*ins)
    assert all(_same(x, y) for x, y in zip(got, ref))
    # new tokens and weights through the same recording
    tok2, w2 = SI.gpt_block(4, **shapes)
    ins2 = [tok2.cuda()] + [w2[k].cuda() for k in GPT_WEIGHTS]
    ref2 = [t.clone() for t in step(*ins2)]
    got2 = rep(*ins2)
    assert all(_same(x, y) for x, y in zip(got2, ref2))
    assert not _same(got2[0], got[0])          # the loss did change with the inputs
