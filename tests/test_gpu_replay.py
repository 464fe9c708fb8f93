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


def test_gpt_train_step_replay_updates_like_eager(G):
    """Forward, backward and AdamW recorded once: replayed twice from the
    same start it gives the eager weights bit for bit."""
    from primitive_sm_graph_gb300.workloads import GPT_WEIGHTS, AdamW, gpt_train_step
    shapes = dict(B=2, T=16, V=64, D=64, H=2, F=128)
    tok, w = SI.gpt_block(6, **shapes)
    dtok = tok.cuda()
    w_eager = {k: v.cuda() for k, v in w.items()}
    opt_e = AdamW([w_eager[k] for k in GPT_WEIGHTS], lr=1e-2)
    for _ in range(2):
        gpt_train_step(dtok, w_eager, 2, opt_e)
    w_rep = {k: v.cuda() for k, v in w.items()}
    opt_r = AdamW([w_rep[k] for k in GPT_WEIGHTS], lr=1e-2)
    snap = {k: v.clone() for k, v in w_rep.items()}
    rep = G.Replay(lambda t: gpt_train_step(t, w_rep, 2, opt_r), dtok)
    # the recording ran the step twice (compile + capture warm-up): restart from the snapshot
    for k in GPT_WEIGHTS:
        w_rep[k].copy_(snap[k])
    for x in opt_r.m + opt_r.v:
        x.zero_()
    opt_r.beta_pow.fill_(1.0)
    for _ in range(2):
        rep.replay()
    torch.cuda.synchronize()
    for k in GPT_WEIGHTS:
        assert _same(w_rep[k], w_eager[k]), k
