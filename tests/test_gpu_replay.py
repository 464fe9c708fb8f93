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


def test_gpt_block_full_size_replay_is_bit_exact(G):
    """The bench's GPT block (B32, T256, d512) recorded once, its independent
    calls on forked streams: every replay gives eager's bits, over several
    replays and new inputs (a missing dependency edge between the streams
    would let a call read a buffer before or after it is written)."""
    from primitive_sm_graph_gb300.workloads import GPT_WEIGHTS, gpt_step
    H = SI.GPT_SHAPES["H"]

    def step(tok, *ws):
        loss, grads = gpt_step(tok, dict(zip(GPT_WEIGHTS, ws)), H)
        return (loss,) + tuple(grads[k] for k in GPT_WEIGHTS)

    tok, w = SI.gpt_block(11, **SI.GPT_SHAPES)
    ins = [tok.cuda()] + [w[k].cuda() for k in GPT_WEIGHTS]
    rep = G.Replay(step, *ins)
    ref = [t.clone() for t in step(*ins)]
    for _ in range(3):
        got = rep(*ins)
        assert all(_same(x, y) for x, y in zip(got, ref))
    tok2, w2 = SI.gpt_block(12, **SI.GPT_SHAPES)
    ins2 = [tok2.cuda()] + [w2[k].cuda() for k in GPT_WEIGHTS]
    ref2 = [t.clone() for t in step(*ins2)]
    for _ in range(3):
        got2 = rep(*ins2)
        assert all(_same(x, y) for x, y in zip(got2, ref2))


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


def test_plan_cache_replays_the_same_calls_bit_for_bit(G):
    """The plan cache (limn, "Reading the schedule": execution plans cached
    by graph structure): a graph whose structure was realized before replays
    the recorded calls with its own buffers, skipping the scheduler.  The
    GPT block step and the tiny graph give the same bits through a recorded
    plan, through the plan on new inputs, and with the cache off (scheduled
    afresh); the hit makes the same calls (the executor's log)."""
    from primitive_sm_graph_gb300.workloads import GPT_WEIGHTS, gpt_step, tiny_graph
    shapes = dict(B=2, T=64, V=128, D=128, H=2, F=256)
    tok, w = SI.gpt_block(8, **shapes)
    dtok, dw = tok.cuda(), {k: v.cuda() for k, v in w.items()}
    ex = G._executor()
    old = G.PLAN_CACHE
    try:
        G.PLAN_CACHE = True
        ex.log.clear()
        first = gpt_step(dtok, dw, 2)
        log_first = list(ex.log)
        n_plans = len(G._PLANS)
        ex.log.clear()
        hit = gpt_step(dtok, dw, 2)
        assert len(G._PLANS) == n_plans and ex.log == log_first
        G.PLAN_CACHE = False
        fresh = gpt_step(dtok, dw, 2)
        for a, b, c in [(first[0], hit[0], fresh[0])] + [(first[1][k], hit[1][k], fresh[1][k]) for k in GPT_WEIGHTS]:
            assert _same(a, b) and _same(a, c)
        # other inputs through the recorded plan
        G.PLAN_CACHE = True
        tok2, w2 = SI.gpt_block(9, **shapes)
        d2 = {k: v.cuda() for k, v in w2.items()}
        via_plan = gpt_step(tok2.cuda(), d2, 2)
        G.PLAN_CACHE = False
        fresh2 = gpt_step(tok2.cuda(), d2, 2)
        assert _same(via_plan[0], fresh2[0]) and not _same(via_plan[0], first[0])
        assert all(_same(via_plan[1][k], fresh2[1][k]) for k in GPT_WEIGHTS)
        G.PLAN_CACHE = True
        a, b = (t.cuda() for t in SI.tiny_graph(0))
        r1 = tiny_graph(G.Tensor.from_torch(a), G.Tensor.from_torch(b)).realize().clone()
        r2 = tiny_graph(G.Tensor.from_torch(a), G.Tensor.from_torch(b)).realize()
        assert _same(r1, r2)
    finally:
        G.PLAN_CACHE = old
