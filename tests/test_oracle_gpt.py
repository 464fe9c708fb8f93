"""Pins of the oracle's GPT block (CPU only).

The block's end-to-end result has no closed form, so the oracle's backward
is pinned by finite differences of its own forward in float64 (a shrunken
block, as Tiki's FlashAttention gate asks for finite-difference checks on
small cases), and its forward by two invariants: with tiny weights the
logits are ~0 and the loss is ln V; the loss is the mean of per-position
cross-entropies, each >= 0."""
import math

import numpy as np
import pytest

SHAPES = dict(B=2, T=6, V=11, D=8, H=2, F=12)


def _weights(O, rng, std, dt, V, T, D, F):
    def r(*shape):
        return O.T(rng.normal(0.0, std, shape).astype(np.float64), "f64") if dt == "f64" else \
            O.cast(O.T(rng.normal(0.0, std, shape), "f64"), dt)
    w = {"E": r(V, D), "P": r(T, D), "Wqkv": r(D, 3 * D), "Wo": r(D, D), "W1": r(D, F),
         "W2": r(F, D), "Wlm": r(D, V)}
    for g in ("g1", "g2", "gf"):
        w[g] = O.cast(O.T(1.0 + rng.normal(0.0, 0.1, (D,)), "f64"), dt)
    return w


def _loss(O, G, tok, w, H):
    return float(G.GPTOracle(tok, w, H, act="f64", acc="f64").run()[0].data[0])


def test_gpt_oracle_backward_matches_finite_differences(O):
    import oracle.gpt as G
    s = SHAPES
    rng = np.random.default_rng(0)
    tok = rng.integers(0, s["V"], (s["B"], s["T"])).astype(np.int32)
    w = _weights(O, rng, 0.5, "f64", s["V"], s["T"], s["D"], s["F"])
    loss, grads = G.GPTOracle(tok, w, s["H"], act="f64", acc="f64").run()
    h = 1e-6
    for name in ("E", "P", "Wqkv", "Wo", "W1", "W2", "Wlm", "g1", "g2", "gf"):
        flat = w[name].data.reshape(-1)
        for i in rng.choice(flat.size, size=min(6, flat.size), replace=False):
            old = flat[i]
            flat[i] = old + h
            lp = _loss(O, G, tok, w, s["H"])
            flat[i] = old - h
            lm = _loss(O, G, tok, w, s["H"])
            flat[i] = old
            fd = (lp - lm) / (2 * h)
            an = grads[name].data.reshape(-1)[i]
            assert abs(fd - an) <= 1e-6 + 1e-5 * abs(fd), (name, i, fd, an)


def test_gpt_oracle_loss_at_tiny_weights_is_ln_v(O):
    import oracle.gpt as G
    s = SHAPES
    rng = np.random.default_rng(1)
    tok = rng.integers(0, s["V"], (s["B"], s["T"])).astype(np.int32)
    w = _weights(O, rng, 1e-4, "f64", s["V"], s["T"], s["D"], s["F"])
    loss, _ = G.GPTOracle(tok, w, s["H"], act="f64", acc="f64").run()
    assert abs(loss.data[0] - math.log(s["V"])) < 1e-3
    # bfloat16 storage / float32 compute gives the same loss to a few units of 2^-8
    wb = {k: O.cast(v, "bf16") for k, v in w.items()}
    lb, gb = G.GPTOracle(tok, wb, s["H"]).run()
    assert abs(float(lb.data[0]) - math.log(s["V"])) < 2e-2
    assert all(np.all(np.isfinite(g.f64())) for g in gb.values())
