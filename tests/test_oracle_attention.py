"""Pins of the attention oracle (CPU): brute force for the forward, finite
differences for the backward, and the cases the mask fixes by itself."""
import numpy as np

from oracle.attention import attention_bwd, attention_fwd


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_forward_against_brute_force_and_mask_cases():
    q, k, v = _rand((2, 5, 3), 1), _rand((2, 5, 3), 2), _rand((2, 5, 3), 3)
    scale = 0.7
    O, L = attention_fwd(q, k, v, scale)
    for h in range(2):
        for i in range(5):
            w = np.array([np.exp(scale * q[h, i] @ k[h, j]) for j in range(i + 1)])
            assert np.allclose(O[h, i], (w[:, None] * v[h, : i + 1]).sum(0) / w.sum(), rtol=1e-13)
            assert np.isclose(L[h, i], np.log(w.sum()), rtol=1e-13)
    # the first query sees only the first key
    assert np.allclose(O[:, 0], v[:, 0], rtol=0, atol=1e-15)
    # without the mask and with equal keys every query averages the values
    kk = np.repeat(k[:, :1], 5, axis=1)
    O2, _ = attention_fwd(q, kk, v, scale, causal=False)
    assert np.allclose(O2, np.repeat(v.mean(axis=1, keepdims=True), 5, axis=1), rtol=1e-13)


def test_backward_matches_finite_differences():
    q, k, v = _rand((2, 6, 4), 4), _rand((2, 6, 4), 5), _rand((2, 6, 4), 6)
    W = _rand((2, 6, 4), 7)           # loss = sum(O * W), so dO = W
    scale = 0.5

    def loss(q_, k_, v_):
        return float((attention_fwd(q_, k_, v_, scale)[0] * W).sum())

    O, L = attention_fwd(q, k, v, scale)
    dq, dk, dv = attention_bwd(q, k, v, O, W, L, scale)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        for idx in [(0, 0, 0), (1, 3, 2), (0, 5, 3), (1, 2, 1)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, g[idx])
