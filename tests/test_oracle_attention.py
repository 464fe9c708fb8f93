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


def test_key_mask_is_dropping_the_masked_keys():
    """A per-key mask (limn, "The op set": masking is a flag per key that
    composes with causal): an all-ones mask changes nothing; without causal,
    masking keys gives exactly the attention over the remaining keys (the
    masked keys removed from K and V); with causal, each query's result is
    its softmax over the keys it sees, brute force; a query that sees no key
    gets O = 0, L = -inf and no gradient."""
    q, k, v = _rand((2, 7, 3), 11), _rand((2, 7, 3), 12), _rand((2, 7, 3), 13)
    scale = 0.6
    ones = np.ones((2, 7), np.int8)
    for causal in (False, True):
        a = attention_fwd(q, k, v, scale, causal)
        b = attention_fwd(q, k, v, scale, causal, key_mask=ones)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    km = np.array([[1, 0, 1, 1, 0, 1, 1], [0, 1, 1, 0, 1, 1, 0]], np.int8)
    O, L = attention_fwd(q, k, v, scale, causal=False, key_mask=km)
    for h in range(2):
        keep = km[h] != 0
        Oh, Lh = attention_fwd(q[h:h + 1], k[h:h + 1, keep], v[h:h + 1, keep], scale, causal=False)
        assert np.allclose(O[h], Oh[0], rtol=1e-13, atol=1e-15) and np.allclose(L[h], Lh[0], rtol=1e-13)
    Oc, Lc = attention_fwd(q, k, v, scale, causal=True, key_mask=km)
    for h in range(2):
        for i in range(7):
            js = [j for j in range(i + 1) if km[h, j]]
            if not js:
                assert np.all(Oc[h, i] == 0) and Lc[h, i] == -np.inf
                continue
            w = np.array([np.exp(scale * q[h, i] @ k[h, j]) for j in js])
            assert np.allclose(Oc[h, i], (w[:, None] * v[h, js]).sum(0) / w.sum(), rtol=1e-13)
            assert np.isclose(Lc[h, i], np.log(w.sum()), rtol=1e-13)
    # head 1's first query sees only key 0, which is masked
    assert Lc[1, 0] == -np.inf
    dO = _rand((2, 7, 3), 14)
    dq, dk, dv = attention_bwd(q, k, v, Oc, dO, Lc, scale, causal=True, key_mask=km)
    assert np.all(np.isfinite(dq)) and np.all(dq[1, 0] == 0)
    # masked keys get no gradient
    assert np.all(dk[0, 1] == 0) and np.all(dv[0, 4] == 0) and np.all(dk[1, 3] == 0)


def test_masked_backward_matches_finite_differences():
    q, k, v = _rand((2, 6, 4), 21), _rand((2, 6, 4), 22), _rand((2, 6, 4), 23)
    km = np.array([[1, 1, 0, 1, 1, 0], [1, 0, 1, 1, 1, 1]], np.int8)
    W = _rand((2, 6, 4), 24)
    scale = 0.5

    def loss(q_, k_, v_):
        return float((attention_fwd(q_, k_, v_, scale, key_mask=km)[0] * W).sum())

    O, L = attention_fwd(q, k, v, scale, key_mask=km)
    dq, dk, dv = attention_bwd(q, k, v, O, W, L, scale, key_mask=km)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        for idx in [(0, 0, 0), (1, 3, 2), (0, 5, 3), (1, 2, 1), (0, 2, 1)]:
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-7 * max(1.0, abs(fd)), (idx, fd, g[idx])
