"""CPU oracle of scaled dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Plain float64 numpy,
one head at a time, written from the definition:

  S = scale * Q K^T, with S[i, j] = -inf where the mask hides key j from
      query i (causal: j > i);
  L[i] = log sum_j exp(S[i, j])            (the logsumexp the forward saves;
                                           limn, "The op set": the fused
                                           attention op saves L);
  P = exp(S - L)                           (each row sums to 1);
  O = P V.

Backward, by the chain rule through O = P V and the row softmax (the form
Tiki's FlashAttention backward target spells out, "Write the attention
kernel at the algorithm level"):

  dV = P^T dO;     dP = dO V^T;     D[i] = sum_d dO[i, d] O[i, d];
  dS = P * (dP - D[:, None]);      dQ = scale * dS K;      dK = scale * dS^T Q.

A library matrix product serves as the step of each contraction.
"""
from __future__ import annotations

import numpy as np


def _mask(T: int, causal: bool) -> np.ndarray:
    """True where query i may see key j."""
    if not causal:
        return np.ones((T, T), dtype=bool)
    return np.tril(np.ones((T, T), dtype=bool))


def attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool = True):
    """q, k, v: [heads, T, hd] -> (O [heads, T, hd], L [heads, T]), float64."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    Hn, T, _ = q.shape
    vis = _mask(T, causal)
    O = np.zeros_like(v)
    L = np.zeros((Hn, T))
    for h in range(Hn):
        S = scale * (q[h] @ k[h].T)
        S = np.where(vis, S, -np.inf)
        m = S.max(axis=1, keepdims=True)
        e = np.exp(S - m)
        s = e.sum(axis=1, keepdims=True)
        L[h] = (m + np.log(s))[:, 0]
        O[h] = (e / s) @ v[h]
    return O, L


def attention_bwd(q, k, v, o, do, L, scale: float, causal: bool = True):
    """Gradients (dQ, dK, dV) of the forward above for the output gradient
    dO, all [heads, T, hd], float64."""
    q, k, v, o, do, L = (np.asarray(x, np.float64) for x in (q, k, v, o, do, L))
    Hn, T, _ = q.shape
    vis = _mask(T, causal)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for h in range(Hn):
        S = np.where(vis, scale * (q[h] @ k[h].T), -np.inf)
        P = np.exp(S - L[h][:, None])
        dv[h] = P.T @ do[h]
        dP = do[h] @ v[h].T
        D = (do[h] * o[h]).sum(axis=1)
        dS = P * (dP - D[:, None])
        dq[h] = scale * (dS @ k[h])
        dk[h] = scale * (dS.T @ q[h])
    return dq, dk, dv
