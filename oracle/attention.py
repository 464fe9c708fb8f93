"""CPU oracle of scaled dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  Plain float64 numpy,
one head at a time, written from the definition:

  S = scale * Q K^T, with S[i, j] = -inf where the mask hides key j from
      query i (causal: j > i; a per-key mask key_mask[j] == 0 hides key j
      from every query, limn, "The op set": masking is a flag per key that
      composes with causal);
  L[i] = log sum_j exp(S[i, j])            (the logsumexp the forward saves;
                                           limn, "The op set": the fused
                                           attention op saves L);
  P = exp(S - L)                           (each row sums to 1);
  O = P V.
A query that sees no key at all (every key masked) has no softmax; the
reading taken here: its O is 0, its L is -inf and its P row is 0.

Backward, by the chain rule through O = P V and the row softmax (the form
Tiki's FlashAttention backward target spells out, "Write the attention
kernel at the algorithm level"):

  dV = P^T dO;     dP = dO V^T;     D[i] = sum_d dO[i, d] O[i, d];
  dS = P * (dP - D[:, None]);      dQ = scale * dS K;      dK = scale * dS^T Q.

A library matrix product serves as the step of each contraction.
"""
from __future__ import annotations

import numpy as np


def _mask(Tq: int, Tk: int, causal: bool, key_mask=None) -> np.ndarray:
    """True where query i may see key j (causal: j <= i)."""
    vis = np.tril(np.ones((Tq, Tk), dtype=bool)) if causal else np.ones((Tq, Tk), dtype=bool)
    if key_mask is not None:
        vis = vis & (np.asarray(key_mask) != 0)[None, :]
    return vis


def _head_masks(Hn, Tq, Tk, causal, key_mask):
    """The visibility of each head: key_mask is None, or one [Tk] row per
    head (a [B, T] mask repeated over the heads of each batch)."""
    if key_mask is None:
        v = _mask(Tq, Tk, causal)
        return [v] * Hn
    km = np.asarray(key_mask).reshape(Hn, Tk)
    return [_mask(Tq, Tk, causal, km[h]) for h in range(Hn)]


def attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, causal: bool = True,
                  key_mask=None):
    """q, k, v: [heads, T, hd] -> (O [heads, T, hd], L [heads, T]), float64.
    key_mask: None or [heads, T] (nonzero: the key is visible)."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    Hn, T, _ = q.shape
    masks = _head_masks(Hn, T, k.shape[1], causal, key_mask)
    O = np.zeros((Hn, T, v.shape[2]))
    L = np.zeros((Hn, T))
    for h in range(Hn):
        vis = masks[h]
        S = scale * (q[h] @ k[h].T)
        S = np.where(vis, S, -np.inf)
        seen = vis.any(axis=1)
        m = np.where(seen, S.max(axis=1), 0.0)[:, None]
        e = np.where(vis, np.exp(S - m), 0.0)
        s = e.sum(axis=1, keepdims=True)
        L[h] = np.where(seen, (m + np.log(np.where(seen[:, None], s, 1.0)))[:, 0], -np.inf)
        O[h] = (e / np.where(seen[:, None], s, 1.0)) @ v[h]
    return O, L


def attention_bwd(q, k, v, o, do, L, scale: float, causal: bool = True, key_mask=None):
    """Gradients (dQ, dK, dV) of the forward above for the output gradient
    dO, all [heads, T, hd], float64."""
    q, k, v, o, do, L = (np.asarray(x, np.float64) for x in (q, k, v, o, do, L))
    Hn, T, _ = q.shape
    masks = _head_masks(Hn, T, k.shape[1], causal, key_mask)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for h in range(Hn):
        vis = masks[h]
        S = np.where(vis, scale * (q[h] @ k[h].T), -np.inf)
        with np.errstate(invalid="ignore"):
            P = np.where(vis, np.exp(S - L[h][:, None]), 0.0)
        dv[h] = P.T @ do[h]
        dP = do[h] @ v[h].T
        D = (do[h] * o[h]).sum(axis=1)
        dS = P * (dP - D[:, None])
        dq[h] = scale * (dS @ k[h])
        dk[h] = scale * (dS.T @ q[h])
    return dq, dk, dv
