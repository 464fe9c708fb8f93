"""Comparison helpers shared by the GPU parity tests (no method arithmetic)."""
import numpy as np
import torch

import seeded_inputs as SI

U = 2.0 ** -24


def gamma(n):
    n = max(int(n), 0)
    return n * U / (1 - n * U)


def ulp_dist_f32(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in float32 ulps (ordered-int difference); NaN==NaN -> 0,
    NaN vs number -> huge."""
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    ia = a.view(np.int32).astype(np.int64)
    ib = b.view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, np.int64(-2**31) - ia, ia)
    ib = np.where(ib < 0, np.int64(-2**31) - ib, ib)
    d = np.abs(ia - ib)
    na, nb = np.isnan(a), np.isnan(b)
    d = np.where(na & nb, 0, d)
    d = np.where(na ^ nb, np.int64(1) << 40, d)
    return d


def same_bits_nan_equal(a: np.ndarray, b: np.ndarray, float_kind: bool):
    """Bitwise equality, except that any two NaNs compare equal."""
    if a.shape != b.shape:
        return False
    if not float_kind:
        return np.array_equal(a, b)
    av, bv = a.view(np.uint8).reshape(a.shape + (-1,)), b.view(np.uint8).reshape(b.shape + (-1,))
    eq = np.all(av == bv, axis=-1)
    return bool(np.all(eq | (_isnan_bits(a) & _isnan_bits(b))))


def _isnan_bits(x: np.ndarray) -> np.ndarray:
    if x.dtype == np.uint16:  # bfloat16 bits
        return ((x & 0x7F80) == 0x7F80) & ((x & 0x007F) != 0)
    if x.dtype.kind == "f":
        return np.isnan(x)
    return np.zeros(x.shape, bool)


def to_np(t: torch.Tensor) -> np.ndarray:
    return SI.bits(t)


def dev(t: torch.Tensor) -> torch.Tensor:
    return t.to("cuda")


def storage_dtype(name):
    return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16, "f64": torch.float64,
            "i32": torch.int32, "i16": torch.int16, "i8": torch.int8}[name]


def first_mismatches(a: np.ndarray, b: np.ndarray, k=5):
    """Positions and values of the first k cells whose bits differ (NaN==NaN)."""
    av = a.reshape(-1)
    bv = b.reshape(-1)
    nan_a, nan_b = _isnan_bits(av), _isnan_bits(bv)
    bad = np.nonzero((av.view(np.uint8).reshape(av.shape + (-1,)) !=
                      bv.view(np.uint8).reshape(bv.shape + (-1,))).any(axis=-1) & ~(nan_a & nan_b))[0]
    return [(int(i), av[i], bv[i]) for i in bad[:k]], int(bad.size)


def _visible(T, causal, km=None):
    v = np.tril(np.ones((T, T), bool)) if causal else np.ones((T, T), bool)
    return v if km is None else v & (np.asarray(km) != 0)[None, :]


def _probs(Q, K, L, scale, vis, h):
    with np.errstate(invalid="ignore", over="ignore"):
        return np.where(vis, np.exp(scale * Q[h] @ K[h].T - L[h][:, None]), 0.0)


def attention_fwd_bounds(Q, K, V, O_ref, L_ref, scale, causal, key_mask=None):
    """Per-cell bound on the fused forward's output O (heads [BH, T, d],
    float64 oracle values): S is a float32 sum of exact bf16 products, P
    rounds to bf16 before P V, and O rounds once to bf16:
        |O - O*| <= 2^-8 * sum_j P*_ij |V_jd| + 2^-7 |O*|.
    key_mask: None or [heads, T] (nonzero: visible)."""
    mag = np.zeros_like(O_ref)
    for h in range(Q.shape[0]):
        vis = _visible(Q.shape[1], causal, None if key_mask is None else key_mask[h])
        P = _probs(Q, K, L_ref, scale, vis, h)
        mag[h] = P @ np.abs(V[h])
    return 2.0 ** -8 * mag + 2.0 ** -7 * np.abs(O_ref)


def attention_bwd_bounds(Q, K, V, O, dO, L, scale, causal, refs, key_mask=None, o_err=None):
    """Per-cell bounds on the fused backward's (dQ, dK, dV) against the
    float64 oracle values refs = (dQ*, dK*, dV*): P and dS round to bf16
    before the second products and every output rounds once to bf16:
        dV:     2^-8 * sum_i P_ij |dO_id|                          + 2^-7 |dV*|
        dQ, dK: 2^-7 * scale * sum_j P_ij (|dP_ij| + |D_i|) |K_jd|   + 2^-7 |dQ*|.
    o_err: None when the backward reads the O the oracle used; else a bound
    on |O_read - O| per cell (the forward's own bar, when refs come from the
    exact O but the backward reads the forward's bf16 output).  Its effect on
    D_i = sum_d dO_id O_id, e_i = sum_d |dO_id| o_err_id, reaches dS as
    P_ij e_i and adds scale * sum_j P_ij e_i |K_jd| to dQ (and the transpose
    to dK); dV does not read O."""
    mq, mk, mv = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
    eq, ek = np.zeros_like(Q), np.zeros_like(K)
    for h in range(Q.shape[0]):
        vis = _visible(Q.shape[1], causal, None if key_mask is None else key_mask[h])
        P = _probs(Q, K, L, scale, vis, h)
        dP = dO[h] @ V[h].T
        D = (dO[h] * O[h]).sum(1)
        G = np.abs(P) * (np.abs(dP) + np.abs(D)[:, None])
        mv[h] = P.T @ np.abs(dO[h])
        mq[h] = scale * (G @ np.abs(K[h]))
        mk[h] = scale * (G.T @ np.abs(Q[h]))
        if o_err is not None:
            E = np.abs(P) * (np.abs(dO[h]) * o_err[h]).sum(1)[:, None]
            eq[h] = scale * (E @ np.abs(K[h]))
            ek[h] = scale * (E.T @ np.abs(Q[h]))
    dq, dk, dv = refs
    return (2.0 ** -7 * mq + 2.0 ** -7 * np.abs(dq) + eq, 2.0 ** -7 * mk + 2.0 ** -7 * np.abs(dk) + ek,
            2.0 ** -8 * mv + 2.0 ** -7 * np.abs(dv))
