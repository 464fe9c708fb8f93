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
