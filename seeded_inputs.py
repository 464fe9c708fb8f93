"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no arithmetic of the method: it only draws random numbers
with ``torch.Generator('cpu').manual_seed(seed)`` and returns CPU tensors
(bfloat16 tensors can be handed to the oracle as uint16 bit patterns with
:func:`bits`).  Draw order within a workload is fixed and documented.
"""
from __future__ import annotations

import numpy as np
import torch


def gen(seed: int = 0) -> torch.Generator:
    g = torch.Generator("cpu")
    g.manual_seed(int(seed))
    return g


def uniform(shape, lo, hi, g, dtype=torch.float32):
    return (torch.rand(shape, generator=g, dtype=torch.float32) * (hi - lo) + lo).to(dtype)


def normal(shape, mean, std, g, dtype=torch.float32):
    return (torch.randn(shape, generator=g, dtype=torch.float32) * std + mean).to(dtype)


def bits(t: torch.Tensor) -> np.ndarray:
    """CPU tensor -> numpy storage array (bfloat16 as uint16 bit patterns)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


DTYPE_NAME = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16",
              torch.float64: "f64", torch.int32: "i32", torch.int16: "i16", torch.int8: "i8"}


# ---- the five workloads (sizes as stated for each) ------------------------

def tiny_graph(seed=0, M=64, K=32, N=48):
    """A[M,K], B[K,N] ~ N(0,1) float32, A drawn first."""
    g = gen(seed)
    return normal((M, K), 0.0, 1.0, g), normal((K, N), 0.0, 1.0, g)


def chain(seed=0, R=4096, C=4096):
    """a[R,C] ~ U(-4,4) float32 and the column b[R] ~ U(-4,4), a drawn first."""
    g = gen(seed)
    return uniform((R, C), -4.0, 4.0, g), uniform((R,), -4.0, 4.0, g)


def transpose_input(seed=0, R=8192, C=8192):
    g = gen(seed)
    return uniform((R, C), -1.0, 1.0, g)


def softmax_input(seed=0, R=4096, N=1024):
    g = gen(seed)
    return uniform((R, N), -1000.0, 1000.0, g)


def rmsnorm_input(seed=0, R=8192, N=4096):
    """x[R,N] ~ N(0,1) and w[N] ~ N(1, 0.1), both bfloat16, x drawn first."""
    g = gen(seed)
    return normal((R, N), 0.0, 1.0, g, torch.bfloat16), normal((N,), 1.0, 0.1, g, torch.bfloat16)


def contraction_bf16(seed=0, M=8192, N=8192, K=8192):
    """A[M,K], B[K,N] bfloat16 ~ N(0, std=1/sqrt(K)), A drawn first."""
    g = gen(seed)
    s = 1.0 / float(np.sqrt(K))
    return normal((M, K), 0.0, s, g, torch.bfloat16), normal((K, N), 0.0, s, g, torch.bfloat16)


def contraction_f32(seed=0, M=4096, N=4096, K=4096):
    g = gen(seed)
    return normal((M, K), 0.0, 1.0, g), normal((K, N), 0.0, 1.0, g)


def contraction_i8(seed=0, M=2048, N=2048, K=2048):
    """A[M,K], B[K,N] int8 uniform over [-128, 127], A drawn first."""
    g = gen(seed)
    a = torch.randint(-128, 128, (M, K), generator=g, dtype=torch.int64).to(torch.int8)
    b = torch.randint(-128, 128, (K, N), generator=g, dtype=torch.int64).to(torch.int8)
    return a, b


GPT_SHAPES = dict(B=32, T=256, V=256, D=512, H=8, F=2048)


def gpt_block(seed=0, B=32, T=256, V=256, D=512, H=8, F=2048, std=0.02):
    """Tokens [B,T] int32 uniform over [0, V) and bfloat16 weights ~ N(0, std)
    in the order E, P, Wqkv, Wo, W1, W2, Wlm; RMSNorm weights are ones."""
    g = gen(seed)
    tok = torch.randint(0, V, (B, T), generator=g, dtype=torch.int64).to(torch.int32)
    w = {}
    for name, shape in (("E", (V, D)), ("P", (T, D)), ("Wqkv", (D, 3 * D)), ("Wo", (D, D)),
                        ("W1", (D, F)), ("W2", (F, D)), ("Wlm", (D, V))):
        w[name] = normal(shape, 0.0, std, g, torch.bfloat16)
    for name in ("g1", "g2", "gf"):
        w[name] = torch.ones((D,), dtype=torch.bfloat16)
    return tok, w


# ---- aimed generators (Litmus, "TargetedFalsification") -------------------

def aimed(kind: str, shape, g, dtype=torch.float32):
    """Value distributions aimed at the bug families a uniform [0,1) draw
    misses: large magnitude, all-negative, subnormal, specials, constant rows,
    cancellation, sorted rows, near-saturation."""
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if kind == "large":
        x = x * 1e30
    elif kind == "negative":
        x = -x.abs() - 1.0
    elif kind == "subnormal":
        x = x * 1e-39
    elif kind == "specials":
        flat = x.reshape(-1)
        n = flat.numel()
        pick = torch.randint(0, n, (max(1, n // 16),), generator=g)
        vals = torch.tensor([float("nan"), float("inf"), float("-inf"), 0.0, -0.0])
        flat[pick] = vals[torch.randint(0, 5, (pick.numel(),), generator=g)]
        x = flat.reshape(shape)
    elif kind == "constant":
        x = x[..., :1].expand(shape).contiguous()
    elif kind == "cancel":
        x = x * 1e4
        x[..., 1::2] = -x[..., 0::2][..., : x[..., 1::2].shape[-1]]
    elif kind == "sorted":
        x = torch.sort(x, dim=-1).values
    elif kind == "saturating":
        x = x.abs() * 80.0
    elif kind != "normal":
        raise ValueError(kind)
    return x.to(dtype)


AIMED_KINDS = ("normal", "large", "negative", "subnormal", "specials", "constant", "cancel",
               "sorted", "saturating")


def shape_classes(block: int):
    """Litmus "SymbolicShapeSpace" size classes for one guarded dim."""
    return sorted({1, block - 1, block, block + 1, 2 * block, 3 * block + 7, 97})
