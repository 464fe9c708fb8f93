"""Node programs for the standard compositions of the op set.

Each function returns psg_node programs spelled only in primitives, the way
limn composes them ("Three rules hold it together": softmax, relu, matmul and
the rest are built from the primitives).
"""
from __future__ import annotations

from ._abi import RED_MAX, RED_SUM, node as N


def where_exp_log_chain():
    """y = WHERE(CMPLT(a, b), EXP(a*0.5), LOG(b*b + 1)); inputs a, b (f32)."""
    return [N("LOAD", 0), N("LOAD", 1), N("CMPLT", 0, 1), N("CONST", cval=0.5), N("MUL", 0, 3),
            N("EXP", 4), N("MUL", 1, 1), N("CONST", cval=1.0), N("ADD", 6, 7), N("LOG", 8),
            N("WHERE", 2, 5, 9)]


def softmax_rows(dt="f32"):
    """Softmax over the last dim as two reductions and an epilogue:
    m = MAX(x); s = SUM(EXP(x + NEG(m))); y = EXP(x + NEG(m)) * RECIP(s)
    (Litmus R1/R2 hold by construction: x - m <= 0 and s >= 1).  x may be a
    half width: it is CAST to f32, and y is CAST back to x's dtype."""
    lx = [N("LOAD", 0, dtype=dt)] + ([N("CAST", 0, dtype="f32")] if dt != "f32" else [])
    x = len(lx) - 1
    stage0 = list(lx)
    stage1 = lx + [N("RED", 0), N("NEG", x + 1), N("ADD", x, x + 2), N("EXP", x + 3)]
    epi = lx + [N("RED", 0), N("NEG", x + 1), N("ADD", x, x + 2), N("EXP", x + 3), N("RED", 1),
                N("RECIP", x + 5), N("MUL", x + 4, x + 6)]
    if dt != "f32":
        epi.append(N("CAST", len(epi) - 1, dtype=dt))
    return [(RED_MAX, stage0), (RED_SUM, stage1)], epi


def rmsnorm(n: int, eps: float = 1e-6, dt="bf16"):
    """Tiki's RMSNorm target: xf = f32(x); inv = RECIP(SQRT(SUM(xf*xf) * (1/n)
    + eps)); y = dt((xf * inv) * f32(w)).  Inputs x [R, n] and w viewed as
    [R, n] with stride 0 over rows."""
    stage = [N("LOAD", 0, dtype=dt), N("CAST", 0, dtype="f32"), N("MUL", 1, 1)]
    epi = [N("LOAD", 0, dtype=dt), N("CAST", 0, dtype="f32"), N("RED", 0), N("CONST", cval=1.0 / n),
           N("MUL", 2, 3), N("CONST", cval=eps), N("ADD", 4, 5), N("SQRT", 6), N("RECIP", 7),
           N("MUL", 1, 8), N("LOAD", 1, dtype=dt), N("CAST", 10, dtype="f32"), N("MUL", 9, 11),
           N("CAST", 12, dtype=dt)]
    return [(RED_SUM, stage)], epi


def sum_rows(dt="f32"):
    """SUM over the last dim, one value per row."""
    return [(RED_SUM, [N("LOAD", 0, dtype=dt)])], None


def relu_square_sum():
    """SUM(relu(x)^2) with relu = WHERE(CMPLT(0, x), x, 0): the tiny graph's
    tail, fused into the reduction's prologue."""
    pro = [N("LOAD", 0), N("CONST", cval=0.0), N("CMPLT", 1, 0), N("WHERE", 2, 0, 1), N("MUL", 3, 3)]
    return [(RED_SUM, pro)], None
