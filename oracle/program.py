"""Oracle evaluation of one library call from its arguments.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py): only the tests, the smoke
check and the bench's CPU legs use it, and it imports nothing of the CUDA
library.  A call is described in plain Python data:

  node   (op, a, b, c, dtype, cval) with op one of LOAD CONST RED ACC NEG EXP
         LOG SQRT RECIP CAST ADD MUL CMPLT WHERE: a postfix program whose
         operands name earlier nodes by index and whose last node is the
         result;
  load   an oracle tensor already read through its View (:func:`read`), at
         the call's iteration shape.

Every node is one primitive of limn's closed op set ("The op set"),
materialised in its own dtype by the node functions of oracle/__init__.py,
one after another, with no fusion (limn, "Three rules hold it together": the
numpy device interprets the graph one call per node and every compiled
backend is diffed against it).  A reduction is SUM or MAX over the last dim
with a float32 running total rounded once (the dtype paragraph of "The op
set"); a contraction is the naive k-ascending loop (Luminal IR blog, "Naive
Matrix Multiplication").

``hook``: an optional callable ``hook(kind, index, value) -> value`` that is
given each node value (kind "node") and each reduced stage value (kind
"stage") as it is produced and returns the value to carry on with.  It is
None for the plain evaluation; the tests pass one to evaluate the same
program with a value moved to the edge of its allowed deviation, which is
how they derive a per-cell tolerance.
"""
from __future__ import annotations

import numpy as np

from . import (_NP, T, add, cast, cmplt, exp, full, log, matmul_bt, mul, neg, recip, reduce_max, reduce_sum, sqrt,
               view, where)

OPS = ("LOAD", "CONST", "RED", "ACC", "NEG", "EXP", "LOG", "SQRT", "RECIP", "CAST", "ADD", "MUL", "CMPLT",
       "WHERE")
_UNARY = {"NEG": neg, "EXP": exp, "LOG": log, "SQRT": sqrt, "RECIP": recip}
_BINARY = {"ADD": add, "MUL": mul, "CMPLT": cmplt}


def read(flat_bits: np.ndarray, dt: str, shape, strides, offset=0, mask=None) -> T:
    """Materialise a View (shape, strides, offset, mask) of a flat buffer
    holding ``dt``'s storage bits."""
    return view(T(np.ascontiguousarray(flat_bits).reshape(-1), dt), shape, strides, offset, mask)


def _expand(x: T, shape) -> T:
    """A [.., 1]-shaped (or scalar) value broadcast to ``shape`` by a
    stride-0 View: the same value in every cell it reaches."""
    flat = x.data.reshape(-1)
    if flat.size == 1:
        return view(T(flat, x.dt), shape, [0] * len(shape))
    rows = flat.size
    n = shape[-1]
    if rows * n != int(np.prod(shape)):
        raise ValueError("stage value of %d rows cannot expand to %s" % (rows, shape))
    return view(T(flat, x.dt), (rows, n), (1, 0)).reshape(shape)


def program(nodes, loads, shape, reds=(), hook=None, acc=None) -> T:
    """Evaluate a postfix program node by node over ``shape``.  loads[k] is
    input k read through its View at ``shape``; reds[s] is stage s's reduced
    value (shape [rows, 1]), broadcast over the row wherever a RED node reads
    it; acc is the float32 value an ACC node reads (a contraction's totals,
    shape ``shape``).  Returns the last node's value."""
    shape = tuple(int(s) for s in shape)
    vals = []
    for i, (op, a, b, c, dt, cval) in enumerate(nodes):
        if op == "LOAD":
            x = loads[a]
            if x.dt != dt:
                raise TypeError("LOAD %d: node dtype %s, input dtype %s" % (a, dt, x.dt))
            if x.shape != shape:
                x = x.reshape(shape)
        elif op == "CONST":
            x = full(shape, cval, dt)
        elif op == "RED":
            x = _expand(reds[a], shape)
            if x.dt != dt:
                raise TypeError("RED %d: node dtype %s, stage dtype %s" % (a, dt, x.dt))
        elif op == "ACC":
            if acc is None or acc.dt != "f32" or dt != "f32":
                raise TypeError("ACC reads a float32 contraction total")
            x = acc if acc.shape == shape else acc.reshape(shape)
        elif op in _UNARY:
            x = _UNARY[op](vals[a])
        elif op == "CAST":
            x = cast(vals[a], dt)
        elif op in _BINARY:
            x = _BINARY[op](vals[a], vals[b])
        elif op == "WHERE":
            x = where(vals[a], vals[b], vals[c])
        else:
            raise ValueError("unknown op %r" % (op,))
        if x.dt != dt:
            raise TypeError("node %d (%s) computed %s, declared %s" % (i, op, x.dt, dt))
        if hook is not None:
            x = hook("node", i, x)
        vals.append(x)
    return vals[-1]


def reduce_rows(stages, epilogue, loads, per_element: bool, hook=None):
    """SUM/MAX row reductions with a prologue per stage and an epilogue.

    stages: sequence of (op, prologue nodes), op "SUM" or "MAX"; loads: the
    inputs read at the iteration shape [.., N] (the last dim is reduced).
    Stage s folds its prologue's values over each row into the prologue's
    dtype (float32 total for floats, wrapping int32 total for ints, rounded
    once); a later prologue may read earlier stage values through RED.
    per_element: the epilogue runs per cell over [.., N] (it may read the
    inputs); otherwise once per row over [.., 1] (constants and stage values
    only), and an empty epilogue returns the last stage's value.
    Returns (output, [stage values [rows, 1]], [prologue values [rows, N]])."""
    shape = tuple(loads[0].shape) if loads else None
    if shape is None:
        raise ValueError("a row reduction needs at least one input")
    N = shape[-1]
    rows = int(np.prod(shape[:-1], dtype=np.int64)) if len(shape) > 1 else 1
    flat = [x.reshape((rows, N)) for x in loads]
    reds, pro = [], []
    for s, (op, nodes) in enumerate(stages):
        p = program(nodes, flat, (rows, N), reds, hook=None if hook is None else
                    (lambda kind, i, x, s=s: hook("prologue%d" % s, i, x)))
        r = reduce_sum(p) if op == "SUM" else reduce_max(p)
        if hook is not None:
            r = hook("stage", s, r)
        reds.append(r)
        pro.append(p)
    if per_element:
        out = program(epilogue, flat, (rows, N), reds, hook=None if hook is None else
                      (lambda kind, i, x: hook("epilogue", i, x)))
        return out.reshape(shape), reds, pro
    if not epilogue:
        return reds[-1], reds, pro
    out = program(epilogue, [], (rows, 1), reds, hook=None if hook is None else
                  (lambda kind, i, x: hook("epilogue", i, x)))
    return out, reds, pro


def contract(a: T, bt: T, out_dt: str) -> T:
    """C[z, m, n] = sum over k ascending of A[z, m, k] * B[z, k, n] for each
    batch index z, with B given transposed (bt[z, n, k]); the float32 total
    rounds once into ``out_dt``."""
    if a.data.ndim != 3 or bt.data.ndim != 3 or a.shape[0] != bt.shape[0] or a.shape[2] != bt.shape[2]:
        raise ValueError("contract wants a [Z, M, K] and bt [Z, N, K]")
    Z, M, _ = a.shape
    N = bt.shape[1]
    out = np.empty((Z, M, N), dtype=_NP[out_dt])
    for z in range(Z):
        out[z] = matmul_bt(T(a.data[z], a.dt), T(bt.data[z], bt.dt), out_dt).data
    return T(out, out_dt)


def contract_epilogue(a: T, bt: T, nodes, loads, hook=None) -> T:
    """A contraction whose cells go through an epilogue program: ACC is each
    cell's float32 total (:func:`contract` before any rounding), LOAD k the
    epilogue's input k at the same cell (loads: [Z, M, N] tensors).  The
    elementwise program then runs node by node over [Z, M, N] (limn,
    "Reading the schedule": elementwise work fused into the kernel that
    produces its operand computes what the separate nodes compute)."""
    tot = contract(a, bt, "f32")
    return program(nodes, loads, tot.shape, hook=hook, acc=tot)
