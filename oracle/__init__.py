"""Plain CPU oracle for the primitive-op graph hot path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this package.  It
shares no code with the CUDA library and never imports it.

Each function is one primitive node of limn's closed op set ("The op set":
sources, VIEW, NEG EXP LOG SQRT RECIP CAST, ADD MUL CMPLT, WHERE, SUM MAX,
GATHER SCATTER), evaluated by one plain C loop nest in ``oracle.c`` over a
materialised buffer, in the spirit of limn's numpy device ("Three rules hold
it together": one call per node, no fusion).  The composed ops at the bottom
(matmul, softmax, RMSNorm, layernorm, the tiny graph and the elementwise
chain) are spelled in those primitives and nothing else.

Tensors are :class:`T`: a numpy array holding the storage bits plus a dtype
name.  bfloat16 is stored as uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")

# the oracle's own dtype numbering (see oracle.c)
_DT = {"f32": 0, "bf16": 1, "f16": 2, "f64": 3, "i32": 4, "i16": 5, "i8": 6}
_NP = {"f32": np.float32, "bf16": np.uint16, "f16": np.float16, "f64": np.float64,
       "i32": np.int32, "i16": np.int16, "i8": np.int8}
_U = {"neg": 0, "exp": 1, "log": 2, "sqrt": 3, "recip": 4}
_B = {"add": 0, "mul": 1, "cmplt": 2}
_R = {"sum": 0, "max": 1}

#: OpenMP team size used by every loop nest (1 = serial).  Output cells are
#: split between threads, so any value gives the same bits.
NTHREADS = 1


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (no FMA contraction)."""
    src = os.path.join(_HERE, "oracle.c")
    if (not force and os.path.exists(_SO)
            and os.path.getmtime(_SO) >= os.path.getmtime(src)):
        return _SO
    tmp = _SO + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_SO)
        i64, i32, vp, dp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p
        L.orc_view_read.argtypes = [i32, vp, i64, i32, dp, dp, i64, dp, dp, vp]
        L.orc_unary.argtypes = [i32, i32, vp, vp, i64, i32]
        L.orc_cast.argtypes = [i32, vp, i32, vp, i64, i32]
        L.orc_binary.argtypes = [i32, i32, vp, vp, vp, i64, i32]
        L.orc_where.argtypes = [i32, vp, i32, vp, vp, vp, i64, i32]
        L.orc_reduce.argtypes = [i32, i32, vp, i64, i64, vp, i32]
        L.orc_matmul.argtypes = [i32, vp, vp, i32, vp, i64, i64, i64, i32]
        L.orc_matmul_bt.argtypes = [i32, vp, vp, i32, vp, i64, i64, i64, i32]
        L.orc_matmul_cells.argtypes = [i32, vp, vp, i64, i64, i64, vp, vp, i64, vp, vp, i32]
        L.orc_gather_rows.argtypes = [i32, vp, i64, i64, vp, i64, vp]
        L.orc_gather_rows.restype = i64
        L.orc_scatter_add_rows.argtypes = [i32, vp, i64, i64, vp, i64, vp]
        L.orc_scatter_add_rows.restype = i64
        L.orc_omp_max_threads.restype = i32
        fl = ctypes.c_float
        L.orc_adamw.argtypes = [i32, vp, vp, vp, vp, i64, fl, fl, fl, fl, fl, fl, fl]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class T:
    """An oracle tensor: contiguous storage bits plus a dtype name."""
    data: np.ndarray
    dt: str

    def __post_init__(self):
        d = np.asarray(self.data, dtype=_NP[self.dt])
        self.data = d if d.flags.c_contiguous else d.copy(order="C")

    @property
    def shape(self):
        return tuple(self.data.shape)

    def numel(self):
        return int(self.data.size)

    def f64(self) -> np.ndarray:
        """Exact float64 copy of the values (for checks)."""
        if self.dt == "bf16":
            return (self.data.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        return self.data.astype(np.float64)

    def reshape(self, shape):
        """A reshape of a contiguous buffer is a View that moves no data."""
        return T(self.data.reshape(shape), self.dt)


def tensor(values, dt: str) -> T:
    """Build an oracle tensor from float/int values, rounding into ``dt`` with
    the oracle's own CAST (float64 -> dt)."""
    v = np.asarray(values)
    if dt in ("i32", "i16", "i8"):
        return T(v.astype(np.int64).astype(_NP[dt]), dt)
    src = T(v.astype(np.float64), "f64")
    return cast(src, dt)


# ---------------------------------------------------------------- VIEW ------

def view(base: T, shape, strides, offset=0, mask=None) -> T:
    """Materialise a View of ``base``'s flat storage (limn, "Three rules":
    a View is shape, strides, offset, mask; masked-out cells read 0)."""
    shape = [int(s) for s in shape]
    nd = len(shape)
    if mask is None:
        mask = [(0, s) for s in shape]
    sh = np.array(shape, np.int64)
    st = np.array([int(s) for s in strides], np.int64)
    lo = np.array([int(m[0]) for m in mask], np.int64)
    hi = np.array([int(m[1]) for m in mask], np.int64)
    out = np.empty(shape, _NP[base.dt])
    flat = np.ascontiguousarray(base.data).reshape(-1)
    rc = lib().orc_view_read(_DT[base.dt], _p(flat), flat.size, nd, _p(sh), _p(st), int(offset),
                             _p(lo), _p(hi), _p(out))
    if rc != 0:
        raise IndexError("view reads outside its buffer")
    return T(out, base.dt)


def expand_last(col: T, n: int) -> T:
    """[R, 1] (or [R]) -> [R, n] by a stride-0 View (limn's expand)."""
    r = col.numel()
    return view(col, (r, n), (1, 0))


def full(shape, value, dt: str) -> T:
    """CONST node broadcast over ``shape``: the python scalar takes the
    tensor's dtype (limn, "The op set", dtype paragraph)."""
    c = tensor([value], dt)
    return view(c, shape, [0] * len(shape))


# --------------------------------------------------------- elementwise ------

def _unary(op, x: T) -> T:
    y = np.empty_like(x.data)
    rc = lib().orc_unary(_U[op], _DT[x.dt], _p(x.data), _p(y), x.numel(), NTHREADS)
    if rc != 0:
        raise TypeError("%s undefined on %s" % (op, x.dt))
    return T(y, x.dt)


def neg(x): return _unary("neg", x)
def exp(x): return _unary("exp", x)
def log(x): return _unary("log", x)
def sqrt(x): return _unary("sqrt", x)
def recip(x): return _unary("recip", x)


def cast(x: T, dt: str) -> T:
    y = np.empty(x.shape, _NP[dt])
    lib().orc_cast(_DT[x.dt], _p(x.data), _DT[dt], _p(y), x.numel(), NTHREADS)
    return T(y, dt)


def _binary(op, a: T, b: T) -> T:
    if a.dt != b.dt or a.shape != b.shape:
        raise TypeError("binary node needs equal dtypes and shapes")
    y = np.empty_like(a.data)
    lib().orc_binary(_B[op], _DT[a.dt], _p(a.data), _p(b.data), _p(y), a.numel(), NTHREADS)
    return T(y, a.dt)


def add(a, b): return _binary("add", a, b)
def mul(a, b): return _binary("mul", a, b)
def cmplt(a, b): return _binary("cmplt", a, b)


def where(c: T, x: T, y: T) -> T:
    if x.dt != y.dt or not (c.shape == x.shape == y.shape):
        raise TypeError("WHERE needs equal shapes and branch dtypes")
    out = np.empty_like(x.data)
    lib().orc_where(_DT[c.dt], _p(c.data), _DT[x.dt], _p(x.data), _p(y.data), _p(out),
                    x.numel(), NTHREADS)
    return T(out, x.dt)


# -------------------------------------------------------------- reduce ------

def _reduce(op, x: T, keepdim=True) -> T:
    cols = x.shape[-1] if x.shape else 1
    rows = int(np.prod(x.shape[:-1], dtype=np.int64)) if x.shape else 1
    out = np.empty(x.shape[:-1] + ((1,) if keepdim else ()), _NP[x.dt])
    lib().orc_reduce(_R[op], _DT[x.dt], _p(x.data), rows, cols, _p(out), NTHREADS)
    return T(out, x.dt)


def reduce_sum(x, keepdim=True): return _reduce("sum", x, keepdim)
def reduce_max(x, keepdim=True): return _reduce("max", x, keepdim)


# ------------------------------------------------------------ contraction ---

def matmul_views(M, N, K):
    """The two broadcast Views that turn a matmul into MUL then SUM over k:
    A [M,K] -> [M,N,K] strides (K,0,1); B [K,N] -> [M,N,K] strides (0,1,N)
    (limn, "Reading the schedule": in0[i0*K + r2], in1[i1 + r2*N];
    Luminal IR blog, "Naive Matrix Multiplication": a stride-0 loop)."""
    return ((M, N, K), (K, 0, 1)), ((M, N, K), (0, 1, N))


def matmul_literal(A: T, B: T) -> T:
    """matmul as the reference interpreter runs it: materialise the (M,N,K)
    broadcast product, then SUM over k (limn, "Three rules": a matmul is a
    broadcast multiply and a reduce).  Result [M, N, 1] in A's dtype."""
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    (sa, ta), (sb, tb) = matmul_views(M, N, K)
    prod = mul(view(A, sa, ta), view(B, sb, tb))
    return reduce_sum(prod)


def matmul(A: T, B: T, out_dt: str | None = None) -> T:
    """The fused naive loop of the Luminal IR blog ("Naive Matrix
    Multiplication"): same products, same k order, same float32 total as
    :func:`matmul_literal`, without the (M,N,K) intermediate."""
    M, K = A.shape
    K2, N = B.shape
    assert K == K2 and A.dt == B.dt
    out_dt = out_dt or A.dt
    C = np.empty((M, N), _NP[out_dt])
    lib().orc_matmul(_DT[A.dt], _p(A.data), _p(B.data), _DT[out_dt], _p(C), M, N, K, NTHREADS)
    return T(C, out_dt)


def matmul_bt(A: T, BT: T, out_dt: str | None = None) -> T:
    """:func:`matmul` with B given transposed ([N, K]): the same products in
    the same k order (so the same bits), walking memory row by row."""
    M, K = A.shape
    N, K2 = BT.shape
    assert K == K2 and A.dt == BT.dt
    out_dt = out_dt or A.dt
    C = np.empty((M, N), _NP[out_dt])
    rc = lib().orc_matmul_bt(_DT[A.dt], _p(A.data), _p(BT.data), _DT[out_dt], _p(C), M, N, K, NTHREADS)
    if rc != 0:
        raise TypeError("matmul_bt on %s" % A.dt)
    return T(C, out_dt)


def matmul_cells(A: T, B: T, ii, jj):
    """Sampled cells of the fused loop: returns (float32 totals, sum |a*b|)."""
    M, K = A.shape
    _, N = B.shape
    ii = np.ascontiguousarray(ii, np.int64)
    jj = np.ascontiguousarray(jj, np.int64)
    acc = np.empty(ii.size, np.float32)
    mag = np.empty(ii.size, np.float64)
    lib().orc_matmul_cells(_DT[A.dt], _p(A.data), _p(B.data), M, N, K, _p(ii), _p(jj), ii.size,
                           _p(acc), _p(mag), NTHREADS)
    return acc, mag


# ------------------------------------------------------------- indexed ------

def gather_rows(src: T, idx: np.ndarray):
    """GATHER along dim 0: out[n,:] = src[idx[n],:].  Returns (out, #bad)."""
    V = src.shape[0]
    D = src.numel() // max(V, 1)
    idx = np.ascontiguousarray(idx, np.int32)
    out = np.empty((idx.size,) + src.shape[1:], _NP[src.dt])
    bad = lib().orc_gather_rows(_DT[src.dt], _p(src.data), V, D, _p(idx), idx.size, _p(out))
    return T(out, src.dt), int(bad)


def scatter_add_rows(dst: T, idx: np.ndarray, upd: T):
    """SCATTER-add along dim 0, n ascending: dst[idx[n],:] += upd[n,:].
    Returns (new dst, #bad)."""
    V = dst.shape[0]
    D = dst.numel() // max(V, 1)
    idx = np.ascontiguousarray(idx, np.int32)
    out = dst.data.copy()
    bad = lib().orc_scatter_add_rows(_DT[dst.dt], _p(out), V, D, _p(idx), idx.size,
                                     _p(upd.data))
    return T(out, dst.dt), int(bad)


# ------------------------------------------------------- composed ops -------

def relu(x: T) -> T:
    """relu = WHERE(CMPLT(0, x), x, 0) (limn: relu is composed, "Three rules")."""
    z = full(x.shape, 0, x.dt)
    return where(cmplt(z, x), x, z)


def softmax_rows(x: T) -> T:
    """Softmax over the last dim in primitives: m = MAX; e = EXP(x + NEG(m));
    s = SUM(e); y = e * RECIP(s)  (limn composes softmax; Litmus R1/R2)."""
    R = x.numel() // x.shape[-1]
    N = x.shape[-1]
    x2 = x.reshape((R, N))
    m = reduce_max(x2)
    e = exp(add(x2, expand_last(neg(m), N)))
    s = reduce_sum(e)
    y = mul(e, expand_last(recip(s), N))
    return y.reshape(x.shape)


def rmsnorm(x: T, w: T, eps: float = 1e-6) -> T:
    """Tiki's RMSNorm target ("Compile model code"): xf = f32(x);
    inv = rsqrt(mean(xf*xf) + eps); y = (xf*inv*f32(w)) in x's dtype, with
    mean = SUM * (1/N), rsqrt = RECIP(SQRT), left-to-right products."""
    R = x.numel() // x.shape[-1]
    N = x.shape[-1]
    xf = cast(x.reshape((R, N)), "f32")
    ss = reduce_sum(mul(xf, xf))
    ms = mul(ss, full(ss.shape, 1.0 / N, "f32"))
    v = add(ms, full(ms.shape, eps, "f32"))
    inv = recip(sqrt(v))
    wf = view(cast(w, "f32"), (R, N), (0, 1))
    y = mul(mul(xf, expand_last(inv, N)), wf)
    return cast(y, x.dt).reshape(x.shape)


def layernorm_centred(x: T) -> T:
    """x - mean(x) over the last dim (the centring step of LayerNorm,
    Litmus lemma R3: its row sum is zero in exact arithmetic)."""
    R = x.numel() // x.shape[-1]
    N = x.shape[-1]
    x2 = x.reshape((R, N))
    mean = mul(reduce_sum(x2), full((R, 1), 1.0 / N, x.dt))
    return add(x2, expand_last(neg(mean), N))


def chain_where_exp_log(a: T, bcol: T) -> T:
    """y = WHERE(CMPLT(a, b), EXP(a*0.5), LOG(b*b + 1)) with b a [R,1] column
    expanded over a's columns (a stride-0 View)."""
    R, N = a.shape
    b = view(bcol, (R, N), (1, 0))
    half = full((R, N), 0.5, a.dt)
    one = full((R, N), 1.0, a.dt)
    return where(cmplt(a, b), exp(mul(a, half)), log(add(mul(b, b), one)))


def transpose(x: T) -> T:
    """CONTIGUOUS(permute(1,0)): a View with swapped strides, materialised."""
    R, C = x.shape
    return view(x, (C, R), (1, C))


def tiny_graph(A: T, B: T) -> T:
    """limn's README example at the tiny-graph size: SUM(relu(A@B)**2), with
    the matmul as broadcast MUL + SUM and the square as MUL(x, x)."""
    M, _ = A.shape
    _, N = B.shape
    c = matmul_literal(A, B).reshape((M, N))
    r = relu(c)
    sq = mul(r, r)
    return reduce_sum(sq.reshape((1, M * N)), keepdim=False).reshape(())


def adamw_step(p: T, g: T, m: np.ndarray, v: np.ndarray, lr: float, b1: float, b2: float, eps: float,
               wd: float, b1t: float, b2t: float):
    """One AdamW step (decoupled decay) over one tensor in float32, the C
    loop's operation order; returns (p', m', v').  b1t, b2t: b1^t, b2^t
    after this step (float32 running products)."""
    pd = np.ascontiguousarray(p.data).copy()
    gd = np.ascontiguousarray(g.data)
    mm = np.ascontiguousarray(m, np.float32).copy()
    vv = np.ascontiguousarray(v, np.float32).copy()
    lib().orc_adamw(_DT[p.dt], pd.ctypes.data, gd.ctypes.data, mm.ctypes.data, vv.ctypes.data, pd.size,
                    lr, b1, b2, eps, wd, b1t, b2t)
    return T(pd, p.dt), mm, vv


def omp_max_threads() -> int:
    return int(lib().orc_omp_max_threads())
