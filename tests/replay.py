"""Node-level replay of library calls on the oracle (test helper, no method
arithmetic of its own beyond tolerances).

While a :class:`Replayer` is active, every call the graph layer makes through
the ctypes binding is wrapped: the wrapper synchronises, copies the bytes of
each input View off the device, makes the call, synchronises again, copies
the output, and evaluates the same call on the oracle from those very input
bytes (oracle/program.py, oracle/attention.py, the node functions of
oracle/__init__.py).  Each call is therefore checked on its own, fed the
GPU's inputs, at the tolerance of its own kind (limn, "Three rules hold it
together": every backend is diffed against the reference interpreter, node
by node):

* GATHER, SCATTER-add, permute, and elementwise programs of correctly
  rounded nodes (no EXP or LOG): the same bits (NaN equal to NaN).
* Contractions: |c - c*| <= (1 + 2^-8) * 2 gamma_{K-1} sum_k |a_k b_k|
  + 2^-8 |c*| for a bfloat16 output (2^-11 for float16), with c* the oracle's
  float32 total: the reduction-order bound (Litmus, "ToleranceBound") plus
  one rounding into the narrow output.  With a fused epilogue program, the
  hull rule below, with the total itself the value moved by that bound.
* Row reductions, and elementwise programs with EXP or LOG: the oracle runs
  the call again with every value that may legitimately differ moved to
  either edge of its allowance, and the GPU cell must lie in the hull of
  those runs widened by one unit of the output dtype.  The values moved are
  each float SUM stage's total (by 2 gamma_{N-1} sum |x|, the reduction-order
  bound, applied to the float32 total before the stage's one rounding) and
  each EXP or LOG node (by 8 float32 ulps, the transcendental bound; by one
  unit of a narrower node dtype, which covers 8 float32 ulps before its
  rounding).  Every node is monotone in each moved value for the programs
  the library runs (products, sums, reciprocals and roots of a moved total,
  differences with it), so the extreme cases bound the GPU's cell.
* Attention: the per-cell bounds of tests/test_gpu_attention.py (float64
  oracle; P and dS rounded to bfloat16 before the second products).
"""
from __future__ import annotations

import itertools

import numpy as np
import torch

from helpers import gamma

NP = {"f32": np.float32, "bf16": np.uint16, "f16": np.float16, "f64": np.float64, "i32": np.int32,
      "i16": np.int16, "i8": np.int8}
FLOAT = ("f32", "bf16", "f16", "f64")
U = 2.0 ** -24


# ------------------------------------------------------------ marshalling ---

def vdesc(A, v):
    """(dtype, shape, strides, offset, mask) of a psg_view."""
    nd = v.ndim
    shape = [int(v.shape[d]) for d in range(nd)]
    mask = [(int(v.mask_lo[d]), int(v.mask_hi[d])) for d in range(nd)]
    if all(lo <= 0 and hi >= s for (lo, hi), s in zip(mask, shape)):
        mask = None
    return A.DTYPE_NAMES[v.dtype], shape, [int(v.strides[d]) for d in range(nd)], int(v.offset), mask


def ndesc(A, nodes):
    names = {k: n for n, k in A.OPS.items()}
    return [(names[n.op], int(n.a), int(n.b), int(n.c), A.DTYPE_NAMES[n.dtype], float(n.cval)) for n in nodes]


def snap(buf, dt, n):
    """The storage bits of the first n elements of dtype dt at buf's data
    pointer (buf: a tensor on any device)."""
    es = np.dtype(NP[dt]).itemsize
    st = buf.untyped_storage()
    off = buf.storage_offset() * buf.element_size()
    nbytes = min(int(n) * es, st.nbytes() - off)
    raw = torch.empty(0, dtype=torch.uint8, device=buf.device)
    raw.set_(st, off, (nbytes,), (1,))
    return raw.cpu().numpy().view(NP[dt]).copy()


def read_view(O, P, A, buf, v):
    dt, shape, strides, offset, mask = vdesc(A, v)
    return P.read(snap(buf, dt, v.extent), dt, shape, strides, offset, mask)


# ------------------------------------------------------- value movements ---

def _ordered(bits, width):
    """Map float bit patterns to integers that order like the values."""
    b = bits.astype(np.int64)
    sign = np.int64(1) << (width - 1)
    return np.where(b & sign, -(b & (sign - 1)), b)


def _unordered(o, width):
    sign = np.int64(1) << (width - 1)
    return np.where(o < 0, (-o) | sign, o)


def step_units(x, sign, k):
    """Move every finite value of oracle tensor x by k units of its dtype in
    the direction of sign (NaN stays NaN; an overflow to inf is allowed)."""
    if x.dt == "f32":
        bits, w, ut = x.data.view(np.uint32), 32, np.uint32
        inf = 0x7F800000
    elif x.dt == "bf16":
        bits, w, ut = x.data, 16, np.uint16
        inf = 0x7F80
    elif x.dt == "f16":
        bits, w, ut = x.data.view(np.uint16), 16, np.uint16
        inf = 0x7C00
    else:
        return x
    o = _ordered(bits, w)
    mag = np.abs(o)
    nan = mag > inf
    moved = np.clip(o + sign * k, -inf, inf)
    o = np.where(nan, o, moved)
    out = _unordered(o, w).astype(ut)
    if x.dt == "f32":
        out = out.view(np.float32)
    elif x.dt == "f16":
        out = out.view(np.float16)
    return type(x)(out, x.dt)


def _round_out_f32(y64, sign):
    """float64 -> float32 rounded away from the centre in the direction of
    sign, so the interval never shrinks."""
    y32 = y64.astype(np.float32)
    if sign > 0:
        low = y32.astype(np.float64) < y64
        y32 = np.where(low, np.nextafter(y32, np.float32(np.inf)), y32)
    else:
        high = y32.astype(np.float64) > y64
        y32 = np.where(high, np.nextafter(y32, np.float32(-np.inf)), y32)
    return y32.astype(np.float32)


# ---------------------------------------------------------------- checks ---

class Record:
    def __init__(self, idx, kind, desc):
        self.idx, self.kind, self.desc = idx, kind, desc
        self.cells = 0
        self.bad = 0
        self.unbounded = 0
        self.worst = 0.0
        self.note = ""

    def __repr__(self):
        return "#%d %s %s cells=%d bad=%d worst=%.3g%s%s" % (
            self.idx, self.kind, self.desc, self.cells, self.bad, self.worst,
            " unbounded=%d" % self.unbounded if self.unbounded else "", " " + self.note if self.note else "")


def _bits_equal(got, ref):
    g = np.ascontiguousarray(got).reshape(-1)
    r = np.ascontiguousarray(ref).reshape(-1)
    if g.dtype.kind == "f" or g.dtype == np.uint16:
        from helpers import _isnan_bits
        same = (g.view(np.uint8).reshape(g.size, -1) == r.view(np.uint8).reshape(r.size, -1)).all(axis=1)
        same |= _isnan_bits(g) & _isnan_bits(r)
    else:
        same = g == r
    return same


def _widen(x64, dt, sign):
    """Values of dtype dt (given as float64) moved one unit of dt outward
    in the direction of sign; infinities stay put."""
    if dt == "f64":
        return x64 + sign * (np.abs(x64) * 2.0 ** -52 + 2.0 ** -1074)
    if dt == "f32":
        bits, w = x64.astype(np.float32).view(np.uint32), 32
    elif dt == "f16":
        bits, w = x64.astype(np.float16).view(np.uint16), 16
    else:  # bf16: the values are bfloat16 values, so the float32 bits end in 16 zeros
        bits, w = (x64.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16), 16
    o = _ordered(bits, w)
    fin = np.isfinite(x64)
    o = np.where(fin, o + sign, o)
    b = _unordered(o, w)
    if dt == "f32":
        return b.astype(np.uint32).view(np.float32).astype(np.float64)
    if dt == "f16":
        return b.astype(np.uint16).view(np.float16).astype(np.float64)
    return (b.astype(np.uint32) << 16).astype(np.uint32).view(np.float32).astype(np.float64)


def check_hull(rec, got, plain, runs, out_dt):
    """got within the hull of the oracle runs, widened by one unit of out_dt;
    NaN exactly where the plain oracle run is NaN."""
    g = got.f64().reshape(-1)
    p = plain.f64().reshape(-1)
    rec.cells = g.size
    if out_dt not in FLOAT:
        rec.bad = int((g != p).sum())
        return
    vals = np.stack([r.f64().reshape(-1) for r in runs])
    nanp = np.isnan(p)
    unb = np.isnan(vals).any(axis=0) & ~nanp
    lo = np.where(np.isnan(vals), np.inf, vals).min(axis=0)
    hi = np.where(np.isnan(vals), -np.inf, vals).max(axis=0)
    lo_w = _widen(np.where(unb | nanp, 0.0, lo), out_dt, -1)
    hi_w = _widen(np.where(unb | nanp, 0.0, hi), out_dt, +1)
    with np.errstate(invalid="ignore"):
        inside = (g >= lo_w) & (g <= hi_w)
    ok = np.where(nanp, np.isnan(g), inside) | unb
    rec.unbounded = int(unb.sum())
    rec.bad = int((~ok).sum())
    width = np.maximum(hi_w - lo_w, 1e-300)
    with np.errstate(invalid="ignore", over="ignore"):
        excess = np.where(nanp | unb | ~np.isfinite(width), 0.0, np.maximum(lo_w - g, g - hi_w) / width)
    rec.worst = float(np.nanmax(excess)) if excess.size else 0.0
    if rec.bad:
        i = int(np.argmax(~ok))
        rec.note = "first bad cell %d: got %r, hull [%r, %r]" % (i, g[i], lo_w[i], hi_w[i])


def perturbed_runs(O, run, items, max_items=10):
    """Evaluate run(signs) for every sign combination of the movable items
    (each +1 or -1); returns the list of outputs."""
    if len(items) > max_items:
        raise AssertionError("too many movable values (%d) for an exhaustive hull" % len(items))
    outs = []
    for signs in itertools.product((-1, 1), repeat=len(items)):
        outs.append(run(dict(zip(items, signs))))
    return outs


def reduce_hook(O, stages, epi, N, signs):
    """The oracle hook that moves each movable value by its allowance in the
    direction signs[item]: stage totals ("stage", s) and EXP/LOG nodes
    (scope, i)."""
    last = {}
    g = 2 * gamma(N - 1)

    def hook(kind, i, x):
        if (kind, i) in signs:
            if kind == "stage":
                p = last[i]
                mag = np.abs(p.f64()).sum(axis=1, keepdims=True)
                t32 = O.reduce_sum(O.cast(p, "f32")) if p.dt != "f32" else x
                y = t32.f64() + signs[(kind, i)] * g * mag * (1 + 2.0 ** -20)
                y32 = O.T(_round_out_f32(y, signs[(kind, i)]), "f32")
                x = O.cast(y32, x.dt) if x.dt != "f32" else y32
            else:
                x = step_units(x, signs[(kind, i)], 8 if x.dt == "f32" else 1)
        if kind.startswith("prologue"):
            s = int(kind[len("prologue"):])
            if i == len(stages[s][1]) - 1:
                last[s] = x
        return x
    return hook


def movable_items(stages, epi, stage_dts):
    items = []
    for s, (op, nodes) in enumerate(stages):
        for i, n in enumerate(nodes):
            if n[0] in ("EXP", "LOG"):
                items.append(("prologue%d" % s, i))
        if op == "SUM" and stage_dts[s] in FLOAT:
            items.append(("stage", s))
    for i, n in enumerate(epi or []):
        if n[0] in ("EXP", "LOG"):
            items.append(("epilogue", i))
    return items


def check_contract(O, P, rec, a3, b3, K, got, out_dt, epi=None):
    """A contraction's cells got ([Z, M, N] oracle tensor of the GPU's C)
    against the oracle's naive loop over the same operands a3 [Z, M, K] and
    b3 [Z, N, K]; epi: None, or (epilogue nodes, its inputs read at
    [Z, M, N]) for a fused epilogue program."""
    acc = "f64" if a3.dt == "f64" else ("i32" if a3.dt.startswith("i") else "f32")
    if acc == "i32":
        raise NotImplementedError("integer contractions are checked by their own tests")
    ref = P.contract(a3, b3, acc)
    r = ref.f64()
    mag = np.abs(a3.f64()) @ np.abs(b3.f64()).transpose(0, 2, 1)
    move = (1 + 2.0 ** -8) * 2 * gamma(K - 1) * mag
    if a3.dt == "f32":
        move = move + 2.0 ** -18 * mag  # three-term TF32 products: a few 2^-20 each
    if epi is not None:
        nodes, loads = epi
        items = ["acc"] + [("epilogue", i) for i, n in enumerate(nodes) if n[0] in ("EXP", "LOG")]

        def run(signs):
            s = signs["acc"]
            total = O.T(_round_out_f32(r + s * move, s), "f32")

            def hook(kind, i, x):
                d = signs.get(("epilogue", i))
                return step_units(x, d, 8 if x.dt == "f32" else 1) if d else x
            return P.program(nodes, loads, total.shape, hook=hook, acc=total)
        plain = P.program(nodes, loads, ref.shape, acc=ref)
        check_hull(rec, got, plain, perturbed_runs(O, run, items), out_dt)
        rec.note = (rec.note + " epilogue %d nodes" % len(nodes)).strip()
        return
    g = got.f64()
    tol = move
    if out_dt == "bf16":
        tol = tol + 2.0 ** -8 * np.abs(r) + 2.0 ** -133
    elif out_dt == "f16":
        tol = tol + 2.0 ** -11 * np.abs(r) + 2.0 ** -25
    else:
        tol = tol + 2.0 ** -149
    err = np.abs(g - r)
    ok = err <= tol
    ok |= np.isnan(g) & np.isnan(r)
    rec.cells = ok.size
    rec.bad = int((~ok).sum())
    rec.worst = float(np.max(np.where(np.isfinite(err), err / tol, 0.0))) if ok.size else 0.0
    if rec.bad:
        i = np.unravel_index(int(np.argmax(~ok)), ok.shape)
        rec.note = "first bad cell %s: got %r, oracle %r, tol %r" % (i, g[i], r[i], tol[i])


def read_epilogue(O, P, A, epilogue, dims):
    """(nodes, inputs read at [Z, M, N]) of an epilogue argument, or None."""
    if not epilogue or not epilogue[0]:
        return None
    prog, ins, views = epilogue
    Z, M, N, _ = dims
    loads = []
    for b, v in zip(ins, views):
        x = read_view(O, P, A, b, v)
        loads.append(O.T(x.data.reshape(Z, M, N), x.dt))
    return ndesc(A, prog), loads


# -------------------------------------------------------------- replayer ---

class Replayer:
    """Context manager: wraps the binding's calls and checks each against the
    oracle as it happens.  records: one Record per call."""

    WRAPPED = ("psg_elementwise", "psg_reduce_rows", "psg_contract", "psg_contract_ws", "psg_gather",
               "psg_scatter_add", "psg_permute", "psg_attention_fwd", "psg_attention_bwd")

    def __init__(self, A, O, nthreads=None, sync=None):
        import oracle.program as P
        self.A, self.O, self.P = A, O, P
        self.records = []
        self.nthreads = nthreads
        self.sync = sync or (torch.cuda.synchronize if torch.cuda.is_available() else (lambda: None))
        self._saved = {}

    def __enter__(self):
        from primitive_sm_graph_gb300 import graph as G
        self._old_threads = self.O.NTHREADS
        if self.nthreads:
            self.O.NTHREADS = self.nthreads
        # a plan recorded earlier would replay its raw C calls past these
        # wrappers: schedule every call afresh while the replay is active
        self._old_plan_cache, G.PLAN_CACHE = G.PLAN_CACHE, False
        for name in self.WRAPPED:
            f = getattr(self.A, name)
            self._saved[name] = f
            setattr(self.A, name, getattr(self, "_" + name[4:])(f))
        return self

    def __exit__(self, *exc):
        from primitive_sm_graph_gb300 import graph as G
        for name, f in self._saved.items():
            setattr(self.A, name, f)
        self.O.NTHREADS = self._old_threads
        G.PLAN_CACHE = self._old_plan_cache
        return False

    def failures(self):
        return [r for r in self.records if r.bad]

    def _rec(self, kind, desc):
        r = Record(len(self.records), kind, desc)
        self.records.append(r)
        return r

    # ---- elementwise ----
    def _elementwise(self, f):
        A, O, P = self.A, self.O, self.P

        def w(prog, ins, in_views, out, out_view, *a, **k):
            self.sync()
            loads = [read_view(O, P, A, b, v) for b, v in zip(ins, in_views)]
            st = f(prog, ins, in_views, out, out_view, *a, **k)
            self.sync()
            nodes = ndesc(A, prog)
            dt, shape, _, _, _ = vdesc(A, out_view)
            rec = self._rec("elementwise", "%s %s %d nodes" % (tuple(shape), dt, len(nodes)))
            got = read_view(O, P, A, out, out_view)
            items = [("epilogue", i) for i, n in enumerate(nodes) if n[0] in ("EXP", "LOG")]
            plain = P.program(nodes, loads, shape)
            if not items:
                same = _bits_equal(got.data, plain.data)
                rec.cells, rec.bad = same.size, int((~same).sum())
                return st

            def run(signs):
                def hook(kind, i, x):
                    s = signs.get(("epilogue", i))
                    return step_units(x, s, 8 if x.dt == "f32" else 1) if s else x
                return P.program(nodes, loads, shape, hook=hook)
            check_hull(rec, got, plain, perturbed_runs(O, run, items), dt)
            return st
        return w

    # ---- reductions ----
    def _reduce_rows(self, f):
        A, O, P = self.A, self.O, self.P

        def w(stages, epilogue, ins, in_views, out, out_view, *a, **k):
            self.sync()
            loads = [read_view(O, P, A, b, v) for b, v in zip(ins, in_views)]
            st = f(stages, epilogue, ins, in_views, out, out_view, *a, **k)
            self.sync()
            st_desc = [("SUM" if op == A.RED_SUM else "MAX", ndesc(A, prog)) for op, prog in stages]
            epi = ndesc(A, epilogue or [])
            odt, oshape, _, _, _ = vdesc(A, out_view)
            N = loads[0].shape[-1]
            per_element = len(oshape) == len(loads[0].shape) and oshape[-1] == N
            rec = self._rec("reduce_rows", "%s -> %s %s, %d stages, %d epilogue nodes" % (
                tuple(loads[0].shape), tuple(oshape), odt, len(st_desc), len(epi)))
            got = read_view(O, P, A, out, out_view)
            plain, reds, _ = P.reduce_rows(st_desc, epi, loads, per_element)
            items = movable_items(st_desc, epi, [r.dt for r in reds])

            def run(signs):
                return P.reduce_rows(st_desc, epi, loads, per_element,
                                     hook=reduce_hook(O, st_desc, epi, N, signs))[0]
            runs = perturbed_runs(O, run, items) if items else [plain]
            check_hull(rec, O.T(got.data.reshape(plain.shape), got.dt), plain,
                       [O.T(r.data.reshape(plain.shape), r.dt) for r in runs], odt)
            rec.note = (rec.note + " items=%d" % len(items)).strip()
            return st
        return w

    # ---- contractions ----
    def _contract_common(self, rec, Ab, Av, Bb, Bv, Cb, Cv):
        A, O, P = self.A, self.O, self.P
        adt, ash, ast, aoff, amask = vdesc(A, Av)
        bdt, bsh, bst, boff, bmask = vdesc(A, Bv)
        if amask or bmask:
            raise NotImplementedError("masked contraction operands are not replayed")
        nb = len(ash) - 3
        M, N, K = ash[-3:]
        Z = int(np.prod(ash[:nb], dtype=np.int64)) if nb else 1
        a3 = P.read(snap(Ab, adt, Av.extent), adt, ash[:nb] + [M, 1, K], ast[:nb] + [ast[-3], 0, ast[-1]], aoff)
        b3 = P.read(snap(Bb, bdt, Bv.extent), bdt, bsh[:nb] + [1, N, K], bst[:nb] + [0, bst[-2], bst[-1]], boff)
        a3 = O.T(a3.data.reshape(Z, M, K), adt)
        b3 = O.T(b3.data.reshape(Z, N, K), bdt)
        return a3, b3, (Z, M, N, K)

    def _contract_check(self, rec, a3, b3, dims, Cb, Cv, epi=None):
        A, O, P = self.A, self.O, self.P
        Z, M, N, K = dims
        cdt, csh, cst, coff, _ = vdesc(A, Cv)
        got = P.read(snap(Cb, cdt, Cv.extent), cdt, csh, cst, coff)
        check_contract(O, P, rec, a3, b3, K, O.T(got.data.reshape(Z, M, N), cdt), cdt, epi)

    def _contract(self, f):
        def w(Ab, Av, Bb, Bv, Cb, Cv, *a, **k):
            self.sync()
            rec = self._rec("contract", "")
            a3, b3, dims = self._contract_common(rec, Ab, Av, Bb, Bv, Cb, Cv)
            epi = read_epilogue(self.O, self.P, self.A, k.get("epilogue"), dims)
            st = f(Ab, Av, Bb, Bv, Cb, Cv, *a, **k)
            self.sync()
            rec.desc = "Z%d M%d N%d K%d -> %s" % (dims + (self.A.DTYPE_NAMES[Cv.dtype],))
            self._contract_check(rec, a3, b3, dims, Cb, Cv, epi)
            return st
        return w

    def _contract_ws(self, f):
        def w(Ab, Av, Bb, Bv, Cb, Cv, ws, ws_bytes, *a, **k):
            self.sync()
            rec = self._rec("contract_ws", "")
            a3, b3, dims = self._contract_common(rec, Ab, Av, Bb, Bv, Cb, Cv)
            epi = read_epilogue(self.O, self.P, self.A, k.get("epilogue"), dims)
            st = f(Ab, Av, Bb, Bv, Cb, Cv, ws, ws_bytes, *a, **k)
            self.sync()
            rec.desc = "Z%d M%d N%d K%d -> %s (split K)" % (dims + (self.A.DTYPE_NAMES[Cv.dtype],))
            self._contract_check(rec, a3, b3, dims, Cb, Cv, epi)
            return st
        return w

    # ---- indexed / movement ----
    def _gather(self, f):
        A, O, P = self.A, self.O, self.P

        def w(src, sv, idx, n, out, ov, *a, **k):
            self.sync()
            s = read_view(O, P, A, src, sv)
            ix = snap(idx, "i32", n)
            st = f(src, sv, idx, n, out, ov, *a, **k)
            self.sync()
            rec = self._rec("gather", "%s by %d" % (s.shape, n))
            ref, _ = O.gather_rows(s, ix)
            got = read_view(O, P, A, out, ov)
            same = _bits_equal(got.data, ref.data)
            rec.cells, rec.bad = same.size, int((~same).sum())
            return st
        return w

    def _scatter_add(self, f):
        A, O, P = self.A, self.O, self.P

        def w(dst, dv, idx, n, upd, uv, *a, **k):
            self.sync()
            before = read_view(O, P, A, dst, dv)
            u = read_view(O, P, A, upd, uv)
            ix = snap(idx, "i32", n)
            st = f(dst, dv, idx, n, upd, uv, *a, **k)
            self.sync()
            rec = self._rec("scatter_add", "%s += %d rows" % (before.shape, n))
            ref, _ = O.scatter_add_rows(before, ix, u)
            got = read_view(O, P, A, dst, dv)
            same = _bits_equal(got.data, ref.data)
            rec.cells, rec.bad = same.size, int((~same).sum())
            return st
        return w

    def _permute(self, f):
        A, O, P = self.A, self.O, self.P

        def w(inp, iv, perm, out, ov, *a, **k):
            self.sync()
            x = read_view(O, P, A, inp, iv)
            st = f(inp, iv, perm, out, ov, *a, **k)
            self.sync()
            rec = self._rec("permute", "%s perm %s" % (x.shape, list(perm)))
            strides = np.cumprod((list(x.shape[1:]) + [1])[::-1])[::-1]
            ref = O.view(x, [x.shape[p] for p in perm], [int(strides[p]) for p in perm])
            got = read_view(O, P, A, out, ov)
            same = _bits_equal(got.data, ref.data)
            rec.cells, rec.bad = same.size, int((~same).sum())
            return st
        return w

    # ---- attention ----
    @staticmethod
    def _heads(x):
        """oracle [B, T, H, d] tensor -> float64 [B*H, T, d]."""
        v = x.f64()
        B, T, H, d = v.shape
        return v.transpose(0, 2, 1, 3).reshape(B * H, T, d)

    def _key_mask(self, km, qv):
        """A [B, T] byte key mask on the device as the oracle's [B*H, T]."""
        if km is None:
            return None
        B, T, H = int(qv.shape[0]), int(qv.shape[1]), int(qv.shape[2])
        m = snap(km, "i8", B * T).reshape(B, T)
        return np.repeat(m, H, axis=0)

    def _attention_fwd(self, f):
        A, O, P = self.A, self.O, self.P

        def w(q, qv, k, kv, v, vv, o, ov, lse, scale, causal=True, *a, **kw):
            from helpers import attention_fwd_bounds
            from oracle.attention import attention_fwd
            self.sync()
            Q, K, V = (self._heads(read_view(O, P, A, b, x)) for b, x in ((q, qv), (k, kv), (v, vv)))
            km = self._key_mask(kw.get("key_mask"), qv)
            st = f(q, qv, k, kv, v, vv, o, ov, lse, scale, causal, *a, **kw)
            self.sync()
            rec = self._rec("attention_fwd", "heads %d T %d" % Q.shape[:2])
            O_ref, L_ref = attention_fwd(Q, K, V, scale, causal, key_mask=km)
            got = self._heads(read_view(O, P, A, o, ov))
            tol = attention_fwd_bounds(Q, K, V, O_ref, L_ref, scale, causal, key_mask=km)
            L = snap(lse, "f32", Q.shape[0] * Q.shape[1]).astype(np.float64).reshape(L_ref.shape)
            ok = np.abs(got - O_ref) <= tol
            with np.errstate(invalid="ignore"):
                okl = (np.abs(L - L_ref) <= 1e-4 + 2.0 ** -16 * np.abs(L_ref)) | (L == L_ref)
            rec.cells = ok.size + okl.size
            rec.bad = int((~ok).sum() + (~okl).sum())
            return st
        return w

    def _attention_bwd(self, f):
        A, O, P = self.A, self.O, self.P

        def w(q, qv, k, kv, v, vv, o, ov, do, dov, lse, delta, dq, dqv, dk, dkv, dv, dvv, scale, causal=True,
              *a, **kw):
            from helpers import attention_bwd_bounds
            from oracle.attention import attention_bwd
            self.sync()
            Q, K, V, Oo, dO = (self._heads(read_view(O, P, A, b, x))
                               for b, x in ((q, qv), (k, kv), (v, vv), (o, ov), (do, dov)))
            L = snap(lse, "f32", Q.shape[0] * Q.shape[1]).astype(np.float64).reshape(Q.shape[:2])
            km = self._key_mask(kw.get("key_mask"), qv)
            st = f(q, qv, k, kv, v, vv, o, ov, do, dov, lse, delta, dq, dqv, dk, dkv, dv, dvv, scale, causal,
                   *a, **kw)
            self.sync()
            rec = self._rec("attention_bwd", "heads %d T %d" % Q.shape[:2])
            refs = attention_bwd(Q, K, V, Oo, dO, L, scale, causal, key_mask=km)
            bounds = attention_bwd_bounds(Q, K, V, Oo, dO, L, scale, causal, refs, key_mask=km)
            cells = bad = 0
            for buf, view, ref, tol in zip((dq, dk, dv), (dqv, dkv, dvv), refs, bounds):
                got = self._heads(read_view(O, P, A, buf, view))
                ok = np.abs(got - ref) <= tol
                cells += ok.size
                bad += int((~ok).sum())
            rec.cells, rec.bad = cells, bad
            return st
        return w
