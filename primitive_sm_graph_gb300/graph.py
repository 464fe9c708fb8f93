"""Lazy tensors over the closed primitive op set, a scheduler that cuts the
graph into the library's five kernel calls, and reverse-mode autograd.

The design follows limn ("Architecture", "Reading the schedule"):
  * Tensor methods never compute; they add nodes.  ``realize()`` runs them.
  * Composed ops (sub, div, relu, matmul, softmax, rmsnorm, ...) are spelled
    in the primitives, so the kernels only ever see primitives.
  * Movement ops compose into Views and cost nothing; a movement of an
    elementwise value is pushed into that value's operands, so it never forces
    a copy.
  * Elementwise work fuses into whatever consumes it; a cut falls where a
    value must exist in memory: a reduction, a contraction, a gather/scatter,
    a value used by several consumers.
  * A SUM over the last axis of MUL(x, y), where x and y are broadcast Views
    of realized buffers, is a contraction and runs as one psg_contract call
    (limn: "a whole matmul is one kernel").
  * Reductions over the same rows fuse into one psg_reduce_rows call with the
    elementwise work that consumes them as its epilogue (softmax, RMSNorm).
  * ``backward()`` walks the graph in reverse and builds the gradients as
    lazy graphs of the same primitives.

Every kernel runs through the C ABI (``_abi``); torch only owns device memory
and the stream.
"""
from __future__ import annotations

import ctypes
import os
import sys
from math import prod

import torch

from . import _abi as A
from .tensor_util import dtype_name, torch_dtype
from .view import View

EW_UNARY = ("NEG", "EXP", "LOG", "SQRT", "RECIP", "CAST")
EW_BINARY = ("ADD", "MUL", "CMPLT")
ELEMENTWISE = EW_UNARY + EW_BINARY + ("WHERE", "CONST")
REDUCE = ("SUM", "MAX")
FLOATS = ("f32", "bf16", "f16")
sys.setrecursionlimit(max(sys.getrecursionlimit(), 20000))


class Tensor:
    """A node of the lazy graph.  ``shape`` is the logical shape; ``arg``
    holds op-specific data; ``_real`` the realized (buffer, View)."""

    __slots__ = ("op", "src", "shape", "dtype", "arg", "requires_grad", "grad", "_real", "_users", "_aux",
                 "__weakref__")

    def __init__(self, op, src, shape, dtype, arg=None, requires_grad=False):
        self.op = op
        self.src = src = tuple(src)
        self.shape = tuple(map(int, shape))
        self.dtype = dtype
        self.arg = arg
        if not requires_grad:
            for s in src:
                if s.requires_grad:
                    requires_grad = True
                    break
        self.requires_grad = requires_grad
        self.grad = None
        self._real = None
        self._users = 0
        self._aux = None  # realization-side data another node needs (ATTN: its row logsumexp)

    def __repr__(self):
        return "Tensor(%s, %s, %s)" % (self.op, self.shape, self.dtype)

    # ---- sources -----------------------------------------------------------
    @staticmethod
    def from_torch(t: torch.Tensor, requires_grad=False) -> "Tensor":
        t = t.contiguous()
        x = Tensor("BUF", (), t.shape, dtype_name(t.dtype), requires_grad=requires_grad)
        x._real = (t, View(t.shape))
        return x

    @staticmethod
    def const(value, shape, dtype="f32") -> "Tensor":
        return Tensor("CONST", (), shape, dtype, arg=float(value))

    @staticmethod
    def zeros(shape, dtype="f32") -> "Tensor":
        return Tensor.const(0.0, shape, dtype)

    def numel(self):
        return prod(self.shape)

    @property
    def ndim(self):
        return len(self.shape)

    # ---- elementwise primitives ---------------------------------------------
    def _un(self, op):
        if op in ("EXP", "LOG", "SQRT", "RECIP") and self.dtype not in FLOATS:
            raise TypeError("%s needs a float dtype" % op)
        return Tensor(op, (self,), self.shape, self.dtype)

    def neg(self): return self._un("NEG")
    def exp(self): return self._un("EXP")
    def log(self): return self._un("LOG")
    def sqrt(self): return self._un("SQRT")
    def recip(self): return self._un("RECIP")

    def cast(self, dtype):
        if dtype == self.dtype:
            return self
        return Tensor("CAST", (self,), self.shape, dtype)

    def _coerce(self, other):
        if isinstance(other, Tensor):
            return other
        return Tensor.const(other, (), self.dtype)

    def _bin(self, op, other):
        b = self._coerce(other)
        a = self
        if a.dtype != b.dtype:
            raise TypeError("%s of %s and %s: cast explicitly" % (op, a.dtype, b.dtype))
        a, b = broadcast(a, b)
        return Tensor(op, (a, b), a.shape, a.dtype)

    def add(self, o): return self._bin("ADD", o)
    def mul(self, o): return self._bin("MUL", o)
    def cmplt(self, o): return self._bin("CMPLT", o)

    def where(self, x, y):
        """WHERE(self, x, y): self nonzero selects x."""
        x = x if isinstance(x, Tensor) else Tensor.const(x, (), y.dtype if isinstance(y, Tensor) else "f32")
        y = y if isinstance(y, Tensor) else Tensor.const(y, (), x.dtype)
        c, x, y = broadcast(self, x, y)
        return Tensor("WHERE", (c, x, y), x.shape, x.dtype)

    # composed elementwise ops (limn, "Three rules": composed from primitives)
    def __add__(self, o): return self.add(o)
    def __radd__(self, o): return self._coerce(o).add(self)
    def __mul__(self, o): return self.mul(o)
    def __rmul__(self, o): return self._coerce(o).mul(self)
    def __neg__(self): return self.neg()
    def __sub__(self, o): return self.add(self._coerce(o).neg())
    def __rsub__(self, o): return self._coerce(o).add(self.neg())
    def __truediv__(self, o): return self.mul(self._coerce(o).recip())
    def __lt__(self, o): return self.cmplt(o)
    def __gt__(self, o): return self._coerce(o).cmplt(self)

    def relu(self):
        zero = Tensor.const(0.0, self.shape, self.dtype)
        return zero.cmplt(self).where(self, zero)

    def square(self):
        return self.mul(self)

    # ---- movement --------------------------------------------------------------
    def _move(self, kind, arg, shape):
        return Tensor("MOVE", (self,), shape, self.dtype, arg=(kind, arg))

    def reshape(self, *shape):
        if len(shape) == 1 and isinstance(shape[0], (tuple, list)):
            shape = tuple(shape[0])
        if shape == self.shape:
            return self
        if -1 not in shape:
            shape = tuple(shape)
            assert prod(shape) == prod(self.shape), (self.shape, shape)
            return Tensor("MOVE", (self,), shape, self.dtype, arg=("reshape", shape))
        shape = list(shape)
        if -1 in shape:
            i = shape.index(-1)
            shape[i] = self.numel() // max(1, prod(s for s in shape if s != -1))
        shape = tuple(shape)
        assert prod(shape) == self.numel(), (self.shape, shape)
        if shape == self.shape:
            return self
        return self._move("reshape", shape, shape)

    def permute(self, *perm):
        if len(perm) == 1 and isinstance(perm[0], (tuple, list)):
            perm = tuple(perm[0])
        if tuple(perm) == tuple(range(self.ndim)):
            return self
        return self._move("permute", tuple(perm), [self.shape[p] for p in perm])

    def transpose(self, a=-2, b=-1):
        p = list(range(self.ndim))
        p[a], p[b] = p[b], p[a]
        return self.permute(p)

    @property
    def T(self):
        return self.transpose()

    def expand(self, *shape):
        if len(shape) == 1 and isinstance(shape[0], (tuple, list)):
            shape = tuple(shape[0])
        if tuple(shape) == self.shape:
            return self
        return self._move("expand", tuple(shape), shape)

    def shrink(self, arg):
        arg = tuple((int(a), int(b)) for a, b in arg)
        if all(a == 0 and b == s for (a, b), s in zip(arg, self.shape)):
            return self
        return self._move("shrink", arg, [b - a for a, b in arg])

    def pad(self, arg):
        arg = tuple((int(a), int(b)) for a, b in arg)
        if all(a == 0 and b == 0 for a, b in arg):
            return self
        return self._move("pad", arg, [s + a + b for s, (a, b) in zip(self.shape, arg)])

    def contiguous(self):
        return Tensor("CONTIG", (self,), self.shape, self.dtype)

    def detach(self):
        """Cut the gradient path: the value, with no backward through it."""
        t = Tensor("MOVE", (self,), self.shape, self.dtype, arg=("detach", None))
        t.requires_grad = False
        return t

    # ---- reductions --------------------------------------------------------------
    def _reduce(self, op, axis=-1, keepdim=True):
        axis = axis % self.ndim
        if axis != self.ndim - 1:
            perm = [d for d in range(self.ndim) if d != axis] + [axis]
            inv = [0] * self.ndim
            for i, p in enumerate(perm):
                inv[p] = i
            r = self.permute(perm)._reduce(op, -1, True).permute(inv)
        else:
            r = Tensor(op, (self,), self.shape[:-1] + (1,), self.dtype)
        if not keepdim:
            r = r.reshape(tuple(s for d, s in enumerate(self.shape) if d != axis))
        return r

    def sum(self, axis=-1, keepdim=True): return self._reduce("SUM", axis, keepdim)
    def max(self, axis=-1, keepdim=True): return self._reduce("MAX", axis, keepdim)

    def mean(self, axis=-1, keepdim=True):
        n = self.shape[axis]
        return self.sum(axis, keepdim) * (1.0 / n)

    # ---- indexed -------------------------------------------------------------------
    def gather(self, idx: "Tensor"):
        """GATHER along dim 0: out[n, ...] = self[idx[n], ...]."""
        assert idx.dtype == "i32" and idx.ndim == 1
        return Tensor("GATHER", (self, idx), (idx.shape[0],) + self.shape[1:], self.dtype)

    def attention(self, k: "Tensor", v: "Tensor", scale: float, causal: bool = True, key_mask=None):
        """Fused scaled dot-product attention (limn, "The op set": the one
        fused node in place of the composed T x T scores; masking is a flag
        per key that composes with causal): self = Q, k, v are bf16
        [B, T, H, hd]; returns O [B, T, H, hd] with O = softmax(scale Q K^T)
        V per head over the keys query i sees (not j > i when causal, not
        where key_mask [B, T] int8 is 0; a query that sees no key gets 0)."""
        assert self.shape == k.shape == v.shape and len(self.shape) == 4
        assert self.dtype == k.dtype == v.dtype == "bf16"
        if self.shape[3] != ATTN_HD:
            if key_mask is not None:
                raise NotImplementedError("a key mask needs the fused attention (head dim %d)" % ATTN_HD)
            return _composed_attention(self, k, v, scale, causal)
        srcs = (self, k, v) + ((_key_mask(key_mask, self.shape),) if key_mask is not None else ())
        return Tensor("ATTN", srcs, self.shape, "bf16", arg=(float(scale), bool(causal), key_mask is not None))

    def attention_packed(self, scale: float, causal: bool = True, key_mask=None):
        """The fused attention over a packed qkv tensor [B, T, 3, H, hd] bf16
        (slot 0 Q, 1 K, 2 V: a fused projection's output): returns O
        [B, T, H, hd].  Its gradient is one tensor in the same packed
        layout, which the backward kernels write in place (no pad-and-add of
        dQ, dK, dV back into the packed tensor).  key_mask as for attention."""
        assert len(self.shape) == 5 and self.shape[2] == 3 and self.dtype == "bf16"
        B, T, _, H, hd = self.shape
        if hd != ATTN_HD:
            if key_mask is not None:
                raise NotImplementedError("a key mask needs the fused attention (head dim %d)" % ATTN_HD)
            q, k, v = (self.shrink(((0, B), (0, T), (i, i + 1), (0, H), (0, hd))).reshape(B, T, H, hd)
                       for i in range(3))
            return _composed_attention(q, k, v, scale, causal)
        srcs = (self,) + ((_key_mask(key_mask, (B, T, H, hd)),) if key_mask is not None else ())
        return Tensor("ATTN", srcs, (B, T, H, hd), "bf16", arg=(float(scale), bool(causal), key_mask is not None))

    def scatter_add(self, idx: "Tensor", upd: "Tensor"):
        """SCATTER-add along dim 0: self + rows of upd added at idx, in order."""
        assert idx.dtype == "i32" and upd.shape[1:] == self.shape[1:] and upd.dtype == self.dtype
        return Tensor("SCATTER", (self, idx, upd), self.shape, self.dtype)

    # ---- composed ops --------------------------------------------------------------
    def matmul(self, other: "Tensor", out_dtype=None):
        """a @ b as SUM over k of MUL of two broadcast Views (limn, "Reading
        the schedule"; Luminal IR blog, "Naive Matrix Multiplication").  Half
        widths widen to float32 first, so the products are exact and the SUM
        keeps a float32 total; the result rounds once into out_dtype.  Two
        float64 or two same-width integer operands keep their dtype (the
        integers wrap)."""
        a, b = self, other
        out_dtype = out_dtype or a.dtype
        assert a.shape[-1] == b.shape[-2], (a.shape, b.shape)
        M, K, N = a.shape[-2], a.shape[-1], b.shape[-1]
        batch = broadcast_shapes(a.shape[:-2], b.shape[:-2])
        keep = a.dtype == b.dtype and a.dtype in ("f64", "i32", "i16", "i8")
        af = a.cast("f32") if a.dtype != "f32" and not keep else a
        bf = b.cast("f32") if b.dtype != "f32" and not keep else b
        af = af.reshape(a.shape[:-2] + (M, 1, K))
        af = _lead(af, len(batch) + 3).expand(batch + (M, N, K))
        bf = bf.permute(tuple(range(b.ndim - 2)) + (b.ndim - 1, b.ndim - 2)).reshape(b.shape[:-2] + (1, N, K))
        bf = _lead(bf, len(batch) + 3).expand(batch + (M, N, K))
        c = af.mul(bf).sum(-1, keepdim=False)
        return c.cast(out_dtype)

    __matmul__ = matmul

    def softmax(self, axis=-1):
        """MAX-shifted softmax: the max is a constant of the gradient (softmax
        does not depend on the shift)."""
        m = self.max(axis).detach()
        e = (self - m).exp()
        return e / e.sum(axis)

    def log_softmax(self, axis=-1):
        m = self.max(axis).detach()
        sh = self - m
        return sh - sh.exp().sum(axis).log()

    def rmsnorm(self, w: "Tensor", eps=1e-6):
        """Tiki's RMSNorm target: (xf * rsqrt(mean(xf*xf) + eps) * f32(w)) in
        x's dtype, with rsqrt = RECIP(SQRT)."""
        xf = self.cast("f32")
        inv = ((xf * xf).mean(-1) + eps).sqrt().recip()
        return (xf * inv * w.cast("f32")).cast(self.dtype)

    # ---- running -----------------------------------------------------------------------
    def realize(self) -> torch.Tensor:
        """Run the graph; returns the value as a torch tensor (a strided view
        of the buffer that holds it)."""
        return realize_all(self)[0]

    def numpy(self):
        return self.realize().float().cpu().numpy() if self.dtype == "bf16" else self.realize().cpu().numpy()

    def item(self):
        return float(self.realize().float().reshape(-1)[0].item())

    def backward(self, grad: "Tensor | None" = None):
        backward(self, grad)


# ---------------------------------------------------------------- helpers -----

def broadcast_shapes(*shapes):
    first = shapes[0]
    if all(s == first for s in shapes):
        return tuple(first)
    n = max(map(len, shapes))
    cols = list(zip(*[(1,) * (n - len(s)) + tuple(s) for s in shapes]))
    out = tuple(max(c) for c in cols)
    for c, m in zip(cols, out):
        for x in c:
            assert x == 1 or x == m, shapes
    return out


def _lead(t: Tensor, nd: int) -> Tensor:
    return t.reshape((1,) * (nd - t.ndim) + t.shape) if t.ndim < nd else t


def broadcast(*ts):
    first = ts[0].shape
    if all(t.shape == first for t in ts):
        return ts
    shape = broadcast_shapes(*[t.shape for t in ts])
    # a constant broadcasts to a constant of the new shape: the same value in
    # every cell, with no movement nodes between
    return tuple(t if t.shape == shape else
                 Tensor("CONST", (), shape, t.dtype, arg=t.arg) if t.op == "CONST" and t._real is None else
                 _lead(t, len(shape)).expand(shape) for t in ts)


def _as_torch(buf: torch.Tensor, v: View, dtype: str) -> torch.Tensor:
    if v.mask is not None:
        raise RuntimeError("a masked View has no torch equivalent; realize a contiguous copy")
    return torch.as_strided(buf, v.shape, v.strides, v.offset)


def _inverse(perm):
    inv = [0] * len(perm)
    for i, p in enumerate(perm):
        inv[p] = i
    return tuple(inv)


# ------------------------------------------------------------ executor --------

# keys the fused attention kernels hold in one block, and their head dim;
# longer sequences and other head dims take the composed form below
ATTN_HD = 64


def _key_mask(m, shape):
    """A per-key mask operand: int8 [B, T] (nonzero: visible)."""
    assert isinstance(m, Tensor) and m.dtype == "i8" and m.shape == (shape[0], shape[1]), "key_mask: int8 [B, T]"
    return m


def _composed_attention(q, k, v, scale, causal):
    """softmax(scale * Q K^T, keys j > i hidden when causal) V per head as
    the composed graph (limn, "The op set": the T x T scores the fused node
    avoids): one contraction for the scores, one fused row reduction for the
    softmax, one contraction for P V.  The scores and weights are float32, P
    rounds to bf16 as the second product's operand (as in the fused kernel),
    and a hidden key gets a bias of -2^100, whose weight exp underflows to
    exactly 0 (every causal row keeps its own key)."""
    B, T, H, hd = q.shape
    qh, kh, vh = (x.permute(0, 2, 1, 3) for x in (q, k, v))  # [B, H, T, hd]
    s = qh.matmul(kh.permute(0, 1, 3, 2), "f32") * float(scale)
    if causal:
        hide = torch.triu(torch.full((T, T), -2.0 ** 100, dtype=torch.float32), diagonal=1)
        s = s + Tensor.from_torch(hide.to("cuda"))
    p = s.softmax(-1).cast("bf16")
    return p.matmul(vh, "bf16").permute(0, 2, 1, 3)


_FLOATS32 = ("bf16", "f16", "f32")
_INTS = ("i32", "i16", "i8")


def _contract_dtypes(ab, c):
    """The operand / result dtype pairs psg_contract takes: float32-summed
    floats into any of them, float64 into float64, the integers (wrapping
    uint32 total) into any integer width."""
    return ((ab in _FLOATS32 and c in _FLOATS32) or (ab == "f64" and c == "f64")
            or (ab in _INTS and c in _INTS))


class Executor:
    """Cuts the graph into library calls and runs them on the current stream.
    ``log`` keeps every call it made (kind, details), for inspection."""

    def __init__(self):
        self.log = []
        self.rec = None    # the plan being recorded (see realize_all), or None
        self.status = None
        self.users = {}
        self.user_nodes = {}
        self.narrow = {}
        self.copies = {}
        self.epi_cut = {}

    def prepare(self, roots):
        """Count, for every unrealized node reachable from roots, how many
        nodes use it: a computed value with several users is a cut (it is
        stored once instead of being recomputed in each consumer)."""
        users, nodes, seen, stack = {}, {}, set(), list(roots)
        while stack:
            t = stack.pop()
            if id(t) in seen or t._real is not None:
                continue
            seen.add(id(t))
            for x in t.src:
                users[id(x)] = users.get(id(x), 0) + 1
                nodes.setdefault(id(x), []).append(t)
                stack.append(x)
        self.users = users
        self.user_nodes = nodes
        self.narrow = {}
        self.copies = {}
        self.epi_cut = {}

    def _only_cast_to(self, x, dt, depth=0):
        """True when every use of x (through movements) is a CAST to dt."""
        us = self.user_nodes.get(id(x))
        if not us or depth > 8:
            return False
        for u in us:
            if u.op == "CAST" and u.dtype == dt:
                continue
            if u.op == "MOVE" and u.arg[0] not in ("pad", "detach") and self._only_cast_to(u, dt, depth + 1):
                continue
            return False
        return True

    def _narrowable(self, t):
        """(contraction node, movements) when t is a CAST to a half width of
        an unrealized contraction whose every use is that CAST (see
        _narrow_contraction), else None; realizes nothing."""
        if t.op != "CAST" or t.dtype not in ("bf16", "f16"):
            return None
        x, inner = t.src[0], []
        while x.op == "MOVE" and x.arg[0] not in ("pad", "detach"):
            inner.append(x.arg)
            x = x.src[0]
        if x.op != "SUM" or x.dtype != "f32":
            return None
        if (id(x), t.dtype) in self.narrow:
            return x, inner
        if x._real is not None or not self._contract_pattern(x) or not self._only_cast_to(x, t.dtype):
            return None
        return x, inner

    def _narrow_contraction(self, t):
        """For t = CAST to a half width of an unrealized contraction (through
        movements) whose every use is that same CAST: the contraction stored
        once in the half width ((buf, View) for t), else None.  Its epilogue
        rounds the float32 total to nearest even, the bits a CAST of the
        float32 result gives, and the float32 tensor is never written."""
        nx = self._narrowable(t)
        if nx is None:
            return None
        x, inner = nx
        key = (id(x), t.dtype)
        if key not in self.narrow:
            r = self._try_contract(x, (), t.dtype, x.shape)
            if r is None:
                return None
            self.narrow[key] = r
        buf, v = self.narrow[key]
        return self._apply_moves(buf, v, list(reversed(inner)), t.dtype)

    def _shared_heavy(self, x):
        """A value with several users is stored once (a cut) when recomputing
        it in each consumer costs more than a store and a load: 4 or more
        elementwise ops above the realized values and reductions it reads
        (a reduction below is computed once either way: its result is
        stored, or it runs as a stage of the one fused reduction call)."""
        if self.users.get(id(x), 0) < 2 or x.op == "CONST" or x._real is not None:
            return False
        # a shared value computed from a contraction is stored once, by the
        # contraction's own epilogue, instead of being recomputed from the
        # contraction's stored result in each consumer
        k = id(x)
        if k not in self.epi_cut:
            self.epi_cut[k] = False  # (a cycle of this question answers no)
            self.epi_cut[k] = x.op in ELEMENTWISE and self._epilogue_contraction(x) is not None
        if self.epi_cut[k]:
            return True
        n = 0
        stack, seen = [x], set()
        while stack and n < 4:
            y = stack.pop()
            if id(y) in seen or y._real is not None or y.op in REDUCE:
                continue
            seen.add(id(y))
            if y.op in ELEMENTWISE + ("MOVE",):
                n += y.op not in ("MOVE", "CONST")
                stack.extend(y.src)
        return n >= 4

    def _status(self):
        if self.status is None or self.status.device != torch.device("cuda", torch.cuda.current_device()):
            self.status = torch.zeros((1,), dtype=torch.int32, device="cuda")
        return self.status

    def check_status(self):
        if self.status is not None:
            s = int(self.status.item())
            if s:
                raise A.PsgError(s, "device")

    def _s(self):
        return torch.cuda.current_stream().cuda_stream

    def _workspace(self, nbytes):
        ws = torch.empty((max(1, int(nbytes)),), dtype=torch.uint8, device="cuda")
        if self.rec is not None:
            self.rec.alloc(ws, ((max(1, int(nbytes)),), torch.uint8))
        return ws

    def _new(self, shape, dtype):
        t = torch.empty(tuple(shape), dtype=torch_dtype(dtype), device="cuda")
        if self.rec is not None:
            self.rec.alloc(t, (tuple(shape), torch_dtype(dtype)))
        return t

    def _lib(self, name):
        """The binding's call `name`; while a plan is recorded, a wrapper
        that also records the call when it succeeds."""
        f = getattr(A, name)
        rec = self.rec
        if rec is None:
            return f

        def call(*args, **kw):
            cap = _RawCapture(A.lib)
            A.lib = cap  # the binding's raw call is forwarded and kept for the plan
            try:
                st = f(*args, **kw)
            finally:
                A.lib = cap.lib
            if st == A.OK:
                rec.call(name, args, kw, cap.calls)
            return st
        return call

    def _pview(self, buf: torch.Tensor, v: View, dtype: str):
        return A.make_view(dtype, v.shape, v.strides, v.offset,
                           None if v.mask is None else list(v.mask), buf.numel())

    # ---- realize ---------------------------------------------------------------
    def realize(self, t: Tensor):
        if t._real is not None:
            return t._real
        op = t.op
        if op == "MOVE":
            r = self._realize_move(t)
        elif op in ELEMENTWISE:
            r = self._realize_ew(t)
        elif op in REDUCE:
            r = self._realize_reduce(t)
        elif op == "CONTIG":
            r = self._copy_contig(*self.realize(t.src[0]), t.dtype)
        elif op == "GATHER":
            r = self._realize_gather(t)
        elif op == "SCATTER":
            r = self._realize_scatter(t)
        elif op == "ATTN":
            r = self._realize_attn(t)
        elif op == "ATTN_BWD":
            r = self._realize_attn_bwd(t)
        else:
            raise RuntimeError("cannot realize %s" % op)
        t._real = r
        return r

    def _realize_move(self, t: Tensor):
        """A movement costs nothing: realize its base, then compose the View
        (a reshape no View can express copies the base first)."""
        chain, base = [], t
        while base.op == "MOVE":
            chain.append(base.arg)
            base = base.src[0]
        buf, v = self.realize(base)
        return self._apply_moves(buf, v, list(reversed(chain)), base.dtype)

    def _apply_moves(self, buf, v, moves, dtype):
        for kind, arg in moves:
            if kind == "detach":
                continue
            nv = getattr(v, kind)(arg)
            if nv is None:  # a reshape no View expresses: copy first
                buf, v = self._copy_contig(buf, v, dtype)
                nv = v.reshape(arg)
            v = nv
        return buf, v

    def _copy_contig(self, buf, v, dtype, fresh=False):
        # the same cells of the same buffer are copied once per schedule (an
        # expanded table reshaped for several consumers, say); the entry holds
        # the source, so its memory cannot be reused under the key meanwhile.
        # fresh: a copy of its own, for a caller that writes into it
        key = (buf.data_ptr(), v.key(), dtype)
        hit = None if fresh else self.copies.get(key)
        if hit is not None and hit[0] is buf:
            return hit[1], View(v.shape)
        out = self._new(v.shape, dtype)
        if not fresh:
            self.copies[key] = (buf, out)
        if out.numel():
            self._lib("psg_permute")(buf, self._pview(buf, v, dtype), list(range(len(v.shape))), out,
                          self._pview(out, View(v.shape), dtype), stream=self._s())
        self.log.append(("permute", v.shape))
        return out, View(v.shape)

    # ---- expression lowering (elementwise programs) ---------------------------
    def _lower(self, root: Tensor, reds=None, acc=None):
        """(program nodes, inputs [(buf, View, dtype)]) for root's value.
        Movements are pushed into elementwise operands; other nodes are
        realized and become LOAD leaves.  reds maps id(REDUCE node) -> stage
        index for reductions fused into the same call (read as RED).  acc:
        the contraction node (or its CAST) whose value a fused contraction
        epilogue reads as ACC (and rounds with a CAST node)."""
        prog, inputs, memo, in_memo = [], [], {}, {}
        reds = reds or {}

        def leaf(buf, v, dt):
            key = (buf.data_ptr(), v.key(), dt)
            if key not in in_memo:
                if len(inputs) >= A.MAX_INPUTS:
                    raise _TooBig()
                in_memo[key] = len(inputs)
                inputs.append((buf, v, dt))
            prog.append(A.node("LOAD", in_memo[key], dtype=dt))
            return len(prog) - 1

        def walk(t: Tensor, moves: tuple):
            key = (id(t), moves)
            if key in memo:
                return memo[key]
            if len(prog) >= A.MAX_NODES - 2:
                raise _TooBig()
            op = t.op
            if acc is not None and t is acc and not moves:
                # the contraction's float32 total, rounded as its CAST rounds
                prog.append(A.node("ACC", dtype="f32"))
                if t.op == "CAST" and t.dtype != "f32":
                    prog.append(A.node("CAST", len(prog) - 1, dtype=t.dtype))
                memo[key] = len(prog) - 1
                return len(prog) - 1
            if t._real is not None and op != "CONST":
                # already in memory: a leaf, whatever computed it
                buf, v = self._apply_moves(*t._real, [m for m in moves], t.dtype)
                r = leaf(buf, v, t.dtype)
                memo[key] = r
                return r
            nr = self._narrow_contraction(t) if op == "CAST" and not any(m[0] == "pad" for m in moves) else None
            if nr is not None:
                buf, v = self._apply_moves(*nr, list(moves), t.dtype)
                r = leaf(buf, v, t.dtype)
                memo[key] = r
                return r
            # a shared value is a cut, except inside one fused reduction,
            # whose stages and epilogue recompute it from registers
            if t is not root and not reds and op in ELEMENTWISE and self._shared_heavy(t):
                buf, v = self.realize(t)
                buf, v = self._apply_moves(buf, v, list(moves), t.dtype)
                r = leaf(buf, v, t.dtype)
            elif op == "MOVE" and t.arg[0] != "pad":
                r = walk(t.src[0], (t.arg,) + moves)
            elif op == "CONST":
                prog.append(A.node("CONST", dtype=t.dtype, cval=t.arg))
                r = len(prog) - 1
            elif op in EW_UNARY and not any(m[0] == "pad" for m in moves):
                a = walk(t.src[0], moves)
                prog.append(A.node(op, a, dtype=t.dtype))
                r = len(prog) - 1
            elif op in EW_BINARY and not any(m[0] == "pad" for m in moves):
                a = walk(t.src[0], moves)
                b = walk(t.src[1], moves)
                prog.append(A.node(op, a, b, dtype=t.dtype))
                r = len(prog) - 1
            elif op == "WHERE" and not any(m[0] == "pad" for m in moves):
                c = walk(t.src[0], moves)
                x = walk(t.src[1], moves)
                y = walk(t.src[2], moves)
                prog.append(A.node("WHERE", c, x, y, dtype=t.dtype))
                r = len(prog) - 1
            elif op in REDUCE and id(t) in reds:
                prog.append(A.node("RED", reds[id(t)], dtype=t.dtype))
                r = len(prog) - 1
            else:
                buf, v = self.realize(t)
                buf, v = self._apply_moves(buf, v, [m for m in moves], t.dtype)
                r = leaf(buf, v, t.dtype)
            memo[key] = r
            return r

        walk(root, ())
        return prog, inputs

    def _realize_ew(self, t: Tensor):
        # a CAST of a contraction (through movements) rounds inside the
        # contraction's epilogue
        base, moves = t, []
        while base.op == "MOVE" and base.arg[0] != "pad":
            moves.append(base.arg)
            base = base.src[0]
        nr = self._narrow_contraction(base)
        if nr is not None:
            return self._apply_moves(*nr, list(reversed(moves)), base.dtype)
        if base.op == "CAST" and base.dtype in ("bf16", "f32"):
            x, inner = base.src[0], []
            while x.op == "MOVE" and x.arg[0] != "pad":
                inner.append(x.arg)
                x = x.src[0]
            if x.op == "SUM" and x._real is None and self._contract_pattern(x):
                r = self._try_contract(x, (), base.dtype, x.shape)
                if r is not None:
                    return self._apply_moves(*r, list(reversed(inner)) + list(reversed(moves)), base.dtype)
        fused = self._try_contract_epilogue(t)
        if fused is not None:
            return fused
        fused = self._try_fused_reduce(t)
        if fused is not None:
            return fused
        while True:
            try:
                prog, inputs = self._lower(t)
                break
            except _TooBig:
                self._split(t)
        out = self._new(t.shape, t.dtype)
        if out.numel():
            self._lib("psg_elementwise")(prog, [b for b, _, _ in inputs], [self._pview(b, v, d) for b, v, d in inputs],
                              out, self._pview(out, View(t.shape), t.dtype), stream=self._s())
        self.log.append(("elementwise", t.shape, len(prog)))
        return out, View(t.shape)

    @staticmethod
    def _unit_moves(x: Tensor):
        """The node below a chain of movements that only add, drop or move
        dims of size 1 (the cells keep their order and their index along
        every other dim), starting at x; x itself when there is none."""
        while x.op == "MOVE" and x._real is None:
            kind, arg = x.arg[0], x.arg[1]
            src = x.src[0]
            if kind == "reshape":
                if [s for s in src.shape if s != 1] != [s for s in x.shape if s != 1]:
                    break
            elif kind == "permute":
                big = [p for p in arg if src.shape[p] != 1]
                if big != sorted(big):
                    break
            else:
                break
            x = src
        return x

    def _pending_contraction(self, s: Tensor):
        """True for a contraction not computed yet in any width."""
        return (s._real is None and not any((id(s), d) in self.narrow for d in ("bf16", "f16"))
                and self._contract_pattern(s) is not None)

    def _epilogue_contraction(self, t: Tensor):
        """(top, SUM node) of the one unrealized contraction that t's
        elementwise program reads directly, through a CAST to a half width or
        as its float32 value, with at most unit-dim movements between (top:
        the node the program reads, a CAST or the float32 value), when every
        use of it lies inside that program; else None."""
        found, region, seen, stack = [], {}, set(), [t]
        while stack:
            x = stack.pop()
            if id(x) in seen or x._real is not None:
                continue
            seen.add(id(x))
            if x is not t and x.op in ELEMENTWISE and self._shared_heavy(x):
                continue  # stored on its own: a leaf of this program
            if x.op == "CAST" and x.dtype in ("bf16", "f16"):
                s = self._unit_moves(x.src[0])
                if s.op == "SUM" and self._pending_contraction(s):
                    found.append((x, s))
                    continue
            s = self._unit_moves(x)
            if s.op == "SUM" and s.dtype == "f32" and self._pending_contraction(s):
                found.append((x, s))
                continue
            if x.op in REDUCE:
                return None  # a row reduction: the fused reduction path takes it
            if x.op in ELEMENTWISE:
                region[id(x)] = x
                stack.extend(x.src)
        if len(found) != 1:
            return None
        top, s = found[0]
        if top is t or any(id(u) not in region for u in self.user_nodes.get(id(top), [])):
            return None
        # no value computed from the contraction below t is read from outside
        # this program (else that reader would need the contraction again)
        dep = {id(top): True}

        def depends(x):
            if id(x) not in dep:
                dep[id(x)] = False
                dep[id(x)] = id(x) in region and any(depends(y) for y in x.src)
            return dep[id(x)]
        for i, x in region.items():
            if x is not t and depends(x) and any(id(u) not in region for u in self.user_nodes.get(i, [])):
                return None
        # the nodes between top and the SUM feed nothing else
        y = top.src[0] if top.op == "CAST" else top
        while y is not s:
            if self.users.get(id(y), 0) != 1:
                return None
            y = y.src[0]
        if self.users.get(id(s), 0) != 1:
            return None
        # a program of nothing but roundings is the contraction's own store
        if not any(x.op not in ("CAST", "CONST") for x in region.values()):
            return None
        out_shape = tuple(s.shape[:-1]) if s.shape and s.shape[-1] == 1 else tuple(s.shape)
        if [d for d in t.shape if d != 1] != [d for d in out_shape if d != 1]:
            return None
        (x, _, wx), (y, _, wy) = self._contract_pattern(s)
        if (wx or x.dtype) not in ("bf16", "f16") or (wy or y.dtype) != (wx or x.dtype):
            return None
        return top, s

    def _try_contract_epilogue(self, t: Tensor):
        """An elementwise value computed from one contraction (a residual add,
        a ReLU, a cast): the contraction's kernel computes it in its epilogue
        (psg_contract's epilogue program, ACC the float32 total), so the
        contraction's result never goes through memory (limn, "Reading the
        schedule": elementwise work fuses into the kernel that produces its
        operand).  None when t is not of that form or the call cannot take
        it (then t is computed the ordinary way)."""
        if t.op not in ELEMENTWISE or t.op == "CONST" or t.dtype not in ("f32", "bf16", "f16"):
            return None
        hit = self._epilogue_contraction(t)
        if hit is None:
            return None
        top, s = hit
        try:
            prog, inputs = self._lower(t, acc=top)
        except _TooBig:
            return None
        if inputs and not FUSE_EPILOGUE_INPUTS:
            return None
        S = s.src[0].shape
        conv = []
        for b, v, d in inputs:
            v2 = v.reshape(tuple(S[:-1])) if v.mask is None else None
            if v2 is None:
                return None
            conv.append((b, v2, d))
        r = self._try_contract(s, (), t.dtype, tuple(S[:-1]), epilogue=(prog, conv))
        if r is None:
            return None
        buf, v = r
        return buf, v.reshape(t.shape)

    def _split(self, t: Tensor):
        """A program too large for one call: realize the operand subtree with
        the most nodes on its own first."""
        best, size = None, -1
        stack = [t]
        seen = set()
        while stack:
            x = stack.pop()
            if id(x) in seen or x._real is not None:
                continue
            seen.add(id(x))
            # only the region this program would cover: elementwise and
            # movement nodes (anything else is already a leaf of it)
            if x.op not in ELEMENTWISE and x.op != "MOVE" and x is not t:
                continue
            if x is not t and x.op in ELEMENTWISE and x.op != "CONST":
                n = _count(x)
                if n > 1 and n > size:
                    best, size = x, n
            stack.extend(x.src)
        if best is None:
            raise RuntimeError("program cannot be split")
        self.realize(best)

    # ---- reductions ---------------------------------------------------------------
    def _collect_reds(self, root: Tensor):
        """Unrealized reductions reachable from root through elementwise and
        movement nodes, each with the movements between it and root."""
        found, seen = {}, set()

        def walk(x, moves):
            key = (id(x), moves)
            if x._real is not None or key in seen:
                return
            seen.add(key)
            if x.op == "MOVE":
                walk(x.src[0], (x.arg,) + moves)
            elif x.op == "CAST" and self._narrowable(x) is not None:
                return  # read from the contraction stored in the half width
            elif x.op in ELEMENTWISE:
                for s in x.src:
                    walk(s, moves)
            elif x.op in REDUCE:
                found.setdefault(id(x), (x, moves))
        walk(root, ())
        return found

    def _stage_order(self, reds, row_shape):
        """Order reductions (and the ones their prologues need) into stages;
        None if any is not a row reduction over row_shape."""
        order, state = [], {}

        def visit(r):
            if state.get(id(r)) == 2:
                return True
            if state.get(id(r)) == 1:
                return False
            state[id(r)] = 1
            if r.src[0].shape != row_shape:
                return False
            inner = self._collect_reds(r.src[0])
            for _, (r2, mv) in inner.items():
                if r2.src[0].shape != row_shape or not _is_row_expand(mv, r2.shape, row_shape):
                    return False
                if not visit(r2):
                    return False
            state[id(r)] = 2
            order.append(r)
            return True

        for r in reds:
            if not visit(r):
                return None
        return order

    def _store_shared_row_values(self, t: Tensor):
        """Per-row values inside t's expression (shape [.., 1], computed from
        reductions) that are shared and heavy and also used outside t (a
        norm's 1/rms, read again by the backward) are stored first, so the
        fused call reads them instead of recomputing them, and the other
        users do not recompute the reduction either."""
        inner, order, seen = {}, [], set()
        stack = [t]
        while stack:
            x = stack.pop()
            if id(x) in seen or x._real is not None:
                continue
            seen.add(id(x))
            order.append(x)
            if x.op in ELEMENTWISE or (x.op == "MOVE" and x.arg[0] != "pad"):
                for y in x.src:
                    inner[id(y)] = inner.get(id(y), 0) + 1
                    stack.append(y)
        for x in order:
            if (x is not t and x.op in ELEMENTWISE and x._real is None and len(x.shape) >= 1 and x.shape[-1] == 1
                    and self.users.get(id(x), 0) > inner.get(id(x), 0) and self._shared_heavy(x)
                    and self._collect_reds(x)):
                self.realize(x)

    def _try_fused_reduce(self, t: Tensor):
        found = self._collect_reds(t)
        if not found:
            return None
        self._store_shared_row_values(t)
        found = self._collect_reds(t)
        if not found:
            return None
        rows = {r.src[0].shape for r, _ in found.values()}
        if len(rows) != 1:
            return None
        row_shape = rows.pop()
        per_elem = t.shape == row_shape
        # one value per row: [.., 1], or any shape of that many cells that
        # the per-row values reach through movements that keep the row-major
        # order (a reshape, a permute of size-1 dims), so cell i is row i
        per_row = not per_elem and prod(t.shape) == prod(row_shape[:-1])
        if not (per_elem or per_row):
            return None
        for r, mv in found.values():
            if per_elem and not _is_row_expand(mv, r.shape, row_shape):
                return None
            if per_row and not _keeps_row_order(mv, r.shape, t.shape):
                return None
        order = self._stage_order([r for r, _ in found.values()], row_shape)
        if order is None or len(order) > 4:
            return None
        if any(self._contract_pattern(r) for r in order):
            return None
        try:
            return self._run_reduce(order, t, per_row)
        except (_NotFusable, _TooBig):
            return None

    def _run_reduce(self, order, epi_root, per_row):
        reds = {}
        stages, inputs, in_index = [], [], {}

        def merge(prog, ins):
            # renumber this program's LOADs into the shared input list
            out = []
            for nd in prog:
                if nd.op == A.OPS["LOAD"]:
                    b, v, d = ins[nd.a]
                    key = (b.data_ptr(), v.key(), d)
                    if key not in in_index:
                        if len(inputs) >= A.MAX_INPUTS:
                            raise _TooBig()
                        in_index[key] = len(inputs)
                        inputs.append((b, v, d))
                    nd = A.node("LOAD", in_index[key], dtype=d)
                out.append(nd)
            return out

        for s, r in enumerate(order):
            prog, ins = self._lower(r.src[0], reds)
            stages.append((A.RED_SUM if r.op == "SUM" else A.RED_MAX, merge(prog, ins)))
            reds[id(r)] = s
        epi = None
        if epi_root is not None and not (per_row and epi_root is order[-1]):
            prog, ins = self._lower(epi_root, reds)
            if per_row and ins:
                raise _NotFusable()
            epi = merge(prog, ins)
        out_shape = epi_root.shape if epi_root is not None else order[-1].shape
        out_dt = epi_root.dtype if epi_root is not None else order[-1].dtype
        out = self._new(out_shape, out_dt)
        if out.numel():
            self._lib("psg_reduce_rows")(stages, epi, [b for b, _, _ in inputs],
                              [self._pview(b, v, d) for b, v, d in inputs], out,
                              self._pview(out, View(out_shape), out_dt), stream=self._s())
        self.log.append(("reduce_rows", order[0].src[0].shape, len(stages), "per_row" if per_row else "per_elem"))
        return out, View(out_shape)

    def _realize_reduce(self, t: Tensor):
        r = self._try_contract(t, (), t.dtype, t.shape)
        if r is not None:
            return r
        order = self._stage_order([t], t.src[0].shape)
        if order is None or len(order) > 4:
            # realize the inner reductions first, then this one alone
            for _, (r2, _) in self._collect_reds(t.src[0]).items():
                self.realize(r2)
            order = [t]
        while True:
            try:
                return self._run_reduce(order, t, True)
            except _TooBig:
                # a prologue past the call's limits: store its largest
                # subexpression first (or, failing that, the whole prologue)
                for r in order:
                    try:
                        self._split(r.src[0])
                        break
                    except RuntimeError:
                        continue
                else:
                    for r in order:
                        self.realize(r.src[0])
                    order = [t]

    # ---- contraction ----------------------------------------------------------------
    def _contract_pattern(self, r: Tensor):
        """SUM over the last axis of MUL(x, y) with x, y movements of
        (widened) non-elementwise values."""
        if r.op != "SUM":
            return None
        m = r.src[0]
        moves = ()
        while m.op == "MOVE" and m.arg[0] != "pad":
            moves = (m.arg,) + moves
            m = m.src[0]
        if m.op != "MUL":
            return None
        if not any(mv[0] == "expand" for x in m.src for mv in _moves_to_base(x)):
            return None
        ops = []
        for x in m.src:
            mv = moves
            widen = None
            while True:
                if x.op == "MOVE" and x.arg[0] != "pad":
                    mv = (x.arg,) + mv
                    x = x.src[0]
                elif x.op == "CAST" and x.dtype == "f32" and x.src[0].dtype in ("bf16", "f16"):
                    widen = x.src[0].dtype
                    x = x.src[0]
                else:
                    break
            if x.op in ELEMENTWISE and x.op != "CAST":
                # a computed operand: realize it as its own value first
                pass
            ops.append((x, mv, widen))
        return ops

    def _try_contract(self, r: Tensor, _moves, out_dtype, out_shape, epilogue=None):
        """r, a contraction, as one psg_contract call writing out_dtype; with
        epilogue = (program, inputs [(buf, View, dtype)] over r's shape) the
        call's epilogue program computes the stored value from the total."""
        if r.op != "SUM" or r._real is not None:
            return None
        pat = self._contract_pattern(r)
        if pat is None:
            return None
        (x, mx, wx), (y, my, wy) = pat
        dx = wx or x.dtype
        dy = wy or y.dtype
        if dx != dy or not _contract_dtypes(dx, out_dtype):
            return None
        S = r.src[0].shape
        bx, vx = self._apply_moves(*self.realize(x), list(mx), x.dtype)
        by, vy = self._apply_moves(*self.realize(y), list(my), y.dtype)
        if vx.mask is not None or vy.mask is not None:
            return None
        L = len(S) - 1
        Mx, Nx, Bx = [], [], []
        for a in range(L):
            if S[a] == 1:
                continue
            sx, sy = vx.strides[a], vy.strides[a]
            if sy == 0 and sx != 0:
                Mx.append(a)
            elif sx == 0 and sy != 0:
                Nx.append(a)
            elif sx != 0 and sy != 0:
                Bx.append(a)
            else:
                return None
        if not Mx and not Nx:
            # no broadcast axis: a plain row reduction with a MUL prologue
            return None
        out = self._new(out_shape, out_dtype)
        # output strides over the leading axes of S (the result shape is S[:-1] + (1,))
        ostr = View.row_major(S[:-1])

        def merged(axes, views):
            """One (size, strides per view) for a group of axes, or None."""
            if not axes:
                return 1, [0] * len(views)
            size = S[axes[0]]
            st = [v[axes[0]] for v in views]
            for a in axes[1:]:
                for i, v in enumerate(views):
                    if st[i] != v[a] * S[a]:
                        return None
                size *= S[a]
                st = [v[a] for v in views]
            return size, st

        estr = [v.strides for _, v, _ in epilogue[1]] if epilogue else []
        gm = merged(Mx, [vx.strides, ostr] + estr)
        gn = merged(Nx, [vy.strides, ostr] + estr)
        if gm is None or gn is None:
            return None
        # batch axes: kept separately when they do not merge (the ABI takes up to 3)
        gb = merged(Bx, [vx.strides, vy.strides, ostr] + estr)
        if Bx and gb is None and epilogue:
            return None
        if Bx and gb is None:
            # batch dims that do not merge (e.g. heads split out of a fused
            # projection): store each operand compactly, so they do
            bx, vx = self._compact(bx, vx, dx, x.dtype)
            by, vy = self._compact(by, vy, dy, y.dtype)
            gm = merged(Mx, [vx.strides, ostr])
            gn = merged(Nx, [vy.strides, ostr])
            gb = merged(Bx, [vx.strides, vy.strides, ostr])
            if gm is None or gn is None or gb is None:
                return None
        batch = [(gb[0], gb[1][0], gb[1][1], gb[1][2])] if Bx else []
        K = S[-1]
        shape = [b[0] for b in batch] + [gm[0], gn[0], K]
        sa = [b[1] for b in batch] + [gm[1][0], 0, vx.strides[-1]]
        sb = [b[2] for b in batch] + [0, gn[1][0], vy.strides[-1]]
        sc = [b[3] for b in batch] + [gm[1][1], gn[1][1]]
        Av = A.make_view(dx, shape, sa, vx.offset, None, bx.numel())
        Bv = A.make_view(dy, shape, sb, vy.offset, None, by.numel())
        Cv = A.make_view(out_dtype, shape[:-1], sc, 0, None, out.numel())
        if epilogue:
            prog, inputs = epilogue
            ev = [A.make_view(d, shape[:-1], [gb[1][3 + k]] * bool(Bx) + [gm[1][2 + k], gn[1][2 + k]], v.offset,
                              None, b.numel()) for k, (b, v, d) in enumerate(inputs)]
            if out.numel():
                st = self._lib("psg_contract")(bx, Av, by, Bv, out, Cv, self._status(), stream=self._s(), check=False,
                                    epilogue=(prog, [b for b, _, _ in inputs], ev))
                if st == A.E_UNSUPPORTED_LAYOUT:
                    return None  # not a tensor-core contraction: computed the ordinary way
                if st != A.OK:
                    raise A.PsgError(st, "psg_contract")
            self.log.append(("contract", tuple(shape), dx, out_dtype, len(prog)))
            return out, View(out_shape)
        if out.numel():
            need = A.psg_contract_workspace(Av, Bv, Cv)
            if need:
                # few output tiles over a long K: the kernel splits K into this workspace
                ws = self._workspace(need)
                self._lib("psg_contract_ws")(bx, Av, by, Bv, out, Cv, ws, ws.numel(), self._status(), stream=self._s())
            else:
                self._lib("psg_contract")(bx, Av, by, Bv, out, Cv, self._status(), stream=self._s())
        self.log.append(("contract", tuple(shape), dx, out_dtype))
        return out, View(out_shape)

    def _compact(self, buf, v, dt, src_dt):
        """Copy the cells a broadcast View reads into a row-major buffer and
        return the same broadcast View over the copy."""
        zero = [a for a, st in enumerate(v.strides) if st == 0 and v.shape[a] > 1]
        small = v.shrink([(0, 1) if a in zero else (0, s) for a, s in enumerate(v.shape)])
        b2, v2 = self._copy_contig(buf, small, src_dt)
        return b2, v2.expand(v.shape)

    # ---- indexed --------------------------------------------------------------------
    def _attn_operand(self, x: Tensor):
        """(buffer, View) of a [B, T, H, 64] bf16 operand the attention
        kernels can read with TMA (head dim contiguous, other strides
        multiples of 8, 16-byte aligned start, no mask); copied first if not."""
        buf, v = self.realize(x)
        ok = (v.mask is None and v.strides[3] == 1 and all(st % 8 == 0 for st in v.strides[:3])
              and (buf.data_ptr() + 2 * v.offset) % 16 == 0)
        if not ok:
            buf, v = self._copy_contig(buf, v, x.dtype)
        return buf, v

    def _attn_slots(self, qkv: Tensor, shape):
        """(buffer, [View of slot 0, 1, 2]) of a packed [B, T, 3, H, 64]
        operand, each slot a [B, T, H, 64] View the kernels can read with TMA
        (the packed tensor is copied contiguous first if a slot is not)."""
        buf, v = self.realize(qkv)
        full = [(0, n) for n in qkv.shape]

        def slots(v):
            return [v.shrink(full[:2] + [(i, i + 1)] + full[3:]).reshape(shape) for i in range(3)]

        vs = slots(v)
        ok = all(x.mask is None and x.strides[3] == 1 and all(st % 8 == 0 for st in x.strides[:3])
                 and (buf.data_ptr() + 2 * x.offset) % 16 == 0 for x in vs)
        if not ok:
            buf, v = self._copy_contig(buf, v, qkv.dtype)
            vs = slots(v)
        return buf, vs

    def _attn_mask(self, fwd: Tensor):
        """The attention node's key mask as a contiguous int8 [B, T] buffer
        starting at its data pointer, or None."""
        if not fwd.arg[2]:
            return None
        buf, v = self.realize(fwd.src[-1])
        if v.mask is not None or v.offset != 0 or not v.contiguous():
            buf, v = self._copy_contig(buf, v, "i8")
        return buf

    def _realize_attn(self, t: Tensor):
        scale, causal, _ = t.arg
        B, T, H, _ = t.shape
        ops = t.src[:-1] if t.arg[2] else t.src
        if len(ops) == 1:  # packed qkv
            b, (vq, vk, vv) = self._attn_slots(ops[0], t.shape)
            bq = bk = bv = b
        else:
            (bq, vq), (bk, vk), (bv, vv) = (self._attn_operand(x) for x in ops)
        km = self._attn_mask(t)
        out = self._new(t.shape, "bf16")
        lse = self._new((B, H, T), "f32")
        self._lib("psg_attention_fwd")(bq, self._pview(bq, vq, "bf16"), bk, self._pview(bk, vk, "bf16"), bv,
                                       self._pview(bv, vv, "bf16"), out, self._pview(out, View(t.shape), "bf16"),
                                       lse, scale, causal, self._status(), stream=self._s(), key_mask=km)
        t._aux = lse
        self.log.append(("attention", t.shape))
        return out, View(t.shape)

    def _realize_attn_bwd(self, t: Tensor):
        fwd, g = t.src[-2:]
        scale, causal, _ = t.arg
        B, T, H, _ = fwd.shape
        bo, vo = self.realize(fwd)
        lse = fwd._aux
        if len(t.src) == 3:
            # packed: dQ, dK, dV land in the slots of one [B, T, 3, H, 64] gradient
            b, vs = self._attn_slots(t.src[0], fwd.shape)
            ops = [(b, x) for x in vs] + [self._attn_operand(g)]
            out = self._new(t.shape, "bf16")
            full = [(0, n) for n in t.shape]
            gv = [View(t.shape).shrink(full[:2] + [(i, i + 1)] + full[3:]).reshape(fwd.shape) for i in range(3)]
        else:
            ops = [self._attn_operand(x) for x in t.src[:3] + (g,)]
            out = self._new(t.shape, "bf16")                  # [3, B, T, H, 64]: dQ, dK, dV
            gv = [View(t.shape).shrink([(i, i + 1)] + [(0, n) for n in fwd.shape]).reshape(fwd.shape)
                  for i in range(3)]
        delta = self._new((B, H, T), "f32")
        pv = lambda bv: self._pview(bv[0], bv[1], "bf16")
        self._lib("psg_attention_bwd")(ops[0][0], pv(ops[0]), ops[1][0], pv(ops[1]), ops[2][0], pv(ops[2]), bo,
                                       pv((bo, vo)), ops[3][0], pv(ops[3]), lse, delta, out, pv((out, gv[0])), out,
                                       pv((out, gv[1])), out, pv((out, gv[2])), scale, causal, self._status(),
                                       stream=self._s(), key_mask=self._attn_mask(fwd))
        self.log.append(("attention_bwd", fwd.shape))
        return out, View(t.shape)

    def _realize_gather(self, t: Tensor):
        src, idx = t.src
        bs, vs = self.realize(src)
        bi, vi = self.realize(idx)
        if not vi.contiguous():
            bi, vi = self._copy_contig(bi, vi, "i32")
        out = self._new(t.shape, t.dtype)
        n = t.shape[0]
        self._lib("psg_gather")(bs, self._pview(bs, vs, src.dtype), bi, n, out, self._pview(out, View(t.shape), t.dtype),
                     self._status(), stream=self._s())
        self.log.append(("gather", t.shape))
        return out, View(t.shape)

    def _realize_scatter(self, t: Tensor):
        dst, idx, upd = t.src
        out = None
        if (dst._real is None and self.users.get(id(dst), 0) == 1 and dst.op in ELEMENTWISE
                and self._narrowable(dst) is None):  # a narrowed contraction's buffer may be shared
            # a value computed for this scatter alone (a zero-filled gradient
            # buffer, say): scatter into its own fresh buffer, no copy
            buf, vd = self.realize(dst)
            if vd.mask is None and vd.offset == 0 and vd.contiguous():
                out, vo = buf, vd
                dst._real = None  # the buffer now holds the scatter's result, not dst's value
        if out is None:
            out, vo = self._copy_contig(*self.realize(dst), dst.dtype, fresh=True)  # scatter-added in place
        bi, vi = self.realize(idx)
        if not vi.contiguous():
            bi, vi = self._copy_contig(bi, vi, "i32")
        bu, vu = self.realize(upd)
        n = idx.shape[0]
        ws = self._workspace(A.psg_scatter_workspace(n))
        self._lib("psg_scatter_add")(out, self._pview(out, vo, t.dtype), bi, n, bu, self._pview(bu, vu, upd.dtype), ws,
                          ws.numel(), self._status(), stream=self._s())
        self.log.append(("scatter_add", t.shape, n))
        return out, vo


def _keeps_row_order(moves, shape, out_shape) -> bool:
    """True when the movements take a contiguous View of `shape` to a
    contiguous View of `out_shape` (cell i stays cell i)."""
    v = View(tuple(shape))
    for kind, arg in moves:
        if kind == "detach":
            continue
        if kind not in ("reshape", "permute"):
            return False
        v = getattr(v, kind)(arg)
        if v is None:
            return False
    return tuple(v.shape) == tuple(out_shape) and v.contiguous()


class _TooBig(Exception):
    pass


class _NotFusable(Exception):
    pass


def _moves_to_base(x):
    """The movements between x and the first non-movement, non-widening node."""
    out = []
    while True:
        if x.op == "MOVE" and x.arg[0] != "pad":
            out.append(x.arg)
            x = x.src[0]
        elif x.op == "CAST" and x.dtype == "f32" and x.src[0].dtype in ("bf16", "f16"):
            x = x.src[0]
        else:
            return out


def _count(t, seen=None):
    seen = seen if seen is not None else set()
    if id(t) in seen or t._real is not None or t.op not in ELEMENTWISE + ("MOVE",):
        return 0
    seen.add(id(t))
    return 1 + sum(_count(s, seen) for s in t.src)


def _is_row_expand(moves, red_shape, row_shape):
    """The movements take a [.., 1] row value to [.., N] by expanding the last axis."""
    mv = [m for m in moves if m[0] != "detach"]
    if not mv:
        return red_shape == row_shape
    v = View(red_shape, [0] * len(red_shape))
    shape = red_shape
    for kind, arg in mv:
        if kind == "expand":
            shape = tuple(arg)
        elif kind == "reshape":
            shape = tuple(arg)
        else:
            return False
    return shape == row_shape and all(m[0] in ("expand", "reshape") for m in mv) and \
        prod(red_shape) == prod(row_shape[:-1])


_EXEC = None


def _executor() -> Executor:
    global _EXEC
    if _EXEC is None:
        _EXEC = Executor()
    return _EXEC


class _Ref:
    """A buffer argument of a recorded call: a leaf of the graph, a buffer
    the schedule allocated, the status word or the current stream."""
    __slots__ = ("kind", "i")

    def __init__(self, kind, i=0):
        self.kind, self.i = kind, i


class _RawCapture:
    """Stands in for the binding's library handle while a call is recorded:
    forwards each raw C call and keeps its function and ctypes arguments."""

    def __init__(self, lib):
        self.lib, self.calls = lib, []

    def __getattr__(self, name):
        f = getattr(self.lib, name)

        def call(*cargs):
            self.calls.append((f, cargs, name))
            return f(*cargs)
        return call


#: Streams a captured replay may spread independent calls over (1: every
#: call on the capturing stream, in order).  Measured on one GB300, the GPT
#: block's replayed step: 0.527 ms on one stream, 0.506 ms on two, 0.520 ms
#: on three (more side streams put more contractions side by side, which
#: then compete for the SMs); keeping contractions off the side streams was
#: slower still (0.520, 0.538 and 0.514 ms on two, three and four streams).
#: Eager calls always run on the current stream.
FORK_STREAMS = int(os.environ.get("PSG_FORK_STREAMS", "2"))

#: The pointer arguments each library call writes, by position; every other
#: buffer argument of the call is only read.
_WRITES = {
    "psg_elementwise": (5,), "psg_reduce_rows": (7,), "psg_permute": (3,), "psg_contract": (4,),
    "psg_contract_ws": (4, 7), "psg_gather": (4,), "psg_scatter_add": (0, 6),
    "psg_attention_fwd": (6, 8), "psg_attention_bwd": (11, 12, 14, 16),
}


class _Fork:
    """The streams of one forked capture: the capturing stream and side
    streams forked from it; each call waits (an event) for its dependencies
    on other streams, and join() brings every side stream back."""

    def __init__(self, sched, main):
        self.where, self.waits = sched
        self.streams = [main] + [torch.cuda.Stream() for _ in range(max(self.where, default=0))]
        for st in self.streams[1:]:
            st.wait_stream(main)
        self.done = {}

    def enter(self, c):
        st = self.streams[self.where[c]]
        for d in self.waits[c]:
            st.wait_event(self.done[d])
        return st.cuda_stream

    def leave(self, c):
        ev = torch.cuda.Event()
        ev.record(self.streams[self.where[c]])
        self.done[c] = ev

    def join(self):
        for st in self.streams[1:]:
            self.streams[0].wait_stream(st)


class _Plan:
    """The library calls one graph structure was realized into, recorded
    once (limn, "Reading the schedule": the compiled devices cache execution
    plans by graph structure).  Replaying it rebinds the buffers and makes
    the same calls: no scheduling, lowering or program building.

    Each call is also kept in its marshalled form (the C function and its
    ctypes arguments: node arrays, Views, sizes) with the places that hold a
    buffer address or the stream; a replay writes the new addresses into
    those places and calls the C function directly.  A call whose arguments
    hold an address the plan cannot name keeps the binding-level path."""

    def __init__(self, ex, leaves):
        self.refs = {id(b): _Ref("leaf", i) for i, b in reversed(list(enumerate(leaves)))}
        self.refs[id(ex._status())] = _Ref("status")
        self.ptrs = {}
        for i, b in reversed(list(enumerate(leaves))):
            self._name_ptr(b, _Ref("leaf", i))
        self._name_ptr(ex._status(), _Ref("status"))
        self.stream_handle = A._stream(ex._s())
        self.allocs, self.keep, self.calls, self.outs, self.log = [], [], [], [], []
        self.fast = []
        self._flat = None  # the slots with flat address indices, made at the first replay
        self._fork = None  # the forked-stream schedule (see _fork_schedule)
        self.ok = True

    def _name_ptr(self, t, ref):
        p = t.data_ptr()
        if p == 0:
            return
        old = self.ptrs.get(p)
        if old is not None and (old.kind, old.i) != (ref.kind, ref.i):
            # leaves that share an address share it in every graph of this
            # structure (the key records the aliasing): either names it
            if not (old.kind == "leaf" and ref.kind == "leaf"):
                self.ptrs[p] = None  # two buffers at one address: not nameable
        elif old is None and p not in self.ptrs:
            self.ptrs[p] = ref

    def alloc(self, t, spec):
        self.refs[id(t)] = _Ref("tmp", len(self.allocs))
        self._name_ptr(t, self.refs[id(t)])
        self.allocs.append(spec)
        self.keep.append(t)

    def _fork_schedule(self, n_leaves):
        """(stream of each call, calls it waits for on other streams), for a
        capture that runs independent calls side by side: a call joins the
        stream whose latest call it depends on, else the stream idle the
        longest.  Dependencies come from the buffers each call reads and
        writes (_WRITES names the written arguments); a call whose buffers
        are not all known depends on every call before it and every later
        call depends on it (computed once per plan)."""
        if self._fork is not None and self._fork[0] == FORK_STREAMS:
            return self._fork[1]
        flat = self._flat_slots(n_leaves)
        n_buf = n_leaves + len(self.allocs)  # status and stream are not buffers
        S = FORK_STREAMS
        last_w, readers = {}, {}
        tail = [-1] * S
        where, waits = [], []
        barrier = -1
        for c, (fast, fslots) in enumerate(zip(self.fast, flat)):
            known = fast is not None and fast[4] in _WRITES
            deps = set() if barrier < 0 else {barrier}
            if known:
                wpos = _WRITES[fast[4]]
                writes = {k for box, at, k in fslots if k < n_buf and box is fast[1] and at in wpos}
                bufs = {k for _, _, k in fslots if k < n_buf}
                for k in bufs:
                    if k in last_w:
                        deps.add(last_w[k])
                for k in writes:
                    deps.update(readers.get(k, ()))
            else:
                deps.update(t for t in tail if t >= 0)
            on = [i for i in range(S) if tail[i] >= 0 and tail[i] in deps]
            if not known:
                s = 0  # a binding-level call runs on the capturing stream
            elif on:
                s = max(on, key=lambda i: tail[i])
            else:
                s = min(range(S), key=lambda i: tail[i])
            # one wait per other stream: its latest call among the dependencies
            w = {}
            for d in deps:
                if where[d] != s and d > w.get(where[d], -1):
                    w[where[d]] = d
            where.append(s)
            waits.append(tuple(sorted(w.values())))
            tail[s] = c
            if known:
                for k in bufs - writes:
                    readers.setdefault(k, set()).add(c)
                for k in writes:
                    last_w[k] = c
                    readers[k] = set()
            else:
                barrier = c
        self._fork = (S, (tuple(where), tuple(waits)))
        return self._fork[1]

    def _flat_slots(self, n_leaves):
        """Each marshalled call's slots as (container, index, k): k indexes
        the leaves' addresses, then the allocated buffers', then the status
        word and the stream (computed once per plan)."""
        flat = self._flat
        if flat is None:
            nt = len(self.allocs)

            def k(r):
                if r.kind == "leaf":
                    return r.i
                if r.kind == "tmp":
                    return n_leaves + r.i
                return n_leaves + nt + (0 if r.kind == "status" else 1)
            flat = [None if f is None else [(box, at, k(r)) for box, at, r in f[2]] for f in self.fast]
            self._flat = flat
        return flat

    def _marshalled(self, raw):
        """(C function, argument list, slots, raw) of one recorded raw call,
        or None; a slot is (container, index, ref).  Which arguments hold
        addresses comes from the C function's declared argument types: a
        void* argument (the last one is the stream), an array of void*
        (input pointers), an epilogue's input array.  A NULL stays as it is;
        any other address must be a buffer the plan names."""
        if len(raw) != 1:
            return None
        f, cargs, cname = raw[0]
        types = getattr(f, "argtypes", None)
        cargs = list(cargs)
        if not types or len(types) != len(cargs):
            return None
        slots = []
        for i, (a, t) in enumerate(zip(cargs, types)):
            if t is ctypes.c_void_p:
                if i == len(cargs) - 1:
                    slots.append((cargs, i, _Ref("stream")))
                elif a:
                    r = self.ptrs.get(a)
                    if r is None:
                        return None
                    slots.append((cargs, i, r))
            elif isinstance(a, ctypes.Array) and a._type_ is ctypes.c_void_p:
                for j in range(len(a)):
                    if a[j]:
                        r = self.ptrs.get(a[j])
                        if r is None:
                            return None
                        slots.append((a, j, r))
            elif type(a).__name__ == "CArgObject" and isinstance(getattr(a, "_obj", None), A.psg_epilogue):
                e = a._obj
                for j in range(e.n_in):
                    if e.in_[j]:
                        r = self.ptrs.get(e.in_[j])
                        if r is None:
                            return None
                        slots.append((e.in_, j, r))
            elif isinstance(a, int) and t is not None and t not in (ctypes.c_int, ctypes.c_int32, ctypes.c_int64,
                                                                    ctypes.c_size_t, ctypes.c_float,
                                                                    ctypes.c_double, ctypes.c_bool):
                return None  # an address-like argument of a type not described here
        return f, cargs, slots, raw, cname

    def sym(self, x, key=None):
        if key == "stream":
            return _Ref("stream")
        if isinstance(x, torch.Tensor):
            r = self.refs.get(id(x))
            if r is None:
                self.ok = False  # a buffer from elsewhere: this schedule is not recorded
            return r
        if isinstance(x, (list, tuple)):
            return type(x)(self.sym(y) for y in x)
        return x

    @staticmethod
    def _has_ref(x):
        if isinstance(x, _Ref):
            return True
        return isinstance(x, (list, tuple)) and any(_Plan._has_ref(y) for y in x)

    def call(self, name, args, kw, raw=()):
        args = self.sym(args)
        kw = {k: self.sym(v, k) for k, v in kw.items()}
        # the arguments that name buffers, rebuilt at each replay; the rest
        # (programs, Views, sizes) are passed as recorded
        dyn = [i for i, x in enumerate(args) if self._has_ref(x)]
        dkw = [k for k, v in kw.items() if self._has_ref(v)]
        self.calls.append((name, args, kw, dyn, dkw))
        self.fast.append(self._marshalled(raw) if raw else None)

    def run(self, ex, leaves, roots):
        status, stream = ex._status(), ex._s()
        tmps = [torch.empty(shape, dtype=dt, device=status.device) for shape, dt in self.allocs]

        def val(x):
            if isinstance(x, _Ref):
                return (leaves[x.i] if x.kind == "leaf" else tmps[x.i] if x.kind == "tmp"
                        else status if x.kind == "status" else stream)
            if isinstance(x, (list, tuple)):
                return type(x)(val(y) for y in x)
            return x
        vals = None
        flat = self._flat_slots(len(leaves))
        fork = None
        if FORK_STREAMS > 1 and torch.cuda.is_available() and torch.cuda.is_current_stream_capturing():
            fork = _Fork(self._fork_schedule(len(leaves)), torch.cuda.current_stream())
        for c, ((name, args, kw, dyn, dkw), fast, fslots) in enumerate(zip(self.calls, self.fast, flat)):
            if fast is not None:
                if vals is None:
                    # every address a slot can take, in the flat order of _flat_slots
                    vals = [b.data_ptr() for b in leaves] + [b.data_ptr() for b in tmps]
                    vals.append(status.data_ptr())
                    vals.append(A._stream(stream))
                if fork is not None:
                    vals[-1] = fork.enter(c)
                f, cargs = fast[0], fast[1]
                for box, at, k in fslots:
                    box[at] = vals[k]
                st = f(*cargs)
                if st != A.OK:
                    A._check(st, name)
                if fork is not None:
                    fork.leave(c)
                continue
            if fork is not None:
                fork.enter(c)  # a binding-level call: on the capturing stream, after everything
            if dyn:
                args = list(args)
                for i in dyn:
                    args[i] = val(args[i])
            if dkw:
                kw = dict(kw)
                for k in dkw:
                    kw[k] = val(kw[k])
            getattr(A, name)(*args, **kw)
            if fork is not None:
                fork.leave(c)
        if fork is not None:
            fork.join()  # before this step's buffers can be freed and reused
        ex.log.extend(self.log)
        out = []
        for t, (ref, v, dt) in zip(roots, self.outs):
            buf = val(ref)
            t._real = (buf, v)
            out.append(_as_torch(buf, v, dt))
        return out


#: Whether a contraction's epilogue program may read further tensors (a
#: residual, a ReLU's saved pre-activation).  Off: only programs of the
#: accumulator alone (a ReLU, a cast) fuse.  Measured on one GB300 at the GPT
#: block's shapes, an input in the epilogue costs about as much as the
#: separate elementwise launch it replaces (the epilogue warps issue the
#: loads and the node arithmetic of every cell): the residual add at 8192 x
#: 512 x 512, 19.1 us fused against 12.3 + 9.0 us; the ReLU-mask gradient at
#: 8192 x 2048 x 512, 43.6 us against 24.6 + 15.8 us; a ReLU alone, 27.3 us
#: against 24.6 + 11.7 us.  The GPT block's replayed step: 0.538 ms unfused,
#: 0.552 ms with its residual adds and ReLU-mask gradient fused, 0.551 ms
#: with the residual adds alone fused (each a win measured on its own: the
#: step's standalone add shares its launch with the work around it).
FUSE_EPILOGUE_INPUTS = False

#: entries the executor's call log keeps (older ones are dropped)
LOG_KEEP = 1 << 14

#: graph structure -> recorded plan; PLAN_CACHE = False (or PSG_NO_PLAN_CACHE
#: in the environment) schedules every realization afresh
_PLANS = {}
PLAN_CACHE = os.environ.get("PSG_NO_PLAN_CACHE") is None
_PLAN_LIMIT = 256


_PLAIN_ARG = (type(None), int, float, str, bool)


def _structure(roots):
    """(key, leaf buffers) of the unrealized graph under roots: every node's
    op, dtype, shape, argument and operands by position, every leaf's
    layout, size, alignment and aliasing; equal keys schedule alike."""
    index, items, leaves, first_ptr = {}, [], [], {}  # nodes hash by identity
    add, add_leaf = items.append, leaves.append
    stack = list(reversed(roots))
    pop, push = stack.pop, stack.append
    while stack:
        t = stack[-1]
        if t in index:
            pop()
            continue
        real = t._real
        if real is not None:
            pop()
            buf, v = real
            p = buf.data_ptr()
            aux = t._aux
            add(("L", t.dtype, t.shape, v.key(), buf.dtype, buf.numel(), p % 256,
                 first_ptr.setdefault(p, len(leaves)), aux is not None))
            add_leaf(buf)
            if aux is not None:
                add_leaf(aux)
            index[t] = len(items) - 1
            continue
        src = t.src
        waiting = False
        for s in reversed(src):
            if s not in index:
                push(s)
                waiting = True
        if waiting:
            continue
        pop()
        arg = t.arg
        ta = type(arg)
        add((t.op, t.dtype, t.shape, arg if ta in _PLAIN_ARG or ta is tuple else repr(arg),
             tuple([index[s] for s in src])))
        index[t] = len(items) - 1
    # the schedule also depends on the fusion switch
    return (tuple(items), tuple([index[r] for r in roots]), FUSE_EPILOGUE_INPUTS), leaves


def realize_all(*ts):
    """Realize several values with one schedule (shared subexpressions are
    computed once) and return them as torch tensors.  The schedule of a
    graph structure seen before is replayed from the plan cache."""
    ex = _executor()
    if len(ex.log) > LOG_KEEP:  # keep the recent calls only: a long eager loop would grow it forever
        del ex.log[:len(ex.log) - LOG_KEEP // 2]
    key = leaves = None
    if PLAN_CACHE:
        key, leaves = _structure(ts)
        try:
            plan = _PLANS.get(key)
        except TypeError:  # an argument tuple holding something unhashable: not cached
            key = plan = None
        if plan is not None:
            return plan.run(ex, leaves, ts)
    ex.prepare(ts)
    rec = _Plan(ex, leaves) if key is not None else None
    ex.rec = rec
    n0 = len(ex.log)
    try:
        out = []
        for t in ts:
            buf, v = ex.realize(t)
            if v.mask is not None:
                buf, v = ex._copy_contig(buf, v, t.dtype, fresh=True)
            out.append(_as_torch(buf, v, t.dtype))
            if rec is not None:
                rec.outs.append((rec.sym(buf), v, t.dtype))
    finally:
        ex.rec = None
    if rec is not None and rec.ok:
        rec.log = ex.log[n0:]
        rec.keep = []
        if len(_PLANS) >= _PLAN_LIMIT:
            _PLANS.pop(next(iter(_PLANS)))
        _PLANS[key] = rec
    return out


class Replay:
    """Capture and replay of one step (limn, "Backends": capture records a
    step's kernel calls once and replays them with new buffers).

    ``fn(*inputs)`` builds and realizes a graph and returns a torch tensor or
    a tuple/list/dict of them.  The first call runs it eagerly, which
    compiles every specialised kernel; the second records it into a CUDA
    Graph on a side stream, with calls that depend on nothing the calls
    before them on a stream write spread over FORK_STREAMS forked streams
    (event edges carry every dependency; all streams join before the step's
    buffers are released).  Each ``replay(*inputs)`` copies the new inputs
    into the recorded input buffers and relaunches the recorded kernels:
    no graph building, scheduling or launch work on the host.  The returned
    outputs are the recorded output buffers, overwritten by the next replay.
    Inputs must keep the example inputs' shapes and dtypes."""

    def __init__(self, fn, *example_inputs):
        self.fn = fn
        self.inputs = [x.detach().clone() for x in example_inputs]
        fn(*self.inputs)                       # compiles the kernels
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn(*self.inputs)                   # allocator warm-up off the capture
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.outputs = fn(*self.inputs)
        torch.cuda.synchronize()

    def replay(self, *inputs):
        for dst, src in zip(self.inputs, inputs):
            if src is not None and src.data_ptr() != dst.data_ptr():
                dst.copy_(src, non_blocking=True)
        self.graph.replay()
        return self.outputs

    __call__ = replay


# ------------------------------------------------------------ autograd -------

def _toposort(root):
    order, seen = [], set()
    stack = [(root, False)]
    while stack:
        t, done = stack.pop()
        if done:
            order.append(t)
            continue
        if id(t) in seen:
            continue
        seen.add(id(t))
        stack.append((t, True))
        for s in t.src:
            if s.requires_grad and id(s) not in seen:
                stack.append((s, False))
    return order


def _sum_to(g: Tensor, shape) -> Tensor:
    """Undo a broadcast: SUM g over the axes where shape has 1."""
    if g.shape == tuple(shape):
        return g
    nd = len(shape)
    while g.ndim > nd:
        g = g.sum(0, keepdim=False)
    for a in range(nd):
        if shape[a] == 1 and g.shape[a] != 1:
            g = g.sum(a, keepdim=True)
    return g


def _is_relu(t: Tensor) -> bool:
    """t = WHERE(CMPLT(0, x), x, 0), the form Tensor.relu builds."""
    if t.op != "WHERE":
        return False
    c, x, y = t.src
    return (c.op == "CMPLT" and c.src[1] is x and c.src[0].op == "CONST" and c.src[0].arg == 0.0
            and y.op == "CONST" and y.arg == 0.0 and c.src[0]._real is None and y._real is None)


def _vjp(t: Tensor, g: Tensor):
    op, s = t.op, t.src
    if op == "ADD":
        return [(s[0], g), (s[1], g)]
    if op == "MUL":
        return [(s[0], g * s[1]), (s[1], g * s[0])]
    if op == "NEG":
        return [(s[0], -g)]
    if op == "EXP":
        return [(s[0], g * t)]
    if op == "LOG":
        return [(s[0], g * s[0].recip())]
    if op == "SQRT":
        return [(s[0], g * 0.5 * t.recip())]
    if op == "RECIP":
        return [(s[0], -g * (t * t))]
    if op == "CAST":
        return [(s[0], g.cast(s[0].dtype))] if s[0].dtype in FLOATS else []
    if op == "WHERE":
        z = Tensor.const(0.0, (), g.dtype)
        c = s[0]
        if _is_relu(t):
            # 0 < x and 0 < relu(x) are the same bit for every x (NaN and -0
            # included), so the mask is taken from the output: the input is
            # then read by nothing but the ReLU itself
            c = Tensor.const(0.0, t.shape, t.dtype).cmplt(t)
        return [(s[1], c.where(g, z)), (s[2], s[0].where(z, g))]
    if op == "SUM":
        return [(s[0], g.expand(s[0].shape))]
    if op == "MAX":
        # gradient to the cells equal to the max
        m = t.expand(s[0].shape)
        eq = (s[0].cmplt(m).cast("f32") + m.cmplt(s[0]).cast("f32")).cmplt(Tensor.const(0.5, (), "f32"))
        return [(s[0], eq.where(g.expand(s[0].shape), Tensor.const(0.0, (), g.dtype)))]
    if op == "MOVE":
        kind, arg = t.arg
        src = s[0]
        if kind == "detach":
            return []
        if kind == "reshape":
            return [(src, g.reshape(src.shape))]
        if kind == "permute":
            return [(src, g.permute(_inverse(arg)))]
        if kind == "expand":
            return [(src, _sum_to(g, src.shape))]
        if kind == "shrink":
            return [(src, g.pad([(a, n - b) for (a, b), n in zip(arg, src.shape)]))]
        if kind == "pad":
            return [(src, g.shrink([(a, a + n) for (a, _), n in zip(arg, src.shape)]))]
    if op == "CONTIG":
        return [(s[0], g)]
    if op == "GATHER":
        return [(s[0], Tensor.zeros(s[0].shape, s[0].dtype).scatter_add(s[1], g))]
    if op == "SCATTER":
        return [(s[0], g), (s[2], g.gather(s[1]))]
    if op == "ATTN":
        # one node computes dQ, dK, dV together (the two-pass backward); the
        # key mask (the last operand, when there is one) has no gradient
        gb = g.cast("bf16") if g.dtype != "bf16" else g
        if t.arg[2]:
            s = s[:-1]
        if len(s) == 1:  # packed qkv: the gradient in the same packed layout
            return [(s[0], Tensor("ATTN_BWD", (s[0], t, gb), s[0].shape, "bf16", arg=t.arg))]
        d = Tensor("ATTN_BWD", (s[0], s[1], s[2], t, gb), (3,) + t.shape, "bf16", arg=t.arg)
        full = [(0, n) for n in t.shape]
        return [(s[i], d.shrink([(i, i + 1)] + full).reshape(t.shape)) for i in range(3)]
    return []


def backward(root: Tensor, grad: Tensor | None = None):
    """Reverse-mode autograd over the lazy graph: every leaf that requires a
    gradient gets ``.grad``, itself a lazy graph of primitives (limn,
    "Architecture": the gradients are lazy graphs like everything else)."""
    if grad is None:
        assert root.numel() == 1, "backward of a non-scalar needs a gradient"
        grad = Tensor.const(1.0, root.shape, root.dtype)
    grads = {id(root): grad}
    for t in reversed(_toposort(root)):
        g = grads.pop(id(t), None)
        if g is None:
            continue
        if not t.src:
            t.grad = g if t.grad is None else t.grad + g
            continue
        for src, gs in _vjp(t, g):
            if not src.requires_grad:
                continue
            if gs.shape != src.shape:
                gs = _sum_to(gs, src.shape)
            prev = grads.get(id(src))
            grads[id(src)] = gs if prev is None else prev + gs
