"""Thin ctypes binding of libpsg.so (include/psg.h), same names as the C ABI.

Argument marshalling only: every step of the hot path runs in the library's
sm_103a kernels.  There is no fallback of any kind: if libpsg.so is missing
the import of this module raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpsg.so")

MAX_DIMS = 8
MAX_NODES = 64
MAX_INPUTS = 8

# psg_status
OK = 0
STATUS = {0: "PSG_OK", 1: "PSG_E_INVALID_ARG", 2: "PSG_E_UNSUPPORTED_DTYPE",
          3: "PSG_E_UNSUPPORTED_LAYOUT", 4: "PSG_E_OUT_OF_BOUNDS_VIEW", 5: "PSG_E_MISALIGNED",
          6: "PSG_E_INDEX_OUT_OF_RANGE", 7: "PSG_E_TIMEOUT", 8: "PSG_E_CUDA",
          9: "PSG_E_UNSUPPORTED_PROGRAM", 10: "PSG_E_WORKSPACE"}
E_INVALID_ARG, E_UNSUPPORTED_DTYPE, E_UNSUPPORTED_LAYOUT, E_OUT_OF_BOUNDS_VIEW = 1, 2, 3, 4
E_MISALIGNED, E_INDEX_OUT_OF_RANGE, E_TIMEOUT, E_CUDA = 5, 6, 7, 8
E_UNSUPPORTED_PROGRAM, E_WORKSPACE = 9, 10

# psg_dtype
DTYPES = {"f32": 0, "bf16": 1, "f16": 2, "f64": 3, "i32": 4, "i16": 5, "i8": 6}
DTYPE_NAMES = {v: k for k, v in DTYPES.items()}
DTYPE_SIZE = {"f32": 4, "bf16": 2, "f16": 2, "f64": 8, "i32": 4, "i16": 2, "i8": 1}

# psg_op
OPS = {"LOAD": 0, "CONST": 1, "RED": 2, "NEG": 3, "EXP": 4, "LOG": 5, "SQRT": 6, "RECIP": 7,
       "CAST": 8, "ADD": 9, "MUL": 10, "CMPLT": 11, "WHERE": 12, "ACC": 13}
RED_SUM, RED_MAX = 0, 1
CALLS = {"elementwise": 0, "reduce_rows": 1, "permute": 2, "contract_bf16": 3,
         "contract_f32": 4, "gather": 5, "scatter_add": 6, "contract_f32_tensor": 7}


class psg_view(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("shape", ctypes.c_int64 * MAX_DIMS), ("strides", ctypes.c_int64 * MAX_DIMS),
                ("offset", ctypes.c_int64), ("mask_lo", ctypes.c_int64 * MAX_DIMS),
                ("mask_hi", ctypes.c_int64 * MAX_DIMS), ("extent", ctypes.c_int64)]


class psg_node(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("a", ctypes.c_int32), ("b", ctypes.c_int32),
                ("c", ctypes.c_int32), ("dtype", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("cval", ctypes.c_double)]


class psg_reduce_stage(ctypes.Structure):
    _fields_ = [("op", ctypes.c_int32), ("n_nodes", ctypes.c_int32),
                ("prologue", ctypes.POINTER(psg_node))]


class psg_epilogue(ctypes.Structure):
    _fields_ = [("prog", ctypes.POINTER(psg_node)), ("n_nodes", ctypes.c_int32), ("n_in", ctypes.c_int32),
                ("in_", ctypes.POINTER(ctypes.c_void_p)), ("in_v", ctypes.POINTER(psg_view))]


class psg_adamw_tensor(ctypes.Structure):
    _fields_ = [("p", ctypes.c_void_p), ("g", ctypes.c_void_p), ("m", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("numel", ctypes.c_int64)]


class PsgError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (call, STATUS.get(status, status),
                                                 status_string(status)))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libpsg.so is not built (%s); run primitive_sm_graph_gb300.build.build()"
                          % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    V = ctypes.POINTER(psg_view)
    N = ctypes.POINTER(psg_node)
    S = ctypes.POINTER(psg_reduce_stage)
    P32 = ctypes.POINTER(ctypes.c_int32)
    L.psg_elementwise.argtypes = [N, i32, ctypes.POINTER(vp), V, i32, vp, V, vp]
    L.psg_reduce_rows.argtypes = [S, i32, N, i32, ctypes.POINTER(vp), V, i32, vp, V, vp, vp]
    L.psg_permute.argtypes = [vp, V, P32, vp, V, vp]
    E = ctypes.POINTER(psg_epilogue)
    L.psg_contract.argtypes = [vp, V, vp, V, vp, V, E, vp, vp]
    L.psg_contract_ws.argtypes = [vp, V, vp, V, vp, V, E, vp, sz, vp, vp]
    L.psg_contract_workspace.argtypes = [V, V, V]
    L.psg_contract_workspace.restype = sz
    L.psg_gather.argtypes = [vp, V, vp, i64, vp, V, vp, vp]
    L.psg_scatter_workspace.argtypes = [i64]
    L.psg_scatter_workspace.restype = sz
    L.psg_scatter_add.argtypes = [vp, V, vp, i64, vp, V, vp, sz, vp, vp]
    L.psg_scatter_add_static.argtypes = [vp, V, vp, i64, vp, V, vp, vp]
    L.psg_scatter_add_static.restype = i32
    L.psg_query_launch.argtypes = [i32, V, P32, P32, P32, P32]
    fl = ctypes.c_float
    L.psg_attention_fwd.argtypes = [vp, V, vp, V, vp, V, vp, V, vp, fl, i32, vp, vp, vp]
    L.psg_adamw_step.argtypes = [ctypes.POINTER(psg_adamw_tensor), i32, i32, fl, fl, fl, fl, fl, vp, vp, vp]
    L.psg_attention_bwd.argtypes = [vp, V, vp, V, vp, V, vp, V, vp, V, vp, vp, vp, V, vp, V, vp, V, fl, i32, vp,
                                    vp, vp]
    L.psg_status_string.argtypes = [i32]
    L.psg_status_string.restype = ctypes.c_char_p
    L.psg_version.restype = ctypes.c_char_p
    for f in ("psg_elementwise", "psg_reduce_rows", "psg_permute", "psg_contract", "psg_contract_ws", "psg_gather",
              "psg_scatter_add", "psg_query_launch", "psg_attention_fwd", "psg_attention_bwd",
              "psg_adamw_step"):
        getattr(L, f).restype = i32
    return L


lib = _load()


def status_string(s: int) -> str:
    return lib.psg_status_string(int(s)).decode()


def version() -> str:
    return lib.psg_version().decode()


def _ptr(x) -> int:
    """A device pointer from a torch tensor or an int (0 = NULL)."""
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def make_view(dtype: str, shape, strides=None, offset: int = 0, mask=None,
              extent: int | None = None) -> psg_view:
    """Build a psg_view; strides default to row-major contiguous, extent to
    the largest element the View reaches plus one."""
    shape = [int(s) for s in shape]
    nd = len(shape)
    if nd > MAX_DIMS:
        raise ValueError("at most %d dims" % MAX_DIMS)
    if strides is None:
        strides, s = [0] * nd, 1
        for d in range(nd - 1, -1, -1):
            strides[d] = s
            s *= shape[d]
    v = psg_view()
    v.ndim = nd
    v.dtype = DTYPES[dtype]
    v.offset = int(offset)
    for d in range(nd):
        v.shape[d] = shape[d]
        v.strides[d] = int(strides[d])
        lo, hi = mask[d] if mask is not None else (0, shape[d])
        v.mask_lo[d] = int(lo)
        v.mask_hi[d] = int(hi)
    if extent is None:
        extent = int(offset) + sum((sh - 1) * st for sh, st in zip(shape, strides)) + 1
        extent = max(extent, 0) if all(s > 0 for s in shape) else 0
    v.extent = int(extent)
    return v


def view_of(t, shape=None, strides=None, offset: int = 0, mask=None) -> psg_view:
    """psg_view over a torch tensor's memory (from its data pointer); by
    default the tensor's own shape and strides."""
    from .tensor_util import dtype_name
    dt = dtype_name(t.dtype)
    es = t.element_size()
    extent = (t.untyped_storage().nbytes() - t.storage_offset() * es) // es
    if shape is None:
        shape, strides = list(t.shape), list(t.stride())
    return make_view(dt, shape, strides, offset, mask, extent)


def node(op: str, a: int = 0, b: int = 0, c: int = 0, dtype: str = "f32",
         cval: float = 0.0) -> psg_node:
    n = psg_node()
    n.op, n.a, n.b, n.c = OPS[op], int(a), int(b), int(c)
    n.dtype = DTYPES[dtype]
    n.cval = float(cval)
    return n


def _nodes(prog):
    arr = (psg_node * max(1, len(prog)))(*prog)
    return arr, len(prog)


def _views(vs):
    return (psg_view * max(1, len(vs)))(*vs)


def _check(st: int, call: str):
    if st != OK:
        raise PsgError(st, call)


# ---------------------------------------------------------------- calls ----

def psg_elementwise(prog, ins, in_views, out, out_view, stream=None, check=True) -> int:
    arr, n = _nodes(prog)
    ptrs = (ctypes.c_void_p * max(1, len(ins)))(*[_ptr(x) for x in ins])
    vs = _views(in_views)
    st = lib.psg_elementwise(arr, n, ptrs, vs, len(ins), _ptr(out), ctypes.byref(out_view),
                             _stream(stream))
    if check:
        _check(st, "psg_elementwise")
    return st


def psg_reduce_rows(stages, epilogue, ins, in_views, out, out_view, d_status=None, stream=None,
                    check=True) -> int:
    """stages: list of (op, prologue node list) with op RED_SUM / RED_MAX."""
    keep = []
    sarr = (psg_reduce_stage * max(1, len(stages)))()
    for i, (op, prog) in enumerate(stages):
        arr, n = _nodes(prog)
        keep.append(arr)
        sarr[i].op = int(op)
        sarr[i].n_nodes = n
        sarr[i].prologue = ctypes.cast(arr, ctypes.POINTER(psg_node))
    earr, ne = _nodes(epilogue or [])
    ptrs = (ctypes.c_void_p * max(1, len(ins)))(*[_ptr(x) for x in ins])
    st = lib.psg_reduce_rows(sarr, len(stages), earr if epilogue else None, ne if epilogue else 0,
                             ptrs, _views(in_views), len(ins), _ptr(out), ctypes.byref(out_view),
                             _ptr(d_status), _stream(stream))
    if check:
        _check(st, "psg_reduce_rows")
    return st


def psg_permute(inp, in_view, perm, out, out_view, stream=None, check=True) -> int:
    p = (ctypes.c_int32 * max(1, len(perm)))(*[int(x) for x in perm])
    st = lib.psg_permute(_ptr(inp), ctypes.byref(in_view), p, _ptr(out), ctypes.byref(out_view),
                         _stream(stream))
    if check:
        _check(st, "psg_permute")
    return st


def _epilogue(epilogue):
    """psg_epilogue from (program nodes, input buffers, input views), or a
    NULL pointer for None; returns (pointer, objects to keep alive)."""
    if not epilogue or not epilogue[0]:
        return None, ()
    prog, ins, views = epilogue
    arr, n = _nodes(prog)
    ptrs = (ctypes.c_void_p * max(1, len(ins)))(*[_ptr(x) for x in ins])
    vs = _views(views)
    e = psg_epilogue(ctypes.cast(arr, ctypes.POINTER(psg_node)), n, len(ins), ctypes.cast(ptrs, ctypes.POINTER(
        ctypes.c_void_p)), ctypes.cast(vs, ctypes.POINTER(psg_view)))
    return ctypes.byref(e), (e, arr, ptrs, vs)


def psg_contract(A, Av, B, Bv, C, Cv, d_status=None, stream=None, check=True, epilogue=None) -> int:
    """epilogue: None, or (program nodes, input buffers, input views): C is
    then the program's value at each cell, with ACC the cell's float32
    total."""
    ep, keep = _epilogue(epilogue)
    st = lib.psg_contract(_ptr(A), ctypes.byref(Av), _ptr(B), ctypes.byref(Bv), _ptr(C),
                          ctypes.byref(Cv), ep, _ptr(d_status), _stream(stream))
    del keep
    if check:
        _check(st, "psg_contract")
    return st


def psg_contract_workspace(Av, Bv, Cv) -> int:
    """Device bytes psg_contract_ws would use to split K for these views (0: no split)."""
    return int(lib.psg_contract_workspace(ctypes.byref(Av), ctypes.byref(Bv), ctypes.byref(Cv)))


def psg_contract_ws(A, Av, B, Bv, C, Cv, workspace, ws_bytes, d_status=None, stream=None, check=True,
                    epilogue=None) -> int:
    ep, keep = _epilogue(epilogue)
    st = lib.psg_contract_ws(_ptr(A), ctypes.byref(Av), _ptr(B), ctypes.byref(Bv), _ptr(C), ctypes.byref(Cv), ep,
                             _ptr(workspace), int(ws_bytes), _ptr(d_status), _stream(stream))
    del keep
    if check:
        _check(st, "psg_contract_ws")
    return st


def psg_attention_fwd(q, qv, k, kv, v, vv, o, ov, lse, scale, causal=True, d_status=None, stream=None,
                      check=True, key_mask=None) -> int:
    """Fused attention forward over [B, T, H, 64] bf16 views; lse: float32
    [B, H, T] device buffer (written); key_mask: None or a device byte
    tensor [B, T] (nonzero: the key is visible)."""
    st = lib.psg_attention_fwd(_ptr(q), ctypes.byref(qv), _ptr(k), ctypes.byref(kv), _ptr(v), ctypes.byref(vv),
                               _ptr(o), ctypes.byref(ov), _ptr(lse), float(scale), 1 if causal else 0,
                               _ptr(key_mask), _ptr(d_status), _stream(stream))
    if check:
        _check(st, "psg_attention_fwd")
    return st


def psg_attention_bwd(q, qv, k, kv, v, vv, o, ov, do, dov, lse, delta, dq, dqv, dk, dkv, dv, dvv, scale,
                      causal=True, d_status=None, stream=None, check=True, key_mask=None) -> int:
    """Fused attention backward: dQ, dK, dV (bf16 [B, T, H, 64] views) from
    dO and the forward's O and lse; delta: float32 [B, H, T] scratch;
    key_mask as for the forward."""
    st = lib.psg_attention_bwd(_ptr(q), ctypes.byref(qv), _ptr(k), ctypes.byref(kv), _ptr(v), ctypes.byref(vv),
                               _ptr(o), ctypes.byref(ov), _ptr(do), ctypes.byref(dov), _ptr(lse), _ptr(delta),
                               _ptr(dq), ctypes.byref(dqv), _ptr(dk), ctypes.byref(dkv), _ptr(dv),
                               ctypes.byref(dvv), float(scale), 1 if causal else 0, _ptr(key_mask),
                               _ptr(d_status), _stream(stream))
    if check:
        _check(st, "psg_attention_bwd")
    return st


def psg_adamw_step(params, grads, ms, vs, lr, beta1, beta2, eps, weight_decay, beta_pow, d_status=None,
                   stream=None, check=True) -> int:
    """One AdamW step over lists of torch tensors (params and grads share a
    dtype; ms, vs float32); beta_pow: float32 device tensor [2]."""
    n = len(params)
    arr = (psg_adamw_tensor * max(1, n))()
    for i, (p, g, m, v) in enumerate(zip(params, grads, ms, vs)):
        arr[i].p, arr[i].g, arr[i].m, arr[i].v = _ptr(p), _ptr(g), _ptr(m), _ptr(v)
        arr[i].numel = p.numel()
    dt = DTYPES[__import__("primitive_sm_graph_gb300.tensor_util", fromlist=["x"]).dtype_name(params[0].dtype)] \
        if n else 0
    st = lib.psg_adamw_step(arr, n, dt, float(lr), float(beta1), float(beta2), float(eps), float(weight_decay),
                            _ptr(beta_pow), _ptr(d_status), _stream(stream))
    if check:
        _check(st, "psg_adamw_step")
    return st


def psg_gather(src, sv, idx, n, out, ov, d_status, stream=None, check=True) -> int:
    st = lib.psg_gather(_ptr(src), ctypes.byref(sv), _ptr(idx), int(n), _ptr(out),
                        ctypes.byref(ov), _ptr(d_status), _stream(stream))
    if check:
        _check(st, "psg_gather")
    return st


def psg_scatter_workspace(n: int) -> int:
    return int(lib.psg_scatter_workspace(int(n)))


def psg_scatter_add(dst, dv, idx, n, upd, uv, workspace, ws_bytes, d_status, stream=None,
                    check=True) -> int:
    st = lib.psg_scatter_add(_ptr(dst), ctypes.byref(dv), _ptr(idx), int(n), _ptr(upd),
                             ctypes.byref(uv), _ptr(workspace), int(ws_bytes), _ptr(d_status),
                             _stream(stream))
    if check:
        _check(st, "psg_scatter_add")
    return st


SCATTER_STATIC_MAX_N = 1 << 20


def psg_scatter_add_static(dst, dv, idx, n, upd, uv, d_status, stream=None, check=True) -> int:
    """psg_scatter_add without a workspace: its keys live in a fixed array
    inside the library (n <= SCATTER_STATIC_MAX_N), for callers that cannot
    allocate device memory."""
    st = lib.psg_scatter_add_static(_ptr(dst), ctypes.byref(dv), _ptr(idx), int(n), _ptr(upd),
                                    ctypes.byref(uv), _ptr(d_status), _stream(stream))
    if check:
        _check(st, "psg_scatter_add_static")
    return st


def psg_query_launch(call: str, v: psg_view):
    g, b, s, r = (ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32())
    st = lib.psg_query_launch(CALLS[call], ctypes.byref(v), ctypes.byref(g), ctypes.byref(b),
                              ctypes.byref(s), ctypes.byref(r))
    _check(st, "psg_query_launch")
    return dict(grid=g.value, block=b.value, smem=s.value, regs=r.value)


def psg_status_string(s: int) -> str:
    return status_string(s)


def psg_version() -> str:
    return version()
