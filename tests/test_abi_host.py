"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/psg.h declares, and refuses bad arguments before any
launch with the documented status codes."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def A():
    from primitive_sm_graph_gb300 import build
    build.build()
    from primitive_sm_graph_gb300 import _abi
    return _abi


def test_exports_every_declared_symbol(A):
    hdr = open(os.path.join(ROOT, "include", "psg.h")).read()
    names = set(re.findall(r"^\s*(?:psg_status|size_t|const char\*)\s+(psg_\w+)\s*\(", hdr, re.M))
    assert {"psg_elementwise", "psg_reduce_rows", "psg_permute", "psg_contract", "psg_gather",
            "psg_scatter_add", "psg_scatter_workspace", "psg_query_launch",
            "psg_status_string", "psg_version"} <= names
    lib = ctypes.CDLL(A.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(A):
    assert A.status_string(0) == "ok"
    assert "index" in A.status_string(A.E_INDEX_OUT_OF_RANGE)
    assert A.status_string(999) == "unknown status"
    assert "sm_103a" in A.version()


def _copy_prog(dt="f32"):
    from primitive_sm_graph_gb300._abi import node
    return [node("LOAD", 0, dtype=dt)]


def test_elementwise_rejects_bad_arguments(A):
    out = A.make_view("f32", (4, 4))
    inp = A.make_view("f32", (4, 4))
    fake = 0x10000  # never dereferenced: every case below fails validation
    st = A.psg_elementwise([], [fake], [inp], fake, out, stream=0, check=False)
    assert st == A.E_INVALID_ARG
    bad = A.make_view("f32", (4, 4), extent=10)  # reaches element 15
    assert A.psg_elementwise(_copy_prog(), [fake], [bad], fake, out, stream=0,
                             check=False) == A.E_OUT_OF_BOUNDS_VIEW
    shape_mismatch = A.make_view("f32", (4, 5))
    assert A.psg_elementwise(_copy_prog(), [fake], [shape_mismatch], fake, out, stream=0,
                             check=False) == A.E_INVALID_ARG
    # a float64 load into a float32 result without a CAST: the dtype rules refuse it
    f64 = A.make_view("f64", (4, 4))
    assert A.psg_elementwise([A.node("LOAD", 0, dtype="f64")], [fake], [f64], fake, out, stream=0,
                             check=False) == A.E_UNSUPPORTED_DTYPE
    # output must be injective: a stride-0 dim of size 4
    aliased = A.make_view("f32", (4, 4), strides=(4, 0), extent=16)
    assert A.psg_elementwise(_copy_prog(), [fake], [inp], fake, aliased, stream=0,
                             check=False) == A.E_UNSUPPORTED_LAYOUT
    # misaligned float pointer
    assert A.psg_elementwise(_copy_prog(), [fake + 2], [inp], fake, out, stream=0,
                             check=False) == A.E_MISALIGNED
    # dtype disagreement between LOAD and its input
    assert A.psg_elementwise(_copy_prog("i32"), [fake], [inp], fake, out, stream=0,
                             check=False) == A.E_UNSUPPORTED_DTYPE
    # EXP of an integer
    i32 = A.make_view("i32", (4, 4))
    prog = [A.node("LOAD", 0, dtype="i32"), A.node("EXP", 0, dtype="i32")]
    assert A.psg_elementwise(prog, [fake], [i32], fake, i32, stream=0,
                             check=False) == A.E_UNSUPPORTED_DTYPE
    # an operand that names a later node
    prog = [A.node("ADD", 1, 1), A.node("LOAD", 0)]
    assert A.psg_elementwise(prog, [fake], [inp], fake, out, stream=0,
                             check=False) == A.E_INVALID_ARG


def _compile_hook(A):
    L = A.lib
    f = L.psg_internal_compile_elementwise
    f.argtypes = [ctypes.POINTER(A.psg_node), ctypes.c_int, ctypes.POINTER(A.psg_view), ctypes.c_int,
                  ctypes.POINTER(A.psg_view), ctypes.c_char_p, ctypes.c_size_t]
    return f


def test_generated_kernels_compile_without_a_gpu(A):
    """Random programs over every dtype plan and compile (NVRTC, sm_103a)."""
    import torch
    f = _compile_hook(A)
    g = torch.Generator().manual_seed(5)
    fdt, idt = ["f32", "bf16", "f16"], ["i32", "i16", "i8"]
    buf = ctypes.create_string_buffer(1 << 16)
    for case in range(12):
        pool = fdt if case % 2 == 0 else idt
        dts = [pool[int(torch.randint(0, 3, (1,), generator=g))] for _ in range(3)]
        prog = [A.node("LOAD", k, dtype=dts[k]) for k in range(3)]
        for _ in range(8):
            i = int(torch.randint(0, len(prog), (1,), generator=g))
            dt = DT_OF(prog[i])
            op = ["ADD", "MUL", "CMPLT", "NEG", "CAST", "WHERE"][int(torch.randint(0, 6, (1,), generator=g))]
            if op == "CAST":
                t = (fdt + idt)[int(torch.randint(0, 6, (1,), generator=g))]
                prog.append(A.node("CAST", i, dtype=t))
            elif op == "NEG":
                prog.append(A.node("NEG", i, dtype=dt))
            elif op == "WHERE":
                prog.append(A.node("WHERE", 0, i, i, dtype=dt))
            else:
                prog.append(A.node(op, i, i, dtype=dt))
        ins = (A.psg_view * 3)(*[A.make_view(d, (7, 33)) for d in dts])
        out = A.make_view(DT_OF(prog[-1]), (7, 33))
        arr = (A.psg_node * len(prog))(*prog)
        st = f(arr, len(prog), ins, 3, ctypes.byref(out), buf, len(buf))
        assert st == 0, (case, A.STATUS.get(st), buf.value.decode()[:2000])


def DT_OF(nd):
    from primitive_sm_graph_gb300._abi import DTYPE_NAMES
    return DTYPE_NAMES[nd.dtype]


def test_permute_rejects_bad_arguments(A):
    fake = 0x10000
    iv = A.make_view("f32", (3, 5))
    ov = A.make_view("f32", (5, 3))
    assert A.psg_permute(fake, iv, [0, 0], fake, ov, stream=0, check=False) == A.E_INVALID_ARG
    assert A.psg_permute(fake, iv, [0, 1], fake, ov, stream=0, check=False) == A.E_INVALID_ARG
    ob = A.make_view("bf16", (5, 3))
    assert A.psg_permute(fake, iv, [1, 0], fake, ob, stream=0, check=False) == A.E_UNSUPPORTED_DTYPE


def test_reduce_rejects_bad_arguments(A):
    fake = 4096
    v = A.make_view("f32", (4, 8))
    bad_out = A.make_view("f32", (3,))
    st = A.psg_reduce_rows([(A.RED_SUM, [A.node("LOAD", 0)])], None, [fake], [v], fake, bad_out,
                           stream=0, check=False)
    assert st == A.E_INVALID_ARG
    # a per-row epilogue may not read inputs
    st = A.psg_reduce_rows([(A.RED_SUM, [A.node("LOAD", 0)])], [A.node("LOAD", 0)], [fake], [v], fake,
                           A.make_view("f32", (4,)), stream=0, check=False)
    assert st == A.E_INVALID_ARG
    # a prologue may not read its own stage
    st = A.psg_reduce_rows([(A.RED_SUM, [A.node("RED", 0)])], None, [fake], [v], fake,
                           A.make_view("f32", (4,)), stream=0, check=False)
    assert st == A.E_INVALID_ARG


def test_scatter_workspace_checks(A):
    fake = 4096
    dv = A.make_view("f32", (4, 2))
    uv = A.make_view("f32", (10, 2))
    need = A.psg_scatter_workspace(10)
    assert need >= 10 * 8
    st = A.psg_scatter_add(fake, dv, fake, 10, fake, uv, fake, need - 8, fake, stream=0, check=False)
    assert st == A.E_WORKSPACE
    # dst and upd of two dtypes, and an unknown dtype, are refused
    st = A.psg_scatter_add(fake, dv, fake, 10, fake, A.make_view("i8", (10, 2)), fake, need, fake,
                           stream=0, check=False)
    assert st == A.E_UNSUPPORTED_DTYPE
    bad, badu = A.make_view("i8", (4, 2)), A.make_view("i8", (10, 2))
    bad.dtype = badu.dtype = 99
    st = A.psg_scatter_add(fake, bad, fake, 10, fake, badu, fake, need, fake, stream=0, check=False)
    assert st == A.E_UNSUPPORTED_DTYPE


def test_columnar_reductions_compile_without_a_gpu(A):
    """Reductions over a leading axis (rows adjacent in memory, the reduced
    axis strided) plan the columnar layout and compile: a weighted column
    sum reading a per-k vector, and a two-stage softmax over a strided axis
    with a per-element epilogue."""
    L = A.lib
    f = L.psg_internal_compile_reduce
    f.argtypes = [ctypes.POINTER(A.psg_reduce_stage), ctypes.c_int, ctypes.POINTER(A.psg_node), ctypes.c_int,
                  ctypes.POINTER(A.psg_view), ctypes.c_int, ctypes.POINTER(A.psg_view), ctypes.c_char_p,
                  ctypes.c_size_t]
    buf = ctypes.create_string_buffer(1 << 16)
    n = A.node

    def run(stages, epi, ins, out):
        keep = []
        sarr = (A.psg_reduce_stage * len(stages))()
        for i, (op, prog) in enumerate(stages):
            arr = (A.psg_node * len(prog))(*prog)
            keep.append(arr)
            sarr[i].op, sarr[i].n_nodes = op, len(prog)
            sarr[i].prologue = ctypes.cast(arr, ctypes.POINTER(A.psg_node))
        earr = (A.psg_node * max(1, len(epi)))(*epi)
        views = (A.psg_view * len(ins))(*ins)
        return f(sarr, len(stages), earr if epi else None, len(epi), views, len(ins), ctypes.byref(out), buf,
                 len(buf))

    # dg[c] = sum_r dy[r, c] * x[r, c] * rstd[r]: rows are c (stride 1), k is r (stride 512)
    R, C = 8192, 512
    dy = A.make_view("bf16", (C, R), (1, C), 0, None, R * C)
    x = A.make_view("bf16", (C, R), (1, C), 0, None, R * C)
    rstd = A.make_view("f32", (C, R), (0, 1), 0, None, R)
    prog = [n("LOAD", 0, dtype="bf16"), n("LOAD", 1, dtype="bf16"), n("CAST", 0), n("CAST", 1),
            n("MUL", 2, 3), n("LOAD", 2), n("MUL", 4, 5)]
    st = run([(A.RED_SUM, prog)], [], [dy, x, rstd], A.make_view("f32", (C,)))
    assert st == 0, (A.STATUS.get(st), buf.value.decode()[:3000])
    # softmax over the leading axis of [64, 300]: MAX, then SUM of EXP(x - m), then EXP(x - m) / s
    v = A.make_view("f32", (300, 64), (1, 300), 0, None, 64 * 300)
    s1 = [n("LOAD", 0)]
    s2 = [n("LOAD", 0), n("RED", 0), n("NEG", 1), n("ADD", 0, 2), n("EXP", 3)]
    epi = s2 + [n("RED", 1), n("RECIP", 5), n("MUL", 4, 6)]
    st = run([(A.RED_MAX, s1), (A.RED_SUM, s2)], epi, [v], A.make_view("f32", (300, 64), (1, 300), 0, None,
                                                                         64 * 300))
    assert st == 0, (A.STATUS.get(st), buf.value.decode()[:3000])
    # staged rows (contiguous, 16-byte aligned, >= 512 bytes a row): the
    # shared-memory ring with its bounded waits and final drain compiles
    v = A.make_view("f32", (300, 1024))
    st = run([(A.RED_MAX, s1), (A.RED_SUM, s2)], epi, [v], A.make_view("f32", (300, 1024)))
    assert st == 0, (A.STATUS.get(st), buf.value.decode()[:3000])


def test_contraction_epilogue_kernels_compile_without_a_gpu(A):
    """A contraction with a fused epilogue program (ACC cast to bf16 plus a
    bf16 residual, then a ReLU) plans and compiles both tensor-core kernels
    (single CTA and CTA pair) through NVRTC; a program that reads a missing
    input is refused before any compile."""
    L = A.lib
    f = L.psg_internal_compile_contract_epilogue
    V = ctypes.POINTER(A.psg_view)
    f.argtypes = [V, V, V, ctypes.POINTER(A.psg_epilogue), ctypes.c_char_p, ctypes.c_size_t]
    M, N, K = 1024, 512, 512
    Av = A.make_view("bf16", (M, N, K), (K, 0, 1), 0, None, M * K)
    Bv = A.make_view("bf16", (M, N, K), (0, 1, N), 0, None, K * N)
    Cv = A.make_view("bf16", (M, N))
    n = A.node
    prog = [n("ACC"), n("CAST", 0, dtype="bf16"), n("LOAD", 0, dtype="bf16"), n("ADD", 1, 2, dtype="bf16"),
            n("CONST", dtype="bf16"), n("CMPLT", 4, 3, dtype="bf16"), n("WHERE", 5, 3, 4, dtype="bf16")]
    arr = (A.psg_node * len(prog))(*prog)
    views = (A.psg_view * 1)(A.make_view("bf16", (M, N)))
    e = A.psg_epilogue(ctypes.cast(arr, ctypes.POINTER(A.psg_node)), len(prog), 1, None,
                       ctypes.cast(views, V))
    buf = ctypes.create_string_buffer(1 << 16)
    st = f(ctypes.byref(Av), ctypes.byref(Bv), ctypes.byref(Cv), ctypes.byref(e), buf, len(buf))
    assert st == 0, (A.STATUS.get(st), buf.value.decode()[:3000])
    bad = (A.psg_node * 1)(n("LOAD", 1, dtype="bf16"))
    e2 = A.psg_epilogue(ctypes.cast(bad, ctypes.POINTER(A.psg_node)), 1, 1, None, ctypes.cast(views, V))
    assert f(ctypes.byref(Av), ctypes.byref(Bv), ctypes.byref(Cv), ctypes.byref(e2), buf, len(buf)) == \
        A.E_INVALID_ARG


def test_float64_programs_compile_and_rows_refuse_them(A):
    """float64 nodes (limn, "The op set": float64 computes natively) compile
    in psg_elementwise with every op and every CAST to and from float64; the
    row reductions, which keep 32-bit totals, refuse a float64 node."""
    f = _compile_hook(A)
    buf = ctypes.create_string_buffer(1 << 16)
    n = A.node
    prog = [n("LOAD", 0, dtype="f64"), n("LOAD", 1, dtype="f32"), n("CAST", 1, dtype="f64"),
            n("ADD", 0, 2, dtype="f64"), n("MUL", 3, 0, dtype="f64"), n("NEG", 4, dtype="f64"),
            n("EXP", 5, dtype="f64"), n("LOG", 6, dtype="f64"), n("SQRT", 0, dtype="f64"),
            n("RECIP", 8, dtype="f64"), n("CMPLT", 7, 9, dtype="f64"), n("CONST", dtype="f64", cval=0.1),
            n("WHERE", 10, 9, 11, dtype="f64"), n("CAST", 12, dtype="bf16"), n("CAST", 13, dtype="f64"),
            n("CAST", 14, dtype="i32"), n("CAST", 15, dtype="f64")]
    views = (A.psg_view * 2)(A.make_view("f64", (37, 301)), A.make_view("f32", (37, 301)))
    arr = (A.psg_node * len(prog))(*prog)
    st = f(arr, len(prog), views, 2, ctypes.byref(A.make_view("f64", (37, 301))), buf, len(buf))
    assert st == 0, (A.STATUS.get(st), buf.value.decode()[:3000])
    rv = A.make_view("f64", (8, 100))
    st = A.psg_reduce_rows([(A.RED_SUM, [n("LOAD", 0, dtype="f64")])], None, [4096], [rv], 4096,
                           A.make_view("f64", (8,)), stream=0, check=False)
    assert st == A.E_UNSUPPORTED_DTYPE
