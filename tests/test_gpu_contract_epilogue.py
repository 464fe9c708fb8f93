"""GPU parity of psg_contract with a fused epilogue program (a residual add,
a ReLU, a bias, a relu-mask gradient, casts) against the oracle: the naive
float32 MUL+SUM loop, then the program node by node (oracle/program.py,
contract_epilogue).  Bar: the hull rule of tests/replay.py: the oracle runs
the program again with each total moved by the reduction-order bound
(1 + 2^-8) * 2 gamma_{K-1} sum_k |a_k b_k| either way (and each EXP / LOG by
its 8 ulps), and every GPU cell lies in the hull of those runs widened by
one unit of C's dtype.  Both tensor-core kernels (single CTA and CTA pair)
run every case, over ragged M, N and K tails (row pitches stay multiples of
16 bytes, which the tensor-core path needs; other layouts refuse an
epilogue, see test_epilogue_refusals).
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
from helpers import dev, storage_dtype, to_np
from replay import Record, check_contract

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from primitive_sm_graph_gb300 import _abi
    return _abi


@pytest.fixture(scope="module")
def P():
    import oracle.program as P
    return P


def N(A, op, a=0, b=0, c=0, dt="f32", cval=0.0):
    return A.node(op, a, b, c, dtype=dt, cval=cval)


def _tuple(A, n):
    names = {k: v for v, k in A.OPS.items()}
    return (names[n.op], n.a, n.b, n.c, A.DTYPE_NAMES[n.dtype], n.cval)


def _run(A, O, P, M, N_, K, prog, epi_inputs, out_dt, batch=None, kernel=None, monkeypatch=None, seed=0,
         alias_out=None):
    """C = prog(ACC = A @ B, LOAD k = epi_inputs[k]) on the GPU and against
    the oracle; epi_inputs: torch tensors of C's shape (host)."""
    g = SI.gen(seed + M + 3 * N_ + 7 * K)
    sh_a = (batch, M, K) if batch else (M, K)
    sh_b = (batch, K, N_) if batch else (K, N_)
    a = SI.normal(sh_a, 0, 1, g, torch.bfloat16)
    b = SI.normal(sh_b, 0, 1, g, torch.bfloat16)
    da, db = dev(a), dev(b)
    if batch:
        shape, sa, sb = [batch, M, N_, K], [M * K, K, 0, 1], [K * N_, 0, 1, N_]
    else:
        shape, sa, sb = [M, N_, K], [K, 0, 1], [0, 1, N_]
    Av = A.view_of(da, shape=shape, strides=sa)
    Bv = A.view_of(db, shape=shape, strides=sb)
    dins = [dev(x) for x in epi_inputs]
    C = dins[alias_out] if alias_out is not None else torch.empty(shape[:-1], dtype=storage_dtype(out_dt),
                                                                 device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    if kernel and monkeypatch is not None:
        monkeypatch.setenv("PSG_GEMM_KERNEL", kernel)
    A.psg_contract(da, Av, db, Bv, C, A.view_of(C), st, epilogue=(prog, dins, [A.view_of(x) for x in dins]))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Z = batch or 1
    a3 = O.T(SI.bits(a).reshape(Z, M, K), "bf16")
    b3 = O.T(np.ascontiguousarray(SI.bits(b).reshape(Z, K, N_).transpose(0, 2, 1)), "bf16")
    names = {torch.bfloat16: "bf16", torch.float32: "f32", torch.float16: "f16"}
    loads = [O.T(SI.bits(x).reshape(Z, M, N_), names[x.dtype]) for x in epi_inputs]
    got = O.T(to_np(C.cpu()).reshape(Z, M, N_), out_dt)
    rec = Record(0, "contract", "epilogue")
    check_contract(O, P, rec, a3, b3, K, got, out_dt, ([_tuple(A, n) for n in prog], loads))
    assert rec.bad == 0 and rec.unbounded == 0, rec
    return C


KERNELS = ["single", "pair"]


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("M,N_,K", [(300, 520, 256), (256, 256, 64), (1000, 712, 1024)])
def test_residual_add(A, O, P, monkeypatch, kernel, M, N_, K):
    """h = residual + bf16(A @ B): the GPT block's residual stream."""
    g = SI.gen(M * N_)
    r = SI.normal((M, N_), 0, 4, g, torch.bfloat16)
    prog = [N(A, "ACC"), N(A, "CAST", 0, dt="bf16"), N(A, "LOAD", 0, dt="bf16"), N(A, "ADD", 2, 1, dt="bf16")]
    _run(A, O, P, M, N_, K, prog, [r], "bf16", kernel=kernel, monkeypatch=monkeypatch)


@pytest.mark.parametrize("kernel", KERNELS)
def test_relu(A, O, P, monkeypatch, kernel):
    """relu(bf16(A @ B)) = WHERE(CMPLT(0, u), u, 0) with no input at all."""
    prog = [N(A, "ACC"), N(A, "CAST", 0, dt="bf16"), N(A, "CONST", dt="bf16"), N(A, "CMPLT", 2, 1, dt="bf16"),
            N(A, "WHERE", 3, 1, 2, dt="bf16")]
    _run(A, O, P, 384, 2048, 512, prog, [], "bf16", kernel=kernel, monkeypatch=monkeypatch)


@pytest.mark.parametrize("kernel", KERNELS)
def test_relu_mask_gradient(A, O, P, monkeypatch, kernel):
    """gu = WHERE(CMPLT(0, u), bf16(gf), 0): the MLP's backward through its
    ReLU, reading the pre-activation u (bf16) as an input."""
    g = SI.gen(5)
    u = SI.normal((512, 640), 0, 1, g, torch.bfloat16)
    prog = [N(A, "CONST", dt="bf16"), N(A, "LOAD", 0, dt="bf16"), N(A, "CMPLT", 0, 1, dt="bf16"), N(A, "ACC"),
            N(A, "CAST", 3, dt="bf16"), N(A, "WHERE", 2, 4, 0, dt="bf16")]
    _run(A, O, P, 512, 640, 320, prog, [u], "bf16", kernel=kernel, monkeypatch=monkeypatch)


def test_bias_rows_and_columns_float32_output(A, O, P):
    """C = (ACC + bias_n) * scale_m, float32 out: a bias along n (a [N] vector
    read through a stride-0 View, one load per cell) and a per-row scale
    along m (a stride-0 View along n: one value per row)."""
    M, N_, K = 200, 296, 192
    g = SI.gen(9)
    bias = SI.normal((N_,), 0, 1, g)
    scale = SI.normal((M,), 1, 0.5, g)
    db, ds = dev(bias), dev(scale)
    da_ = SI.normal((M, K), 0, 1, g, torch.bfloat16)
    dbm = SI.normal((K, N_), 0, 1, g, torch.bfloat16)
    dA, dB = dev(da_), dev(dbm)
    Av = A.view_of(dA, shape=[M, N_, K], strides=[K, 0, 1])
    Bv = A.view_of(dB, shape=[M, N_, K], strides=[0, 1, N_])
    C = torch.empty((M, N_), device="cuda")
    vb = A.view_of(db, shape=(M, N_), strides=(0, 1))
    vs = A.view_of(ds, shape=(M, N_), strides=(1, 0))
    prog = [N(A, "ACC"), N(A, "LOAD", 0), N(A, "ADD", 0, 1), N(A, "LOAD", 1), N(A, "MUL", 2, 3)]
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), None, epilogue=(prog, [db, ds], [vb, vs]))
    torch.cuda.synchronize()
    a3 = O.T(SI.bits(da_).reshape(1, M, K), "bf16")
    b3 = O.T(np.ascontiguousarray(SI.bits(dbm).T).reshape(1, N_, K), "bf16")
    loads = [O.T(np.broadcast_to(bias.numpy(), (M, N_)).reshape(1, M, N_).copy(), "f32"),
             O.T(np.broadcast_to(scale.numpy()[:, None], (M, N_)).reshape(1, M, N_).copy(), "f32")]
    rec = Record(0, "contract", "bias")
    check_contract(O, P, rec, a3, b3, K, O.T(C.cpu().numpy().reshape(1, M, N_), "f32"), "f32",
                   ([_tuple(A, n) for n in prog], loads))
    assert rec.bad == 0, rec


def test_batched_with_exp_and_in_place_residual(A, O, P, monkeypatch):
    """A batch of three products, an EXP node in the program (held to its 8
    ulps), and C written in place over its residual input (an identical
    View: each cell is read before it is written)."""
    g = SI.gen(11)
    r = SI.normal((3, 256, 320), 0, 1, g, torch.bfloat16)
    prog = [N(A, "ACC"), N(A, "CONST", cval=0.25), N(A, "MUL", 0, 1), N(A, "EXP", 2), N(A, "CAST", 3, dt="bf16"),
            N(A, "LOAD", 0, dt="bf16"), N(A, "ADD", 4, 5, dt="bf16")]
    _run(A, O, P, 256, 320, 128, prog, [r], "bf16", batch=3, alias_out=0)


def test_epilogue_refusals(A):
    """An epilogue runs only in the bf16 / f16 tensor-core kernel: float32
    operands, a masked epilogue input, an input of another shape and a
    result dtype other than C's are refused before anything launches."""
    M, N_, K = 64, 64, 256
    x = torch.zeros((M, K), device="cuda")
    y = torch.zeros((K, N_), device="cuda")
    C = torch.empty((M, N_), device="cuda")
    Av = A.view_of(x, shape=[M, N_, K], strides=[K, 0, 1])
    Bv = A.view_of(y, shape=[M, N_, K], strides=[0, 1, N_])
    acc = [N(A, "ACC")]
    st = A.psg_contract(x, Av, y, Bv, C, A.view_of(C), None, check=False, epilogue=(acc, [], []))
    assert st == A.E_UNSUPPORTED_LAYOUT
    xb, yb = x.bfloat16(), y.bfloat16()
    Avb = A.view_of(xb, shape=[M, N_, K], strides=[K, 0, 1])
    Bvb = A.view_of(yb, shape=[M, N_, K], strides=[0, 1, N_])
    r = torch.zeros((M, N_), device="cuda")
    masked = A.view_of(r, shape=(M, N_), strides=(N_, 1), mask=[(0, M - 1), (0, N_)])
    prog = [N(A, "ACC"), N(A, "LOAD", 0), N(A, "ADD", 0, 1)]
    st = A.psg_contract(xb, Avb, yb, Bvb, C, A.view_of(C), None, check=False, epilogue=(prog, [r], [masked]))
    assert st == A.E_UNSUPPORTED_LAYOUT
    small = torch.zeros((M, N_ - 1), device="cuda")
    st = A.psg_contract(xb, Avb, yb, Bvb, C, A.view_of(C), None, check=False,
                        epilogue=(prog, [small], [A.view_of(small)]))
    assert st == A.E_INVALID_ARG
    st = A.psg_contract(xb, Avb, yb, Bvb, C, A.view_of(C), None, check=False,
                        epilogue=([N(A, "ACC"), N(A, "CAST", 0, dt="bf16")], [], []))
    assert st == A.E_UNSUPPORTED_DTYPE
    # LOAD of an input that is not there, and RED, are invalid
    st = A.psg_contract(xb, Avb, yb, Bvb, C, A.view_of(C), None, check=False,
                        epilogue=([N(A, "LOAD", 0)], [], []))
    assert st == A.E_INVALID_ARG
