"""GPU parity of psg_contract beyond the float tensor-core path: masked
(padded) operand Views, float64 and the integer dtypes, all against the
oracle's broadcast product (MUL of the two materialised Views, then SUM over
k; limn, "Three rules hold it together": a matmul is a broadcast multiply and
a reduce, a masked cell reads zero, integers wrap modulo 2^width).

Bars: integers bit-exact; float32 totals within the reduction-order term
2*gamma_{K-1} * sum_k |a_k b_k| (Litmus, "ToleranceBound"); float64 the same
term with the float64 unit roundoff.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
from helpers import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from primitive_sm_graph_gb300 import _abi
    return _abi


_TORCH = {"f32": torch.float32, "f64": torch.float64, "i32": torch.int32, "i16": torch.int16, "i8": torch.int8,
          "bf16": torch.bfloat16}


def _rand(dt, shape, g):
    """Seeded values of a dtype (integers span the whole range, so products
    and totals wrap)."""
    if dt in ("i32", "i16", "i8"):
        info = torch.iinfo(_TORCH[dt])
        return torch.randint(info.min, info.max + 1, shape, generator=g, dtype=torch.int64).to(_TORCH[dt]).numpy()
    return SI.normal(shape, 0.0, 1.0, g, torch.float64 if dt == "f64" else torch.float32).numpy()


def _operands(dt, M, N, K, seed):
    """Seeded A [M, K] and B [K, N]."""
    g = SI.gen(seed)
    return _rand(dt, (M, K), g), _rand(dt, (K, N), g)


def _broadcast(M, N, K):
    """[M, N, K] strides of A [M, K] (broadcast over n) and B [K, N] (over m)."""
    return [K, 0, 1], [0, 1, N]


def _run(A, a, b, dt, out_dt, shape, sa, sb, ma=None, mb=None, batch_c=None):
    dA = dev(torch.from_numpy(np.ascontiguousarray(a)))
    dB = dev(torch.from_numpy(np.ascontiguousarray(b)))
    Av = A.make_view(dt, shape, sa, 0, ma, a.size)
    Bv = A.make_view(dt, shape, sb, 0, mb, b.size)
    C = torch.full(tuple(shape[:-1]), 77, dtype=_TORCH[out_dt], device="cuda")
    Cv = A.view_of(C)
    A.psg_contract(dA, Av, dB, Bv, C, Cv, None, stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return C.cpu().numpy()


def _oracle(O, a, b, dt, shape, sa, sb, ma=None, mb=None, out_dt=None):
    """MUL of the two masked broadcast Views, SUM over the last dim."""
    pa = O.view(O.T(np.ascontiguousarray(a), dt), shape, sa, 0, ma)
    pb = O.view(O.T(np.ascontiguousarray(b), dt), shape, sb, 0, mb)
    s = O.reduce_sum(O.mul(pa, pb), keepdim=False)
    return s, (np.abs(pa.data.astype(np.float64)) * np.abs(pb.data.astype(np.float64))).sum(-1)


def _close(got, ref, mag, K, u=2.0 ** -24):
    n = max(K - 1, 0)
    tol = 2 * (n * u / (1 - n * u)) * mag + 1e-300
    bad = np.abs(got.astype(np.float64) - ref.astype(np.float64)) > tol
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:3], got[bad][:3], ref[bad][:3])


@pytest.mark.parametrize("dt", ["f32", "i32", "i16", "i8", "f64"])
@pytest.mark.parametrize("M,N,K,ma,mb", [
    # A masked along m and k, B along n and k: zero factors as the tiles load
    (70, 130, 45, [(3, 60), (0, 130), (0, 40)], [(0, 70), (5, 120), (2, 45)]),
    # masks across the other operand's broadcast axis: whole cells are 0
    (129, 140, 33, [(0, 129), (0, 100), (0, 33)], [(10, 129), (0, 140), (0, 33)]),
    # windows past the shape are clipped; an empty k window reads nothing
    (40, 20, 17, [(-5, 500), (0, 20), (0, 17)], [(0, 40), (0, 20), (9, 9)]),
])
def test_masked_contraction_matches_broadcast_product(A, O, dt, M, N, K, ma, mb):
    a, b = _operands(dt, M, N, K, 7 + M)
    sa, sb = _broadcast(M, N, K)
    shape = [M, N, K]
    got = _run(A, a, b, dt, dt, shape, sa, sb, ma, mb)
    ref, mag = _oracle(O, a, b, dt, shape, sa, sb, ma, mb)
    if dt in ("i32", "i16", "i8"):
        np.testing.assert_array_equal(got, ref.data.reshape(M, N))
    else:
        _close(got, ref.data.reshape(M, N), mag, K, 2.0 ** -53 if dt == "f64" else 2.0 ** -24)


def test_masked_bf16_operands_take_the_fp32_pipes(A, O):
    """bf16 operands with a padded k: exact products summed in float32, as
    the float32 broadcast product of the same (widened) values."""
    M, N, K = 96, 200, 70
    a, b = _operands("f32", M, N, K, 3)
    ab = torch.from_numpy(a).to(torch.bfloat16)
    bb = torch.from_numpy(b).to(torch.bfloat16)
    sa, sb = _broadcast(M, N, K)
    shape, ma, mb = [M, N, K], [(0, M), (0, N), (0, 64)], [(0, M), (0, N), (0, K)]
    Av = A.make_view("bf16", shape, sa, 0, ma, ab.numel())
    Bv = A.make_view("bf16", shape, sb, 0, mb, bb.numel())
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    A.psg_contract(dev(ab), Av, dev(bb), Bv, C, A.view_of(C), None, stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    ref, mag = _oracle(O, ab.float().numpy(), bb.float().numpy(), "f32", shape, sa, sb, ma, mb)
    _close(C.cpu().numpy(), ref.data.reshape(M, N), mag, K)


@pytest.mark.parametrize("dt,out_dt", [("i32", "i32"), ("i16", "i32"), ("i8", "i32"), ("i32", "i8"), ("i8", "i16")])
@pytest.mark.parametrize("M,N,K", [(130, 257, 70), (1, 1, 1), (5, 3, 0)])
def test_integer_contraction_wraps(A, O, dt, out_dt, M, N, K):
    """Integer MUL+SUM: products and totals wrap modulo 2^32, the store wraps
    to the output's width; bit-exact against the oracle's integer loop."""
    a, b = _operands(dt, M, N, K, 11 + K)
    sa, sb = _broadcast(M, N, K)
    got = _run(A, a, b, dt, out_dt, [M, N, K], sa, sb)
    ref = O.matmul(O.T(a, dt), O.T(b, dt), out_dt).data
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("M,N,K", [(65, 70, 300), (128, 129, 16)])
def test_f64_contraction(A, O, M, N, K):
    a, b = _operands("f64", M, N, K, 5)
    sa, sb = _broadcast(M, N, K)
    got = _run(A, a, b, "f64", "f64", [M, N, K], sa, sb)
    ref = O.matmul(O.T(a, "f64"), O.T(b, "f64")).data
    _close(got, ref, np.abs(a) @ np.abs(b), K, 2.0 ** -53)


@pytest.mark.parametrize("dt", ["f32", "i32"])
def test_masked_batch_dims(A, O, dt):
    """A batch dim masked on A (index 0 reads nothing) and one masked on B,
    over two batch dims that do not merge: one launch per batch index."""
    b1, b2, M, N, K = 3, 2, 33, 40, 19
    g = SI.gen(21)
    a = _rand(dt, (b1, b2, M, K), g)
    b = _rand(dt, (b1, b2, K, N), g)
    shape = [b1, b2, M, N, K]
    # A batch-major with b2 outermost in memory (the dims do not merge)
    a_store = np.ascontiguousarray(a.transpose(1, 0, 2, 3))
    sa = [M * K, b1 * M * K, K, 0, 1]
    sb = [b2 * K * N, K * N, 0, 1, N]
    ma = [(1, b1), (0, b2), (0, M), (0, N), (0, K)]
    mb = [(0, b1), (0, 1), (0, M), (0, N), (0, K)]
    got = _run(A, a_store, b, dt, dt, shape, sa, sb, ma, mb)
    ref, mag = _oracle(O, a_store, b, dt, shape, sa, sb, ma, mb)
    if dt == "i32":
        np.testing.assert_array_equal(got, ref.data.reshape(b1, b2, M, N))
    else:
        _close(got, ref.data.reshape(b1, b2, M, N), mag, K)
    assert not got[0].any() and not got[:, 1].any()


def test_unsupported_dtype_pairings_are_refused(A):
    M, N, K = 4, 4, 4
    sa, sb = _broadcast(M, N, K)
    x = torch.zeros(64, dtype=torch.int32, device="cuda")
    for ab, c in [("i32", "f32"), ("f32", "i32"), ("f64", "f32"), ("f32", "f64")]:
        Av = A.make_view(ab, [M, N, K], sa, 0, None, 16)
        Bv = A.make_view(ab, [M, N, K], sb, 0, None, 16)
        Cv = A.make_view(c, [M, N], None, 0, None, 16)
        st = A.psg_contract(x, Av, x, Bv, x, Cv, None, stream=torch.cuda.current_stream().cuda_stream,
                            check=False)
        assert st == A.E_UNSUPPORTED_DTYPE, (ab, c, st)


@pytest.mark.parametrize("dt", ["i32", "i8", "f64", "f16"])
def test_graph_matmul_of_every_dtype_is_one_contraction(O, dt):
    """The graph layer recognises MUL+SUM of any operand dtype psg_contract
    takes as one contraction call, with the oracle's result."""
    from primitive_sm_graph_gb300 import graph as G
    M, K, N = 70, 90, 130
    g = SI.gen(4)
    if dt == "f16":
        a = SI.normal((M, K), 0.0, 1.0, g, torch.float16)
        b = SI.normal((K, N), 0.0, 1.0, g, torch.float16)
    else:
        a, b = torch.from_numpy(_rand(dt, (M, K), g)), torch.from_numpy(_rand(dt, (K, N), g))
    ex = G._executor()
    ex.log.clear()
    c = G.Tensor.from_torch(a.cuda()).matmul(G.Tensor.from_torch(b.cuda())).realize().cpu()
    assert [e[0] for e in ex.log].count("contract") == 1, ex.log
    if dt == "f16":
        ref = O.matmul(O.T(a.float().numpy(), "f32"), O.T(b.float().numpy(), "f32")).data
        mag = a.double().abs().numpy() @ b.double().abs().numpy()
        tol = 2 * (89 * 2.0 ** -24) * mag + 2.0 ** -10 * np.abs(ref) + 2.0 ** -24
        assert (np.abs(c.float().numpy() - ref) <= tol).all()
    elif dt == "f64":
        ref = O.matmul(O.T(a.numpy(), dt), O.T(b.numpy(), dt)).data
        _close(c.numpy(), ref, np.abs(a.numpy()) @ np.abs(b.numpy()), K, 2.0 ** -53)
    else:
        np.testing.assert_array_equal(c.numpy(), O.matmul(O.T(a.numpy(), dt), O.T(b.numpy(), dt)).data)


def test_full_size_int8_contraction_sampled_rows(A, O):
    """The bench's int8 [2048, 2048] @ [2048, 2048] -> int32 contraction in
    its own launch configuration: sampled rows bit-exact against the
    oracle's integer loop over those rows."""
    a, b = SI.contraction_i8(0)
    M, K = a.shape
    N = b.shape[1]
    da, db = a.cuda(), b.cuda()
    va = A.view_of(da, shape=(M, N, K), strides=(K, 0, 1))
    vb = A.view_of(db, shape=(M, N, K), strides=(0, 1, N))
    c = torch.empty((M, N), dtype=torch.int32, device="cuda")
    A.psg_contract(da, va, db, vb, c, A.view_of(c), None, stream=torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    rows = np.array([0, 1, 127, 128, 1000, 2047])
    ref = O.matmul(O.T(a.numpy()[rows], "i8"), O.T(b.numpy(), "i8"), "i32").data
    np.testing.assert_array_equal(c.cpu().numpy()[rows], ref)
