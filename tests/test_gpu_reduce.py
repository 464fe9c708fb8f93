"""GPU parity of psg_reduce_rows against the CPU oracle.

Bars (derived from the per-node budgets; Litmus, "ToleranceBound"):
  * MAX, integer SUM and every integer result: bit-exact;
  * float SUM: |gpu - oracle| <= 2*gamma_{N-1} * sum|x| (two association
    orders), plus one rounding of the stage dtype for half widths;
  * softmax: |y - y_ref| <= y_ref * (24u + 2*gamma_{N-1}) + 4*2^-149, from the
    EXP (8 ulp), RECIP and MUL roundings and the SUM bound on the denominator;
  * RMSNorm (bfloat16 out): within 2^-7 relative of the oracle (one bf16 unit).
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
from helpers import U, dev, gamma, storage_dtype, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from primitive_sm_graph_gb300 import _abi
    return _abi


@pytest.fixture(scope="module")
def PR():
    from primitive_sm_graph_gb300 import programs
    return programs


def _softmax_check(O, x_np, y_gpu):
    N = x_np.shape[-1]
    ref = O.softmax_rows(O.T(x_np, "f32")).data.astype(np.float64)
    got = y_gpu.astype(np.float64)
    tol = ref * (24 * U + 2 * gamma(N - 1)) + 4 * 2.0 ** -149
    bad = np.abs(got - ref) > tol
    assert not bad.any(), (np.argwhere(bad)[:3], got[bad][:3], ref[bad][:3])
    # rows sum to 1; the max of each row is exactly 0 after the shift (R1)
    assert np.all(np.abs(got.sum(axis=-1) - 1.0) <= N * 2.0 ** -23 + 2 * gamma(N - 1))


@pytest.mark.parametrize("R,N", [(7, 1024), (33, 100), (1, 1), (5, 3000), (64, 257), (3, 50000)])
def test_softmax_matches_oracle(A, O, PR, R, N):
    g = SI.gen(R * 7 + N)
    x = SI.uniform((R, N), -1000.0, 1000.0, g)
    dx = dev(x)
    y = torch.empty_like(dx)
    stages, epi = PR.softmax_rows()
    A.psg_reduce_rows(stages, epi, [dx], [A.view_of(dx)], y, A.view_of(y))
    torch.cuda.synchronize()
    _softmax_check(O, x.numpy(), y.cpu().numpy())


def test_softmax_full_size_and_aimed_rows(A, O, PR):
    x = SI.softmax_input(0)
    dx = dev(x)
    y = torch.empty_like(dx)
    stages, epi = PR.softmax_rows()
    A.psg_reduce_rows(stages, epi, [dx], [A.view_of(dx)], y, A.view_of(y))
    torch.cuda.synchronize()
    _softmax_check(O, x.numpy(), y.cpu().numpy())
    # all-negative, constant and large-magnitude rows (Litmus's aimed generators)
    g = SI.gen(3)
    for kind in ("negative", "constant", "saturating", "large"):
        x = SI.aimed(kind, (16, 1024), g)
        if kind == "large":
            x = x.clamp(-3e38, 3e38)
        dx = dev(x)
        y = torch.empty_like(dx)
        A.psg_reduce_rows(stages, epi, [dx], [A.view_of(dx)], y, A.view_of(y))
        torch.cuda.synchronize()
        _softmax_check(O, x.numpy(), y.cpu().numpy())


@pytest.mark.parametrize("R,N", [(8192, 4096), (5, 4096), (3, 300), (17, 8)])
def test_rmsnorm_matches_oracle(A, O, PR, R, N):
    x, w = SI.rmsnorm_input(0, R, N)
    dx, dw = dev(x), dev(w)
    y = torch.empty_like(dx)
    stages, epi = PR.rmsnorm(N)
    A.psg_reduce_rows(stages, epi, [dx, dw], [A.view_of(dx), A.view_of(dw, shape=(R, N), strides=(0, 1))],
                      y, A.view_of(y))
    torch.cuda.synchronize()
    got = O.T(to_np(y.cpu()), "bf16").f64()
    ref = O.rmsnorm(O.T(SI.bits(x), "bf16"), O.T(SI.bits(w), "bf16")).f64()
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30)
    # and most cells are bit-identical (only SUM-order ties can move a rounding)
    assert np.mean(got == ref) > 0.99


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16", "i32", "i16", "i8"])
@pytest.mark.parametrize("shape", [(9, 37), (4, 5, 1000), (1, 1), (2, 0), (3, 20000)])
def test_sum_and_max_rows(A, O, dt, shape):
    g = SI.gen(len(shape) * 100 + shape[-1])
    if dt.startswith("i"):
        lim = {"i32": 1 << 20, "i16": 300, "i8": 100}[dt]
        x = torch.randint(-lim, lim, shape, generator=g).to(storage_dtype(dt))
    else:
        x = SI.normal(shape, 0, 3, g).to(storage_dtype(dt))
    dx = dev(x)
    rows_shape = shape[:-1]
    ox = O.T(SI.bits(x), dt)
    for op, red in ((A.RED_SUM, O.reduce_sum), (A.RED_MAX, O.reduce_max)):
        out = torch.empty(rows_shape, dtype=storage_dtype(dt), device="cuda")
        A.psg_reduce_rows([(op, [A.node("LOAD", 0, dtype=dt)])], None, [dx], [A.view_of(dx)], out,
                          A.view_of(out))
        torch.cuda.synchronize()
        got = to_np(out.cpu())
        ref = red(ox, keepdim=False)
        if op == A.RED_MAX or dt.startswith("i"):
            assert np.array_equal(got.view(np.uint8), ref.data.view(np.uint8)), (op, dt, shape)
        else:
            g64 = O.T(got, dt).f64()
            r64 = ref.f64()
            mag = np.abs(ox.f64()).sum(axis=-1)
            n = shape[-1]
            half = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}[dt]
            assert np.all(np.abs(g64 - r64) <= 2 * gamma(n - 1) * mag + 2 * half * np.abs(r64) + 1e-30)


def test_max_specials_bit_exact(A, O):
    x = torch.tensor([[-0.0, 0.0, -0.0], [-0.0, -0.0, -0.0], [1.0, float("nan"), 5.0],
                      [-5.0, -3.0, -7.0], [float("-inf"), float("-inf"), float("-inf")]])
    dx = dev(x)
    out = torch.empty((5,), device="cuda")
    A.psg_reduce_rows([(A.RED_MAX, [A.node("LOAD", 0)])], None, [dx], [A.view_of(dx)], out,
                      A.view_of(out))
    torch.cuda.synchronize()
    ref = O.reduce_max(O.T(x.numpy(), "f32"), keepdim=False).data
    got = out.cpu().numpy()
    assert np.array_equal(np.signbit(got), np.signbit(ref))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.nan_to_num(got), np.nan_to_num(ref))


@pytest.mark.parametrize("N", [1000, 1024, 4096, 5000])
def test_max_specials_long_rows(A, O, N):
    """Signed zeros, NaNs and -inf spread over rows long enough for warp and
    block folds (and the staged ring): MAX must match the oracle's sign bit
    and NaN-ness in every row whatever the fold order."""
    g = SI.gen(N)
    R = 12
    x = torch.where(torch.rand((R, N), generator=g) < 0.5, torch.tensor(-0.0), torch.tensor(0.0))
    x[0] = -0.0                                             # all -0 -> -0
    x[1] = -0.0
    x[1, int(torch.randint(0, N, (1,), generator=g))] = 0.0  # a single +0 wins
    x[2] = float("-inf")                                     # all -inf
    x[3, int(torch.randint(0, N, (1,), generator=g))] = float("nan")
    x[4] = -0.0
    x[4, -1] = float("nan")                                  # NaN in the last cell
    x[5] = -torch.rand((N,), generator=g) - 1.0              # all negative
    x[6] = -torch.rand((N,), generator=g) - 1.0
    x[6, 0] = float("nan")                                   # NaN in the first cell
    x[7] = float("-inf")
    x[7, N // 2] = -0.0
    dx = dev(x)
    out = torch.empty((R,), device="cuda")
    A.psg_reduce_rows([(A.RED_MAX, [A.node("LOAD", 0)])], None, [dx], [A.view_of(dx)], out, A.view_of(out))
    torch.cuda.synchronize()
    ref = O.reduce_max(O.T(x.numpy(), "f32"), keepdim=False).data
    got = out.cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(ref[~np.isnan(ref)]))
    assert np.array_equal(np.nan_to_num(got), np.nan_to_num(ref))


def test_strided_and_broadcast_inputs(A, O):
    g = SI.gen(9)
    base = SI.normal((300 * 40,), 0, 1, g)
    d = dev(base)
    # reduce over the columns of a [40, 300] row-major buffer viewed transposed
    v = A.view_of(d, shape=(300, 40), strides=(1, 300))
    out = torch.empty((300,), device="cuda")
    A.psg_reduce_rows([(A.RED_MAX, [A.node("LOAD", 0)])], None, [d], [v], out, A.view_of(out))
    torch.cuda.synchronize()
    ref = O.reduce_max(O.view(O.T(base.numpy(), "f32"), (300, 40), (1, 300)), keepdim=False).data
    assert np.array_equal(out.cpu().numpy(), ref)
    # a row of a broadcast value: SUM of N copies folds like any row
    c = dev(torch.tensor([0.1]))
    out1 = torch.empty((3, 1), device="cuda")
    A.psg_reduce_rows([(A.RED_SUM, [A.node("LOAD", 0)])], None, [c],
                      [A.view_of(c, shape=(3, 1000), strides=(0, 0))], out1, A.view_of(out1))
    torch.cuda.synchronize()
    ref = O.reduce_sum(O.full((3, 1000), 0.1, "f32")).data
    mag = 1000 * 0.1
    assert np.all(np.abs(out1.cpu().numpy() - ref) <= 2 * gamma(999) * mag)


def test_per_row_epilogue_and_tiny_graph_tail(A, O, PR):
    A_, B_ = SI.tiny_graph(0)
    C = O.matmul_literal(O.T(A_.numpy(), "f32"), O.T(B_.numpy(), "f32")).data.reshape(64, 48)
    dc = dev(torch.from_numpy(C.copy()))
    out = torch.empty((), device="cuda")
    stages, _ = PR.relu_square_sum()
    A.psg_reduce_rows(stages, None, [dc], [A.view_of(dc, shape=(1, 3072), strides=(3072, 1))], out,
                      A.make_view("f32", (1,), extent=1))
    torch.cuda.synchronize()
    r = O.relu(O.T(C, "f32"))
    sq = O.mul(r, r)
    ref = float(O.reduce_sum(sq.reshape((1, 3072)), keepdim=False).data[0])
    assert abs(float(out.cpu()) - ref) <= 2 * gamma(3071) * ref
    # mean over rows via a per-row epilogue: RED * (1/N)
    x = SI.normal((10, 96), 0, 1, SI.gen(4))
    dx = dev(x)
    m = torch.empty((10, 1), device="cuda")
    epi = [A.node("RED", 0), A.node("CONST", cval=1.0 / 96), A.node("MUL", 0, 1)]
    A.psg_reduce_rows([(A.RED_SUM, [A.node("LOAD", 0)])], epi, [dx], [A.view_of(dx)], m, A.view_of(m))
    torch.cuda.synchronize()
    s = O.reduce_sum(O.T(x.numpy(), "f32"))
    mref = O.mul(s, O.full(s.shape, 1.0 / 96, "f32")).data
    mag = np.abs(x.numpy().astype(np.float64)).sum(axis=1, keepdims=True) / 96
    assert np.all(np.abs(m.cpu().numpy() - mref) <= 2 * gamma(95) * mag + np.spacing(np.abs(mref)))




# ---- reductions over a leading axis (the columnar layout) -------------------

@pytest.mark.parametrize("rows,k,dt", [(512, 8192, "f32"), (512, 4096, "bf16"), (100, 37, "f32"),
                                       (33, 1000, "bf16"), (1000, 3, "f32"),
                                       (40, 777, "bf16"), (8, 20000, "f32"), (2056, 300, "bf16")])
def test_column_sum_weighted(A, O, rows, k, dt):
    """out[c] = sum_r dy[r, c] * x[r, c] * w[r] over a row-major [k, rows]
    pair (an RMSNorm weight's gradient): within the SUM bound of the
    oracle's float32 total of the same products."""
    g = SI.gen(rows + k)
    dy = SI.normal((k, rows), 0, 1, g).to(storage_dtype(dt))
    x = SI.normal((k, rows), 0, 1, g).to(storage_dtype(dt))
    w = SI.uniform((k,), 0.5, 2.0, g)
    ddy, dx, dw = dev(dy), dev(x), dev(w)
    vdy = A.make_view(dt, (rows, k), (1, rows), 0, None, rows * k)
    vx = A.make_view(dt, (rows, k), (1, rows), 0, None, rows * k)
    vw = A.make_view("f32", (rows, k), (0, 1), 0, None, k)
    n = A.node
    prog = [n("LOAD", 0, dtype=dt), n("LOAD", 1, dtype=dt), n("CAST", 0), n("CAST", 1), n("MUL", 2, 3),
            n("LOAD", 2), n("MUL", 4, 5)]
    out = torch.empty((rows,), device="cuda")
    A.psg_reduce_rows([(A.RED_SUM, prog)], None, [ddy, dx, dw], [vdy, vx, vw], out, A.view_of(out))
    torch.cuda.synchronize()
    ody = O.cast(O.view(O.T(SI.bits(dy), dt), (rows, k), (1, rows)), "f32")
    ox = O.cast(O.view(O.T(SI.bits(x), dt), (rows, k), (1, rows)), "f32")
    ow = O.view(O.T(w.numpy(), "f32"), (rows, k), (0, 1))
    prod = O.mul(O.mul(ody, ox), ow)
    ref = O.reduce_sum(prod, keepdim=False).data.astype(np.float64)
    mag = np.abs(prod.f64()).sum(axis=-1)
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= 2 * gamma(k - 1) * mag + 1e-30)
    # the same bits on a second call
    out2 = torch.empty_like(out)
    A.psg_reduce_rows([(A.RED_SUM, prog)], None, [ddy, dx, dw], [vdy, vx, vw], out2, A.view_of(out2))
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), out2.view(torch.int32))


@pytest.mark.parametrize("rows,k", [(300, 64), (64, 5000), (40, 1)])
def test_column_softmax(A, O, PR, rows, k):
    """Softmax over the leading axis of a row-major [k, rows] tensor, written
    back in the same layout (two stages and a per-element epilogue)."""
    g = SI.gen(rows * 3 + k)
    x = SI.uniform((k, rows), -50.0, 50.0, g)
    dx = dev(x)
    y = torch.empty_like(dx)
    v = A.make_view("f32", (rows, k), (1, rows), 0, None, rows * k)
    stages, epi = PR.softmax_rows()
    A.psg_reduce_rows(stages, epi, [dx], [v], y, A.make_view("f32", (rows, k), (1, rows), 0, None, rows * k))
    torch.cuda.synchronize()
    _softmax_check(O, x.numpy().T.copy(), y.cpu().numpy().T.copy())


@pytest.mark.parametrize("k", [40, 3000, 9000])
def test_column_max_specials(A, O, k):
    """MAX over a strided axis with signed zeros, NaNs and -inf, across
    warps and cluster ranks: bit-exact."""
    g = SI.gen(k + 1)
    rows = 96
    x = torch.where(torch.rand((k, rows), generator=g) < 0.5, torch.tensor(-0.0), torch.tensor(0.0))
    x[:, 0] = -0.0
    x[k // 2, 1] = 0.0
    x[:, 2] = float("-inf")
    x[k - 1, 3] = float("nan")
    x[:, 4] = -torch.rand((k,), generator=g) - 1.0
    x[0, 5] = float("nan")
    dx = dev(x)
    out = torch.empty((rows,), device="cuda")
    v = A.make_view("f32", (rows, k), (1, rows), 0, None, rows * k)
    A.psg_reduce_rows([(A.RED_MAX, [A.node("LOAD", 0)])], None, [dx], [v], out, A.view_of(out))
    torch.cuda.synchronize()
    ref = O.reduce_max(O.view(O.T(x.numpy(), "f32"), (rows, k), (1, rows)), keepdim=False).data
    got = out.cpu().numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(ref[~np.isnan(ref)]))
    assert np.array_equal(np.nan_to_num(got), np.nan_to_num(ref))


def test_column_sum_over_batch_of_3d(A, O):
    """A sum over the batch axis of [B, T, D] (a position embedding's
    gradient): rows are the (T, D) cells, two row dims."""
    B, T, D = 8, 40, 96
    g = SI.gen(77)
    x = SI.normal((B, T, D), 0, 1, g).to(torch.bfloat16)
    dx = dev(x)
    v = A.make_view("bf16", (T, D, B), (D, 1, T * D), 0, None, B * T * D)
    out = torch.empty((T, D), device="cuda")
    A.psg_reduce_rows([(A.RED_SUM, [A.node("LOAD", 0, dtype="bf16"), A.node("CAST", 0)])], None, [dx], [v],
                      out, A.view_of(out))
    torch.cuda.synchronize()
    ox = O.cast(O.view(O.T(SI.bits(x), "bf16"), (T, D, B), (D, 1, T * D)), "f32")
    ref = O.reduce_sum(ox, keepdim=False).data.astype(np.float64)
    mag = np.abs(ox.f64()).sum(axis=-1)
    assert np.all(np.abs(out.cpu().numpy().astype(np.float64) - ref) <= 2 * gamma(B - 1) * mag + 1e-30)


def test_staged_wait_gives_up_with_timeout_status_then_recovers(A, O, PR, monkeypatch):
    """The staged ring's bounded wait, made to run out.  The library's test
    hook PSG_TEST_RING_TIMEOUT=1 leaves every team's first ring slot unfilled
    (a phase nothing completes) and bounds each wait by about a millisecond:
    the waits give up, PSG_E_TIMEOUT reaches the status word, and the kernel
    still ends, after the copies it did issue have landed, with the context
    usable.  The same call without the hook is then correct again."""
    x = SI.softmax_input(7, 300, 4096)  # 16 KB rows, wider than a warp holds: the staged ring
    dx = dev(x)
    y = torch.empty_like(dx)
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    stages, epi = PR.softmax_rows()
    monkeypatch.setenv("PSG_TEST_RING_TIMEOUT", "1")
    A.psg_reduce_rows(stages, epi, [dx], [A.view_of(dx)], y, A.view_of(y), st)
    torch.cuda.synchronize()
    assert int(st.item()) == A.E_TIMEOUT
    monkeypatch.delenv("PSG_TEST_RING_TIMEOUT")
    st.zero_()
    A.psg_reduce_rows(stages, epi, [dx], [A.view_of(dx)], y, A.view_of(y), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _softmax_check(O, x.numpy(), y.cpu().numpy())
