"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every test here runs without a GPU.  Each pin is chosen so that a plausible
mistake in the oracle (a dropped term, a wrong sign or index, a transposed
operand, a wrong identity or rounding) fails it: closed forms, exact rational
arithmetic on tiny inputs, library routines for special cases (numpy views,
torch's bfloat16 conversion, Python's math), the invariants Litmus states as
lemmas R1-R3, and the printed examples under tests/golden/.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import seeded_inputs as SI

GOLD = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24


def gamma(n):
    return n * U / (1 - n * U)


def f32(x):
    return np.asarray(x, dtype=np.float32)


def spacing32(y):
    return float(np.spacing(np.float32(abs(y)))) if y != 0 else 2.0 ** -149


# ------------------------------------------------------------------ View ---

def _oracle_view_of(O, arr, shape, strides, offset=0, mask=None):
    return O.view(O.T(arr, "f32"), shape, strides, offset, mask).data


def test_view_matches_numpy_movement_ops(O):
    """reshape / permute / expand / pad / shrink expressed as (shape, strides,
    offset, mask) read the same values numpy's own movement ops produce."""
    g = np.random.default_rng(1)
    base = g.standard_normal(60).astype(np.float32)
    a = base.reshape(3, 4, 5)
    # permute (2,0,1)
    got = _oracle_view_of(O, base, (5, 3, 4), (1, 20, 5))
    np.testing.assert_array_equal(got, np.transpose(a, (2, 0, 1)))
    # shrink a[1:3, 0:4, 2:5]
    got = _oracle_view_of(O, base, (2, 4, 3), (20, 5, 1), offset=1 * 20 + 2)
    np.testing.assert_array_equal(got, a[1:3, 0:4, 2:5])
    # expand a middle broadcast dim: [3,1,5] -> [3,7,5]
    b = a[:, 1:2, :]
    got = _oracle_view_of(O, base, (3, 7, 5), (20, 0, 1), offset=5)
    np.testing.assert_array_equal(got, np.broadcast_to(b, (3, 7, 5)))
    # pad last dim by (2, 1) and first dim by (1, 0): masked cells read 0
    got = _oracle_view_of(O, base, (4, 4, 8), (20, 5, 1), offset=-20 - 2,
                          mask=[(1, 4), (0, 4), (2, 7)])
    np.testing.assert_array_equal(got, np.pad(a, ((1, 0), (0, 0), (2, 1))))
    # reshape of a permuted tensor needs a copy: compose permute then a View
    # over the materialised buffer
    p = _oracle_view_of(O, base, (5, 3, 4), (1, 20, 5))
    got = _oracle_view_of(O, p.reshape(-1), (15, 4), (4, 1))
    np.testing.assert_array_equal(got, np.transpose(a, (2, 0, 1)).reshape(15, 4))


def test_view_out_of_range_is_refused(O):
    with pytest.raises(IndexError):
        _oracle_view_of(O, np.zeros(10, np.float32), (4, 4), (4, 1))
    # a negative offset is fine when the mask keeps every read in range
    got = _oracle_view_of(O, np.arange(3, dtype=np.float32), (5,), (1,), offset=-1,
                          mask=[(1, 4)])
    np.testing.assert_array_equal(got, [0, 0, 1, 2, 0])


# ----------------------------------------------------------- elementwise ---

def test_unary_special_values(O):
    x = O.T(f32([0.0, 1.0, 4.0, 2.0]), "f32")
    assert O.exp(x).data[0] == 1.0
    assert O.log(x).data[1] == 0.0
    assert O.sqrt(x).data[2] == 2.0
    assert O.recip(x).data[3] == 0.5
    s = O.T(f32([np.inf, -np.inf, np.nan, -0.0, 0.0, -1.0]), "f32")
    e = O.exp(s).data
    assert e[0] == np.inf and e[1] == 0.0 and np.isnan(e[2]) and e[3] == 1.0
    lg = O.log(s).data
    assert lg[0] == np.inf and np.isnan(lg[1]) and lg[4] == -np.inf and np.isnan(lg[5])
    r = O.recip(s).data
    assert r[0] == 0.0 and np.signbit(r[1]) and r[3] == -np.inf and r[4] == np.inf
    n = O.neg(s).data
    assert n[0] == -np.inf and not np.signbit(n[3]) and np.signbit(n[4])


def test_transcendentals_within_one_ulp_of_double(O):
    """exp/log/sqrt of the oracle are within 1 float32 ulp of the double result
    rounded to float32 (glibc's float functions are nearly correctly rounded)."""
    g = np.random.default_rng(2)
    x = f32(np.concatenate([g.uniform(-80, 80, 400), g.uniform(-1e-3, 1e-3, 100)]))
    e = O.exp(O.T(x, "f32")).data
    ref = f32([math.exp(float(v)) for v in x])
    assert np.all(np.abs(e.astype(np.float64) - ref) <= np.spacing(np.abs(ref)).astype(np.float64))
    xp = f32(np.abs(x) + 1e-30)
    lg = O.log(O.T(xp, "f32")).data
    ref = f32([math.log(float(v)) for v in xp])
    assert np.all(np.abs(lg.astype(np.float64) - ref) <= np.spacing(np.abs(ref)).astype(np.float64))


def test_sqrt_and_recip_correctly_rounded_exact_rationals(O):
    """IEEE division and square root are correctly rounded: checked against
    exact rational arithmetic (half an ulp)."""
    g = np.random.default_rng(3)
    x = f32(g.uniform(0.001, 1000.0, 300))
    r = O.recip(O.T(x, "f32")).data
    s = O.sqrt(O.T(x, "f32")).data
    for xi, ri, si in zip(x, r, s):
        exact = Fraction(1) / Fraction(float(xi))
        assert abs(Fraction(float(ri)) - exact) <= Fraction(spacing32(ri)) / 2
        # sqrt: |s^2 - x| bound via s +- half ulp bracketing
        h = Fraction(spacing32(si)) / 2
        lo, hi = Fraction(float(si)) - h, Fraction(float(si)) + h
        assert lo * lo <= Fraction(float(xi)) <= hi * hi


def test_tiki_vector_add_exact(O):
    """Tiki's first native result: 4,096 float32 additions exactly right."""
    spec = json.load(open(os.path.join(GOLD, "tiki_vector_add_4096.json")))
    g = SI.gen(0)
    a = SI.uniform((spec["n"],), -1.0, 1.0, g).numpy()
    b = SI.uniform((spec["n"],), -1.0, 1.0, g).numpy()
    y = O.add(O.T(a, "f32"), O.T(b, "f32")).data
    for ai, bi, yi in zip(a[:512], b[:512], y[:512]):
        exact = Fraction(float(ai)) + Fraction(float(bi))
        assert abs(Fraction(float(yi)) - exact) <= Fraction(spacing32(yi)) / 2
    # the float64 sum of two float32 values of this range is exact
    np.testing.assert_array_equal(y, (a.astype(np.float64) + b.astype(np.float64)).astype(np.float32))


def test_luminal_element_wise_mul_reading(O):
    """The blog's element_wise_mul indexes C[i*m + j]; the oracle's MUL is the
    row-major loop with i*n + j, which is the only reading valid for m != n."""
    spec = json.load(open(os.path.join(GOLD, "luminal_element_wise_mul.json")))
    g = np.random.default_rng(4)
    for m, n in spec["cases"]:
        A = f32(g.integers(-9, 9, (m, n)))
        B = f32(g.integers(-9, 9, (m, n)))
        C = O.mul(O.T(A, "f32"), O.T(B, "f32")).data
        Af, Bf = A.reshape(-1), B.reshape(-1)
        ref = np.zeros(m * n, np.float32)
        for i in range(m):
            for j in range(n):
                ref[i * n + j] = Af[i * n + j] * Bf[i * n + j]
        np.testing.assert_array_equal(C.reshape(-1), ref)
        if 1 < m < n:  # the printed index aliases two cells
            cells = {i * m + j for i in range(m) for j in range(n)}
            assert len(cells) < m * n


def test_cast_bf16_round_to_nearest_even(O):
    """float32 -> bfloat16 matches torch's conversion (round to nearest even)
    and the hand-worked ties."""
    g = SI.gen(5)
    x = torch.cat([torch.randn(20000, generator=g) * 100, torch.tensor([
        1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.0e38, -3.0e38, 1e-40, 0.0, -0.0])])
    got = O.cast(O.T(x.numpy(), "f32"), "bf16").data
    ref = SI.bits(x.to(torch.bfloat16))
    np.testing.assert_array_equal(got, ref)
    # ties: 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert got[20000] == 0x3F80
    assert got[20001] == 0x3F82  # 1 + 3*2^-8 -> 1 + 2^-6 (even)
    nan = O.cast(O.T(f32([np.nan]), "f32"), "bf16")
    assert np.isnan(nan.f64()[0])
    # bf16 -> f32 is exact
    back = O.cast(O.T(got, "bf16"), "f32").data
    np.testing.assert_array_equal(back, x.to(torch.bfloat16).to(torch.float32).numpy())


def test_cast_float_to_int_and_int_wraparound(O):
    x = O.T(f32([2.9, -2.9, np.nan, 3e9, -3e9, 127.5, 128.0, -129.0]), "f32")
    i32 = O.cast(x, "i32").data
    assert list(i32) == [2, -2, 0, 2**31 - 1, -2**31, 127, 128, -129]
    i8 = O.cast(x, "i8").data
    assert list(i8[:2]) == [2, -2] and i8[5] == 127 and i8[6] == -128 and i8[7] == 127
    a = O.T(np.array([127, -128, 100], np.int8), "i8")
    b = O.T(np.array([1, -1, 100], np.int8), "i8")
    assert list(O.add(a, b).data) == [-128, 127, -56]
    assert list(O.mul(a, b).data) == [127, -128, 16]  # 10000 mod 256 = 16
    assert list(O.neg(a).data) == [-127, -128, -100]
    big = O.T(np.array([2**31 - 1], np.int32), "i32")
    assert O.add(big, big).data[0] == -2
    # int -> float
    assert O.cast(O.T(np.array([16777217], np.int32), "i32"), "f32").data[0] == 16777216.0


def test_cmplt_and_where_semantics(O):
    a = O.T(f32([1, 2, np.nan, 3, -0.0]), "f32")
    b = O.T(f32([2, 2, 1, np.nan, 0.0]), "f32")
    assert list(O.cmplt(a, b).data) == [1, 0, 0, 0, 0]
    c = O.T(f32([0.0, -0.0, np.nan, 2.0, 1e-45]), "f32")
    x = O.T(f32([1, 1, 1, 1, 1]), "f32")
    y = O.T(f32([7, 7, 7, 7, 7]), "f32")
    assert list(O.where(c, x, y).data) == [7, 7, 1, 1, 1]


# ---------------------------------------------------------------- reduce ---

def test_sum_of_ones_is_exact_and_sum_within_gamma(O):
    n = 1 << 20
    s = O.reduce_sum(O.T(np.ones((2, n), np.float32), "f32")).data
    assert s[0, 0] == n and s[1, 0] == n
    g = np.random.default_rng(6)
    x = f32(g.standard_normal((8, 3000)) * g.uniform(0.1, 1e3, (8, 1)))
    s = O.reduce_sum(O.T(x, "f32")).data[:, 0]
    for r in range(8):
        exact = math.fsum(float(v) for v in x[r])
        bound = gamma(x.shape[1] - 1) * float(np.abs(x[r].astype(np.float64)).sum())
        assert abs(float(s[r]) - exact) <= bound + spacing32(s[r]) / 2


def test_sum_folds_in_ascending_order(O):
    """The fold is sequential and left to right: 2^24 + 1 + 1 + ... stays at
    2^24 in float32 (every +1 is a tie that rounds to even), whereas a
    reversed or pairwise order would keep the ones."""
    x = f32([2.0 ** 24] + [1.0] * 64)
    assert O.reduce_sum(O.T(x[None, :], "f32")).data[0, 0] == 2.0 ** 24
    assert O.reduce_sum(O.T(x[::-1].copy()[None, :], "f32")).data[0, 0] == 2.0 ** 24 + 64


def test_bf16_sum_keeps_float32_total_and_rounds_once(O):
    """limn's dtype paragraph: a reduce keeps its running total in float32 and
    rounds back once.  1 + 256 * 2^-9 = 1.5; rounding every step to bfloat16
    would lose each 2^-9 (less than half a bf16 ulp at 1.0) and give 1.0."""
    x = O.tensor([1.0] + [2.0 ** -9] * 256, "bf16").reshape((1, 257))
    s = O.reduce_sum(x)
    assert s.dt == "bf16" and s.f64()[0, 0] == 1.5


def test_integer_sum_wraps_exactly(O):
    x = np.full((1, 1000), 2**30, np.int32)
    s = O.reduce_sum(O.T(x, "i32")).data[0, 0]
    assert s == np.int32((1000 * 2**30) % 2**32 - (2**32 if (1000 * 2**30) % 2**32 >= 2**31 else 0))
    x8 = np.full((1, 300), 1, np.int8)
    assert O.reduce_sum(O.T(x8, "i8")).data[0, 0] == 300 - 256


def test_max_identity_nan_and_signed_zero(O):
    neg = f32([[-5.0, -3.0, -7.0]])
    assert O.reduce_max(O.T(neg, "f32")).data[0, 0] == -3.0  # not 0 (reduction_init)
    assert O.reduce_max(O.T(np.zeros((1, 0), np.float32), "f32")).data[0, 0] == -np.inf
    nan = f32([[1.0, np.nan, 5.0]])
    assert np.isnan(O.reduce_max(O.T(nan, "f32")).data[0, 0])
    for row in ([-0.0, 0.0], [0.0, -0.0], [-0.0, -0.0, 0.0, -0.0]):
        m = O.reduce_max(O.T(f32([row]), "f32")).data[0, 0]
        assert m == 0.0 and not np.signbit(m)
    assert np.signbit(O.reduce_max(O.T(f32([[-0.0, -0.0]]), "f32")).data[0, 0])
    ints = np.array([[-100, -3, -50]], np.int8)
    assert O.reduce_max(O.T(ints, "i8")).data[0, 0] == -3


def test_threaded_equals_serial_bit_for_bit(O):
    g = np.random.default_rng(7)
    x = f32(g.standard_normal((64, 2000)))
    A = f32(g.standard_normal((40, 70)))
    B = f32(g.standard_normal((70, 30)))
    old = O.NTHREADS
    try:
        O.NTHREADS = 1
        s1, m1 = O.reduce_sum(O.T(x, "f32")).data, O.matmul(O.T(A, "f32"), O.T(B, "f32")).data
        e1 = O.exp(O.T(x, "f32")).data
        O.NTHREADS = 4
        s4, m4 = O.reduce_sum(O.T(x, "f32")).data, O.matmul(O.T(A, "f32"), O.T(B, "f32")).data
        e4 = O.exp(O.T(x, "f32")).data
    finally:
        O.NTHREADS = old
    assert s1.tobytes() == s4.tobytes() and m1.tobytes() == m4.tobytes()
    assert e1.tobytes() == e4.tobytes()


# ----------------------------------------------------------- contraction ---

def test_limn_printed_matmul_nest(O):
    """The printed nest of (4,5) @ (5,3): the loads are in0[i0*5 + r2] and
    in1[i1 + r2*3], the (4,3,1) output aliases the (4,3) sink, and the
    reduce is a SUM from 0.0."""
    spec = json.load(open(os.path.join(GOLD, "limn_ir_matmul_4x5x3.json")))
    M, N, K = spec["loop"]
    (sa, ta), (sb, tb) = O.matmul_views(M, N, K)
    assert list(sa) == spec["loop"] and list(sb) == spec["loop"]
    c0, c1 = spec["in0"]["index_coeff"], spec["in1"]["index_coeff"]
    assert list(ta) == [c0["i0"], c0["i1"], c0["r2"]]
    assert list(tb) == [c1["i0"], c1["i1"], c1["r2"]]
    g = np.random.default_rng(8)
    A = f32(g.integers(-20, 20, spec["in0"]["shape"]))
    B = f32(g.integers(-20, 20, spec["in1"]["shape"]))
    lit = O.matmul_literal(O.T(A, "f32"), O.T(B, "f32"))
    assert lit.shape == tuple(spec["out"]["shape"])
    exact = A.astype(np.int64) @ B.astype(np.int64)  # small ints: exact in float32
    np.testing.assert_array_equal(lit.data.reshape(spec["sink"]), exact.astype(np.float32))


def test_luminal_kernel0_matches_oracle_matmul(O):
    """kernel0's pointer arithmetic (block (f, i), A row f*2, B column i, k
    walking A by 1 and B by 2) computes the same cells as the oracle's
    A @ B: a transposed operand in the oracle would fail this."""
    spec = json.load(open(os.path.join(GOLD, "luminal_kernel0_2x2.json")))
    g = np.random.default_rng(9)
    for _ in range(5):
        A = f32(g.integers(-9, 9, (2, 2)))
        B = f32(g.integers(-9, 9, (2, 2)))
        a, b = A.reshape(-1), B.reshape(-1)
        ref = np.zeros(4, np.float32)
        for f in range(spec["grid"][0]):
            for i in range(spec["grid"][1]):
                acc = np.float32(0.0)  # the acc input, here a zero buffer
                for l in range(spec["loop_extent"]):
                    acc = np.float32(acc + a[f * spec["a_row_stride"] + l * spec["a_k_stride"]]
                                     * b[i * spec["b_col_stride"] + l * spec["b_k_stride"]])
                ref[f * spec["out_row_stride"] + i * spec["out_col_stride"]] = acc
        got = O.matmul(O.T(A, "f32"), O.T(B, "f32")).data.reshape(-1)
        np.testing.assert_array_equal(got, ref)
        assert not np.array_equal(ref, (A @ B.T).reshape(-1)) or np.array_equal(B, B.T)


def test_fused_loop_equals_literal_broadcast_mul_sum(O):
    """The naive fused loop and the literal (M,N,K) MUL + SUM give the same
    bits (same products, same k order) at the tiny graph's size."""
    A, B = SI.tiny_graph(0)
    a, b = O.T(A.numpy(), "f32"), O.T(B.numpy(), "f32")
    lit = O.matmul_literal(a, b).data.reshape(64, 48)
    fused = O.matmul(a, b).data
    assert lit.tobytes() == fused.tobytes()
    # non-square and K = 1 edge
    g = np.random.default_rng(10)
    for (M, K, N) in ((3, 7, 5), (1, 1, 1), (6, 1, 2), (2, 9, 1)):
        A = f32(g.standard_normal((M, K)))
        B = f32(g.standard_normal((K, N)))
        l2 = O.matmul_literal(O.T(A, "f32"), O.T(B, "f32")).data.reshape(M, N)
        f2 = O.matmul(O.T(A, "f32"), O.T(B, "f32")).data
        assert l2.tobytes() == f2.tobytes()


def test_matmul_within_reduction_bound_of_exact(O):
    g = np.random.default_rng(11)
    M, K, N = 6, 257, 5
    A = f32(g.standard_normal((M, K)))
    B = f32(g.standard_normal((K, N)))
    C = O.matmul(O.T(A, "f32"), O.T(B, "f32")).data
    for i in range(M):
        for j in range(N):
            exact = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K))
            mag = sum(abs(float(A[i, k]) * float(B[k, j])) for k in range(K))
            assert abs(float(Fraction(float(C[i, j])) - exact)) <= gamma(K) * mag
    ident = np.eye(5, dtype=np.float32)
    X = f32(g.standard_normal((5, 5)))
    np.testing.assert_array_equal(O.matmul(O.T(ident, "f32"), O.T(X, "f32")).data, X)
    np.testing.assert_array_equal(O.matmul(O.T(X, "f32"), O.T(ident, "f32")).data, X)


def test_bf16_matmul_products_exact_and_cells_agree(O):
    A, B = SI.contraction_bf16(0, 48, 40, 64)
    a, b = O.T(SI.bits(A), "bf16"), O.T(SI.bits(B), "bf16")
    C32 = O.matmul(a, b, "f32").data
    ref = (A.double() @ B.double()).numpy()
    mag = (A.double().abs() @ B.double().abs()).numpy()
    assert np.all(np.abs(C32 - ref) <= gamma(63) * mag + 1e-30)
    ii = np.array([0, 5, 47, 20]); jj = np.array([0, 39, 3, 20])
    acc, m2 = O.matmul_cells(a, b, ii, jj)
    np.testing.assert_array_equal(acc, C32[ii, jj])
    np.testing.assert_allclose(m2, mag[ii, jj], rtol=1e-12)
    Cb = O.matmul(a, b, "bf16")
    np.testing.assert_array_equal(Cb.data, O.cast(O.T(C32, "f32"), "bf16").data)


def test_integer_matmul_exact(O):
    g = np.random.default_rng(12)
    A = g.integers(-128, 127, (5, 9)).astype(np.int8)
    B = g.integers(-128, 127, (9, 4)).astype(np.int8)
    C = O.matmul(O.T(A, "i8"), O.T(B, "i8"), "i32").data
    np.testing.assert_array_equal(C, A.astype(np.int64) @ B.astype(np.int64))


def test_integer_matmul_wraps_modulo_the_width(O):
    """Full-range int32 operands: every product and the total wrap modulo
    2^32 (limn, "Three rules hold it together": integers wrap), and a
    narrower output keeps the low bits.  numpy's uint64 matmul wraps modulo
    2^64, which reduces to the same residues."""
    g = np.random.default_rng(13)
    A = g.integers(-2**31, 2**31, (6, 11), dtype=np.int64).astype(np.int32)
    B = g.integers(-2**31, 2**31, (11, 5), dtype=np.int64).astype(np.int32)
    exact = A.astype(np.int64).astype(np.uint64) @ B.astype(np.int64).astype(np.uint64)
    np.testing.assert_array_equal(O.matmul(O.T(A, "i32"), O.T(B, "i32"), "i32").data,
                                  exact.astype(np.uint32).view(np.int32))
    np.testing.assert_array_equal(O.matmul(O.T(A, "i32"), O.T(B, "i32"), "i8").data,
                                  (exact & np.uint64(0xff)).astype(np.uint8).view(np.int8))
    A16 = g.integers(-2**15, 2**15, (4, 7), dtype=np.int64).astype(np.int16)
    B16 = g.integers(-2**15, 2**15, (7, 3), dtype=np.int64).astype(np.int16)
    e16 = A16.astype(np.int64).astype(np.uint64) @ B16.astype(np.int64).astype(np.uint64)
    np.testing.assert_array_equal(O.matmul(O.T(A16, "i16"), O.T(B16, "i16"), "i16").data,
                                  (e16 & np.uint64(0xffff)).astype(np.uint16).view(np.int16))


def test_float64_matmul_exact_on_small_integers(O):
    """Small-integer float64 operands: every product and partial sum is an
    exact double, so the oracle's float64 loop must equal the exact integer
    product (a transposed operand or a dropped term would not)."""
    g = np.random.default_rng(14)
    A = g.integers(-1000, 1000, (7, 13)).astype(np.float64)
    B = g.integers(-1000, 1000, (13, 9)).astype(np.float64)
    got = O.matmul(O.T(A, "f64"), O.T(B, "f64")).data
    np.testing.assert_array_equal(got, (A.astype(np.int64) @ B.astype(np.int64)).astype(np.float64))


# ------------------------------------------------------- composed ops ------

def test_softmax_lemmas_r1_r2_and_row_sums(O):
    x = O.T(SI.softmax_input(0, 64, 1024).numpy(), "f32")
    m = O.reduce_max(x)
    sh = O.add(x, O.expand_last(O.neg(m), 1024))
    assert np.all(sh.data <= 0) and np.all(sh.data.max(axis=1) == 0)  # R1, bit-exact
    e = O.exp(sh)
    s = O.reduce_sum(e)
    assert np.all(s.data >= 1.0)  # R2
    y = O.softmax_rows(x).data.astype(np.float64)
    N = 1024
    tol = N * 2.0 ** -23 + 2 * gamma(N - 1)
    assert np.all(np.abs(y.sum(axis=1) - 1.0) <= tol)
    # the argmax cell of each row equals RECIP(s) up to an ulp
    r = O.recip(s).data[:, 0]
    am = y[np.arange(64), x.data.argmax(axis=1)]
    assert np.all(np.abs(am - r) <= np.spacing(r))
    # a constant row gives exactly 1/N for N a power of two
    c = O.softmax_rows(O.T(np.full((2, 256), 3.5, np.float32), "f32")).data
    assert np.all(c == np.float32(1.0 / 256))
    # closed form on a two-element row: [0, log 3] -> [1/4, 3/4]
    t = O.softmax_rows(O.T(f32([[0.0, math.log(3.0)]]), "f32")).data[0]
    assert abs(t[0] - 0.25) < 1e-7 and abs(t[1] - 0.75) < 1e-7


def test_softmax_against_double_precision(O):
    xs = SI.softmax_input(1, 16, 1024).double()
    ref = torch.softmax(xs, dim=-1).numpy()
    y = O.softmax_rows(O.T(xs.float().numpy(), "f32")).data.astype(np.float64)
    # per-element: exp + recip + two muls + the SUM bound on the denominator
    tol = ref * ((8 + 4 + 4) * U + 2 * gamma(1023)) + 4 * 2.0 ** -149
    assert np.all(np.abs(y - ref) <= tol + 1e-45)


def test_rmsnorm_invariants(O):
    N = 4096
    w1 = O.tensor(np.ones(N), "bf16")
    for c in (3.0, -0.75, 1e-2):
        x = O.tensor(np.full((1, N), c), "bf16")
        y = O.rmsnorm(x, w1).f64()
        assert np.all(np.abs(y - math.copysign(1.0, c)) <= 2.0 ** -7 + 1e-6 / (c * c))
    X, _ = SI.rmsnorm_input(0, 32, N)
    y = O.rmsnorm(O.T(SI.bits(X), "bf16"), w1).f64()
    ms = (y * y).mean(axis=1)
    assert np.all(np.abs(ms - 1.0) < 2e-2)
    # against the formula in double precision, including the weight
    Xd, Wd = X.double(), SI.rmsnorm_input(0, 32, N)[1].double()
    ref = (Xd * torch.rsqrt((Xd * Xd).mean(-1, keepdim=True) + 1e-6) * Wd).numpy()
    y = O.rmsnorm(O.T(SI.bits(X), "bf16"), O.T(SI.bits(SI.rmsnorm_input(0, 32, N)[1]), "bf16")).f64()
    assert np.all(np.abs(y - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30)


def test_layernorm_centring_r3(O):
    g = np.random.default_rng(13)
    x = f32(g.uniform(-10, 10, (16, 768)))
    xc = O.layernorm_centred(O.T(x, "f32")).data.astype(np.float64)
    row_abs = np.abs(x.astype(np.float64)).sum(axis=1)
    # exact arithmetic gives 0; the computed mean carries the SUM bound
    assert np.all(np.abs(xc.sum(axis=1)) <= 4 * gamma(768) * row_abs + 768 * 2.0 ** -23 * 10)
    # dropping the NEG (a plausible slip) would give 2*x - ... far from zero
    assert np.all(np.abs(xc.mean(axis=1)) < 1e-3)


def test_chain_where_exp_log_elementwise_against_double(O):
    a, b = SI.chain(0, 64, 96)
    y = O.chain_where_exp_log(O.T(a.numpy(), "f32"), O.T(b.numpy(), "f32")).data
    A = a.double().numpy(); Bc = b.double().numpy()[:, None]
    ref = np.where(A < Bc, np.exp(A * 0.5), np.log(Bc * Bc + 1.0))
    # EXP branch: a*0.5 is exact, so only exp's rounding; LOG branch: b*b and
    # +1 each round once (relative 2u on an argument >= 1, i.e. 2u absolute
    # after log), then log's own rounding
    tol = np.where(A < Bc, 1.0, 0.0) * np.spacing(np.abs(ref).astype(np.float32)) \
        + np.where(A < Bc, 0.0, 1.0) * (np.spacing(np.abs(ref).astype(np.float32)) + 2.5 * U)
    assert np.all(np.abs(y - ref) <= tol)
    # a dropped WHERE branch or a swapped comparison would fail this
    assert np.array_equal(y == y, np.ones_like(y, dtype=bool))
    sel = (A < Bc)
    assert np.all(np.abs(y[sel] - np.exp(A[sel] * 0.5)) <= np.spacing(np.abs(ref[sel]).astype(np.float32)))


def test_transpose_is_exact(O):
    x = SI.transpose_input(0, 37, 53).numpy()
    np.testing.assert_array_equal(O.transpose(O.T(x, "f32")).data, x.T)


def test_tiny_graph_against_double(O):
    A, B = SI.tiny_graph(0)
    got = float(O.tiny_graph(O.T(A.numpy(), "f32"), O.T(B.numpy(), "f32")).data)
    C = A.double() @ B.double()
    ref = float((torch.relu(C) ** 2).sum())
    mag_c = (A.double().abs() @ B.double().abs())
    # bound: the matmul cells' SUM error propagated through the square, plus
    # the final SUM's own bound
    dc = gamma(32) * mag_c
    sq_err = float(((2 * C.abs() + dc) * dc).sum()) + 2 * U * ref
    assert abs(got - ref) <= sq_err + gamma(3071) * ref * 2


# ---------------------------------------------------------------- indexed ---

def test_gather_rows(O):
    g = np.random.default_rng(14)
    src = f32(g.standard_normal((10, 7)))
    idx = g.integers(0, 10, 25).astype(np.int32)
    out, bad = O.gather_rows(O.T(src, "f32"), idx)
    assert bad == 0
    np.testing.assert_array_equal(out.data, np.take(src, idx, axis=0))
    out, bad = O.gather_rows(O.T(src, "f32"), np.arange(10, dtype=np.int32))
    np.testing.assert_array_equal(out.data, src)
    out, bad = O.gather_rows(O.T(src, "f32"), np.array([1, 10, -1, 2], np.int32))
    assert bad == 2 and np.all(out.data[1] == 0) and np.all(out.data[2] == 0)
    np.testing.assert_array_equal(out.data[3], src[2])


def test_scatter_add_rows(O):
    g = np.random.default_rng(15)
    V, D, n = 6, 5, 40
    dst = f32(g.standard_normal((V, D)))
    upd = f32(g.standard_normal((n, D)))
    # a permutation-free single row: every update lands on row 3, in order
    idx = np.full(n, 3, np.int32)
    out, bad = O.scatter_add_rows(O.T(dst, "f32"), idx, O.T(upd, "f32"))
    acc = dst[3].copy()
    for r in range(n):
        acc = (acc + upd[r]).astype(np.float32)
    np.testing.assert_array_equal(out.data[3], acc)
    np.testing.assert_array_equal(np.delete(out.data, 3, axis=0), np.delete(dst, 3, axis=0))
    # a permutation is a pure placement
    perm = g.permutation(V).astype(np.int32)
    out, _ = O.scatter_add_rows(O.T(np.zeros((V, D), np.float32), "f32"), perm,
                                O.T(upd[:V], "f32"))
    np.testing.assert_array_equal(out.data[perm], upd[:V])
    # matches numpy's unbuffered in-order add.at for float32
    idx = g.integers(0, V, n).astype(np.int32)
    ref = dst.copy()
    np.add.at(ref, idx, upd)
    out, _ = O.scatter_add_rows(O.T(dst, "f32"), idx, O.T(upd, "f32"))
    np.testing.assert_array_equal(out.data, ref)
    # bad indices are skipped and counted
    out, bad = O.scatter_add_rows(O.T(dst, "f32"), np.array([0, 6, -1], np.int32),
                                  O.T(upd[:3], "f32"))
    assert bad == 2
    np.testing.assert_array_equal(out.data[0], (dst[0] + upd[0]).astype(np.float32))


def test_scatter_add_bf16_rounds_once(O):
    dst = O.tensor(np.ones((1, 1)), "bf16")
    upd = O.tensor(np.full((256, 1), 2.0 ** -9), "bf16")
    out, _ = O.scatter_add_rows(dst, np.zeros(256, np.int32), upd)
    assert out.f64()[0, 0] == 1.5


def test_matmul_bt_float_path_equals_fused_loop_and_exact_values(O):
    """The transposed-operand loop (the one the GPT oracle uses) against the
    plain loop and against exact values.  Its products and k order are those
    of the naive loop (Luminal IR blog, "Naive Matrix Multiplication"), so
    both give the same bits for float32, bfloat16 and float16 operands and
    every output dtype; on small-integer operands every product and partial
    sum is an exact float32, so the result equals the exact integer product
    (a transposed operand, a dropped term or a wrong index would not)."""
    g = np.random.default_rng(21)
    for (M, K, N) in ((3, 7, 5), (1, 1, 1), (17, 130, 9), (2, 513, 33)):
        A64 = g.standard_normal((M, K))
        B64 = g.standard_normal((K, N))
        for dt in ("f32", "bf16", "f16"):
            a = O.tensor(A64, dt)
            b = O.tensor(B64, dt)
            bt = O.transpose(b)
            for out in ("f32", "bf16", "f16"):
                ref = O.matmul(a, b, out).data
                got = O.matmul_bt(a, bt, out).data
                assert got.tobytes() == ref.tobytes(), (M, K, N, dt, out)
        Ai = g.integers(-60, 60, (M, K))
        Bi = g.integers(-60, 60, (K, N))
        exact = (Ai @ Bi).astype(np.float64)
        for dt in ("f32", "bf16", "f16"):
            got = O.matmul_bt(O.tensor(Ai, dt), O.T(O.tensor(Bi.T.copy(), dt).data, dt), "f32").data
            np.testing.assert_array_equal(got.astype(np.float64), exact)
    # a non-square case with rows and columns told apart: C[i, j] = sum_k
    # A[i, k] * B[k, j], never A[j, k] or B[j, k]
    A = f32([[1, 2, 3], [4, 5, 6]])
    B = f32([[1, 0], [0, 10], [100, 0]])
    got = O.matmul_bt(O.T(A, "f32"), O.T(B.T.copy(), "f32"), "f32").data
    np.testing.assert_array_equal(got, f32([[301, 20], [604, 50]]))


def test_cast_f16_round_to_nearest_even(O):
    """float32 -> float16 matches numpy's conversion (IEEE round to nearest
    even) on a wide random sweep and on hand-worked cases: ties to even,
    overflow to inf at the halfway point above the largest finite half,
    the subnormal range and its ties; float16 -> float32 is exact."""
    g = SI.gen(22)
    x = torch.cat([torch.randn(20000, generator=g) * 300,
                   torch.randn(4000, generator=g) * 1e-5,
                   torch.randn(2000, generator=g) * 5e4]).numpy().astype(np.float32)
    got = O.cast(O.T(x, "f32"), "f16").data
    with np.errstate(over="ignore"):  # values past 65520 overflow to inf on both sides
        want = x.astype(np.float16)
    np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))
    cases = {
        1.0 + 2 ** -11: 1.0,                    # halfway between 1 and 1 + 2^-10 -> even (1)
        1.0 + 3 * 2 ** -11: 1.0 + 2 ** -9,      # halfway -> even (1 + 2^-9)
        -(1.0 + 2 ** -11): -1.0,
        65504.0: 65504.0,                       # largest finite half
        65519.0: 65504.0,                       # below the halfway point
        65520.0: np.inf,                        # halfway to 65536 rounds to even: inf
        2.0 ** -25: 0.0,                        # half the smallest subnormal -> even (0)
        3 * 2.0 ** -25: 2.0 ** -23,             # 1.5 subnormal steps -> even (2 steps)
        2.0 ** -24: 2.0 ** -24,                 # smallest subnormal is exact
        -0.0: -0.0,
    }
    src = f32(list(cases.keys()))
    out = O.cast(O.T(src, "f32"), "f16").data
    for s, o, want in zip(src, out, cases.values()):
        assert float(o) == want and np.signbit(o) == np.signbit(np.float16(want)), (float(s), float(o), want)
    nan = O.cast(O.T(f32([np.nan]), "f32"), "f16").data
    assert np.isnan(nan[0])
    back = O.cast(O.T(got, "f16"), "f32").data
    np.testing.assert_array_equal(back, got.astype(np.float32))


def test_float64_nodes_against_exact_values(O):
    """float64 nodes compute in double: ADD, MUL exact on small integers,
    SQRT and RECIP correctly rounded (exact rationals), EXP and LOG within
    one float64 ulp of 40-digit values (sympy, an independent
    arbitrary-precision evaluation), NEG flips the sign, CMPLT/WHERE as for
    float32, CAST to float32 rounds to nearest."""
    sympy = pytest.importorskip("sympy")
    g = np.random.default_rng(31)
    a = g.integers(-10**6, 10**6, 200).astype(np.float64)
    b = g.integers(-10**6, 10**6, 200).astype(np.float64)
    A, B = O.T(a, "f64"), O.T(b, "f64")
    np.testing.assert_array_equal(O.add(A, B).data, a + b)
    np.testing.assert_array_equal(O.mul(A, B).data, a * b)
    np.testing.assert_array_equal(O.neg(A).data, -a)
    x = np.abs(g.standard_normal(50)) * 10 + 1e-3
    X = O.T(x, "f64")
    for xi, si, ri in zip(x, O.sqrt(X).data, O.recip(X).data):
        fx = Fraction(float(xi))
        # the correctly rounded square root: the nearest double, checked by
        # the exact squares of its neighbours
        below, above = np.nextafter(si, -np.inf), np.nextafter(si, np.inf)
        assert abs(Fraction(float(si)) ** 2 - fx) <= min(abs(Fraction(float(below)) ** 2 - fx),
                                                         abs(Fraction(float(above)) ** 2 - fx))
        err = abs(Fraction(1) / fx - Fraction(float(ri)))
        assert err <= abs(Fraction(1) / fx - Fraction(float(np.nextafter(ri, np.inf))))
        assert err <= abs(Fraction(1) / fx - Fraction(float(np.nextafter(ri, -np.inf))))
    y = g.uniform(-20, 20, 40)
    for yi, ei in zip(y, O.exp(O.T(y, "f64")).data):
        exact = float(sympy.exp(sympy.Float(float(yi), 60)).evalf(40))
        assert abs(ei - exact) <= np.spacing(exact)
    for xi, li in zip(x, O.log(X).data):
        exact = float(sympy.log(sympy.Float(float(xi), 60)).evalf(40))
        assert abs(li - exact) <= np.spacing(abs(exact))
    c = O.cmplt(O.T(np.array([1.0, np.nan, 2.0]), "f64"), O.T(np.array([2.0, 1.0, np.nan]), "f64")).data
    assert list(c) == [1.0, 0.0, 0.0]
    v = np.array([1.0 + 2.0 ** -24, 1.0 + 3 * 2.0 ** -24, 1e300], np.float64)
    with np.errstate(over="ignore"):   # 1e300 rounds to +inf, as it should
        np.testing.assert_array_equal(O.cast(O.T(v, "f64"), "f32").data, v.astype(np.float32))
