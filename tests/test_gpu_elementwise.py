"""GPU parity of psg_elementwise against the CPU oracle.

Bar: programs of correctly rounded nodes (ADD MUL NEG CMPLT WHERE RECIP SQRT
CAST) and every integer program are bit-exact; an EXP or LOG result is within
8 float32 ulps of the oracle's (the elementwise bound for transcendentals).
Inputs use every View form: contiguous, transposed, expanded rows and
columns, scalars, offset slices and masked (padded) reads, at shapes with
ragged chunk tails.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
from helpers import dev, first_mismatches, same_bits_nan_equal, storage_dtype, to_np, ulp_dist_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from primitive_sm_graph_gb300 import _abi
    return _abi


def _run(A, prog, ins, in_views, shape, out_dt):
    out = torch.empty(shape, dtype=storage_dtype(out_dt), device="cuda")
    A.psg_elementwise(prog, ins, in_views, out, A.view_of(out))
    torch.cuda.synchronize()
    return out


# ---------------------------------------------------------- the chain --------

def _chain_prog(A):
    n = A.node
    return [n("LOAD", 0), n("LOAD", 1), n("CMPLT", 0, 1), n("CONST", cval=0.5), n("MUL", 0, 3),
            n("EXP", 4), n("MUL", 1, 1), n("CONST", cval=1.0), n("ADD", 6, 7), n("LOG", 8),
            n("WHERE", 2, 5, 9)]


@pytest.mark.parametrize("R,C", [(37, 1003), (5, 8), (1, 1), (64, 4096), (3, 7)])
def test_chain_matches_oracle(A, O, R, C):
    a, b = SI.chain(1, R, C)
    da, db = dev(a), dev(b)
    bview = A.view_of(db, shape=(R, C), strides=(1, 0))
    y = _run(A, _chain_prog(A), [da, db], [A.view_of(da), bview], (R, C), "f32")
    ref = O.chain_where_exp_log(O.T(a.numpy(), "f32"), O.T(b.numpy(), "f32")).data
    d = ulp_dist_f32(to_np(y.cpu()), ref)
    assert d.max() <= 8, d.max()
    # the CMPLT / WHERE decision itself is exact: the EXP branch is taken
    # exactly where a < b
    sel = a.numpy() < b.numpy()[:, None]
    e = np.exp(a.numpy()[sel].astype(np.float64) * 0.5)
    assert np.all(np.abs(to_np(y.cpu())[sel] - e) <= 8 * np.spacing(e.astype(np.float32)))


def test_chain_full_size(A, O):
    a, b = SI.chain(0)
    da, db = dev(a), dev(b)
    bview = A.view_of(db, shape=(4096, 4096), strides=(1, 0))
    y = _run(A, _chain_prog(A), [da, db], [A.view_of(da), bview], (4096, 4096), "f32")
    ref = O.chain_where_exp_log(O.T(a.numpy(), "f32"), O.T(b.numpy(), "f32")).data
    assert ulp_dist_f32(to_np(y.cpu()), ref).max() <= 8
    # same bits twice
    y2 = _run(A, _chain_prog(A), [da, db], [A.view_of(da), bview], (4096, 4096), "f32")
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))


# ------------------------------------------------------ random programs ------

FLOAT_DT = ("f32", "bf16", "f16")
INT_DT = ("i32", "i16", "i8")


def _make_inputs(g, shape, dts):
    """Random base buffers and View layouts over them, for a 2-D shape."""
    R, C = shape
    out = []
    for k, dt in enumerate(dts):
        form = ["contig", "transposed", "row_bcast", "col_bcast", "scalar", "slice",
                "padded"][int(torch.randint(0, 7, (1,), generator=g))]
        if form == "contig":
            n, shp, st, off, mask = R * C, (R, C), (C, 1), 0, None
        elif form == "transposed":
            n, shp, st, off, mask = R * C, (R, C), (1, R), 0, None
        elif form == "row_bcast":
            n, shp, st, off, mask = C, (R, C), (0, 1), 0, None
        elif form == "col_bcast":
            n, shp, st, off, mask = R, (R, C), (1, 0), 0, None
        elif form == "scalar":
            n, shp, st, off, mask = 1, (R, C), (0, 0), 0, None
        elif form == "slice":
            n, shp, st, off, mask = (R + 1) * (C + 3) + 5, (R, C), (C + 3, 1), 5, None
        else:  # padded by (1, 2) on rows and (3, 1) on columns of an inner block
            r0, c0 = 1, 3
            ir, ic = max(R - 3, 0), max(C - 4, 0)
            n = max(ir * ic, 1)
            shp, st, off = (R, C), (ic, 1), -(r0 * ic + c0)
            mask = [(r0, r0 + ir), (c0, c0 + ic)]
        if dt in INT_DT:
            lim = {"i32": 2**31 - 1, "i16": 2**15 - 1, "i8": 127}[dt]
            base = torch.randint(-lim, lim, (n,), generator=g, dtype=torch.int64).to(storage_dtype(dt))
        else:
            kind = SI.AIMED_KINDS[int(torch.randint(0, len(SI.AIMED_KINDS), (1,), generator=g))]
            base = SI.aimed(kind, (n,), g).to(storage_dtype(dt)) if kind not in ("constant", "cancel", "sorted") \
                else SI.aimed("normal", (n,), g).to(storage_dtype(dt))
        out.append((base, shp, st, off, mask, dt))
    return out


def _random_program(g, n_in, in_dts, int_mode, n_ops, transcendental_last, pool=None):
    """A random DAG as (op, args, dtype) in topological order."""
    P = [("LOAD", (k,), in_dts[k]) for k in range(n_in)]
    dts_pool = pool or (INT_DT if int_mode else FLOAT_DT)

    def pick(pred=None):
        cands = [i for i in range(len(P)) if pred is None or pred(P[i][2])]
        if not cands:
            return None
        # prefer recent values so the program stays deep rather than wide
        w = torch.tensor([1.0 + i for i in range(len(cands))])
        return cands[int(torch.multinomial(w, 1, generator=g))]

    unary = ["NEG", "CAST"] if int_mode else ["NEG", "RECIP", "SQRT", "CAST"]
    binary = ["ADD", "MUL", "CMPLT"]
    for _ in range(n_ops):
        r = float(torch.rand(1, generator=g))
        if r < 0.3:
            op = unary[int(torch.randint(0, len(unary), (1,), generator=g))]
            i = pick()
            if op == "CAST":
                dt = dts_pool[int(torch.randint(0, len(dts_pool), (1,), generator=g))]
                if not int_mode and float(torch.rand(1, generator=g)) < 0.2:
                    dt = "i32"
                P.append(("CAST", (i,), dt))
            else:
                if P[i][2] in INT_DT and op != "NEG":
                    op = "NEG"
                P.append((op, (i,), P[i][2]))
        elif r < 0.8:
            op = binary[int(torch.randint(0, 3, (1,), generator=g))]
            i = pick()
            j = pick(lambda d, di=P[i][2]: d == di)
            if float(torch.rand(1, generator=g)) < 0.2:
                c = float(torch.randn(1, generator=g)) * 3
                P.append(("CONST", (round(c) if P[i][2] in INT_DT else c,), P[i][2]))
                j = len(P) - 1
            P.append((op, (i, j), P[i][2]))
        else:
            c = pick()
            x = pick()
            y = pick(lambda d, dx=P[x][2]: d == dx)
            P.append(("WHERE", (c, x, y), P[x][2]))
    last = len(P) - 1
    if transcendental_last:
        if P[last][2] not in (pool or FLOAT_DT):
            P.append(("CAST", (last,), "f32"))
            last += 1
        P.append((["EXP", "LOG"][int(torch.randint(0, 2, (1,), generator=g))], (last,), P[last][2]))
    return P


def _to_psg(A, P):
    prog = []
    for op, args, dt in P:
        if op == "CONST":
            prog.append(A.node("CONST", dtype=dt, cval=args[0]))
        else:
            a = list(args) + [0, 0, 0]
            prog.append(A.node(op, a[0], a[1], a[2], dtype=dt))
    return prog


def _oracle_eval(O, P, inputs, shape):
    vals = []
    for op, args, dt in P:
        if op == "LOAD":
            base, shp, st, off, mask, idt = inputs[args[0]]
            vals.append(O.view(O.T(SI.bits(base), idt), shp, st, off, mask))
        elif op == "CONST":
            vals.append(O.full(shape, args[0], dt))
        elif op in ("NEG", "EXP", "LOG", "SQRT", "RECIP"):
            vals.append(getattr(O, op.lower())(vals[args[0]]))
        elif op == "CAST":
            vals.append(O.cast(vals[args[0]], dt))
        elif op in ("ADD", "MUL", "CMPLT"):
            vals.append(getattr(O, op.lower())(vals[args[0]], vals[args[1]]))
        elif op == "WHERE":
            vals.append(O.where(vals[args[0]], vals[args[1]], vals[args[2]]))
    return vals[-1]


def _fuzz(A, O, seed, int_mode, transcendental_last, n_cases, pool=None):
    g = SI.gen(seed)
    ran = 0
    for case in range(n_cases):
        R = int(torch.randint(1, 40, (1,), generator=g))
        C = int(torch.randint(1, 300, (1,), generator=g))
        n_in = int(torch.randint(1, 4, (1,), generator=g))
        dpool = pool or (INT_DT if int_mode else FLOAT_DT)
        in_dts = [dpool[int(torch.randint(0, len(dpool), (1,), generator=g))] for _ in range(n_in)]
        inputs = _make_inputs(g, (R, C), in_dts)
        P = _random_program(g, n_in, in_dts, int_mode, int(torch.randint(2, 10, (1,), generator=g)),
                            transcendental_last, pool)
        prog = _to_psg(A, P)
        dins = [dev(x[0]) for x in inputs]
        views = [A.view_of(d, shape=x[1], strides=x[2], offset=x[3], mask=x[4])
                 for d, x in zip(dins, inputs)]
        out_dt = P[-1][2]
        out = torch.empty((R, C), dtype=storage_dtype(out_dt), device="cuda")
        st = A.psg_elementwise(prog, dins, views, out, A.view_of(out), check=False)
        if st == A.E_UNSUPPORTED_PROGRAM:
            continue
        assert st == 0, (case, A.STATUS[st], P)
        torch.cuda.synchronize()
        ref = _oracle_eval(O, P, inputs, (R, C))
        got = to_np(out.cpu())
        if transcendental_last:
            if out_dt == "f64":
                # float64 EXP / LOG: CUDA's and the C library's are both within
                # an ulp or so of the exact value; 4 float64 ulps bound them
                g64, r64 = got.astype(np.float64), ref.data.astype(np.float64)
                fin = np.isfinite(r64)
                assert np.all(np.abs(g64[fin] - r64[fin]) <= 4 * np.spacing(np.abs(r64[fin]))), (case, P)
                assert np.array_equal(np.isnan(g64), np.isnan(r64)) and np.array_equal(g64[~fin & ~np.isnan(r64)],
                                                                                        r64[~fin & ~np.isnan(r64)])
            elif out_dt == "f32":
                assert ulp_dist_f32(got, ref.data).max() <= 8, (case, P)
            else:  # a narrow float result: within one unit of its own rounding
                g64 = O.T(got, out_dt).f64()
                r64 = ref.f64()
                rel = 2.0 ** -7 if out_dt == "bf16" else 2.0 ** -10
                fin = np.isfinite(r64)
                assert np.all(np.abs(g64[fin] - r64[fin]) <= rel * np.abs(r64[fin]) + 1e-30), (case, P)
                assert np.array_equal(np.isnan(g64), np.isnan(r64))
        else:
            assert same_bits_nan_equal(got, ref.data, not int_mode or out_dt in FLOAT_DT), \
                (case, P, [x[4] for x in inputs], first_mismatches(got, ref.data))
        ran += 1
    assert ran >= n_cases * 0.7


def test_random_float_programs_bit_exact(A, O):
    _fuzz(A, O, seed=11, int_mode=False, transcendental_last=False, n_cases=120)


def test_random_int_programs_bit_exact(A, O):
    _fuzz(A, O, seed=12, int_mode=True, transcendental_last=False, n_cases=120)


def test_random_programs_ending_in_exp_or_log(A, O):
    _fuzz(A, O, seed=13, int_mode=False, transcendental_last=True, n_cases=80)


def test_random_float64_programs(A, O):
    """float64 nodes (limn, "The op set": float64 computes natively at its own
    width) mixed with float32 inputs and CASTs both ways: programs of
    correctly rounded nodes give the oracle's bits; a final EXP or LOG in
    float64 is within 4 float64 ulps of the C library's."""
    _fuzz(A, O, seed=14, int_mode=False, transcendental_last=False, n_cases=80, pool=("f64", "f32"))
    _fuzz(A, O, seed=15, int_mode=False, transcendental_last=True, n_cases=60, pool=("f64", "f32"))


def test_rank3_broadcast_and_empty(A, O):
    g = SI.gen(3)
    x = SI.normal((4, 1, 9), 0, 1, g)
    y = SI.normal((1, 5, 9), 0, 1, g)
    dx, dy = dev(x), dev(y)
    vx = A.view_of(dx, shape=(4, 5, 9), strides=(9, 0, 1))
    vy = A.view_of(dy, shape=(4, 5, 9), strides=(0, 9, 1))
    out = _run(A, [A.node("LOAD", 0), A.node("LOAD", 1), A.node("MUL", 0, 1)], [dx, dy], [vx, vy],
               (4, 5, 9), "f32")
    ref = O.mul(O.view(O.T(x.numpy(), "f32"), (4, 5, 9), (9, 0, 1)),
                O.view(O.T(y.numpy(), "f32"), (4, 5, 9), (0, 9, 1)))
    assert np.array_equal(to_np(out.cpu()), ref.data)
    # an empty output launches nothing and succeeds
    e = torch.empty((0, 7), device="cuda")
    A.psg_elementwise([A.node("LOAD", 0)], [e], [A.view_of(e)], e, A.view_of(e))


def test_exp_dense_sweep_within_8_ulp(A, O):
    """EXP over every 251st float32 bit pattern of [-104, 89] (every binade,
    overflow to inf, underflow through the subnormals to 0) plus the special
    values, against the oracle's expf: within 8 float32 ulps, NaN for NaN."""
    def bits(v):
        return int(np.array([v], np.float32).view(np.int32)[0])
    pos = np.arange(0, bits(89.0), 251, dtype=np.int64)
    neg = np.arange(0, bits(104.0), 251, dtype=np.int64) | np.int64(0x80000000)
    x = np.concatenate([pos, neg]).astype(np.uint32).view(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 88.72283, 88.72284, -87.33654, -87.33655,
                        -103.97208, -103.97209, 1e-45, -1e-45, 1e30, -1e30, 0.5, -0.5, 1.0, -1.0],
                       dtype=np.float32)
    x = np.concatenate([x, special])
    dx = torch.from_numpy(x).cuda()
    out = torch.empty_like(dx)
    v = A.view_of(dx)
    A.psg_elementwise([A.node("LOAD", 0), A.node("EXP", 0)], [dx], [v], out, A.view_of(out))
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = O.exp(O.T(x, "f32")).data
    d = ulp_dist_f32(got, ref)
    worst = int(np.argmax(d))
    assert d.max() <= 8, (float(x[worst]), float(got[worst]), float(ref[worst]), int(d.max()))
