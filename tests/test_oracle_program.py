"""Pins of the oracle's call evaluator (oracle/program.py) on the CPU.

The evaluator runs a call's node program, row reduction or contraction one
primitive node at a time.  Each case here spells a composed op whose oracle
form is already pinned (the elementwise chain, softmax, RMSNorm, the naive
matmul loop) as the program the library would be given, and asks for the
same bits: a wrong operand, stage order, broadcast or epilogue mode would
not give them.
"""
import numpy as np
import pytest

import seeded_inputs as SI


def N(op, a=0, b=0, c=0, dt="f32", cval=0.0):
    return (op, a, b, c, dt, cval)


@pytest.fixture(scope="module")
def P(O):
    import oracle.program as P
    return P


def test_chain_program_equals_composed_chain(O, P):
    a, b = SI.chain(1, 37, 301)
    a_, b_ = O.T(a.numpy(), "f32"), O.T(b.numpy(), "f32")
    prog = [N("LOAD", 0), N("LOAD", 1), N("CMPLT", 0, 1), N("CONST", cval=0.5), N("MUL", 0, 3), N("EXP", 4),
            N("MUL", 1, 1), N("CONST", cval=1.0), N("ADD", 6, 7), N("LOG", 8), N("WHERE", 2, 5, 9)]
    loads = [P.read(a_.data, "f32", (37, 301), (301, 1)), P.read(b_.data, "f32", (37, 301), (1, 0))]
    got = P.program(prog, loads, (37, 301))
    ref = O.chain_where_exp_log(a_, b_)
    assert got.data.tobytes() == ref.data.tobytes()


def test_softmax_as_two_stage_reduction(O, P):
    x = O.T(SI.softmax_input(2, 19, 130).numpy(), "f32")
    stages = [("MAX", [N("LOAD", 0)]),
              ("SUM", [N("LOAD", 0), N("RED", 0), N("NEG", 1), N("ADD", 0, 2), N("EXP", 3)])]
    epi = [N("LOAD", 0), N("RED", 0), N("NEG", 1), N("ADD", 0, 2), N("EXP", 3), N("RED", 1), N("RECIP", 5),
           N("MUL", 4, 6)]
    out, reds, pro = P.reduce_rows(stages, epi, [x], per_element=True)
    ref = O.softmax_rows(x)
    assert out.data.tobytes() == ref.data.tobytes()
    assert reds[0].data.tobytes() == O.reduce_max(x).data.tobytes()
    assert pro[1].shape == (19, 130)


def test_rmsnorm_as_one_stage_reduction_with_row_broadcast_weight(O, P):
    xr, wr = SI.rmsnorm_input(3, 12, 256)
    x, w = O.T(SI.bits(xr), "bf16"), O.T(SI.bits(wr), "bf16")
    stages = [("SUM", [N("LOAD", 0, dt="bf16"), N("CAST", 0), N("MUL", 1, 1)])]
    epi = [N("LOAD", 0, dt="bf16"), N("CAST", 0), N("RED", 0), N("CONST", cval=1.0 / 256), N("MUL", 2, 3),
           N("CONST", cval=1e-6), N("ADD", 4, 5), N("SQRT", 6), N("RECIP", 7), N("MUL", 1, 8),
           N("LOAD", 1, dt="bf16"), N("CAST", 10), N("MUL", 9, 11), N("CAST", 12, dt="bf16")]
    loads = [x, P.read(w.data, "bf16", (12, 256), (0, 1))]
    out, _, _ = P.reduce_rows(stages, epi, loads, per_element=True)
    assert out.data.tobytes() == O.rmsnorm(x, w).data.tobytes()


def test_per_row_epilogue_and_bare_stage(O, P):
    g = SI.gen(4)
    x = O.T(SI.normal((7, 33), 0, 1, g).numpy(), "f32")
    stages = [("SUM", [N("LOAD", 0)])]
    out, reds, _ = P.reduce_rows(stages, [N("RED", 0), N("CONST", cval=1.0 / 33), N("MUL", 0, 1)], [x],
                                 per_element=False)
    ref = O.mul(O.reduce_sum(x), O.full((7, 1), 1.0 / 33, "f32"))
    assert out.shape == (7, 1) and out.data.tobytes() == ref.data.tobytes()
    bare, _, _ = P.reduce_rows(stages, [], [x], per_element=False)
    assert bare.data.tobytes() == O.reduce_sum(x).data.tobytes()
    # rank-3 iteration shape: the leading dims are the rows
    x3 = O.T(x.data.reshape(7, 1, 33), "f32")
    out3, _, _ = P.reduce_rows([("MAX", [N("LOAD", 0)])], [], [x3], per_element=False)
    assert out3.data.reshape(-1).tobytes() == O.reduce_max(x).data.reshape(-1).tobytes()


def test_hook_sees_every_value_and_identity_changes_nothing(O, P):
    x = O.T(SI.softmax_input(5, 4, 40).numpy(), "f32")
    stages = [("MAX", [N("LOAD", 0)]), ("SUM", [N("LOAD", 0), N("RED", 0), N("NEG", 1), N("ADD", 0, 2),
                                                N("EXP", 3)])]
    epi = [N("LOAD", 0), N("RED", 0), N("NEG", 1), N("ADD", 0, 2), N("EXP", 3), N("RED", 1), N("RECIP", 5),
           N("MUL", 4, 6)]
    seen = []

    def hook(kind, i, v):
        seen.append((kind, i))
        return v
    out, _, _ = P.reduce_rows(stages, epi, [x], per_element=True, hook=hook)
    assert out.data.tobytes() == O.softmax_rows(x).data.tobytes()
    assert ("stage", 0) in seen and ("stage", 1) in seen and ("epilogue", 7) in seen and ("prologue1", 4) in seen

    # moving the sum up moves every probability down
    def bump(kind, i, v):
        if kind == "stage" and i == 1:
            return O.T((v.data * np.float32(1.01)).astype(np.float32), v.dt)
        return v
    lo, _, _ = P.reduce_rows(stages, epi, [x], per_element=True, hook=bump)
    assert np.all(lo.data <= out.data)


def test_contract_equals_naive_loop_per_batch(O, P):
    g = np.random.default_rng(5)
    A = g.standard_normal((3, 9, 17)).astype(np.float32)
    B = g.standard_normal((3, 17, 6)).astype(np.float32)
    got = P.contract(O.T(A, "f32"), O.T(np.ascontiguousarray(B.transpose(0, 2, 1)), "f32"), "bf16")
    for z in range(3):
        ref = O.matmul(O.T(A[z], "f32"), O.T(B[z], "f32"), "bf16")
        assert got.data[z].tobytes() == ref.data.tobytes()
    with pytest.raises(ValueError):
        P.contract(O.T(A, "f32"), O.T(B, "f32"), "f32")


def test_contract_epilogue_equals_matmul_then_elementwise(O, P):
    """ACC + residual, cast and relu through the evaluator give the bits of
    the separate nodes: the float32 matmul, its CAST, the ADD, the WHERE."""
    g = np.random.default_rng(6)
    A = O.tensor(g.standard_normal((2, 7, 33)), "bf16")
    B = O.tensor(g.standard_normal((2, 33, 5)), "bf16")
    R = O.tensor(g.standard_normal((2, 7, 5)), "bf16")
    bt = O.T(np.ascontiguousarray(B.data.transpose(0, 2, 1)), "bf16")
    prog = [N("ACC"), N("CAST", 0, dt="bf16"), N("LOAD", 0, dt="bf16"), N("ADD", 1, 2, dt="bf16"),
            N("CONST", dt="bf16"), N("CMPLT", 4, 3, dt="bf16"), N("WHERE", 5, 3, 4, dt="bf16")]
    got = P.contract_epilogue(A, bt, prog, [R])
    for z in range(2):
        c = O.matmul(O.T(A.data[z], "bf16"), O.T(B.data[z], "bf16"), "f32")
        h = O.add(O.cast(c, "bf16"), O.T(R.data[z], "bf16"))
        ref = O.relu(h)
        assert got.data[z].tobytes() == ref.data.tobytes()
    with pytest.raises(TypeError):
        P.program([N("ACC")], [], (2, 2))
