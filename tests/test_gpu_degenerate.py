"""Degenerate sizes through the C ABI, against the oracle where it defines a
result: a contraction over an empty K (an empty SUM is its identity, so every
cell is 0; Luminal IR blog, "Naive Matrix Multiplication": the k loop runs no
times) and over empty M or N; a permute with a zero-length dim; a scatter-add
of no rows (dst unchanged); attention over an empty batch, sequence or head
axis (nothing to compute, nothing written).  Each call returns PSG_OK and
writes no cell outside its (empty) result.  Empty elementwise programs, a
reduction over an empty axis, a gather of no rows, an integer K = 0 product
and an AdamW tensor of no elements are covered beside their rows' other cases.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
from helpers import dev, storage_dtype, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from primitive_sm_graph_gb300 import _abi
    return _abi


def _status():
    return torch.zeros((1,), dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("dt,out_dt", [("bf16", "bf16"), ("bf16", "f32"), ("f32", "f32"), ("f16", "f16")])
def test_contraction_over_empty_k_is_zero(A, O, dt, out_dt):
    M, N, K = 37, 70, 0
    a = torch.empty((M, K), dtype=storage_dtype(dt))
    b = torch.empty((K, N), dtype=storage_dtype(dt))
    da, db = dev(a), dev(b)
    C = torch.full((M, N), 7.0, device="cuda").to(storage_dtype(out_dt))
    st = _status()
    A.psg_contract(da, A.view_of(da, shape=[M, N, K], strides=[K, 0, 1]), db,
                   A.view_of(db, shape=[M, N, K], strides=[0, 1, N]), C, A.view_of(C), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = O.matmul(O.T(SI.bits(a), dt), O.T(SI.bits(b), dt), out_dt)
    assert np.array_equal(to_np(C.cpu()).view(np.uint8), ref.data.view(np.uint8))
    assert not np.any(ref.f64())


@pytest.mark.parametrize("M,N", [(0, 64), (64, 0), (0, 0)])
def test_contraction_with_empty_result(A, M, N):
    K = 128
    a = torch.ones((max(M, 1), K), dtype=torch.bfloat16, device="cuda")[:M]
    b = torch.ones((K, max(N, 1)), dtype=torch.bfloat16, device="cuda")[:, :N].contiguous()
    C = torch.empty((M, N), device="cuda")
    st = _status()
    A.psg_contract(a, A.view_of(a, shape=[M, N, K], strides=[K, 0, 1]), b,
                   A.view_of(b, shape=[M, N, K], strides=[0, 1, max(N, 1)]), C, A.view_of(C), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


@pytest.mark.parametrize("shape,perm", [((0, 7), [1, 0]), ((5, 0), [1, 0]), ((3, 0, 4), [2, 0, 1])])
def test_permute_with_a_zero_length_dim(A, shape, perm):
    x = torch.empty(shape, device="cuda")
    out = torch.empty([shape[p] for p in perm], device="cuda")
    A.psg_permute(x, A.view_of(x), perm, out, A.view_of(out))
    torch.cuda.synchronize()
    assert out.numel() == 0


@pytest.mark.parametrize("dt", ["f32", "bf16", "i32"])
def test_scatter_add_of_no_rows_leaves_dst(A, O, dt):
    g = SI.gen(4)
    V, D = 9, 40
    base = (torch.randint(-50, 50, (V, D), generator=g) if dt == "i32" else SI.normal((V, D), 0, 1, g))
    base = base.to(storage_dtype(dt))
    dst = dev(base)
    idx = torch.empty((0,), dtype=torch.int32, device="cuda")
    upd = torch.empty((0, D), dtype=storage_dtype(dt), device="cuda")
    ws = torch.empty((max(1, A.psg_scatter_workspace(0)),), dtype=torch.uint8, device="cuda")
    st = _status()
    A.psg_scatter_add(dst, A.view_of(dst), idx, 0, upd, A.view_of(upd), ws, ws.numel(), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, bad = O.scatter_add_rows(O.T(SI.bits(base), dt), np.zeros((0,), np.int32),
                                  O.T(np.zeros((0, D), SI.bits(base).dtype), dt))
    assert bad == 0
    assert np.array_equal(to_np(dst.cpu()).view(np.uint8), ref.data.view(np.uint8))


@pytest.mark.parametrize("B,T,H", [(0, 128, 2), (2, 0, 2), (2, 128, 0)])
def test_attention_over_an_empty_axis(A, B, T, H):
    q = torch.empty((B, T, H, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((max(1, B * H * T),), device="cuda")
    guard = lse.clone()
    st = _status()
    vq = A.view_of(q)
    A.psg_attention_fwd(q, vq, q, vq, q, vq, o, A.view_of(o), lse, 0.125, True, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(lse.view(torch.int32), guard.view(torch.int32))
