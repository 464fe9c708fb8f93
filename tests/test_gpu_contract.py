"""GPU parity of psg_contract (matmul as SUM over k of MUL of two broadcast
Views) against the oracle's naive MUL+SUM loop.

Bar (the reduction-order term of Litmus's ToleranceBound, per output cell):
  |c - c_ref| <= 2*gamma_{K-1} * sum_k |a_k b_k|           (float32 output)
  |c - c_ref| <= 2^-7 |c_ref| + 2*gamma_{K-1} * sum|a b|    (bfloat16 output)
where c_ref is the oracle's float32 total.
"""
import os

import numpy as np
import pytest
import torch

import seeded_inputs as SI
from helpers import dev, gamma, storage_dtype, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from primitive_sm_graph_gb300 import _abi
    return _abi


def _views(A, dA, dB, M, N, K, a_layout="mk", b_layout="kn", batch=None):
    """Broadcast Views [batch.., M, N, K] of A and B over their storage."""
    a_ms, a_ks = (K, 1) if a_layout == "mk" else (1, M)
    b_ns, b_ks = (1, N) if b_layout == "kn" else (K, 1)
    shape, sa, sb = [M, N, K], [a_ms, 0, a_ks], [0, b_ns, b_ks]
    if batch:
        shape = [batch] + shape
        sa = [M * K] + sa
        sb = [K * N] + sb
    return A.view_of(dA, shape=shape, strides=sa), A.view_of(dB, shape=shape, strides=sb)


def _check(got, ref32, mag, K, out_dt):
    g = got.astype(np.float64)
    r = ref32.astype(np.float64)
    tol = 2 * gamma(K - 1) * mag + 1e-30
    if out_dt == "bf16":
        tol = tol + 2.0 ** -7 * np.abs(r)
    bad = np.abs(g - r) > tol
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:3], g[bad][:3], r[bad][:3])


def _storage(t, layout):
    return t if layout in ("mk", "kn") else t.t().contiguous()


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 300, 100), (1, 1, 1), (64, 48, 32), (257, 513, 1000),
                                   (512, 256, 4096)])
@pytest.mark.parametrize("out_dt", ["bf16", "f32"])
def test_bf16_contraction_matches_oracle(A, O, M, N, K, out_dt):
    a, b = SI.contraction_bf16(M + N + K, M, N, K)
    ref = O.matmul(O.T(SI.bits(a), "bf16"), O.T(SI.bits(b), "bf16"), "f32").data
    mag = (a.double().abs() @ b.double().abs()).numpy()
    dA, dB = dev(a), dev(b)
    Av, Bv = _views(A, dA, dB, M, N, K)
    C = torch.empty((M, N), dtype=storage_dtype(out_dt), device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = O.T(to_np(C.cpu()), out_dt).f64()
    _check(got, ref, mag, K, out_dt)


@pytest.mark.parametrize("a_layout,b_layout", [("mk", "kn"), ("km", "kn"), ("mk", "nk"), ("km", "nk")])
def test_every_operand_major(A, O, a_layout, b_layout):
    M, N, K = 300, 520, 200
    a, b = SI.contraction_bf16(7, M, N, K)
    ref = O.matmul(O.T(SI.bits(a), "bf16"), O.T(SI.bits(b), "bf16"), "f32").data
    mag = (a.double().abs() @ b.double().abs()).numpy()
    dA, dB = dev(_storage(a, a_layout)), dev(_storage(b, b_layout))
    Av, Bv = _views(A, dA, dB, M, N, K, a_layout, b_layout)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), torch.zeros((1,), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    _check(C.cpu().numpy(), ref, mag, K, "f32")


def test_batched_contraction_and_kept_dim(A, O):
    Bt, M, N, K = 5, 70, 130, 96
    g = SI.gen(5)
    a = SI.normal((Bt, M, K), 0, 0.1, g, torch.bfloat16)
    b = SI.normal((Bt, K, N), 0, 0.1, g, torch.bfloat16)
    dA, dB = dev(a), dev(b)
    Av, Bv = _views(A, dA, dB, M, N, K, batch=Bt)
    C = torch.empty((Bt, M, N, 1), dtype=torch.bfloat16, device="cuda")  # the (M,N,1) sink form
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), torch.zeros((1,), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    got = O.T(to_np(C.cpu()), "bf16").f64().reshape(Bt, M, N)
    for i in range(Bt):
        ref = O.matmul(O.T(SI.bits(a[i]), "bf16"), O.T(SI.bits(b[i]), "bf16"), "f32").data
        mag = (a[i].double().abs() @ b[i].double().abs()).numpy()
        _check(got[i], ref, mag, K, "bf16")


@pytest.mark.parametrize("M,N,K", [(64, 48, 32), (129, 131, 257), (1, 5, 3)])
def test_f32_contraction_simt(A, O, M, N, K):
    a, b = SI.contraction_f32(M * N + K, M, N, K)
    ref = O.matmul(O.T(a.numpy(), "f32"), O.T(b.numpy(), "f32"), "f32").data
    mag = (a.double().abs() @ b.double().abs()).numpy()
    dA, dB = dev(a), dev(b)
    Av, Bv = _views(A, dA, dB, M, N, K)
    C = torch.empty((M, N), device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), torch.zeros((1,), dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    _check(C.cpu().numpy(), ref, mag, K, "f32")


def test_tiny_graph_literal_shape(A, O):
    """The tiny graph's 64x32 @ 32x48 float32 contraction through the same call."""
    a, b = SI.tiny_graph(0)
    ref = O.matmul_literal(O.T(a.numpy(), "f32"), O.T(b.numpy(), "f32")).data.reshape(64, 48)
    dA, dB = dev(a), dev(b)
    Av, Bv = _views(A, dA, dB, 64, 48, 32)
    C = torch.empty((64, 48), device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), None)
    torch.cuda.synchronize()
    mag = (a.double().abs() @ b.double().abs()).numpy()
    _check(C.cpu().numpy(), ref, mag, 32, "f32")


def _sampled_full(A, O, a, b, out_dt, n_cells, seed):
    M, K = a.shape
    N = b.shape[1]
    dA, dB = dev(a), dev(b)
    Av, Bv = _views(A, dA, dB, M, N, K)
    C = torch.empty((M, N), dtype=storage_dtype(out_dt), device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    g = np.random.default_rng(seed)
    ii = g.integers(0, M, n_cells)
    jj = g.integers(0, N, n_cells)
    # include the corners and the last tile's edges
    ii = np.concatenate([ii, [0, M - 1, M - 1, 0]])
    jj = np.concatenate([jj, [0, N - 1, 0, N - 1]])
    dt = "bf16" if a.dtype == torch.bfloat16 else "f32"
    acc, mag = O.matmul_cells(O.T(SI.bits(a), dt), O.T(SI.bits(b), dt), ii, jj)
    got = O.T(to_np(C.cpu()), out_dt).f64()[ii, jj]
    _check(got, acc, mag, K, out_dt)
    return C


def test_full_size_bf16_sampled(A, O):
    a, b = SI.contraction_bf16(0)
    C = _sampled_full(A, O, a, b, "bf16", 3000, 1)
    # same bits twice
    dA, dB = dev(a), dev(b)
    Av, Bv = _views(A, dA, dB, 8192, 8192, 8192)
    C2 = torch.empty_like(C)
    A.psg_contract(dA, Av, dB, Bv, C2, A.view_of(C2), None)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))


def test_full_size_f32_sampled(A, O):
    a, b = SI.contraction_f32(0)
    _sampled_full(A, O, a, b, "f32", 2000, 2)


def _host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def _full_matrix(A, O, a, b, out_dt):
    """Every cell of the workload's product against the oracle's naive loop
    (float32 totals, k ascending), run on all the host's cores; the bound per
    cell is the one above, with sum |a b| from a float64 product of the
    magnitudes."""
    M, K = a.shape
    N = b.shape[1]
    dA, dB = dev(a), dev(b)
    Av, Bv = _views(A, dA, dB, M, N, K)
    C = torch.empty((M, N), dtype=storage_dtype(out_dt), device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = O.T(to_np(C.cpu()), out_dt).f64()
    del C, dA, dB
    dt = "bf16" if a.dtype == torch.bfloat16 else "f32"
    old = O.NTHREADS
    O.NTHREADS = _host_threads()
    try:
        ref = O.matmul_bt(O.T(SI.bits(a), dt), O.transpose(O.T(SI.bits(b), dt)), "f32").data
    finally:
        O.NTHREADS = old
    mag = np.abs(a.double().numpy()) @ np.abs(b.double().numpy())
    _check(got, ref, mag, K, out_dt)


def test_full_size_bf16_every_cell(A, O):
    """C4a at its full size (8192^3, bf16 in, bf16 out): all 67,108,864 cells."""
    a, b = SI.contraction_bf16(0)
    _full_matrix(A, O, a, b, "bf16")


def test_full_size_f32_every_cell(A, O):
    """C4b at its full size (4096^3 float32, 3xTF32 on the tensor cores): all
    16,777,216 cells."""
    a, b = SI.contraction_f32(0)
    _full_matrix(A, O, a, b, "f32")


def _f32_tc_case(A, O, M, N, K, a_layout="mk", b_layout="kn", out_dt="f32", seed=0):
    a, b = SI.contraction_f32(seed + M + 3 * N + 7 * K, M, N, K)
    ref = O.matmul(O.T(a.numpy(), "f32"), O.T(b.numpy(), "f32"), "f32").data
    mag = (a.double().abs() @ b.double().abs()).numpy()
    dA, dB = dev(_storage(a, a_layout)), dev(_storage(b, b_layout))
    Av, Bv = _views(A, dA, dB, M, N, K, a_layout, b_layout)
    C = torch.empty((M, N), dtype=storage_dtype(out_dt), device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check(O.T(to_np(C.cpu()), out_dt).f64(), ref, mag, K, out_dt)


@pytest.mark.parametrize("M,N,K", [(256, 128, 256), (300, 200, 512), (128, 384, 1000), (1, 130, 260)])
def test_f32_tensor_core_3xtf32(A, O, M, N, K):
    """float32 with K >= 256 and 16-byte aligned operands: the 3xTF32
    tensor-core kernel (ragged M, N and K tails), within the SUM bound."""
    _f32_tc_case(A, O, M, N, K)


@pytest.mark.parametrize("a_layout,b_layout", [("mk", "kn"), ("km", "kn"), ("mk", "nk"), ("km", "nk")])
def test_f32_tensor_core_every_operand_major(A, O, a_layout, b_layout):
    _f32_tc_case(A, O, 256, 192, 512, a_layout, b_layout)


def test_f32_tensor_core_bf16_output_and_batch(A, O):
    _f32_tc_case(A, O, 200, 256, 384, out_dt="bf16")
    B_, M, N, K = 3, 128, 128, 256
    g = SI.gen(77)
    a = SI.normal((B_, M, K), 0, 1, g)
    b = SI.normal((B_, K, N), 0, 1, g)
    dA, dB = dev(a), dev(b)
    Av, Bv = _views(A, dA, dB, M, N, K, batch=B_)
    C = torch.empty((B_, M, N), device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), None)
    torch.cuda.synchronize()
    got = C.cpu().numpy()
    for i in range(B_):
        ref = O.matmul(O.T(a[i].numpy(), "f32"), O.T(b[i].numpy(), "f32"), "f32").data
        mag = (a[i].double().abs() @ b[i].double().abs()).numpy()
        _check(got[i], ref, mag, K, "f32")


def test_f32_tensor_core_launch_query(A):
    q = A.psg_query_launch("contract_f32_tensor", A.make_view("f32", (4096, 4096)))
    assert q["block"] == 448 and q["smem"] > 190000 and 1 <= q["grid"] <= 152


@pytest.mark.parametrize("M,N,K,a_layout,b_layout,out_dt", [(256, 256, 128, "mk", "kn", "f32"),
                                                             (200, 300, 100, "km", "nk", "f16"),
                                                             (130, 70, 64, "mk", "nk", "bf16")])
def test_f16_contraction_tensor_cores(A, O, M, N, K, a_layout, b_layout, out_dt):
    """float16 operands (both f16: the tensor cores take one type for A and
    B) on the tcgen05 path, within the SUM bound plus the output rounding."""
    g = SI.gen(M + N + K)
    s = 1.0 / float(np.sqrt(K))
    a = SI.normal((M, K), 0.0, s, g).to(torch.float16)
    b = SI.normal((K, N), 0.0, s, g).to(torch.float16)
    ref = O.matmul(O.T(a.numpy(), "f16"), O.T(b.numpy(), "f16"), "f32").data
    mag = (a.double().abs() @ b.double().abs()).numpy()
    dA, dB = dev(_storage(a, a_layout)), dev(_storage(b, b_layout))
    Av, Bv = _views(A, dA, dB, M, N, K, a_layout, b_layout)
    C = torch.empty((M, N), dtype=storage_dtype(out_dt), device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), None)
    torch.cuda.synchronize()
    got = O.T(to_np(C.cpu()), out_dt).f64()
    tol = 2 * gamma(K - 1) * mag + 1e-30
    if out_dt == "bf16":
        tol = tol + 2.0 ** -7 * np.abs(ref)
    elif out_dt == "f16":
        tol = tol + 2.0 ** -10 * np.abs(ref) + 2.0 ** -24
    assert np.all(np.abs(got - ref) <= tol)


def test_f16_contraction_simt_unaligned(A, O):
    """Rows of odd length (not TMA-addressable): the FP32-pipe kernel."""
    M, N, K = 33, 17, 45
    g = SI.gen(3)
    a = SI.normal((M, K), 0.0, 1.0, g).to(torch.float16)
    b = SI.normal((K, N), 0.0, 1.0, g).to(torch.float16)
    ref = O.matmul(O.T(a.numpy(), "f16"), O.T(b.numpy(), "f16"), "f32").data
    mag = (a.double().abs() @ b.double().abs()).numpy()
    dA, dB = dev(a), dev(b)
    Av, Bv = _views(A, dA, dB, M, N, K)
    C = torch.empty((M, N), device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), None)
    torch.cuda.synchronize()
    assert np.all(np.abs(C.cpu().numpy().astype(np.float64) - ref) <= 2 * gamma(K - 1) * mag + 1e-30)


def _split_case(A, M, N, K, a_layout, b_layout, out_dt, batch, seed):
    g = SI.gen(seed)
    s = 1.0 / float(np.sqrt(K))
    shp_a, shp_b = ((batch, M, K), (batch, K, N)) if batch else ((M, K), (K, N))
    a = SI.normal(shp_a, 0.0, s, g, torch.bfloat16)
    b = SI.normal(shp_b, 0.0, s, g, torch.bfloat16)
    if batch:
        dA, dB = dev(a), dev(b)
    else:
        dA, dB = dev(_storage(a, a_layout)), dev(_storage(b, b_layout))
    Av, Bv = _views(A, dA, dB, M, N, K, a_layout, b_layout, batch=batch)
    C = torch.empty(((batch,) if batch else ()) + (M, N), dtype=storage_dtype(out_dt), device="cuda")
    return a, b, dA, dB, Av, Bv, C


@pytest.mark.parametrize("M,N,K,a_layout,b_layout,out_dt,batch", [
    (256, 512, 4096, "mk", "kn", "f32", None),      # 4 tiles, 8 splits of 8 K blocks
    (200, 300, 3000, "km", "nk", "bf16", None),     # ragged tiles and a short last split
    (130, 70, 1000, "mk", "nk", "f32", None),
    (128, 256, 2048, "mk", "kn", "bf16", 3)])       # batched: 3 tiles
def test_split_k_matches_oracle(A, O, M, N, K, a_layout, b_layout, out_dt, batch):
    """Few output tiles over a long K: psg_contract_ws splits K; the result
    stays within the SUM bound, and is the same bits on every call."""
    a, b, dA, dB, Av, Bv, C = _split_case(A, M, N, K, a_layout, b_layout, out_dt, batch, M + N + K)
    need = A.psg_contract_workspace(Av, Bv, A.view_of(C))
    assert need > 0
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    A.psg_contract_ws(dA, Av, dB, Bv, C, A.view_of(C), ws, need, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    first = C.clone()
    ws.fill_(0xFF)   # the partials are written before they are read
    A.psg_contract_ws(dA, Av, dB, Bv, C, A.view_of(C), ws, need, st)
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16 if C.element_size() == 2 else torch.int32),
                       C.view(torch.int16 if C.element_size() == 2 else torch.int32))
    got = O.T(to_np(C.cpu()), out_dt).f64()
    for i in range(batch or 1):
        ai, bi = (a[i], b[i]) if batch else (a, b)
        ref = O.matmul(O.T(SI.bits(ai), "bf16"), O.T(SI.bits(bi), "bf16"), "f32").data
        mag = (ai.double().abs() @ bi.double().abs()).numpy()
        _check(got[i] if batch else got, ref, mag, K, out_dt)


def test_split_k_short_workspace_runs_unsplit(A):
    """A workspace smaller than the query asks for: the unsplit kernel runs,
    bit for bit what psg_contract gives."""
    M, N, K = 256, 256, 2048
    a, b, dA, dB, Av, Bv, C = _split_case(A, M, N, K, "mk", "kn", "f32", None, 11)
    need = A.psg_contract_workspace(Av, Bv, A.view_of(C))
    assert need > 0
    ref = torch.empty_like(C)
    A.psg_contract(dA, Av, dB, Bv, ref, A.view_of(ref), None)
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    A.psg_contract_ws(dA, Av, dB, Bv, C, A.view_of(C), ws, need - 16, None)
    torch.cuda.synchronize()
    assert torch.equal(C.view(torch.int32), ref.view(torch.int32))


def test_split_k_not_used_for_many_tiles(A):
    """An output that already fills the GPU with tiles asks for no workspace."""
    M, N, K = 4096, 4096, 4096
    Av = A.make_view("bf16", [M, N, K], [K, 0, 1], 0, None, M * K)
    Bv = A.make_view("bf16", [M, N, K], [0, 1, N], 0, None, K * N)
    Cv = A.make_view("f32", [M, N], [N, 1], 0, None, M * N)
    assert A.psg_contract_workspace(Av, Bv, Cv) == 0


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("M,N,K,a_layout,b_layout,out_dt", [
    (300, 520, 200, "mk", "kn", "f32"), (300, 520, 200, "km", "kn", "bf16"),
    (300, 520, 200, "mk", "nk", "f32"), (300, 520, 200, "km", "nk", "bf16"),
    (257, 513, 1000, "mk", "kn", "bf16"),   # the second CTA of the last pair reads only zero fill
    (640, 256, 2048, "km", "nk", "f32")])
def test_pair_and_single_cta_kernels(A, O, monkeypatch, kernel, M, N, K, a_layout, b_layout, out_dt):
    """The two bf16 tensor-core kernels (one CTA a 128 x 256 tile; two CTAs a
    256 x 256 tile) on every operand major and ragged edges, each against the
    oracle, and the same bits from both."""
    monkeypatch.setenv("PSG_GEMM_KERNEL", kernel)
    a, b = SI.contraction_bf16(M * 3 + N + K, M, N, K)
    ref = O.matmul(O.T(SI.bits(a), "bf16"), O.T(SI.bits(b), "bf16"), "f32").data
    mag = (a.double().abs() @ b.double().abs()).numpy()
    dA, dB = dev(_storage(a, a_layout)), dev(_storage(b, b_layout))
    Av, Bv = _views(A, dA, dB, M, N, K, a_layout, b_layout)
    C = torch.empty((M, N), dtype=storage_dtype(out_dt), device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    A.psg_contract(dA, Av, dB, Bv, C, A.view_of(C), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check(O.T(to_np(C.cpu()), out_dt).f64(), ref, mag, K, out_dt)
    # the other kernel sums the same exact products in the same K order
    monkeypatch.setenv("PSG_GEMM_KERNEL", "single" if kernel == "pair" else "pair")
    C2 = torch.empty_like(C)
    A.psg_contract(dA, Av, dB, Bv, C2, A.view_of(C2), st)
    torch.cuda.synchronize()
    iv = torch.int16 if C.element_size() == 2 else torch.int32
    assert torch.equal(C.view(iv), C2.view(iv))


@pytest.mark.parametrize("kernel", ["pair", "single"])
def test_pair_and_single_cta_split_k(A, O, monkeypatch, kernel):
    monkeypatch.setenv("PSG_GEMM_KERNEL", kernel)
    M, N, K = 384, 512, 4096
    a, b, dA, dB, Av, Bv, C = _split_case(A, M, N, K, "km", "kn", "bf16", None, 77)
    need = A.psg_contract_workspace(Av, Bv, A.view_of(C))
    assert need > 0
    ws = torch.empty((need,), dtype=torch.uint8, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    A.psg_contract_ws(dA, Av, dB, Bv, C, A.view_of(C), ws, need, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = O.matmul(O.T(SI.bits(a), "bf16"), O.T(SI.bits(b), "bf16"), "f32").data
    mag = (a.double().abs() @ b.double().abs()).numpy()
    _check(O.T(to_np(C.cpu()), "bf16").f64(), ref, mag, K, "bf16")
