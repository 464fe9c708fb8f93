"""GPU parity of the fused attention calls against the attention oracle.

Q, K, V are Views into one packed [B, T, 3, H, 64] bf16 buffer (the GPT
block's qkv layout).  Bars, from the roundings the kernels make (S and dP
are float32 sums of exact bf16 products; P and dS round to bf16 before the
second products; outputs round once to bf16), per cell:
  O:      |O - O*|   <= 2^-8 * sum_j P*_ij |V_jd|               + 2^-7 |O*|
  dV:     |dV - dV*| <= 2^-8 * sum_i P*_ij |dO_id|              + 2^-7 |dV*|
  dQ, dK: |dQ - dQ*| <= 2^-7 * scale * sum_j |P*_ij| (|dP*_ij| + |D*_i|) |K_jd| + 2^-7 |dQ*|
with * the oracle's float64 values; L within 1e-4 + 2^-16 |L*|.
"""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
from helpers import attention_bwd_bounds, attention_fwd_bounds
from oracle.attention import attention_bwd, attention_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from primitive_sm_graph_gb300 import _abi
    return _abi


def _heads(x):
    """[B, T, H, 64] -> [B*H, T, 64] float64."""
    B, T, H, d = x.shape
    return x.float().cpu().permute(0, 2, 1, 3).reshape(B * H, T, d).double().numpy()


def _setup(A, B, T, H, seed):
    g = SI.gen(seed)
    qkv = SI.normal((B, T, 3, H, 64), 0, 1, g, torch.bfloat16).cuda()
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    views = [A.view_of(qkv, shape=(B, T, H, 64), strides=q.stride(), offset=i * H * 64) for i in range(3)]
    return qkv, (q, k, v), views


def _fwd(A, B, T, H, causal, seed):
    qkv, (q, k, v), (qv, kv, vv) = _setup(A, B, T, H, seed)
    o = torch.empty((B, T, H, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    scale = 0.125
    A.psg_attention_fwd(qkv, qv, qkv, kv, qkv, vv, o, A.view_of(o), lse, scale, causal, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return qkv, (q, k, v), (qv, kv, vv), o, lse, scale


@pytest.mark.parametrize("B,T,H,causal", [(2, 256, 2, True), (1, 200, 3, True), (2, 64, 1, True),
                                          (1, 256, 2, False), (1, 130, 1, False)])
def test_attention_forward_matches_oracle(A, B, T, H, causal):
    qkv, (q, k, v), _, o, lse, scale = _fwd(A, B, T, H, causal, seed=T + H)
    Q, K, V = _heads(q), _heads(k), _heads(v)
    O_ref, L_ref = attention_fwd(Q, K, V, scale, causal)
    got = _heads(o)
    tol = attention_fwd_bounds(Q, K, V, O_ref, L_ref, scale, causal)
    bad = np.abs(got - O_ref) > tol
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:3])
    L = lse.cpu().numpy().reshape(B * H, T)
    assert np.all(np.abs(L - L_ref) <= 1e-4 + 2.0 ** -16 * np.abs(L_ref))


@pytest.mark.parametrize("B,T,H,causal", [(2, 256, 2, True), (1, 200, 3, True), (1, 256, 1, False)])
def test_attention_backward_matches_oracle(A, B, T, H, causal):
    qkv, (q, k, v), (qv, kv, vv), o, lse, scale = _fwd(A, B, T, H, causal, seed=7 * T + H)
    g = SI.gen(99)
    do = SI.normal((B, T, H, 64), 0, 1, g, torch.bfloat16).cuda()
    dqkv = torch.empty_like(qkv)
    dq, dk, dv = dqkv[:, :, 0], dqkv[:, :, 1], dqkv[:, :, 2]
    dviews = [A.view_of(dqkv, shape=(B, T, H, 64), strides=dq.stride(), offset=i * H * 64) for i in range(3)]
    delta = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    A.psg_attention_bwd(qkv, qv, qkv, kv, qkv, vv, o, A.view_of(o), do, A.view_of(do), lse, delta,
                        dqkv, dviews[0], dqkv, dviews[1], dqkv, dviews[2], scale, causal, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Q, K, V, O, dO = _heads(q), _heads(k), _heads(v), _heads(o), _heads(do)
    _, L_ref = attention_fwd(Q, K, V, scale, causal)
    refs = attention_bwd(Q, K, V, O, dO, L_ref, scale, causal)
    bounds = attention_bwd_bounds(Q, K, V, O, dO, L_ref, scale, causal, refs)
    for name, got, ref, tol in zip(("dq", "dk", "dv"), (dq, dk, dv), refs, bounds):
        g64 = _heads(got)
        bad = np.abs(g64 - ref) > tol
        assert not bad.any(), (name, int(bad.sum()), np.argwhere(bad)[:3])


def test_attention_rejects_unsupported_shapes(A):
    x = torch.empty((1, 300, 1, 64), dtype=torch.bfloat16, device="cuda")
    v = A.view_of(x)
    lse = torch.empty((300,), dtype=torch.float32, device="cuda")
    assert A.psg_attention_fwd(x, v, x, v, x, v, x, v, lse, 0.125, True, check=False) == A.E_UNSUPPORTED_LAYOUT
    y = torch.empty((1, 16, 1, 32), dtype=torch.bfloat16, device="cuda")
    w = A.view_of(y)
    assert A.psg_attention_fwd(y, w, y, w, y, w, y, w, lse, 0.125, True, check=False) == A.E_UNSUPPORTED_LAYOUT


@pytest.mark.parametrize("T,hd,causal", [(384, 64, True), (300, 64, False), (130, 32, True), (96, 128, False)])
def test_long_sequence_attention_composes(T, hd, causal):
    """Past one key block (T > 256), or at a head dim other than 64, the
    graph's attention is the composed form (score contraction, fused
    softmax, P V contraction); forward and the three gradients meet the same
    bars as the fused kernels."""
    from primitive_sm_graph_gb300 import graph as G
    B, H, scale = 1, 2, hd ** -0.5
    g = SI.gen(T + hd)
    qkv = SI.normal((B, T, 3, H, hd), 0, 1, g, torch.bfloat16)
    do = SI.normal((B, T, H, hd), 0, 1, g, torch.bfloat16)
    ex = G._executor()
    ex.log.clear()
    x = G.Tensor.from_torch(qkv.cuda(), requires_grad=True)
    o = x.attention_packed(scale, causal)
    o.backward(G.Tensor.from_torch(do.cuda()))
    o_t, dx = G.realize_all(o, x.grad)
    assert not any(e[0].startswith("attention") for e in ex.log) and any(e[0] == "contract" for e in ex.log)
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    Q, K, V, dO = _heads(q), _heads(k), _heads(v), _heads(do)
    O_ref, L_ref = attention_fwd(Q, K, V, scale, causal)
    refs = attention_bwd(Q, K, V, O_ref, dO, L_ref, scale, causal)
    bounds = attention_bwd_bounds(Q, K, V, O_ref, dO, L_ref, scale, causal, refs)
    dxc = dx.cpu()
    checks = [("o", o_t.cpu(), O_ref, attention_fwd_bounds(Q, K, V, O_ref, L_ref, scale, causal))]
    checks += [(n, dxc[:, :, i], r, t) for n, i, r, t in zip(("dq", "dk", "dv"), (0, 1, 2), refs, bounds)]
    for name, got, ref, tol in checks:
        g64 = _heads(got)
        bad = np.abs(g64 - ref) > tol
        assert not bad.any(), (name, int(bad.sum()), np.argwhere(bad)[:3])
