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
    lse = torch.empty((16,), dtype=torch.float32, device="cuda")
    y = torch.empty((1, 16, 1, 32), dtype=torch.bfloat16, device="cuda")
    w = A.view_of(y)
    assert A.psg_attention_fwd(y, w, y, w, y, w, y, w, lse, 0.125, True, check=False) == A.E_UNSUPPORTED_LAYOUT


def _key_mask(B, T, seed, pad=True):
    """[B, T] int8: batch b's last keys masked (a padded batch of
    sequences of different lengths) plus a scattering of masked keys."""
    g = SI.gen(seed)
    m = (torch.rand((B, T), generator=g) > 0.15).to(torch.int8)
    if pad:
        for b in range(B):
            m[b, T - (17 * (b + 1)) % (T // 2):] = 0
    return m


def _check_fwd(q, k, v, o, lse, scale, causal, km=None):
    Q, K, V = _heads(q), _heads(k), _heads(v)
    B, T, H, _ = q.shape
    kmh = None if km is None else np.repeat(km.numpy(), H, axis=0)
    O_ref, L_ref = attention_fwd(Q, K, V, scale, causal, key_mask=kmh)
    tol = attention_fwd_bounds(Q, K, V, O_ref, L_ref, scale, causal, key_mask=kmh)
    bad = np.abs(_heads(o) - O_ref) > tol
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:3])
    L = lse.cpu().numpy().reshape(B * H, T).astype(np.float64)
    with np.errstate(invalid="ignore"):
        okl = (np.abs(L - L_ref) <= 1e-4 + 2.0 ** -16 * np.abs(L_ref)) | (L == L_ref)
    assert okl.all(), np.argwhere(~okl)[:3]
    return Q, K, V, L_ref, kmh


@pytest.mark.parametrize("B,T,H,causal,masked", [(1, 512, 2, True, False), (2, 1000, 1, False, False),
                                                 (1, 300, 2, True, True), (2, 640, 1, False, True),
                                                 (1, 200, 2, True, True), (1, 256, 1, False, True)])
def test_attention_long_sequences_and_key_mask(A, B, T, H, causal, masked):
    """Past one key block (T > 256) the forward walks 128-key blocks with a
    running max and sum (rescaling the partial output), and the backward
    streams the other operand's tiles through a two-slot ring; a per-key
    mask (padded sequences) composes with causal at every length.  Forward,
    L and all three gradients against the float64 oracle at the bars above."""
    qkv, (q, k, v), (qv, kv, vv) = _setup(A, B, T, H, seed=T + 3 * H)
    km = _key_mask(B, T, T) if masked else None
    dkm = km.cuda() if masked else None
    scale = 0.125
    o = torch.empty((B, T, H, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    st = torch.zeros((1,), dtype=torch.int32, device="cuda")
    A.psg_attention_fwd(qkv, qv, qkv, kv, qkv, vv, o, A.view_of(o), lse, scale, causal, st, key_mask=dkm)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    Q, K, V, _, kmh = _check_fwd(q, k, v, o, lse, scale, causal, km)
    g = SI.gen(T + 1)
    do = SI.normal((B, T, H, 64), 0, 1, g, torch.bfloat16).cuda()
    dqkv = torch.empty_like(qkv)
    dq, dk, dv = dqkv[:, :, 0], dqkv[:, :, 1], dqkv[:, :, 2]
    dviews = [A.view_of(dqkv, shape=(B, T, H, 64), strides=dq.stride(), offset=i * H * 64) for i in range(3)]
    delta = torch.empty((B, H, T), dtype=torch.float32, device="cuda")
    A.psg_attention_bwd(qkv, qv, qkv, kv, qkv, vv, o, A.view_of(o), do, A.view_of(do), lse, delta,
                        dqkv, dviews[0], dqkv, dviews[1], dqkv, dviews[2], scale, causal, st, key_mask=dkm)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O, dO = _heads(o), _heads(do)
    L = lse.cpu().numpy().reshape(B * H, T).astype(np.float64)
    refs = attention_bwd(Q, K, V, O, dO, L, scale, causal, key_mask=kmh)
    bounds = attention_bwd_bounds(Q, K, V, O, dO, L, scale, causal, refs, key_mask=kmh)
    for name, got, ref, tol in zip(("dq", "dk", "dv"), (dq, dk, dv), refs, bounds):
        bad = np.abs(_heads(got) - ref) > tol
        assert not bad.any(), (name, int(bad.sum()), np.argwhere(bad)[:3])


@pytest.mark.parametrize("T,hd,causal", [(384, 64, True), (300, 64, False), (130, 32, True), (96, 128, False)])
def test_graph_attention_at_any_length(T, hd, causal):
    """The graph's attention op: at head dim 64 the fused kernels at any
    length (one key block, or the running softmax over many); at other head
    dims the composed form (score contraction, fused softmax, P V
    contraction).  Forward and the three gradients meet the fused kernels'
    bars either way."""
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
    fused = any(e[0].startswith("attention") for e in ex.log)
    assert fused == (hd == 64), ex.log
    assert fused or any(e[0] == "contract" for e in ex.log)
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    Q, K, V, dO = _heads(q), _heads(k), _heads(v), _heads(do)
    O_ref, L_ref = attention_fwd(Q, K, V, scale, causal)
    refs = attention_bwd(Q, K, V, O_ref, dO, L_ref, scale, causal)
    tol_o = attention_fwd_bounds(Q, K, V, O_ref, L_ref, scale, causal)
    # the fused backward forms D from the forward's bf16 O (within tol_o)
    bounds = attention_bwd_bounds(Q, K, V, O_ref, dO, L_ref, scale, causal, refs, o_err=tol_o if fused else None)
    dxc = dx.cpu()
    checks = [("o", o_t.cpu(), O_ref, tol_o)]
    checks += [(n, dxc[:, :, i], r, t) for n, i, r, t in zip(("dq", "dk", "dv"), (0, 1, 2), refs, bounds)]
    for name, got, ref, tol in checks:
        g64 = _heads(got)
        bad = np.abs(g64 - ref) > tol
        assert not bad.any(), (name, int(bad.sum()), np.argwhere(bad)[:3])


def test_graph_attention_with_key_mask(A):
    """Tensor.attention with a key mask (int8 [B, T]) over many key blocks:
    the fused forward and backward calls, against the float64 oracle."""
    from primitive_sm_graph_gb300 import graph as G
    B, T, H, scale = 2, 320, 2, 0.125
    g = SI.gen(77)
    x = [SI.normal((B, T, H, 64), 0, 1, g, torch.bfloat16) for _ in range(4)]
    km = _key_mask(B, T, 78)
    ex = G._executor()
    ex.log.clear()
    q, k, v = (G.Tensor.from_torch(t.cuda(), requires_grad=True) for t in x[:3])
    o = q.attention(k, v, scale, causal=True, key_mask=G.Tensor.from_torch(km.cuda()))
    o.backward(G.Tensor.from_torch(x[3].cuda()))
    out, gq, gk, gv = G.realize_all(o, q.grad, k.grad, v.grad)
    kinds = [e[0] for e in ex.log]
    assert kinds.count("attention") == 1 and kinds.count("attention_bwd") == 1, kinds
    Q, K, V, dO = (_heads(t) for t in x)
    kmh = np.repeat(km.numpy(), H, axis=0)
    O_ref, L_ref = attention_fwd(Q, K, V, scale, True, key_mask=kmh)
    bad = np.abs(_heads(out) - O_ref) > attention_fwd_bounds(Q, K, V, O_ref, L_ref, scale, True, key_mask=kmh)
    assert not bad.any(), int(bad.sum())
    refs = attention_bwd(Q, K, V, _heads(out), dO, L_ref, scale, True, key_mask=kmh)
    bounds = attention_bwd_bounds(Q, K, V, _heads(out), dO, L_ref, scale, True, refs, key_mask=kmh)
    for name, got, ref, tol in zip(("dq", "dk", "dv"), (gq, gk, gv), refs, bounds):
        bad = np.abs(_heads(got) - ref) > tol
        assert not bad.any(), (name, int(bad.sum()))
