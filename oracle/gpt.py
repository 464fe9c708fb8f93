"""CPU oracle of the one-layer byte-level GPT block (forward and backward).

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).  It restates the block
from its definition with the oracle's primitive nodes; nothing here imports
or mirrors the product's graph code.  The reading of the block (none of the
pages fixes it; limn's examples/train_stories.py is only named):
  h0 = E[tok] + P[pos]            (GATHER, learned position table)
  h1 = h0 + attn(rmsnorm(h0)) Wo  (pre-norm, H heads, causal, scale hd^-1/2)
  h2 = h1 + relu(rmsnorm(h1) W1) W2
  logits = rmsnorm(h2) Wlm, then float32
  loss = mean over positions t < T-1 of -log_softmax(logits)[next token]
Storage dtype `act` (bfloat16 in the workload, float64 for the
finite-difference pin) at node boundaries, float32 compute inside a node and
float32 running totals (`acc`; float64 in the f64 pin).  A matmul's products
are exact (bfloat16 products fit float32) and its total rounds once into
`act`.  The softmax max is a constant of the gradient.

The backward is written out by hand, node by node, as the chain rule of the
forward above.  With attention="fused" the attention is the fused op instead
of its composition: exact softmax attention (oracle/attention.py, float64)
between bf16-rounded inputs and a bf16-rounded output, and likewise its
gradients.
"""
from __future__ import annotations

import numpy as np

from . import (T, add, cast, exp, expand_last, full, gather_rows, log, mul, neg, recip,
               reduce_max, reduce_sum, scatter_add_rows, sqrt, tensor, view, where, cmplt,
               matmul_bt)


def _tr(x: T) -> T:
    """Materialised transpose of a 2-D tensor (a permute View)."""
    r, c = x.shape
    return view(x, (c, r), (1, c))


def _mm(a: T, b: T, out: str) -> T:
    """a [M,K] @ b [K,N]: the naive MUL+SUM loop, total rounded into out."""
    return matmul_bt(a, _tr(b), out)


def _rows(x: T, n: int) -> T:
    """[D] -> [R, D] by a stride-0 View."""
    d = x.numel()
    return view(x, (n, d), (0, 1))


class GPTOracle:
    def __init__(self, tok: np.ndarray, w: dict, H: int, act="bf16", acc="f32", eps=1e-6,
                 relu_mask: np.ndarray | None = None, attention: str = "composed"):
        self.tok = np.asarray(tok, np.int32)
        self.B, self.T = self.tok.shape
        self.w = w                     # name -> oracle T (dtype act)
        self.H = H
        self.act, self.acc, self.eps = act, acc, eps
        self.V, self.D = w["E"].shape
        self.hd = self.D // H
        self.cache = {}  # intermediate values by name, for inspection
        # optional [B*T, F] bool: which MLP units count as active in the
        # backward.  relu is discontinuous at 0, so two runs whose
        # pre-activations differ by rounding can disagree on units at ~0;
        # handing the other run's mask in compares the rest like for like.
        self.relu_mask = relu_mask
        # "composed": scores, mask, softmax and the weighted sum as nodes;
        # "fused": the fused attention op, defined as exact (float64) softmax
        # attention between act-rounded inputs and an act-rounded output
        # (the forward and backward of oracle/attention.py)
        self.attention = attention

    # ---- pieces ---------------------------------------------------------------
    def rmsnorm_fwd(self, x: T, g: T):
        R, D = x.shape
        xf = cast(x, self.acc)
        ss = reduce_sum(mul(xf, xf))
        ms = mul(ss, full(ss.shape, 1.0 / D, self.acc))
        v = add(ms, full(ms.shape, self.eps, self.acc))
        q = sqrt(v)
        inv = recip(q)
        a = mul(xf, expand_last(inv, D))
        wf = _rows(cast(g, self.acc), R)
        y = cast(mul(a, wf), self.act)
        return y, (xf, q, inv, a, wf)

    def rmsnorm_bwd(self, gy: T, g: T, saved):
        xf, q, inv, a, wf = saved
        R, D = xf.shape
        g1 = cast(gy, self.acc)
        ga = mul(g1, wf)
        gw = cast(reduce_sum(_tr(mul(g1, a)), keepdim=False).reshape((D,)), self.act)
        gxf = mul(ga, expand_last(inv, D))
        ginv = reduce_sum(mul(ga, xf))
        gq = mul(neg(ginv), mul(inv, inv))
        gv = mul(mul(gq, full(gq.shape, 0.5, self.acc)), recip(q))
        gss = mul(gv, full(gv.shape, 1.0 / D, self.acc))
        gsq = expand_last(gss, D)
        gxf = add(gxf, add(mul(gsq, xf), mul(gsq, xf)))
        return cast(gxf, self.act), gw

    def softmax_fwd(self, x: T):
        R, N = x.shape
        m = reduce_max(x)
        e = exp(add(x, expand_last(neg(m), N)))
        s = reduce_sum(e)
        r = recip(s)
        y = mul(e, expand_last(r, N))
        return y, (e, r)

    def softmax_bwd(self, gy: T, saved):
        e, r = saved
        R, N = e.shape
        ge = mul(gy, expand_last(r, N))
        gr = reduce_sum(mul(gy, e))
        gs = mul(neg(gr), mul(r, r))
        ge = add(ge, expand_last(gs, N))
        return mul(ge, e)

    def _head(self, qkv: T, which: int, b: int, h: int) -> T:
        """[T, hd] slice of head h of q/k/v for sequence b (a View)."""
        D, hd, Tn = self.D, self.hd, self.T
        off = b * Tn * 3 * D + which * D + h * hd
        return view(qkv, (Tn, hd), (3 * D, 1), off)

    # ---- forward + backward ---------------------------------------------------------
    def run(self):
        act, acc = self.act, self.acc
        B, Tn, V, D, H, hd = self.B, self.T, self.V, self.D, self.H, self.hd
        BT = B * Tn
        w = self.w
        flat = self.tok.reshape(-1)
        emb, _ = gather_rows(w["E"], flat)
        pos = view(w["P"], (B, Tn, D), (0, D, 1)).reshape((BT, D))
        h0 = add(emb, pos)
        n1, s1 = self.rmsnorm_fwd(h0, w["g1"])
        qkv = _mm(n1, w["Wqkv"], act)                           # [BT, 3D]
        mask = np.tril(np.ones((Tn, Tn), np.float32))
        mk = T(mask, "f32") if acc == "f32" else T(mask.astype(np.float64), acc)
        scale = full((Tn, Tn), 1.0 / np.sqrt(hd), acc)
        ninf = full((Tn, Tn), -np.inf, acc)
        attn = np.zeros((B, Tn, H, hd), dtype=qkv.data.dtype)
        saved_h = {}
        if self.attention == "fused":
            from .attention import attention_fwd
            q5 = qkv.f64().reshape(B, Tn, 3, H, hd)
            heads = [np.ascontiguousarray(q5[:, :, i].transpose(0, 2, 1, 3)).reshape(B * H, Tn, hd)
                     for i in range(3)]
            O, Lse = attention_fwd(*heads, 1.0 / np.sqrt(hd), causal=True)
            o_act = cast(T(O.reshape(B, H, Tn, hd).transpose(0, 2, 1, 3).reshape(B * Tn, D).copy(), "f64"), act)
            saved_fused = (heads, O, Lse, o_act)
        for b in range(B if self.attention != "fused" else 0):
            for h in range(H):
                q = self._head(qkv, 0, b, h)
                k = self._head(qkv, 1, b, h)
                v = self._head(qkv, 2, b, h)
                sc = cast(_mm(q, _tr(k), act), acc)
                sc = mul(sc, scale)
                sm = where(mk, sc, ninf)
                p, sv = self.softmax_fwd(sm)
                pb = cast(p, act)
                o = _mm(pb, v, act)
                attn[b, :, h, :] = o.data
                saved_h[(b, h)] = (q, k, v, sv, pb)
        o2 = T(attn.reshape(BT, D), act) if self.attention != "fused" else o_act
        h1 = add(h0, _mm(o2, w["Wo"], act))
        n2, s2 = self.rmsnorm_fwd(h1, w["g2"])
        u = _mm(n2, w["W1"], act)
        zero = full(u.shape, 0.0, act)
        pos_u = cmplt(zero, u)
        f = where(pos_u, u, zero)
        h2 = add(h1, _mm(f, w["W2"], act))
        n3, s3 = self.rmsnorm_fwd(h2, w["gf"])
        logits = cast(_mm(n3, w["Wlm"], act), acc)             # [BT, V]
        self.cache.update(h0=h0, n1=n1, qkv=qkv, o2=o2, h1=h1, h2=h2, n3=n3, logits=logits)
        m = reduce_max(logits)
        sh = add(logits, expand_last(neg(m), V))
        e = exp(sh)
        s = reduce_sum(e)
        lse = log(s)
        lsm = add(sh, expand_last(neg(lse), V))
        rows = (np.arange(B)[:, None] * Tn + np.arange(Tn - 1)[None, :]).reshape(-1)
        tgt = self.tok[:, 1:].reshape(-1)
        pick = (rows * V + tgt).astype(np.int32)
        picked, _ = gather_rows(lsm.reshape((BT * V, 1)), pick)
        n = pick.size
        tot = reduce_sum(picked.reshape((1, n)), keepdim=False)
        loss = mul(tot, full(tot.shape, -1.0 / n, acc))

        # ---------------- backward ----------------
        grads = {}
        gtot = full((1,), -1.0 / n, acc)
        gpick = view(gtot, (n, 1), (0, 0))
        glsm_flat, _ = scatter_add_rows(full((BT * V, 1), 0.0, acc), pick, gpick)
        glsm = glsm_flat.reshape((BT, V))
        # lsm = sh + NEG(lse) expanded; lse = LOG(SUM(EXP(sh)))
        gnl = reduce_sum(glsm)
        gl = neg(gnl)
        gs = mul(gl, recip(s))
        gsh = add(glsm, mul(expand_last(gs, V), e))
        glogits = gsh                                           # the max is a constant
        gmm = cast(glogits, act)
        self.cache.update(glogits=glogits)
        gn3 = _mm(gmm, _tr(w["Wlm"]), act)
        grads["Wlm"] = _mm(_tr(n3), gmm, act)
        gh2, grads["gf"] = self.rmsnorm_bwd(gn3, w["gf"], s3)
        self.cache.update(gn3=gn3, gh2=gh2)
        # h2 = h1 + f W2
        gf = _mm(gh2, _tr(w["W2"]), act)
        grads["W2"] = _mm(_tr(f), gh2, act)
        if self.relu_mask is not None:
            pos_u = T(np.asarray(self.relu_mask, np.float64), "f64")
            pos_u = cast(pos_u, act)
        gu = where(pos_u, gf, zero)
        self.cache.update(gf=gf, gu=gu, n2=n2, u=u, f=f)
        gn2 = _mm(gu, _tr(w["W1"]), act)
        grads["W1"] = _mm(_tr(n2), gu, act)
        gh1n, grads["g2"] = self.rmsnorm_bwd(gn2, w["g2"], s2)
        gh1 = add(gh2, gh1n)
        # h1 = h0 + o2 Wo
        go2 = _mm(gh1, _tr(w["Wo"]), act)
        grads["Wo"] = _mm(_tr(o2), gh1, act)
        go = go2.data.reshape(B, Tn, H, hd)
        gqkv = np.zeros((BT, 3 * D), dtype=qkv.data.dtype)
        if self.attention == "fused":
            from .attention import attention_bwd
            heads, _, Lse, o_act = saved_fused
            ohead = o_act.f64().reshape(B, Tn, H, hd).transpose(0, 2, 1, 3).reshape(B * H, Tn, hd)
            dohead = go2.f64().reshape(B, Tn, H, hd).transpose(0, 2, 1, 3).reshape(B * H, Tn, hd)
            grads3 = attention_bwd(*heads, ohead, dohead, Lse, 1.0 / np.sqrt(hd), causal=True)
            g5 = np.zeros((B, Tn, 3, H, hd))
            for i in range(3):
                g5[:, :, i] = grads3[i].reshape(B, H, Tn, hd).transpose(0, 2, 1, 3)
            gqkv = cast(T(g5.reshape(BT, 3 * D), "f64"), act).data
        for b in range(B if self.attention != "fused" else 0):
            for h in range(H):
                q, k, v, sv, pb = saved_h[(b, h)]
                gpv = T(np.ascontiguousarray(go[b, :, h, :]), act)
                gpb = _mm(gpv, _tr(v), act)
                gv = _mm(_tr(pb), gpv, act)
                gsm = self.softmax_bwd(cast(gpb, acc), sv)
                gsc = mul(where(mk, gsm, full((Tn, Tn), 0.0, acc)), scale)
                gs_act = cast(gsc, act)
                gq = _mm(gs_act, k, act)
                gk = _mm(_tr(gs_act), q, act)
                r0 = b * Tn
                gqkv[r0:r0 + Tn, h * hd:(h + 1) * hd] = gq.data
                gqkv[r0:r0 + Tn, D + h * hd:D + (h + 1) * hd] = gk.data
                gqkv[r0:r0 + Tn, 2 * D + h * hd:2 * D + (h + 1) * hd] = gv.data
        gqkv = T(gqkv, act)
        gn1 = _mm(gqkv, _tr(w["Wqkv"]), act)
        grads["Wqkv"] = _mm(_tr(n1), gqkv, act)
        gh0n, grads["g1"] = self.rmsnorm_bwd(gn1, w["g1"], s1)
        gh0 = add(gh1, gh0n)
        # h0 = E[tok] + P[pos]
        grads["P"] = reduce_sum(_tr(gh0.reshape((B, Tn * D))).reshape((Tn * D, B)), keepdim=False) \
            .reshape((Tn, D))
        grads["E"], _ = scatter_add_rows(full((V, D), 0.0, act), flat, gh0)
        return loss, grads
