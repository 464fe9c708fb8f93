"""The two graph workloads of the hot path, written only with the lazy
Tensor API (so every kernel they launch comes from the scheduler):

* ``tiny_graph``: limn's README example at a small size, SUM(relu(A @ B)^2),
  with the matmul as broadcast MUL + SUM over k;
* ``gpt_block_loss``: a one-layer byte-level GPT block, forward and the
  graph its backward builds: embedding GATHER plus a learned position table,
  pre-norm RMSNorm, causal softmax attention in the composed form (the full
  T x T scores), a relu MLP, a final RMSNorm, an LM head and the mean
  next-token cross-entropy.  Weights and activations are bfloat16 at node
  boundaries; softmax, the logits and the loss are float32.
"""
from __future__ import annotations

import numpy as np
import torch

from .graph import Tensor, backward, realize_all

GPT_WEIGHTS = ("E", "P", "Wqkv", "Wo", "W1", "W2", "Wlm", "g1", "g2", "gf")


def tiny_graph(A: Tensor, B: Tensor) -> Tensor:
    """SUM(relu(A @ B) ** 2) as a scalar [1]."""
    c = A.matmul(B)
    return c.relu().square().reshape(1, -1).sum(-1, keepdim=False)


def causal_mask(T: int) -> torch.Tensor:
    """[T, T] float32: 1 where key j <= query i (data for WHERE)."""
    return torch.tril(torch.ones((T, T), dtype=torch.float32))


_STATIC = {}


def _static(key, make, device):
    """Shape-only tables (no data in them) kept on the device, so a recorded
    step (Replay) reads them from the same place every replay."""
    k = key + (str(device),)
    if k not in _STATIC:
        _STATIC[k] = make().to(device)
    return _STATIC[k]


def target_index(tok: Tensor, V: int, device) -> Tensor:
    """Flat indices r*V + tok[b, t+1] of the target logits, for positions
    t < T-1 (r = b*T + t), computed on the device as an int32 ADD of a
    shape-only table of r*V and the shifted token View."""
    Bn, T = tok.shape
    base = _static(("rowbase", Bn, T, V), lambda: torch.from_numpy(
        ((np.arange(Bn)[:, None] * T + np.arange(T - 1)[None, :]) * V).astype(np.int32)), device)
    nxt = tok.shrink(((0, Bn), (1, T)))
    return (Tensor.from_torch(base) + nxt).reshape(Bn * (T - 1))


def fused_attention_applies(T: int, D: int, H: int) -> bool:
    """The fused attention op covers head dim 64 at any sequence length;
    other head dims use the composed form."""
    return D // H == 64


def gpt_block_loss(tok: torch.Tensor, w: dict, H: int, eps: float = 1e-6,
                   pick: torch.Tensor | None = None, mask: torch.Tensor | None = None,
                   taps: dict | None = None, fused_attention: bool = True):
    """Mean next-token cross-entropy of the block on tokens [B, T] (int32,
    on the device).  w maps GPT_WEIGHTS to Tensors.  Returns the loss node
    (shape [1], float32).  If taps is a dict, the MLP pre-activation is put
    there as taps["mlp_pre"] (for inspection).  fused_attention picks the
    fused attention op where it applies (head dim 64, T <= 256) over the
    composed form."""
    Bn, T = tok.shape
    V, D = w["E"].shape
    hd = D // H
    BT = Bn * T
    tok_t = Tensor.from_torch(tok)
    pick_t = target_index(tok_t, V, tok.device) if pick is None else Tensor.from_torch(pick)
    if mask is None:
        mask = _static(("causal", T), lambda: causal_mask(T), tok.device)
    idx = Tensor.from_torch(tok.reshape(-1))
    h0 = (w["E"].gather(idx).reshape(Bn, T, D) + w["P"].reshape(1, T, D)).reshape(BT, D)

    # attention (pre-norm): the fused op, or composed from scores, causal
    # WHERE, softmax and the weighted sum
    n1 = h0.rmsnorm(w["g1"], eps)
    qkv = n1.matmul(w["Wqkv"]).reshape(Bn, T, 3, H, hd)

    def head(i):
        return qkv.shrink(((0, Bn), (0, T), (i, i + 1), (0, H), (0, hd))).reshape(Bn, T, H, hd)

    q, k, v = head(0), head(1), head(2)
    if fused_attention and fused_attention_applies(T, D, H):
        o = qkv.attention_packed(1.0 / np.sqrt(hd), causal=True).reshape(BT, D)
    else:
        q, k, v = (x.permute(0, 2, 1, 3) for x in (q, k, v))
        s = q.matmul(k.transpose(-1, -2)).cast("f32") * (1.0 / np.sqrt(hd))
        s = Tensor.from_torch(mask).where(s, float("-inf"))
        p = s.softmax(-1).cast("bf16")
        o = p.matmul(v).permute(0, 2, 1, 3).reshape(BT, D)
    h1 = h0 + o.matmul(w["Wo"])

    # MLP (pre-norm)
    n2 = h1.rmsnorm(w["g2"], eps)
    u = n2.matmul(w["W1"])
    if taps is not None:
        taps["mlp_pre"] = u
    h2 = h1 + u.relu().matmul(w["W2"])

    # head and loss
    logits = h2.rmsnorm(w["gf"], eps).matmul(w["Wlm"]).cast("f32")
    lsm = logits.log_softmax(-1)
    picked = lsm.reshape(BT * V, 1).gather(pick_t)
    n = pick_t.shape[0]
    return picked.reshape(1, n).sum(-1, keepdim=False) * (-1.0 / n)


def gpt_step(tok: torch.Tensor, weights: dict, H: int, pick=None, mask=None, taps=None, fused_attention=True):
    """One forward + backward pass: returns (loss, {name: grad}) as torch
    tensors.  weights maps GPT_WEIGHTS to device bf16 torch tensors.  With a
    taps dict, the tapped intermediates come back realized in it too."""
    w = {k: Tensor.from_torch(weights[k], requires_grad=True) for k in GPT_WEIGHTS}
    tp = {} if taps is not None else None
    loss = gpt_block_loss(tok, w, H, pick=pick, mask=mask, taps=tp, fused_attention=fused_attention)
    backward(loss)
    names = list(tp) if tp else []
    outs = realize_all(loss, *[w[k].grad for k in GPT_WEIGHTS], *[tp[k] for k in names])
    if taps is not None:
        taps.update(zip(names, outs[1 + len(GPT_WEIGHTS):]))
    return outs[0], dict(zip(GPT_WEIGHTS, outs[1:1 + len(GPT_WEIGHTS)]))


class AdamW:
    """Decoupled-weight-decay Adam over a fixed list of parameter tensors:
    float32 moments and the running beta powers live on the device, and a
    step is one psg_adamw_step call (one launch for all the tensors)."""

    def __init__(self, params, lr=3e-4, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1):
        from . import _abi as A
        self._A = A
        self.params = list(params)
        self.lr, self.betas, self.eps, self.wd = lr, betas, eps, weight_decay
        self.m = [torch.zeros(p.numel(), dtype=torch.float32, device=p.device) for p in self.params]
        self.v = [torch.zeros_like(m) for m in self.m]
        self.beta_pow = torch.ones(2, dtype=torch.float32, device=self.params[0].device)

    def step(self, grads):
        self._A.psg_adamw_step(self.params, [g.contiguous() for g in grads], self.m, self.v, self.lr, self.betas[0],
                               self.betas[1], self.eps, self.wd, self.beta_pow,
                               stream=torch.cuda.current_stream().cuda_stream)


def gpt_train_step(tok: torch.Tensor, weights: dict, H: int, opt: AdamW, fused_attention=True):
    """Forward, backward and one AdamW step of the block (weights updated in
    place); returns the loss tensor."""
    loss, grads = gpt_step(tok, weights, H, fused_attention=fused_attention)
    opt.step([grads[k] for k in GPT_WEIGHTS])
    return loss
