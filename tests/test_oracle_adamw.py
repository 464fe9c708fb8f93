"""Pins of the oracle's AdamW step (CPU): torch.optim.AdamW as the library
routine over several steps, and the closed form of a first step."""
import numpy as np
import torch


def test_adamw_matches_torch_adamw_over_steps(O):
    g = torch.Generator().manual_seed(0)
    p0 = torch.randn(2000, generator=g)
    grads = [torch.randn(2000, generator=g) for _ in range(4)]
    pt = p0.clone().requires_grad_(True)
    opt = torch.optim.AdamW([pt], lr=1e-2, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.1)
    P = O.T(p0.numpy().copy(), "f32")
    m = np.zeros(2000, np.float32)
    v = np.zeros(2000, np.float32)
    b1t, b2t = np.float32(1), np.float32(1)
    for gr in grads:
        pt.grad = gr.clone()
        opt.step()
        b1t, b2t = np.float32(b1t * np.float32(0.9)), np.float32(b2t * np.float32(0.999))
        P, m, v = O.adamw_step(P, O.T(gr.numpy(), "f32"), m, v, 1e-2, 0.9, 0.999, 1e-8, 0.1, float(b1t), float(b2t))
    ref = pt.detach().numpy().astype(np.float64)
    assert np.all(np.abs(P.data - ref) <= 2.0 ** -20 * (1.0 + np.abs(ref)))


def test_adamw_first_step_closed_form(O):
    """From m = v = 0, one step moves each parameter by lr * g / (|g| + eps)
    after the decay: the sign step of Adam."""
    g = np.array([0.5, -2.0, 1e-3, -1e-6, 3.0], np.float32)
    p = np.array([1.0, -1.0, 0.25, 2.0, 0.0], np.float32)
    lr, wd = 0.01, 0.05
    P, m, v = O.adamw_step(O.T(p.copy(), "f32"), O.T(g, "f32"), np.zeros(5, np.float32), np.zeros(5, np.float32),
                           lr, 0.9, 0.999, 1e-8, wd, 0.9, 0.999)
    expect = p.astype(np.float64) * (1 - lr * wd) - lr * g / (np.abs(g) + 1e-8)
    assert np.allclose(P.data, expect, rtol=1e-5, atol=1e-7)
    # the coefficients are formed in float32: 1 - 0.9f, 1 - 0.999f
    c1 = np.float64(np.float32(1) - np.float32(0.9))
    c2 = np.float64(np.float32(1) - np.float32(0.999))
    assert np.allclose(m, c1 * g, rtol=1e-6) and np.allclose(v, c2 * g.astype(np.float64) ** 2, rtol=1e-6)
