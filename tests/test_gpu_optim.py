"""GPU parity of psg_adamw_step: every operation is an IEEE float32 rounding
in the oracle's order (sqrt and division correctly rounded on both sides),
so parameters and moments must match the oracle bit for bit, step after
step, across more tensors than one launch takes."""
import numpy as np
import pytest
import torch

import seeded_inputs as SI
from helpers import storage_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from primitive_sm_graph_gb300 import _abi
    return _abi


@pytest.mark.parametrize("dt", ["bf16", "f32", "f16"])
def test_adamw_bit_exact_against_oracle(A, O, dt):
    g = SI.gen(len(dt))
    sizes = [int(s) for s in torch.randint(1, 3000, (37,), generator=g)] + [0, 5000]   # two launch groups
    tdt = storage_dtype(dt)
    params = [SI.normal((n,), 0, 1, g, tdt) for n in sizes]
    m = [np.zeros(n, np.float32) for n in sizes]
    v = [np.zeros(n, np.float32) for n in sizes]
    dp = [p.cuda() for p in params]
    dm = [torch.zeros(n, device="cuda") for n in sizes]
    dv = [torch.zeros(n, device="cuda") for n in sizes]
    bpow = torch.ones(2, device="cuda")
    ref = [O.T(SI.bits(p), dt) for p in params]
    lr, b1, b2, eps, wd = 3e-3, 0.9, 0.95, 1e-8, 0.1
    b1t = b2t = np.float32(1)
    for step in range(3):
        grads = [SI.normal((n,), 0, 1, g, tdt) for n in sizes]
        A.psg_adamw_step(dp, [x.cuda() for x in grads], dm, dv, lr, b1, b2, eps, wd, bpow)
        b1t, b2t = np.float32(b1t * np.float32(b1)), np.float32(b2t * np.float32(b2))
        for i in range(len(sizes)):
            ref[i], m[i], v[i] = O.adamw_step(ref[i], O.T(SI.bits(grads[i]), dt), m[i], v[i], lr, b1, b2, eps, wd,
                                              float(b1t), float(b2t))
    torch.cuda.synchronize()
    for i in range(len(sizes)):
        assert np.array_equal(SI.bits(dp[i]).view(np.uint8), ref[i].data.view(np.uint8)), (dt, i)
        assert np.array_equal(dm[i].cpu().numpy(), m[i]) and np.array_equal(dv[i].cpu().numpy(), v[i])
    assert np.array_equal(bpow.cpu().numpy(), np.array([b1t, b2t], np.float32))
