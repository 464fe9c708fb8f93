"""psg_scatter_add_static: the scatter-add for callers that cannot allocate
device memory (its sort keys live in a fixed array inside the library, so it
takes no workspace).  Checked through the C ABI against psg_scatter_add, which
uses a caller-provided workspace: the two must give the same bits, on two
calls in a row (the second call reuses the array the first one left behind).
Collected last on purpose: it is independent of every other test, and a run
that stops at the first failure has run all the others before it."""
import numpy as np
import pytest
import torch

import seeded_inputs as SI

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    from primitive_sm_graph_gb300 import _abi
    return _abi


def _status():
    return torch.zeros((1,), dtype=torch.int32, device="cuda")


def _with_workspace(A, dst, idx, upd):
    n = idx.numel()
    ws = torch.empty((A.psg_scatter_workspace(n),), dtype=torch.uint8, device="cuda")
    st = _status()
    A.psg_scatter_add(dst, A.view_of(dst), idx, n, upd, A.view_of(upd), ws, ws.numel(), st)
    torch.cuda.synchronize()
    return int(st.item())


def _static(A, dst, idx, upd):
    st = _status()
    A.psg_scatter_add_static(dst, A.view_of(dst), idx, idx.numel(), upd, A.view_of(upd), st)
    torch.cuda.synchronize()
    return int(st.item())


@pytest.mark.parametrize("dt,V,D,n", [(torch.float32, 256, 512, 8192), (torch.bfloat16, 37, 9, 20000)])
def test_static_scratch_matches_workspace_call_twice(A, dt, V, D, n):
    g = SI.gen(V + n)
    dst0 = SI.normal((V, D), 0, 1, g).to(dt).cuda()
    idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32).cuda()
    upd = SI.normal((n, D), 0, 1, g).to(dt).cuda()
    ref = dst0.clone()
    assert _with_workspace(A, ref, idx, upd) == 0
    for _ in range(2):  # the second call runs over the keys the first left behind
        out = dst0.clone()
        assert _static(A, out, idx, upd) == 0
        assert torch.equal(out.view(torch.int16 if dt == torch.bfloat16 else torch.int32),
                           ref.view(torch.int16 if dt == torch.bfloat16 else torch.int32))


def test_static_scratch_limit_is_refused(A):
    n = A.SCATTER_STATIC_MAX_N + 1
    fake = 4096
    st = A.psg_scatter_add_static(fake, A.make_view("f32", (4, 1)), fake, n, fake,
                                  A.make_view("f32", (n, 1)), fake, check=False)
    assert st == A.E_WORKSPACE
    # a smaller call after the refusal still works
    dst = torch.zeros((3, 2), device="cuda")
    idx = torch.tensor([2, 0, 2], dtype=torch.int32, device="cuda")
    upd = torch.ones((3, 2), device="cuda")
    assert _static(A, dst, idx, upd) == 0
    assert np.array_equal(dst.cpu().numpy(), [[1, 1], [0, 0], [2, 2]])
