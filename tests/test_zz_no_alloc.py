"""psg_scatter_add_static: the scatter-add for callers that cannot allocate
device memory (its sort keys live in a fixed array inside the library, so it
takes no workspace).  Checked through the C ABI against psg_scatter_add, which
uses a caller-provided workspace, and against the oracle's serial loop: all
three must give the same bits, on two calls in a row (the second call reuses
the array the first one left behind).  The cases reach each of the library's
scatter paths: few destination rows (owner scan), a planned radix order
(n <= 16384 with many destination rows), the bitonic key sort, and the sort
at the array's full capacity (n = PSG_SCATTER_STATIC_MAX_N).
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


def _bits(t):
    return t.view(torch.int16 if t.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("dt,V,D,n", [
    (torch.float32, 256, 512, 8192),        # few destination rows: the owner scan
    (torch.float32, 8192, 64, 4096),        # many destination rows, n <= 16384: the planned radix order
    (torch.bfloat16, 37, 9, 20000),         # a longer list: the bitonic key sort
    (torch.float32, 1024, 4, 1 << 20),      # the key array at its full capacity
])
def test_static_scratch_matches_workspace_call_and_oracle_twice(A, O, dt, V, D, n):
    g = SI.gen(V + n)
    dst0 = SI.normal((V, D), 0, 1, g).to(dt)
    idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
    upd = SI.normal((n, D), 0, 1, g).to(dt)
    name = "bf16" if dt == torch.bfloat16 else "f32"
    want, bad = O.scatter_add_rows(O.T(SI.bits(dst0), name), idx.numpy(), O.T(SI.bits(upd), name))
    assert bad == 0
    d_dst0, d_idx, d_upd = dst0.cuda(), idx.cuda(), upd.cuda()
    ref = d_dst0.clone()
    assert _with_workspace(A, ref, d_idx, d_upd) == 0
    assert np.array_equal(SI.bits(ref.cpu()), want.data)
    for _ in range(2):  # the second call runs over the keys the first left behind
        out = d_dst0.clone()
        assert _static(A, out, d_idx, d_upd) == 0
        assert torch.equal(_bits(out), _bits(ref))
        assert np.array_equal(SI.bits(out.cpu()), want.data)


def test_static_scratch_limit_is_refused(A):
    n = A.SCATTER_STATIC_MAX_N + 1
    dst = torch.zeros((4, 1), device="cuda")
    idx = torch.zeros((n,), dtype=torch.int32, device="cuda")
    upd = torch.ones((n, 1), device="cuda")
    st_word = _status()
    st = A.psg_scatter_add_static(dst, A.view_of(dst), idx, n, upd, A.view_of(upd), st_word, check=False)
    assert st == A.E_WORKSPACE
    torch.cuda.synchronize()
    assert int(st_word.item()) == 0 and not dst.any()  # nothing was launched
    # a smaller call after the refusal still works
    dst = torch.zeros((3, 2), device="cuda")
    idx = torch.tensor([2, 0, 2], dtype=torch.int32, device="cuda")
    upd = torch.ones((3, 2), device="cuda")
    assert _static(A, dst, idx, upd) == 0
    assert np.array_equal(dst.cpu().numpy(), [[1, 1], [0, 0], [2, 2]])
