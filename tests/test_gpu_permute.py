"""GPU parity of psg_permute (bit-exact: only bytes move)."""
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


def _base(g, n, dt):
    if dt in ("i32", "i16", "i8"):
        return torch.randint(-100, 100, (n,), generator=g).to(storage_dtype(dt))
    return SI.normal((n,), 0, 1, g).to(storage_dtype(dt))


def _check(A, O, base, dt, shape, strides, offset, mask, perm):
    d = dev(base)
    iv = A.view_of(d, shape=shape, strides=strides, offset=offset, mask=mask)
    oshape = [shape[p] for p in perm]
    out = torch.empty(oshape, dtype=storage_dtype(dt), device="cuda")
    A.psg_permute(d, iv, perm, out, A.view_of(out))
    torch.cuda.synchronize()
    pshape = [shape[p] for p in perm]
    pstr = [strides[p] for p in perm]
    pmask = None if mask is None else [mask[p] for p in perm]
    ref = O.view(O.T(SI.bits(base), dt), pshape, pstr, offset, pmask).data
    assert np.array_equal(to_np(out.cpu()).view(np.uint8), ref.view(np.uint8))


@pytest.mark.parametrize("R,C", [(64, 64), (65, 63), (1, 300), (300, 1), (130, 70), (7, 1000)])
@pytest.mark.parametrize("dt", ["f32", "bf16", "i8", "f64"])
def test_transpose_shapes_and_dtypes(A, O, R, C, dt):
    g = SI.gen(R * 1000 + C)
    base = _base(g, R * C, dt)
    _check(A, O, base, dt, (R, C), (C, 1), 0, None, [1, 0])


@pytest.mark.parametrize("perm", [[0, 2, 1], [2, 1, 0], [1, 0, 2], [2, 0, 1], [1, 2, 0], [0, 1, 2]])
def test_rank3_permutes(A, O, perm):
    g = SI.gen(7)
    shape = (5, 67, 33)
    base = _base(g, 5 * 67 * 33, "f32")
    _check(A, O, base, "f32", shape, (67 * 33, 33, 1), 0, None, perm)


def test_permute_of_sliced_and_padded_views(A, O):
    g = SI.gen(8)
    base = _base(g, 50 * 40, "f32")
    # a slice with an offset
    _check(A, O, base, "f32", (30, 20), (40, 1), 45, None, [1, 0])
    # a padded read: zeros outside the mask
    _check(A, O, base, "f32", (52, 44), (40, 1), -(1 * 40 + 2), [(1, 51), (2, 42)], [1, 0])
    _check(A, O, base, "f64" if False else "f32", (52, 44), (40, 1), -(1 * 40 + 2),
           [(1, 51), (2, 42)], [0, 1])


def test_full_size_transpose(A, O):
    x = SI.transpose_input(0)
    d = dev(x)
    out = torch.empty((8192, 8192), device="cuda")
    A.psg_permute(d, A.view_of(d), [1, 0], out, A.view_of(out))
    torch.cuda.synchronize()
    assert torch.equal(out.cpu(), x.t().contiguous())
    # spot-check against the oracle's View read on a band of rows
    ref = O.view(O.T(x.numpy(), "f32"), (8192, 8192), (1, 8192)).data
    assert np.array_equal(out.cpu().numpy(), ref)


@pytest.mark.parametrize("shape,strides,offset,perm", [
    ((96, 200), (200, 1), 0, [1, 0]),            # ragged 64x64 tiles both ways
    ((260, 132), (132, 1), 0, [1, 0]),
    ((3, 100, 68), (6800, 68, 1), 0, [0, 2, 1]),  # one batch dim
    ((40, 52), (72, 1), 8, [1, 0]),               # a slice: row pitch 72, 32-byte offset
    ((2, 3, 64, 16), (4096, 1024, 16, 1), 0, [0, 1, 3, 2]),  # two batch dims that do not collapse
])
def test_tiled_transposes_ragged_batched_and_sliced(A, O, shape, strides, offset, perm):
    """The tiled transpose over ragged edge tiles, batch dims and a slice
    with an offset.  Bit-exact."""
    g = SI.gen(sum(shape) + offset)
    n = offset + sum((s - 1) * st for s, st in zip(shape, strides)) + 1
    base = _base(g, n, "f32")
    _check(A, O, base, "f32", shape, strides, offset, None, perm)
