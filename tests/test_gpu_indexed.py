"""GPU parity of psg_gather / psg_scatter_add: bit-exact against the oracle
(gather moves bytes; scatter adds colliding rows in ascending n into a float32
total seeded with the destination and rounds once, so the result is unique)."""
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


def _vals(g, shape, dt):
    if dt.startswith("i"):
        return torch.randint(-1000, 1000, shape, generator=g).to(storage_dtype(dt))
    return SI.normal(shape, 0, 1, g).to(storage_dtype(dt))


def _status():
    return torch.zeros((1,), dtype=torch.int32, device="cuda")


@pytest.mark.parametrize("dt", ["f32", "bf16", "i8", "f64"])
@pytest.mark.parametrize("V,D,n", [(256, 512, 8192), (10, 7, 25), (3, 1, 100), (5, 33, 0), (1000, 24, 77)])
def test_gather_matches_oracle(A, O, dt, V, D, n):
    g = SI.gen(V + D + n)
    src = _vals(g, (V, D), dt)
    idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
    ds, di = dev(src), dev(idx)
    out = torch.empty((n, D), dtype=storage_dtype(dt), device="cuda")
    st = _status()
    A.psg_gather(ds, A.view_of(ds), di, n, out, A.view_of(out), st)
    torch.cuda.synchronize()
    ref, bad = O.gather_rows(O.T(SI.bits(src), dt), idx.numpy())
    assert bad == 0 and int(st.item()) == 0
    assert np.array_equal(to_np(out.cpu()).view(np.uint8), ref.data.view(np.uint8))


def test_gather_out_of_range_and_strided(A, O):
    g = SI.gen(2)
    src = _vals(g, (6, 40), "f32")
    ds = dev(src)
    idx = torch.tensor([0, 6, -1, 5, 2], dtype=torch.int32)
    out = torch.full((5, 40), 7.0, device="cuda")
    st = _status()
    A.psg_gather(ds, A.view_of(ds), dev(idx), 5, out, A.view_of(out), st)
    torch.cuda.synchronize()
    ref, bad = O.gather_rows(O.T(src.numpy(), "f32"), idx.numpy())
    assert bad == 2 and int(st.item()) == A.E_INDEX_OUT_OF_RANGE
    assert np.array_equal(out.cpu().numpy(), ref.data)
    # a column-strided source (every other column of an [6, 80] buffer)
    wide = _vals(g, (6, 80), "f32")
    dw = dev(wide)
    sv = A.view_of(dw, shape=(6, 40), strides=(80, 2))
    out2 = torch.empty((5, 40), device="cuda")
    idx2 = torch.tensor([5, 0, 0, 3, 1], dtype=torch.int32)
    A.psg_gather(dw, sv, dev(idx2), 5, out2, A.view_of(out2), _status())
    torch.cuda.synchronize()
    ref2, _ = O.gather_rows(O.view(O.T(wide.numpy(), "f32"), (6, 40), (80, 2)), idx2.numpy())
    assert np.array_equal(out2.cpu().numpy(), ref2.data)


def _scatter(A, dst, idx, upd):
    n = idx.numel()
    ws = torch.empty((max(1, A.psg_scatter_workspace(n)),), dtype=torch.uint8, device="cuda")
    st = _status()
    du = dev(upd)
    A.psg_scatter_add(dst, A.view_of(dst), dev(idx), n, du, A.view_of(du), ws, ws.numel(), st)
    torch.cuda.synchronize()
    return int(st.item())


@pytest.mark.parametrize("dt", ["f32", "bf16", "f16", "i32", "i16", "i8", "f64"])
@pytest.mark.parametrize("case", ["embedding_grad", "single_row", "permutation", "ragged", "large", "long_runs",
                                  "wide_small", "wide", "wide_max", "target_pick", "deep_keys", "one_row", "one"])
def test_scatter_add_matches_oracle(A, O, dt, case):
    g = SI.gen(sum(map(ord, dt + case)))
    if case == "embedding_grad":   # [8192, 512] into [256, 512], ~32 collisions per row
        V, D, n = 256, 512, 8192
        idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
    elif case == "single_row":     # every update lands on one row (collisions on a single row)
        V, D, n = 9, 17, 3000
        idx = torch.full((n,), 4, dtype=torch.int32)
    elif case == "permutation":
        V, D, n = 300, 5, 300
        idx = torch.randperm(V, generator=g).to(torch.int32)
    elif case == "ragged":
        V, D, n = 50, 3, 1234
        idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
    elif case == "large":          # past one sorting block: global bitonic steps
        V, D, n = 4000, 2, 20000
        idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
    elif case == "long_runs":      # runs of ~33,000 equal indices (run ends found 32 keys at a time)
        V, D, n = 3, 4, 100000
        idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
    elif case == "target_pick":    # the cross-entropy pick's gradient: sorted, distinct, one cell a row
        V, D, n = 2032 * 256, 1, 2032
        idx = (torch.arange(n, dtype=torch.int32) * 256 + torch.randint(0, 256, (n,), generator=g,
                                                                          dtype=torch.int32))
    elif case == "deep_keys":      # 23-bit destinations: six radix passes of the one-block sort
        V, D, n = 5_000_000, 2, 12000
        idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
    elif case == "one_row":        # V = 1: no key bits at all
        V, D, n = 1, 40, 777
        idx = torch.zeros((n,), dtype=torch.int32)
    elif case == "one":
        V, D, n = 7, 9, 1
        idx = torch.tensor([3], dtype=torch.int32)
    else:                          # many destination rows: the one-block sort (1, 16 keys a thread)
        V, D, n = {"wide_small": (50000, 3, 700), "wide": (100000, 2, 9000), "wide_max": (60000, 2, 16384)}[case]
        idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
    dst0 = _vals(g, (V, D), dt)
    upd = _vals(g, (n, D), dt)
    dst = dev(dst0)
    assert _scatter(A, dst, idx, upd) == 0
    ref, bad = O.scatter_add_rows(O.T(SI.bits(dst0), dt), idx.numpy(), O.T(SI.bits(upd), dt))
    assert bad == 0
    got = to_np(dst.cpu())
    assert np.array_equal(got.view(np.uint8), ref.data.view(np.uint8)), \
        np.argwhere(got != ref.data)[:5]
    # same bits on a second run from the same start
    dst2 = dev(dst0)
    _scatter(A, dst2, idx, upd)
    assert np.array_equal(to_np(dst2.cpu()).view(np.uint8), got.view(np.uint8))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_scatter_padded_update_rows(A, O, dt):
    """Update rows that are a column slice of wider rows: 16-byte vectors
    for the full segments, single cells for the ragged last one."""
    g = SI.gen(21)
    V, D, W, n = 40, 19, 24, 3000
    idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
    dst0 = _vals(g, (V, D), dt)
    wide = _vals(g, (n, W), dt)
    dst = dev(dst0)
    du = dev(wide)
    uv = A.view_of(du, shape=(n, D), strides=(W, 1))
    ws = torch.empty((A.psg_scatter_workspace(n),), dtype=torch.uint8, device="cuda")
    st = _status()
    A.psg_scatter_add(dst, A.view_of(dst), dev(idx), n, du, uv, ws, ws.numel(), st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, _ = O.scatter_add_rows(O.T(SI.bits(dst0), dt), idx.numpy(), O.T(SI.bits(wide[:, :D].contiguous()), dt))
    assert np.array_equal(to_np(dst.cpu()).view(np.uint8), ref.data.view(np.uint8))


def test_scatter_bad_indices_power_of_two_rows(A, O):
    """Out-of-range indices equal to V (= 2^8) and negative ones among valid
    rows: they sort after row 255 and are skipped; the rest is exact."""
    g = SI.gen(22)
    V, D, n = 256, 8, 5000
    idx = torch.randint(0, V, (n,), generator=g, dtype=torch.int32)
    idx[::97] = V
    idx[5::131] = -1
    dst0 = _vals(g, (V, D), "f32")
    upd = _vals(g, (n, D), "f32")
    dst = dev(dst0)
    assert _scatter(A, dst, idx, upd) == A.E_INDEX_OUT_OF_RANGE
    ref, bad = O.scatter_add_rows(O.T(dst0.numpy(), "f32"), idx.numpy(), O.T(upd.numpy(), "f32"))
    assert bad > 0
    assert np.array_equal(dst.cpu().numpy(), ref.data)


def test_scatter_bad_indices_are_skipped(A, O):
    g = SI.gen(4)
    dst0 = _vals(g, (5, 3), "f32")
    upd = _vals(g, (6, 3), "f32")
    idx = torch.tensor([0, 5, -2, 4, 0, 9], dtype=torch.int32)
    dst = dev(dst0)
    assert _scatter(A, dst, idx, upd) == A.E_INDEX_OUT_OF_RANGE
    ref, bad = O.scatter_add_rows(O.T(dst0.numpy(), "f32"), idx.numpy(), O.T(upd.numpy(), "f32"))
    assert bad == 3
    assert np.array_equal(dst.cpu().numpy(), ref.data)


