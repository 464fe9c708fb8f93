"""The plan cache's marshalled replay, on the CPU with the C calls faked.

A repeated eager step replays its recorded library calls with their ctypes
arguments kept and only the buffer addresses and the stream rewritten
(graph._Plan).  This checks, with no GPU, that a replay makes the same C
calls as a schedule built afresh for the same inputs: the same functions in
the same order, every non-address argument identical (node arrays, Views,
sizes, scalars compared by value), and every address naming the same
buffer: an input leaf is the new input's address, a buffer the schedule
allocates is a fresh allocation used at the same places.
"""
import ctypes

import pytest
import torch

from primitive_sm_graph_gb300 import _abi as A
from primitive_sm_graph_gb300 import graph as G
from primitive_sm_graph_gb300.workloads import tiny_graph


class _FakeLib:
    """Stands in for libpsg: every launch call succeeds and is logged with
    its arguments (struct and array arguments copied by value); each call
    carries the real function's declared argument types."""

    def __init__(self, real):
        self.log, self.real = [], real

    def __getattr__(self, name):
        def call(*cargs):
            self.log.append((name, [_snap(a) for a in cargs]))
            return 0
        call.argtypes = getattr(self.real, name).argtypes
        return call


def _snap(a):
    if isinstance(a, ctypes.Array):
        if a._type_ is ctypes.c_void_p:
            return ("ptrs", tuple(int(x or 0) for x in a))
        if a._type_ is A.psg_reduce_stage:  # by value: each stage's op and its nodes
            return ("stages", tuple((st.op, st.n_nodes, bytes(memoryview(
                (A.psg_node * st.n_nodes).from_address(ctypes.addressof(st.prologue.contents))))) for st in a))
        return ("bytes", bytes(memoryview(a)))
    obj = getattr(a, "_obj", None)
    if obj is not None:  # byref(struct)
        if isinstance(obj, A.psg_epilogue):
            return ("epi", obj.n_nodes, obj.n_in, tuple(int(obj.in_[j] or 0) for j in range(obj.n_in)))
        return ("struct", bytes(memoryview(obj)))
    if isinstance(a, ctypes._Pointer):
        return ("ptr", ctypes.cast(a, ctypes.c_void_p).value)
    return a


@pytest.fixture
def cpu_graph(monkeypatch):
    fake = _FakeLib(A.lib)
    monkeypatch.setattr(A, "lib", fake)
    monkeypatch.setattr(A, "psg_contract_workspace", lambda *a: 0)
    status = torch.zeros((1,), dtype=torch.int32)
    monkeypatch.setattr(G.Executor, "_s", lambda self: 0)
    monkeypatch.setattr(G.Executor, "_status", lambda self: status)

    def _new(self, shape, dtype):
        t = torch.empty(tuple(shape), dtype=G.torch_dtype(dtype))
        if self.rec is not None:
            self.rec.alloc(t, (tuple(shape), t.dtype))
        return t

    def _ws(self, n):
        t = torch.empty((max(1, int(n)),), dtype=torch.uint8)
        if self.rec is not None:
            self.rec.alloc(t, ((max(1, int(n)),), torch.uint8))
        return t
    monkeypatch.setattr(G.Executor, "_new", _new)
    monkeypatch.setattr(G.Executor, "_workspace", _ws)
    monkeypatch.setattr(G, "_PLANS", {})
    monkeypatch.setattr(G, "_EXEC", None)
    return fake, status


def _canon(log, leaves, status, real):
    """The log with the addresses (the void* arguments, by the real
    functions' declared types, and pointer arrays) named: leaf k, the status
    word, or the j-th distinct other address in order of first use."""
    names = {t.data_ptr(): "leaf%d" % k for k, t in enumerate(leaves)}
    names[status.data_ptr()] = "status"
    seen = {}

    def name(v):
        if not v:
            return v
        if v in names:
            return names[v]
        return seen.setdefault(v, "tmp%d" % len(seen))
    out = []
    for fn, args in log:
        types = getattr(real, fn).argtypes
        row = []
        for a, t in zip(args, types):
            if isinstance(a, tuple) and a and a[0] == "ptrs":
                row.append(("ptrs",) + tuple(name(x) for x in a[1]))
            elif isinstance(a, tuple) and a and a[0] == "epi":
                row.append(a[:3] + tuple(name(x) for x in a[3]))
            elif t is ctypes.c_void_p:
                row.append(name(a))
            else:
                row.append(a)
        out.append((fn, row))
    return out


def _run(x, y):
    return tiny_graph(G.Tensor.from_torch(x), G.Tensor.from_torch(y)).realize()


def test_replay_makes_the_calls_of_a_fresh_schedule(cpu_graph):
    fake, status = cpu_graph
    g = torch.Generator().manual_seed(3)
    x0, y0 = torch.randn((64, 32), generator=g), torch.randn((32, 48), generator=g)
    _run(x0, y0)                       # records the plan
    assert len(G._PLANS) == 1
    plan = next(iter(G._PLANS.values()))
    assert plan.fast and all(f is not None for f in plan.fast)

    x1, y1 = torch.randn((64, 32), generator=g), torch.randn((32, 48), generator=g)
    fake.log.clear()
    _run(x1, y1)                       # replayed from the plan, marshalled
    replayed = _canon(fake.log, [x1, y1], status, fake.real)

    fake.log.clear()
    G.PLAN_CACHE = False
    try:
        _run(x1, y1)                   # scheduled afresh
    finally:
        G.PLAN_CACHE = True
    fresh = _canon(fake.log, [x1, y1], status, fake.real)
    assert len(replayed) == len(fresh) > 0
    assert replayed == fresh
    # the new inputs' addresses were written in: no address of the first step remains
    old = {x0.data_ptr(), y0.data_ptr()}
    for _, args in fake.log:
        for a in args:
            assert not (isinstance(a, int) and a in old)


def test_gpt_step_replay_covers_every_call_kind(cpu_graph):
    """The one-layer GPT block's forward and backward (gather, contractions
    with workspaces, reductions, elementwise programs, permutes, fused
    attention, scatter-add): every call of the step takes the marshalled
    path and a replay makes the calls of a fresh schedule."""
    import seeded_inputs as SI
    from primitive_sm_graph_gb300.workloads import gpt_step
    fake, status = cpu_graph
    tok, w = SI.gpt_block(6, 2, 64, 128, 128, 2, 256)
    gpt_step(tok, w, 2)
    assert len(G._PLANS) == 1
    plan = next(iter(G._PLANS.values()))
    kinds = {c[0] for c in plan.calls}
    assert {"psg_gather", "psg_reduce_rows", "psg_elementwise", "psg_attention_fwd",
            "psg_attention_bwd", "psg_scatter_add"} <= kinds, kinds
    assert all(f is not None for f in plan.fast)
    tok2, w2 = SI.gpt_block(7, 2, 64, 128, 128, 2, 256)
    leaves = None

    def step():
        fake.log.clear()
        gpt_step(tok2, w2, 2)
        return list(fake.log)
    replayed = step()
    G.PLAN_CACHE = False
    try:
        fresh = step()
    finally:
        G.PLAN_CACHE = True
    assert [fn for fn, _ in replayed] == [fn for fn, _ in fresh]
    # the same inputs are read at the same places: name the step's input tensors
    ins = [tok2] + [w2[k] for k in sorted(w2)]
    a, b = _canon(replayed, ins, status, fake.real), _canon(fresh, ins, status, fake.real)
    assert a == b


def test_executor_log_stays_bounded(cpu_graph, monkeypatch):
    """A long eager loop keeps only the recent calls in the executor's log."""
    monkeypatch.setattr(G, "LOG_KEEP", 8)
    g = torch.Generator().manual_seed(5)
    x, y = torch.randn((16, 8), generator=g), torch.randn((8, 4), generator=g)
    for _ in range(40):
        _run(x, y)
    assert 0 < len(G._executor().log) <= 8 + 2   # one step's two calls past the trim


def _header_writes():
    """Per C function, the positions of its non-const pointer parameters
    (other than the status word and the stream): what it writes, read from
    include/psg.h's declarations."""
    import os
    import re
    src = open(os.path.join(os.path.dirname(__file__), "..", "include", "psg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"psg_status\s+(psg_\w+)\s*\(([^)]*)\)\s*;", src):
        params = [p.strip() for p in m.group(2).split(",")]
        w = []
        for i, p in enumerate(params):
            name = re.split(r"[\s*]+", p)[-1]
            if "*" in p and not p.startswith("const") and name not in ("d_status", "stream"):
                w.append(i)
        out[m.group(1)] = tuple(w)
    return out


def test_written_arguments_match_the_header():
    hw = _header_writes()
    for fn, pos in G._WRITES.items():
        assert hw[fn] == pos, (fn, hw[fn], pos)


@pytest.mark.parametrize("streams", [2, 3])
def test_forked_schedule_orders_every_conflicting_pair(cpu_graph, monkeypatch, streams):
    """The forked-stream schedule of the GPT block's recorded step: every
    pair of calls that touch one buffer, one of them writing it (writes from
    the header's non-const pointers), is ordered by stream order or by the
    waits; the step's independent calls spread over more than one stream."""
    import seeded_inputs as SI
    from primitive_sm_graph_gb300.workloads import gpt_step
    monkeypatch.setattr(G, "FORK_STREAMS", streams)
    tok, w = SI.gpt_block(6, 2, 64, 128, 128, 2, 256)
    gpt_step(tok, w, 2)
    plan = next(iter(G._PLANS.values()))
    n_leaves = 1 + max(r.i for r in plan.refs.values() if r.kind == "leaf")
    where, waits = plan._fork_schedule(n_leaves)
    hw = _header_writes()
    flat = plan._flat_slots(n_leaves)
    nb = n_leaves + len(plan.allocs)
    acc = []
    for fast, fs in zip(plan.fast, flat):
        bufs = {k for _, _, k in fs if k < nb}
        wr = {k for box, at, k in fs if k < nb and box is fast[1] and at in hw[fast[4]]} if fast[4] in hw else bufs
        acc.append((bufs, wr))
    n = len(acc)
    # happens-before: stream order plus the waits, closed transitively
    before = [set() for _ in range(n)]
    last_on = {}
    for c in range(n):
        preds = set(waits[c])
        if where[c] in last_on:
            preds.add(last_on[where[c]])
        for p in preds:
            before[c] |= before[p] | {p}
        last_on[where[c]] = c
    for j in range(n):
        for i in range(j):
            bi, wi = acc[i]
            bj, wj = acc[j]
            if (wi & bj) or (wj & bi):
                assert i in before[j], (i, j, plan.fast[i][4], plan.fast[j][4])
    assert len(set(where)) > 1
