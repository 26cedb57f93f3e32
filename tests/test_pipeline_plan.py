"""The schedule of the streamed stack (QCFuse Figure 9, pipeline cache fusion;
PCR, layer-wise overlapping), checked on the CPU: the library's plan is run
through a model of two CUDA streams with events (a wait binds to the
event's latest record issued before it), and the resulting happens-before
order must (1) put every layer's uploads before its kernels, (2) never
refill a slot before every earlier user of it has finished, (3) let one
layer's upload run beside the previous layer's kernels when they use
different slots, and (4) run the scoring layer first, then the others in
index order.  A plan with a wait removed is shown to fail the check."""

import itertools

import pytest


@pytest.fixture(scope="module")
def fk():
    from rag_kv_cache_rerotate_gb300 import _build, fusekv
    _build.build()
    fusekv.load()
    return fusekv


def _order(fk, ops):
    """Happens-before closure of a plan: nodes are op indices."""
    copy_kinds = {fk.OP_WAIT_FREE, fk.OP_COPY, fk.OP_MARK_READY}
    n = len(ops)
    pred = [set() for _ in range(n)]
    last = {"copy": None, "compute": None}
    latest = {}                                 # (event, slot) -> op index of its latest record
    for i, (kind, layer, slot) in enumerate(ops):
        stream = "copy" if kind in copy_kinds else "compute"
        if last[stream] is not None:
            pred[i].add(last[stream])
        last[stream] = i
        if kind == fk.OP_WAIT_FREE and ("free", slot) in latest:
            pred[i].add(latest[("free", slot)])
        if kind == fk.OP_WAIT_READY and ("ready", slot) in latest:
            pred[i].add(latest[("ready", slot)])
        if kind == fk.OP_MARK_READY:
            latest[("ready", slot)] = i
        if kind == fk.OP_MARK_FREE:
            latest[("free", slot)] = i
    before = [set() for _ in range(n)]
    for i in range(n):
        for p in pred[i]:
            before[i] |= before[p] | {p}
    return before


def _check(fk, ops, n_layers, score_layer, slots):
    before = _order(fk, ops)
    at = {}
    for i, (kind, layer, slot) in enumerate(ops):
        assert slot == slots[layer]
        at.setdefault((kind, layer), []).append(i)
    order = [score_layer] + [l for l in range(n_layers) if l != score_layer]
    computes = [layer for kind, layer, _ in ops if kind == fk.OP_COMPUTE]
    assert computes == order
    for l in range(n_layers):
        (cp,), (cm,) = at[(fk.OP_COPY, l)], at[(fk.OP_COMPUTE, l)]
        assert cp in before[cm], ("kernels before uploads", l)
    for a, b in itertools.combinations(range(n_layers), 2):
        ia, ib = order.index(a), order.index(b)
        first, second = (a, b) if ia < ib else (b, a)
        if slots[a] == slots[b]:
            assert at[(fk.OP_COMPUTE, first)][0] in before[at[(fk.OP_COPY, second)][0]], (
                "slot refilled while in use", first, second)
    return before, at, order


@pytest.mark.parametrize("n_layers,score_layer,n_slots",
                         [(1, 0, 1), (3, 1, 1), (3, 1, 2), (5, 0, 2), (6, 5, 3), (36, 2, 2),
                          (8, 3, 8), (9, 4, 4)])
def test_round_robin_plans_are_safe_and_overlap(fk, n_layers, score_layer, n_slots):
    order = [score_layer] + [l for l in range(n_layers) if l != score_layer]
    slots = [0] * n_layers
    for i, l in enumerate(order):
        slots[l] = i % n_slots
    ops = fk.stack_pipeline_plan(n_layers, score_layer, slots, n_slots)
    reuses = n_layers - min(n_layers, n_slots)
    assert len(ops) == 5 * n_layers + reuses
    before, at, order = _check(fk, ops, n_layers, score_layer, slots)
    for x, y in zip(order, order[1:]):
        serial = at[(fk.OP_COMPUTE, x)][0] in before[at[(fk.OP_COPY, y)][0]]
        assert serial == (n_slots == 1), (x, y)


def test_uneven_slot_assignments(fk):
    # any assignment is safe: a layer waits for the previous users of its slot
    for slots in ([0, 0, 1, 0, 2], [2, 2, 2, 0, 1], [1, 0, 1, 0, 1]):
        ops = fk.stack_pipeline_plan(5, 2, slots, 3)
        _check(fk, ops, 5, 2, slots)


def test_a_plan_without_its_slot_wait_fails_the_check(fk):
    slots = [0, 1, 0, 1]
    ops = fk.stack_pipeline_plan(4, 0, slots, 2)
    _check(fk, ops, 4, 0, slots)
    broken = [o for o in ops if not (o[0] == fk.OP_WAIT_FREE and o[1] == 2)]
    with pytest.raises(AssertionError):
        _check(fk, broken, 4, 0, slots)


def test_plan_argument_errors(fk):
    with pytest.raises(fk.FuseError) as e:
        fk.stack_pipeline_plan(3, 1, [0, 2, 0], 2)             # slot out of range
    assert e.value.status == fk.FUSE_ERR_INVALID_ARG
    with pytest.raises(fk.FuseError) as e:
        fk.stack_pipeline_plan(3, 3, [0, 1, 0], 2)             # scoring layer out of range
    assert e.value.status == fk.FUSE_ERR_INVALID_ARG
    with pytest.raises(fk.FuseError) as e:
        fk.stack_pipeline_plan(3, 0, [0, 0, 0], 65)            # more slots than events allowed
    assert e.value.status == fk.FUSE_ERR_INVALID_ARG
    import ctypes
    n = ctypes.c_int32(0)
    slots = (ctypes.c_int32 * 3)(0, 1, 0)
    ops = (fk.PipelineOp * 4)()
    st = fk.load().fuse_stack_pipeline_plan(3, 0, slots, 2, ops, 4, ctypes.byref(n))
    assert st == fk.FUSE_ERR_WORKSPACE and n.value == 16
