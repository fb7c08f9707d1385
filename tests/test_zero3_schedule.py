"""The ZeRO-3 schedule (per-unit gathers with next-unit prefetch on a side
stream, per-unit reduce-scatter fused with AdamW), run on the CPU against a
backend that executes the oracle's unit calls and records every stream
operation.  Checks the call counts of "Data parallelism, ZeRO and FSDP",
"5. In code", third block (two units: four all-gathers, two reduce-scatters),
the prefetch order and buffer reuse of "How FSDP implements ZeRO-3", step 5,
and that the result equals DDP bit for bit."""
import numpy as np
import pytest

from zero3_model import Zero3Schedule
from schedule_check import check_zero3_kept_trace, check_zero3_trace

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


class OracleBackend:
    """Streams and events are names in a trace; the two calls run the oracle."""

    main, side = "main", "side"

    def __init__(self, orc, n_ranks, shards, master, m, v):
        self.orc, self.N = orc, n_ranks
        self.shards, self.master, self.m, self.v = shards, master, m, v
        self.trace = []
        self._n = 0

    def event(self):
        self._n += 1
        return "ev%d" % self._n

    def record(self, ev, stream):
        self.trace.append(("record", stream, ev))

    def wait(self, stream, ev):
        self.trace.append(("wait", stream, ev))

    def gather(self, ui, unit, full, stream):
        self.trace.append(("gather", stream, ui, id(full.base) if full.base is not None else id(full)))
        self.orc.zero3_gather_unit(unit, self.shards, full)

    def reduce_scatter(self, ui, unit, grads, hp, stream):
        self.trace.append(("rs", stream, ui))
        g = np.ascontiguousarray(np.stack(grads))
        self.orc.zero3_reduce_scatter_unit(unit, g, self.master, self.m, self.v, self.shards, hp)


def _setup(orc, sizes, N, seed):
    units, total = orc.layout(sizes, N)
    master = orc.gen_master(seed, 0.02, units, N)
    m, v = np.zeros_like(master), np.zeros_like(master)
    shards = orc.bf16_rne(master)
    be = OracleBackend(orc, N, shards, master, m, v)
    max_unit = max(u.n_padded for u in units)
    full = [np.zeros(max_unit, np.uint16), np.zeros(max_unit, np.uint16)]
    grads = [np.zeros(max_unit, np.uint16) for _ in range(N)]
    return units, be, Zero3Schedule(units, be, full, grads), full


def _make_grads(orc, seed, step, N):
    def make(ui, unit, views, stream):
        g = orc.gen_grads_unit(seed, step, 1e-3, 0, unit, N)
        for r in range(N):
            views[r][:] = g[r]
    return make


@pytest.mark.parametrize("sizes,N,T", [([64 * 16 + 64, 4 * 64 + 4], 2, 1), ([300, 50, 1000, 7, 64], 4, 3),
                                       ([5000], 8, 2)])
def test_schedule_equals_ddp_and_counts_calls(orc, sizes, N, T):
    seed = 21
    units, be, sched, full = _setup(orc, sizes, N, seed)
    for t in range(1, T + 1):
        sched.step(orc.hparams(**HP, step=t), _make_grads(orc, seed, t, N))
    U = len(units)
    assert sched.calls == {"allgather": 2 * U * T, "reduce_scatter": U * T}
    # the updated shards, gathered, equal T DDP steps on the whole model
    ddp = orc.sim_ddp(N, sum(sizes), seed, 0.02, 1e-3, 0, orc.hparams(**HP, step=1), T)
    got = []
    for u in units:
        f = np.zeros(u.n_padded, np.uint16)
        orc.zero3_gather_unit(u, be.shards, f)
        got.append(f[:u.n_params])
    np.testing.assert_array_equal(np.concatenate(got), ddp[0])


def test_two_units_four_gathers_two_reduce_scatters(orc):
    units, be, sched, _ = _setup(orc, [64 * 16 + 64, 4 * 64 + 4], 2, 0)
    sched.step(orc.hparams(**HP, step=1), _make_grads(orc, 0, 1, 2))
    ops = [e[0] for e in be.trace if e[0] in ("gather", "rs")]
    assert ops.count("gather") == 4 and ops.count("rs") == 2


def test_prefetch_order_and_buffer_safety(orc):
    units, be, sched, full = _setup(orc, [100, 200, 300, 400, 64], 2, 0)
    slot_of = lambda view: id(view.base) if view.base is not None else id(view)
    use = lambda tag: (lambda ui, unit, f: be.trace.append(("use", "main", ui, slot_of(f), tag)))
    for t in (1, 2):
        sched.step(orc.hparams(**HP, step=t), _make_grads(orc, 0, t, 2), forward=use("fwd"),
                   backward=use("bwd"))
    check_zero3_trace(be.trace, len(units), 2)


STREAMS = {0: "main", 1: "side", 2: "aux", 3: "side2"}


def _native_trace(n_units, n_steps, regen=False, clip=False, reshard=True):
    from fsdp_sharded_optimizer_gb300 import _binding as B
    names = STREAMS
    trace = []
    for _ in range(n_steps):
        for kind, stream, unit, arg in B.zero3_plan(n_units, regen, clip, reshard):
            st = names[stream]
            if kind in ("record", "wait"):
                trace.append((kind, st, "ev%d" % arg))
            elif kind == "gather":
                trace.append(("gather", st, unit, arg))
            elif kind == "use":
                trace.append(("use", st, unit, arg))
            elif kind == "reduce_scatter":
                trace.append(("rs", st, unit))
            else:
                trace.append((kind, st, unit))
        trace.append(("end", "main"))
    return trace


@pytest.mark.parametrize("n_units,n_steps,regen,clip", [(1, 1, False, False), (2, 1, False, True),
                                                        (5, 3, False, False), (33, 2, True, True),
                                                        (23, 2, False, True), (4, 2, True, False)])
def test_native_plan_is_safe(n_units, n_steps, regen, clip):
    """The native scheduler's plan (zero3_plan, the operations zero3_step
    executes) obeys the same happens-before rules as the Python schedule."""
    trace = _native_trace(n_units, n_steps, regen, clip)
    check_zero3_trace(trace, n_units, n_steps)
    if clip:
        # each step: every unit's norm, then the coefficient, before any reduce-scatter
        per = len(trace) // n_steps
        for s0 in range(0, len(trace), per):
            st = trace[s0:s0 + per]
            kinds = [e[0] for e in st]
            first_rs, coef = kinds.index("rs"), kinds.index("clip_coef")
            norms = [i for i, k in enumerate(kinds) if k == "norm"]
            assert len(norms) == n_units and max(norms) < coef < first_rs
            assert all(e[1] == "main" for e in st if e[0] in ("norm", "clip_coef"))
        _assert_rs_after_coef(trace)


def _assert_rs_after_coef(trace):
    """Every reduce-scatter, on either compute stream, happens after the
    coefficient kernel of its step (it scales by the coefficient)."""
    from schedule_check import happens_before_graph, hb
    pos, edges = happens_before_graph(trace)
    order_of = {id(e): i for i, e in enumerate(trace)}
    nodes = sorted(pos, key=lambda n: order_of.get(id(pos[n]), 0))
    coef = None
    for n in nodes:
        if pos[n][0] == "clip_coef":
            coef = n
        elif pos[n][0] == "rs":
            assert coef is not None and hb(edges, coef, n), "update before its coefficient"


def test_checks_catch_a_missing_join_of_the_second_compute_stream():
    """The plan's second compute stream hands its end back to the main stream
    (event 6): without that join the step could return, and the next step
    start, before a unit's update, and the checks see it.  Its updates follow
    the clip coefficient (through the side stream's waits on the forward
    pass's releases, and explicitly through event 5)."""
    trace = _native_trace(5, 2, clip=True)
    assert any(e[:2] == ("wait", "main") and e[2] == "ev6" for e in trace)
    assert any(e[:2] == ("wait", "aux") and e[2] == "ev5" for e in trace)
    no_join = [e for e in trace if not (e[:2] == ("wait", "main") and e[2] == "ev6")]
    with pytest.raises(AssertionError):
        check_zero3_trace(no_join, 5, 2)
    check_zero3_trace(trace, 5, 2)
    _assert_rs_after_coef(trace)


def test_checks_catch_a_second_side_stream_that_does_not_wait_for_the_start():
    """The second side stream's gathers read shards the previous step updated:
    it waits for the step's start event like the first side stream, and
    without that wait the checks see a gather overtake its unit's update."""
    trace = _native_trace(5, 2)
    assert any(e[:2] == ("wait", "side2") and e[2] == "ev0" for e in trace)
    no_start = [e for e in trace if not (e[:2] == ("wait", "side2") and e[2] == "ev0")]
    with pytest.raises(AssertionError):
        check_zero3_trace(no_start, 5, 2)
    kept = _native_trace(4, 2, reshard=False)
    no_start = [e for e in kept if not (e[:2] == ("wait", "side2") and e[2] == "ev0")]
    with pytest.raises(AssertionError):
        check_zero3_kept_trace(no_start, 4, 2)


def test_plan_length_stays_within_the_header_bound():
    """include/zero.h sizes the caller's op array: 13 n + 7 operations, plus n
    with regeneration, n + 1 with clipping and n more with both; a micro-batch
    plan stays within 13 n + 7.  An array one entry short is rejected."""
    import ctypes as C

    from fsdp_sharded_optimizer_gb300 import _binding as B
    for n in list(range(1, 41)) + [64, 257]:
        for regen in (0, 1):
            for clip in (0, 1):
                for reshard in (0, 1):
                    L = len(B.zero3_plan(n, regen, clip, reshard))
                    bound = 13 * n + 7 + regen * n + clip * (n + 1) + regen * clip * n
                    assert L <= bound, (n, regen, clip, reshard, L, bound)
                    ops = (B.zero_op_t * L)()
                    got = C.c_int32()
                    assert B.lib.zero3_plan(n, regen, clip, reshard, ops, L, C.byref(got)) == 0
                    assert got.value == L
                    assert B.lib.zero3_plan(n, regen, clip, reshard, ops, L - 1,
                                            C.byref(got)) == B.ZERO_EINVAL
        for m in (1, 2, 4):
            for mb in range(m):
                for reshard in (True, False):
                    assert len(B.zero3_plan_microbatch(n, mb, m, reshard)) <= 13 * n + 7


def test_native_plan_counts_and_regen():
    from fsdp_sharded_optimizer_gb300 import _binding as B
    ops = B.zero3_plan(2, False)
    kinds = [o[0] for o in ops]
    assert kinds.count("gather") == 4 and kinds.count("reduce_scatter") == 2
    assert "regen" not in kinds and "norm" not in kinds and len(ops) <= 13 * 2 + 7
    assert all(o[3] == 0 for o in ops if o[0] == "reduce_scatter")
    ops = B.zero3_plan(3, True, True)
    assert len(ops) <= 13 * 3 + 7 + 3 + 3 + 1 + 3
    assert all(o[3] == 1 for o in ops if o[0] == "reduce_scatter")
    norms = [o for o in ops if o[0] == "norm"]
    assert [o[3] for o in norms] == [0, 1, 1]  # the first unit overwrites the partials
    ops = B.zero3_plan(4, True)
    kinds = [o[0] for o in ops]
    assert kinds.count("regen") == 4 and len(ops) <= 14 * 4 + 7
    # every regeneration immediately precedes its unit's reduce-scatter on the main stream
    for i, o in enumerate(ops):
        if o[0] == "regen":
            assert ops[i + 1][0] == "reduce_scatter" and ops[i + 1][2] == o[2]
            assert o[1] == 0



@pytest.mark.parametrize("n_units,n_steps,regen,clip", [(1, 1, False, False), (2, 2, False, False),
                                                        (7, 3, True, True), (33, 2, False, True)])
def test_native_kept_plan_is_safe(n_units, n_steps, regen, clip):
    check_zero3_kept_trace(_native_trace(n_units, n_steps, regen, clip, reshard=False), n_units,
                           n_steps)


def test_no_reshard_saves_one_gather_per_unit(orc):
    """"With reshard_after_forward=False ... you would see one all-gather less"
    ("Data parallelism, ZeRO and FSDP", "5. In code", third block): two units give
    two all-gathers and two reduce-scatters, the 2P volume of the accounting."""
    from fsdp_sharded_optimizer_gb300 import _binding as B
    kinds = [o[0] for o in B.zero3_plan(2, False, False, False)]
    assert kinds.count("gather") == 2 and kinds.count("reduce_scatter") == 2
    assert orc.comm_volume(3, 1, False, 1.0) == 2.0
    assert all(o[3] == 2 for o in B.zero3_plan(4, False, False, False) if o[0] in ("gather", "use"))


@pytest.mark.parametrize("regen,clip", [(False, False), (False, True), (True, False), (True, True)])
def test_which_main_stream_launches_follow_one_another(regen, clip):
    """zero3_step chains a norm pass to a norm pass issued right before it on
    the main stream, and a unit update to an update right before it, where
    nothing else was issued between them (USE issues nothing; an event record
    or wait, a regeneration or a gather's release does).  The plan fixes
    where that happens: the norm passes follow one another unless the
    regeneration of the gradients each reads sits between; without
    resharding the backward updates follow one another unless regenerations
    separate them; with resharding an event record and wait always separate
    two updates, so those stay unchained."""
    from fsdp_sharded_optimizer_gb300 import _binding as B
    n = 6
    for reshard in (True, False):
        main = [o for o in B.zero3_plan(n, regen, clip, reshard) if o[1] == 0 and o[0] != "use"]
        pairs = list(zip(main, main[1:]))
        rs_pairs = [(a, b) for a, b in pairs if a[0] == b[0] == "reduce_scatter"]
        norm_pairs = [(a, b) for a, b in pairs if a[0] == b[0] == "norm"]
        assert len(rs_pairs) == (n - 1 if not reshard and not regen else 0)
        assert len(norm_pairs) == (n - 1 if clip and not regen else 0)
        # chained neighbours always work on different units
        assert all(a[2] != b[2] for a, b in rs_pairs + norm_pairs)
        # a norm pass that adds to the partials (arg 1) is never the first of the step
        assert all(b[3] == 1 for _, b in norm_pairs)


@pytest.mark.parametrize("n_units,micro,reshard", [(1, 2, True), (5, 3, True), (23, 4, True),
                                                   (5, 3, False), (7, 1, True)])
def test_microbatch_plans_are_safe_and_accumulate(n_units, micro, reshard):
    """Each micro-batch of an accumulated step has zero3_plan's operations and
    order, with the backward units accumulating (the first micro-batch
    starting the accumulator) until the last, which reduce-scatters into the
    update (arg 2).  The happens-before rules hold for every micro-batch."""
    from fsdp_sharded_optimizer_gb300 import _binding as B
    trace = []
    for mb in range(micro):
        ops = B.zero3_plan_microbatch(n_units, mb, micro, reshard)
        plain = B.zero3_plan(n_units, False, False, reshard)
        assert len(ops) == len(plain)
        for o, p in zip(ops, plain):
            if p[0] == "reduce_scatter":
                if mb < micro - 1:
                    assert o == ("accumulate", p[1], p[2], 1 if mb == 0 else 0)
                else:
                    assert o == ("reduce_scatter", p[1], p[2], 2 if micro > 1 else 0)
            else:
                assert o == p
        for kind, stream, unit, arg in ops:
            st = STREAMS[stream]
            if kind in ("record", "wait"):
                trace.append((kind, st, "ev%d" % arg))
            elif kind in ("gather", "use"):
                trace.append((kind, st, unit, arg))
            elif kind in ("reduce_scatter", "accumulate"):  # both read the unit's gradients
                trace.append(("rs", st, unit))
            else:
                trace.append((kind, st, unit))
    if reshard:
        check_zero3_trace(trace, n_units, micro)
    else:
        check_zero3_kept_trace(trace, n_units, micro)
    with pytest.raises(B.ZeroError):
        B.zero3_plan_microbatch(n_units, micro, micro, reshard)
    with pytest.raises(B.ZeroError):
        B.zero3_plan_microbatch(n_units, -1, micro, reshard)
