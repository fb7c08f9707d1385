"""The ZeRO-3 schedule (per-unit gathers with next-unit prefetch on a side
stream, per-unit reduce-scatter fused with AdamW), run on the CPU against a
backend that executes the oracle's unit calls and records every stream
operation.  Checks the call counts of "Data parallelism, ZeRO and FSDP",
"5. In code", third block (two units: four all-gathers, two reduce-scatters),
the prefetch order and buffer reuse of "How FSDP implements ZeRO-3", step 5,
and that the result equals DDP bit for bit."""
import numpy as np
import pytest

from fsdp_sharded_optimizer_gb300.zero3 import Zero3Schedule

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


def _happens_before_graph(trace):
    """Ops per stream in program order, plus edges from each wait to the op just
    before the awaited event's record on the other stream."""
    pos = {}            # (stream, i) -> trace entry
    last_op = {}        # stream -> (stream, i) of its latest op
    event_src = {}      # event -> op that precedes its record (or None)
    edges = {}
    count = {"main": 0, "side": 0}
    pending_wait = {"main": [], "side": []}
    for e in trace:
        kind, stream = e[0], e[1]
        if kind == "record":
            event_src[e[2]] = last_op.get(stream)
            continue
        if kind == "wait":
            if event_src.get(e[2]) is not None:
                pending_wait[stream].append(event_src[e[2]])
            continue
        node = (stream, count[stream])
        count[stream] += 1
        pos[node] = e
        preds = list(pending_wait[stream])
        pending_wait[stream].clear()
        if stream in last_op:
            preds.append(last_op[stream])
        edges[node] = preds
        last_op[stream] = node
    return pos, edges


def _hb(edges, a, b):
    """True when op a happens before op b."""
    stack, seen = [b], set()
    while stack:
        n = stack.pop()
        for p in edges.get(n, []):
            if p == a:
                return True
            if p not in seen:
                seen.add(p)
                stack.append(p)
    return False


def test_prefetch_order_and_buffer_safety(orc):
    units, be, sched, full = _setup(orc, [100, 200, 300, 400, 64], 2, 0)
    slot_of = lambda view: id(view.base) if view.base is not None else id(view)
    use = lambda tag: (lambda ui, unit, f: be.trace.append(("use", "main", ui, slot_of(f), tag)))
    for t in (1, 2):
        sched.step(orc.hparams(**HP, step=t), _make_grads(orc, 0, t, 2), forward=use("fwd"),
                   backward=use("bwd"))
    pos, edges = _happens_before_graph(be.trace)
    gathers = [n for n, e in pos.items() if e[0] == "gather"]
    uses = [n for n, e in pos.items() if e[0] == "use"]
    rss = [n for n, e in pos.items() if e[0] == "rs"]
    U = len(units)
    assert len(gathers) == 2 * 2 * U and len(uses) == 2 * 2 * U and len(rss) == 2 * U
    # gathers on the side stream, uses and reduce-scatters on the main stream
    assert all(n[0] == "side" for n in gathers) and all(n[0] == "main" for n in uses + rss)
    # order: forward 0..U-1 then backward U-1..0, every step
    order = [pos[n][2] for n in sorted(gathers, key=lambda n: n[1])]
    assert order == (list(range(U)) + list(range(U - 1, -1, -1))) * 2
    # only two full buffers exist
    assert len({pos[n][3] for n in gathers}) == 2
    # every use sees its own gather, and the buffer is not overwritten before the use
    # ends: the next gather into the same buffer happens after the use
    gathers_sorted = sorted(gathers, key=lambda n: n[1])
    uses_sorted = sorted(uses, key=lambda n: n[1])
    for g, u in zip(gathers_sorted, uses_sorted):
        assert pos[g][2] == pos[u][2] and pos[g][3] == pos[u][3]
        assert _hb(edges, g, u), "use of unit %d may run before its gather" % pos[u][2]
        later = [h for h in gathers_sorted if h[1] > g[1] and pos[h][3] == pos[g][3]]
        if later:
            assert _hb(edges, u, later[0]), "buffer of unit %d overwritten while in use" % pos[u][2]
    # backward prefetch: unit u-1's gather is issued before unit u's reduce-scatter,
    # and the reduce-scatter of unit u does not wait for it
    trace_index = {id(e): i for i, e in enumerate(be.trace)}
    for r in rss:
        u = pos[r][2]
        if u == 0:
            continue
        pre = [g for g in gathers if pos[g][2] == u - 1 and trace_index[id(pos[g])] < trace_index[id(pos[r])]]
        assert pre, "no prefetch of unit %d before the reduce-scatter of unit %d" % (u - 1, u)
        assert not _hb(edges, pre[-1], r)
    # a step's first gather happens after the previous step's last reduce-scatter
    first_of_step2 = gathers_sorted[2 * U]
    assert _hb(edges, sorted(rss, key=lambda n: n[1])[U - 1], first_of_step2)
