"""Happens-before checks of a ZeRO-3 step trace (test helper).

A trace is a list of entries in host issue order:
  ("record", stream, event)   ("wait", stream, event)
  ("gather", stream, unit, buffer)   ("use", stream, unit, buffer, ...)
  ("rs", stream, unit)   ("regen", stream, unit)   ("end", stream)
with stream "main", "side", "aux" (the second compute stream of the native
scheduler) or "side2" (its second side stream), and "end" marking where a
step returns (on "main").  A
wait orders the waiting stream's later operations after the operation that
preceded the event's most recent record at the time of the wait (CUDA's
semantics for a re-recorded event); a record right after waits also carries
them, as a CUDA event record carries everything before it on its stream."""
from collections import defaultdict

COMPUTE = ("main", "aux")
SIDE = ("side", "side2")


def happens_before_graph(trace):
    pos, last_op, event_src, edges = {}, {}, {}, {}
    count = defaultdict(int)
    pending = defaultdict(list)
    for e in trace:
        kind, stream = e[0], e[1]
        if kind == "record":
            if pending[stream]:
                # a record after waits captures them too: it becomes a node of
                # its own, after the waited-for operations and the stream's last
                node = (stream, count[stream])
                count[stream] += 1
                pos[node] = ("sync", stream)
                edges[node] = list(pending[stream]) + ([last_op[stream]] if stream in last_op else [])
                pending[stream].clear()
                last_op[stream] = node
            event_src[e[2]] = last_op.get(stream)
            continue
        if kind == "wait":
            if event_src.get(e[2]) is not None:
                pending[stream].append(event_src[e[2]])
            continue
        node = (stream, count[stream])
        count[stream] += 1
        pos[node] = e
        preds = list(pending[stream])
        pending[stream].clear()
        if stream in last_op:
            preds.append(last_op[stream])
        edges[node] = preds
        last_op[stream] = node
    return pos, edges


def hb(edges, a, b):
    """True when operation a happens before operation b."""
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


def check_zero3_trace(trace, n_units, n_steps):
    """Assert the ZeRO-3 schedule properties of "Data parallelism, ZeRO and FSDP",
    "How FSDP implements ZeRO-3", steps 2-5, on a trace of n_steps steps."""
    U = n_units
    pos, edges = happens_before_graph(trace)
    order_of = {id(e): i for i, e in enumerate(trace)}
    by_issue = lambda nodes: sorted(nodes, key=lambda n: order_of[id(pos[n])])
    gathers = by_issue([n for n, e in pos.items() if e[0] == "gather"])
    uses = by_issue([n for n, e in pos.items() if e[0] == "use"])
    rss = by_issue([n for n, e in pos.items() if e[0] == "rs"])
    ends = by_issue([n for n, e in pos.items() if e[0] == "end"])
    assert len(gathers) == 2 * U * n_steps and len(uses) == 2 * U * n_steps
    assert len(rss) == U * n_steps
    assert all(n[0] in SIDE for n in gathers) and all(n[0] in COMPUTE for n in uses + rss)
    # each full buffer's gathers stay on one side stream
    for b in {pos[n][3] for n in gathers}:
        assert len({n[0] for n in gathers if pos[n][3] == b}) == 1
    # the forward pass runs on the main stream; a unit's backward use and
    # reduce-scatter share one compute stream
    fwd_uses = [u for k, u in enumerate(uses) if (k // U) % 2 == 0]
    assert all(n[0] == "main" for n in fwd_uses)
    # forward 0..U-1, backward U-1..0, every step
    assert [pos[n][2] for n in gathers] == (list(range(U)) + list(range(U - 1, -1, -1))) * n_steps
    assert [pos[n][2] for n in uses] == (list(range(U)) + list(range(U - 1, -1, -1))) * n_steps
    # two full buffers, alternating (a single unit may always use the same one)
    slots = {pos[n][3] for n in gathers}
    assert len(slots) <= 2 and (len(slots) == 2 or U == 1)
    for g, u in zip(gathers, uses):
        assert pos[g][2] == pos[u][2] and pos[g][3] == pos[u][3]
        assert hb(edges, g, u), "unit %d used before it was gathered" % pos[u][2]
        later = [h for h in gathers if order_of[id(pos[h])] > order_of[id(pos[g])]
                 and pos[h][3] == pos[g][3]]
        if later:
            assert hb(edges, u, later[0]), "buffer of unit %d overwritten in use" % pos[u][2]
    # each reduce-scatter follows its unit's backward use; backward prefetch:
    # the gather of unit u-1 is issued before unit u's reduce-scatter and does
    # not delay it
    bwd_uses = [u for k, u in enumerate(uses) if (k // U) % 2 == 1]
    for r, u in zip(rss, bwd_uses):
        assert pos[r][2] == pos[u][2] and hb(edges, u, r)
        unit = pos[r][2]
        if unit > 0:
            pre = [g for g in gathers if pos[g][2] == unit - 1
                   and order_of[id(pos[g])] < order_of[id(pos[r])]]
            assert pre, "no prefetch of unit %d before unit %d's reduce-scatter" % (unit - 1, unit)
            assert not hb(edges, pre[-1], r)
    # the next step's first gather sees every reduce-scatter of the step before,
    # and every gather of a unit sees that unit's update of the step before
    for s in range(1, n_steps):
        for r in rss[(s - 1) * U:s * U]:
            assert hb(edges, r, gathers[s * 2 * U]), "next step overtakes unit %d" % pos[r][2]
            for g in gathers[s * 2 * U:(s + 1) * 2 * U]:
                if pos[g][2] == pos[r][2]:
                    assert hb(edges, r, g), "unit %d gathered before its update" % pos[r][2]
    # where the trace marks the step's return on the main stream, every
    # reduce-scatter of the step happens before it
    if ends:
        assert len(ends) == n_steps and all(n[0] == "main" for n in ends)
        for s in range(n_steps):
            for r in rss[s * U:(s + 1) * U]:
                assert hb(edges, r, ends[s]), "step ends before unit %d's update" % pos[r][2]
    # at most two units gathered and not yet released at any time is implied by
    # the two buffers and the overwrite check above
    return True


def check_zero3_kept_trace(trace, n_units, n_steps):
    """The reshard_after_forward = False schedule ("How FSDP implements ZeRO-3",
    step 6): one gather per unit per step into the unit's own region, kept from
    the forward to the backward pass; the backward reuses it."""
    U = n_units
    pos, edges = happens_before_graph(trace)
    order_of = {id(e): i for i, e in enumerate(trace)}
    by_issue = lambda nodes: sorted(nodes, key=lambda n: order_of[id(pos[n])])
    gathers = by_issue([n for n, e in pos.items() if e[0] == "gather"])
    uses = by_issue([n for n, e in pos.items() if e[0] == "use"])
    rss = by_issue([n for n, e in pos.items() if e[0] == "rs"])
    assert len(gathers) == U * n_steps and len(uses) == 2 * U * n_steps
    assert len(rss) == U * n_steps
    assert all(n[0] in SIDE for n in gathers) and all(n[0] == "main" for n in uses + rss)
    assert [pos[n][2] for n in gathers] == list(range(U)) * n_steps
    assert [pos[n][2] for n in uses] == (list(range(U)) + list(range(U - 1, -1, -1))) * n_steps
    for s in range(n_steps):
        g = gathers[s * U:(s + 1) * U]
        us = uses[s * 2 * U:(s + 1) * 2 * U]
        r = rss[s * U:(s + 1) * U]
        for u in range(U):
            fwd, bwd = us[u], us[2 * U - 1 - u]
            assert hb(edges, g[u], fwd) and hb(edges, g[u], bwd)
            rs = r[U - 1 - u]
            assert pos[rs][2] == u and hb(edges, bwd, rs)
            if u + 1 < U:  # forward prefetch: unit u+1's gather issued before unit u's use
                assert order_of[id(pos[g[u + 1]])] < order_of[id(pos[fwd])]
            if s + 1 < n_steps:  # the next step gathers only after this step updated the shard
                assert hb(edges, rs, gathers[(s + 1) * U + u])
    return True
