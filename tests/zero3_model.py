"""A Python model of the ZeRO-3 step schedule, for the tests: per-unit gathers
with next-unit prefetch on a side stream, and per-unit reduce-scatter fused
with AdamW.

TEST-SIDE CHECKER, NOT THE PRODUCT.  The library's schedule is the native one
in csrc/zero3_sched.cpp (zero3_plan, zero3_step) and its CUDA-graph form
(zero3_graph_create); the benchmark times those, and the tests compare them
with the oracle.  This model issues the same order through a pluggable backend,
so that a test can (a) run it on the CPU against a backend that executes the
oracle's unit calls and records every stream operation, and (b) run it on the
GPU with a consumer callback between a unit's gather and its release, which
copies the gathered weights and poisons the buffer -- a race check the native
scheduler, which runs no Python between its launches, cannot host.

Method ("Data parallelism, ZeRO and FSDP", "How FSDP implements ZeRO-3",
steps 2-5):
  2. forward of a unit: all-gather its bf16 parameters, run it, free them;
  3. backward in reverse unit order: all-gather again, compute the gradients,
     free the parameters, reduce-scatter the gradients;
  4. the optimizer updates each rank's local shards with no communication;
  5. the all-gathers run on a separate stream, the next unit's gather is issued
     before the current unit's work (forward and backward prefetch), and at
     most about two units of full parameters are resident.
("Data parallelism, collectives and ZeRO/FSDP", the per-unit FSDP step figure,
shows the same order.)

On one GPU the "ranks" are buffers: the gather is ``zero3_gather_unit`` into
one of two full-unit buffers (double buffering bounds residency at two units),
and the reduce-scatter is ``zero3_reduce_scatter_unit``, which also applies
AdamW to each owner's shard of the unit and writes its new bf16 shard.  Fusing
the update into the unit's reduce-scatter gives the same bits as updating
after the whole backward pass: unit u's shard is last read by unit u's own
backward gather, which comes before its reduce-scatter, and the prefetch of
unit u-1 reads a disjoint region.
"""


class CudaBackend:
    """The library's kernels on two torch CUDA streams (main + gather side stream)."""

    def __init__(self, n_ranks, shards, master, m, v, device=None):
        import torch

        from fsdp_sharded_optimizer_gb300 import _binding as B

        self._torch, self._B = torch, B
        self.n_ranks = n_ranks
        self.shards, self.master, self.m, self.v = shards, master, m, v
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        self.main = torch.cuda.current_stream(dev)
        self.side = torch.cuda.Stream(device=dev)

    # stream/event primitives
    def event(self):
        return self._torch.cuda.Event()

    def record(self, ev, stream):
        ev.record(stream)

    def wait(self, stream, ev):
        stream.wait_event(ev)

    # the two collectives
    def gather(self, ui, unit, full, stream):
        self._B.zero3_gather_unit(unit, self.shards, full, stream=stream)

    def reduce_scatter(self, ui, unit, grads, hp, stream):
        self._B.zero3_reduce_scatter_unit(unit, grads, self.master, self.m, self.v, self.shards,
                                          hp, stream=stream)


class Zero3Schedule:
    """One ZeRO-3 step per ``step()`` call.

    units         unit layouts (``zero_layout``), model order
    backend       provides gather / reduce_scatter / event / record / wait and
                  the ``main`` and ``side`` streams
    full_bufs     two buffers, each at least the largest unit's n_padded bf16;
                  a callable ``full_view(buf, unit)`` cuts the unit's view
    grad_bufs     per-rank gradient buffers of at least the largest unit
    """

    def __init__(self, units, backend, full_bufs, grad_bufs, full_view=None, grad_view=None):
        if len(full_bufs) != 2:
            raise ValueError("ZeRO-3 double-buffers the gathered units: two full buffers")
        self.units = list(units)
        self.be = backend
        self.full_bufs = full_bufs
        self.grad_bufs = grad_bufs
        self.full_view = full_view or (lambda buf, unit: buf[:unit.n_padded])
        self.grad_view = grad_view or (lambda bufs, unit: [b[:unit.n_padded] for b in bufs])
        self.calls = {"allgather": 0, "reduce_scatter": 0}
        # free[b]: the main stream finished with full buffer b
        self._free = [None, None]

    def _gather(self, order, pos, slot):
        """Issue the gather of units[order[pos]] into full buffer `slot` on the side stream."""
        be = self.be
        if self._free[slot] is not None:
            be.wait(be.side, self._free[slot])
        ui = order[pos]
        unit = self.units[ui]
        be.gather(ui, unit, self.full_view(self.full_bufs[slot], unit), be.side)
        self.calls["allgather"] += 1
        ready = be.event()
        be.record(ready, be.side)
        return ready

    def _pass(self, order, body):
        """Walk the units in `order`: gather each one (prefetching the next on the
        side stream), run body(ui, unit, full) on the main stream, release it."""
        be = self.be
        ready = {0: self._gather(order, 0, 0)}
        for pos, ui in enumerate(order):
            slot = pos % 2
            if pos + 1 < len(order):  # prefetch the next unit before this unit's work
                ready[pos + 1] = self._gather(order, pos + 1, 1 - slot)
            be.wait(be.main, ready.pop(pos))
            unit = self.units[ui]
            body(ui, unit, self.full_view(self.full_bufs[slot], unit))
            done = be.event()
            be.record(done, be.main)
            self._free[slot] = done

    def step(self, hp_for_step, make_grads, forward=None, backward=None):
        """One step.  make_grads(ui, unit, grad_views, stream) writes unit ui's
        per-rank gradients on the main stream (the backward compute stand-in);
        forward/backward(ui, unit, full_view) optionally consume the gathered
        weights.  hp_for_step is the zero_hparams_t of this step."""
        be = self.be
        # the first gather of this step must see the previous step's updates
        start = be.event()
        be.record(start, be.main)
        be.wait(be.side, start)

        def fwd(ui, unit, full):
            if forward is not None:
                forward(ui, unit, full)

        def bwd(ui, unit, full):
            if backward is not None:
                backward(ui, unit, full)
            grads = self.grad_view(self.grad_bufs, unit)
            make_grads(ui, unit, grads, be.main)
            be.reduce_scatter(ui, unit, grads, hp_for_step, be.main)
            self.calls["reduce_scatter"] += 1

        n = len(self.units)
        self._pass(list(range(n)), fwd)
        self._pass(list(range(n - 1, -1, -1)), bwd)
