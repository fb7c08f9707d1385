"""The package's usage example, as a module the tests import and run (the
user documentation prints the body of run()): ZeRO-1, ZeRO-2 with clipping
through the fp32 gradient shard, and a ZeRO-3 step captured as a CUDA graph,
on seeded synthetic inputs."""


def run():
    import torch
    import fsdp_sharded_optimizer_gb300 as Z

    N = 8                                                   # emulated data-parallel ranks
    (unit,), _ = Z.zero_layout([10_000_000], N)             # one flat buffer, padded to N * 64
    P, S = unit.n_padded, unit.shard_len                    # rank k owns [k*S, (k+1)*S)
    grads = torch.empty((N, P), dtype=torch.int16, device="cuda")    # rank r's bf16 gradient
    master = torch.empty((N, S), dtype=torch.float32, device="cuda")  # fp32 master shards
    m, v = torch.zeros_like(master), torch.zeros_like(master)         # AdamW state shards
    params = torch.empty(P, dtype=torch.int16, device="cuda")         # replicated bf16 weights
    Z.zero_gen_master(0, 0.02, [unit], master)              # seeded synthetic inputs
    Z.zero_gen_grads_unit(0, 1, 1e-3, 0, unit, grads)

    # ZeRO-1: reduce-scatter (rank-order fp32 mean) + AdamW + bf16 all-gather, one pass
    Z.zero_step_stage12(1, grads, master, m, v, params, Z.hparams(lr=1e-3, step=1))

    # ZeRO-2 with 25 MiB buckets and global-norm clipping through the fp32 gradient shard
    scratch = torch.empty(Z.zero_clip_scratch_bytes() // 8, dtype=torch.float64, device="cuda")
    norm_coef = torch.empty(4, dtype=torch.float32, device="cuda")[:2]
    grad_shard = torch.empty_like(master)
    Z.zero_grad_reduce_sqnorm(grads, grad_shard, scratch)   # norm pass that keeps the mean
    Z.zero_clip_coef(scratch, 1.0, norm_coef)               # max_norm 1.0
    Z.zero_step_stage12_reduced(2, grad_shard, master, m, v, params, Z.hparams(step=2), norm_coef,
                                bucket_elems=13_107_200)

    # ZeRO-3: units, per-unit gathers on a side stream, captured once as a CUDA graph
    units, total = Z.zero_layout([4_000_000] * 3 + [6_000_000], N)
    shards = torch.empty((N, total // N), dtype=torch.int16, device="cuda")
    w3 = torch.empty((N, total // N), dtype=torch.float32, device="cuda")
    m3, v3 = torch.zeros_like(w3), torch.zeros_like(w3)
    g3 = torch.empty((N, total), dtype=torch.int16, device="cuda")    # every unit's gradients
    full = [torch.empty(max(u.n_padded for u in units), dtype=torch.int16, device="cuda")
            for _ in range(2)]
    Z.zero_gen_master(0, 0.02, units, w3)
    for k in range(N):
        Z.zero_cast_bf16(w3[k], shards[k])                  # each rank's initial bf16 shard
    for u in units:
        Z.zero_gen_grads_unit(0, 1, 1e-3, 0, u, [r[u.offset:u.offset + u.n_padded] for r in g3])
    graph = Z.zero3_graph_create(units, g3, w3, m3, v3, shards, full[0], full[1], Z.hparams(),
                                 torch.cuda.Stream(), torch.cuda.Stream())
    for t in range(1, 4):
        graph.launch(Z.hparams(step=t))                     # new AdamW scalars every step
    torch.cuda.synchronize()
    graph.close()                                           # after the last replay has finished
