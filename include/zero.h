/*
 * zero.h -- C ABI of the GB300 fused ZeRO/FSDP sharded optimizer step.
 *
 * The N_d data-parallel ranks of one training job are emulated on ONE GPU:
 * each rank is a separate set of device buffers (its bf16 gradient, its fp32
 * master/m/v shard and, for ZeRO-3, its bf16 parameter shard).  The
 * "collectives" are memory traffic inside one kernel: the reduce-scatter is
 * each owner's fixed-order fp32 sum over the N_d gradient buffers, the
 * all-gather is the owner writing its new bf16 slice into the replicated
 * buffer (ZeRO-1/2) or into its shard that the unit gather later copies
 * (ZeRO-3).
 *
 * Sources (page title and section; the method is theirs, the code is not):
 *  [DZF] "Data parallelism, ZeRO and FSDP" (ML Systems, lesson 8):
 *        "2. The picture" (what is redundant; the communication is already
 *        there), "3. Definitions and main results" (Theorem: ZeRO memory and
 *        communication; How FSDP implements ZeRO-3), "5. In code" (the
 *        AdamW update of the ZeRO-1 simulator).
 *  [DDF] "Distributed Training Basics -- DDP and FSDP": "Memory accounting:
 *        derive the table from bytes", "Communication and a roofline sanity
 *        check".
 *  [COL] "Data parallelism, collectives and ZeRO/FSDP": "Collectives",
 *        "ZeRO and FSDP" (the per-unit FSDP step figure).
 *
 * Conventions shared by every call:
 *  - Return ZERO_OK (0) or a negative ZERO_E* code; no exception crosses the
 *    ABI.  zero_strerror() names a code.
 *  - Device calls are asynchronous on the caller's stream and allocate no
 *    memory.  The caller owns every buffer.  Pointer tables ("n_ranks device
 *    pointers") are HOST arrays holding DEVICE addresses; the library copies
 *    them into the kernel's parameters, so the tables may be freed as soon as
 *    the call returns.
 *  - bf16 values travel as uint16_t bit patterns.  Every device pointer must
 *    be 16-byte aligned (ZERO_EALIGN otherwise).  A "device pointer" may also
 *    address pinned (page-locked) host memory: the kernels then read or write
 *    it in place over the host link, with no staging copy (unified virtual
 *    addressing; NVLink-C2C on Grace-Blackwell).
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument launches nothing.  ZERO_ECUDA reports a launch failure.
 *  - Stateless and re-entrant, with three documented exceptions: zero3_step
 *    keeps a per-thread cache of seven CUDA events and two CUDA streams,
 *    zero_clip_coef_units_noalloc
 *    works in a library-internal device array, and a zero3_graph_t holds the
 *    graph it captured.  1 <= n_ranks <= ZERO_MAX_RANKS.
 *
 * Layout (zero_layout): a unit of P true parameters is padded to
 * P' = ceil(P / (n_ranks*align)) * n_ranks*align; S = P'/n_ranks; rank k owns
 * [k*S, (k+1)*S).  Padding holds +0 gradients and +0 state and stays +0.
 */
#ifndef ZERO_H
#define ZERO_H

#include <stdint.h>

#include <cuda_runtime_api.h> /* cudaStream_t */

#ifdef __cplusplus
extern "C" {
#endif

#define ZERO_OK 0
#define ZERO_EINVAL (-1)   /* an argument is out of range or null */
#define ZERO_EALIGN (-2)   /* a device pointer is not 16-byte aligned */
#define ZERO_ECUDA (-3)    /* the CUDA runtime reported an error */
#define ZERO_ETIMEOUT (-4) /* a bounded host wait ran out */

#define ZERO_MAX_RANKS 64
#define ZERO_DEFAULT_ALIGN 64 /* elements per shard granule */

/* Launch granularity of the fused step.  A call (or a ZeRO-2 bucket) of n
 * elements is covered by ceil(n / ZERO_CHUNK_ELEMS) launches, consecutive
 * chunks of ZERO_CHUNK_ELEMS elements with a shorter last one, each after the
 * first a programmatic dependent launch on the one before (the chunks touch
 * disjoint elements).  A block that finishes its share of a chunk early hands
 * its SM to the next chunk, which one persistent launch over the whole range
 * cannot do.  The results do not depend on it.  The value is 25 MiB of bf16
 * gradients, the DDP bucket default ([DZF] "How DDP overlaps the all-reduce
 * with the backward pass", step 1). */
#define ZERO_CHUNK_ELEMS 13107200

/* AdamW hyper-parameters ([DZF] "5. In code": lr, b1, b2, eps, wd) and the
 * 1-based step counter t used by the bias correction 1 - b^t. */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;
} zero_hparams_t;

/* One FSDP unit ([DZF] "How FSDP implements ZeRO-3", step 1): its parameters
 * flattened, padded and cut into n_ranks equal chunks. */
typedef struct {
    int64_t n_params;     /* true parameters of the unit */
    int64_t n_padded;     /* multiple of n_ranks*align */
    int64_t shard_len;    /* n_padded / n_ranks */
    int64_t offset;       /* start of the unit in the concatenated padded buffer */
    int64_t shard_offset; /* start of the unit inside each rank's shard storage */
    int64_t param_offset; /* start of the unit's true parameters in the model */
    int64_t pad;          /* n_padded - n_params */
} zero_unit_t;

/* Per-rank accounting ([DZF] Theorem; [DDF] "Memory accounting"). */
typedef struct {
    double weight_bytes;    /* bf16 weights one rank keeps */
    double grad_bytes;      /* bf16 gradients one rank keeps */
    double optim_bytes;     /* optimizer state (K bytes per parameter) one rank keeps */
    double state_bytes;     /* their sum: model states per GPU */
    double comm_volume;     /* elements per step: 2P (DDP, ZeRO-1/2) or 3P (ZeRO-3) */
    double comm_sent_elems; /* ring elements sent per rank: volume*(N-1)/N */
    double comm_sent_bytes; /* the same at 2 bytes per element */
    double hbm_bytes;       /* algorithmic HBM bytes of the one-GPU emulated step:
                               (26 + 2N) per parameter, + 8 per parameter for
                               ZeRO-3's two unit gathers */
} zero_bytes_t;

/* zero_layout -- host only.  [DZF] "What is redundant" (GPU k owns slice k);
 * "How FSDP implements ZeRO-3", step 1 (equal chunks of the flat unit).
 *   unit_sizes[n_units]  true parameter count of each unit (> 0)
 *   n_ranks, align_elems shards are multiples of align_elems elements
 *   out_units[n_units]   filled with each unit's layout; units are padded one
 *                        by one and concatenated in order
 *   out_total_padded     sum of the units' n_padded
 * ZERO_EINVAL on a null pointer, n_units < 1, n_ranks outside [1, 64],
 * align_elems < 1 or not a multiple of 8, or a unit size <= 0. */
int zero_layout(const int64_t* unit_sizes, int32_t n_units, int32_t n_ranks,
                int32_t align_elems, zero_unit_t* out_units,
                int64_t* out_total_padded);

/* zero_step_stage12 -- the fused ZeRO-1/ZeRO-2 step, one pass over HBM.
 * [DZF] Theorem, proof steps 2, 3, 6; "The communication is already there".
 * For every element i of the flat padded buffer, with owner k = i / S:
 *   g   = (sum over r = 0..n_ranks-1, in that order, of fp32(grads[r][i]))
 *         * (float)(1/n_ranks)                                [reduce-scatter]
 *   AdamW on master[k], m[k], v[k] at i - k*S in fp32:          [update]
 *     m = b1*m + (1-b1)*g;  v = b2*v + ((1-b2)*g)*g;
 *     w = w - lr*((m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps) + wd*w)
 *   params_bf16[i] = bf16_round_nearest_even(w)                [all-gather]
 * Every operation is one IEEE fp32 operation, none fused; the fp32 scalars
 * are computed in double from *hp and rounded once.
 *   stage          1 (ZeRO-1) or 2 (ZeRO-2); identical results
 *   n_padded       P' (multiple of 8*n_ranks); S = n_padded / n_ranks
 *   grads          n_ranks device pointers, each n_padded bf16 (read only)
 *   master, m, v   n_ranks device pointers, each S fp32 (read and written)
 *   params_bf16    device pointer, n_padded bf16 (written): the replicated
 *                  weights every rank holds after the all-gather
 *   bucket_elems   stage 2: reduce-scatter+update bucket by bucket, in the
 *                  launches of one bucket of this many elements after another
 *                  (multiple of 8; 0 = whole buffer); ignored for stage 1.
 *                  Every launch after the call's first is a programmatic
 *                  dependent launch on the one before it (ZERO_CHUNK_ELEMS), so
 *                  it may start while that one drains; the call as a whole is
 *                  still ordered on the stream like one kernel.
 * Buffers must not overlap.  ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero_step_stage12(int32_t stage, int32_t n_ranks, int64_t n_padded,
                      const uint16_t* const* grads, float* const* master,
                      float* const* m, float* const* v, uint16_t* params_bf16,
                      const zero_hparams_t* hp, int64_t bucket_elems,
                      cudaStream_t stream);

/* zero3_gather_unit -- ZeRO-3 all-gather of one unit's bf16 parameters.
 * [DZF] "How FSDP implements ZeRO-3", steps 2-3; [COL] "Collectives" (every
 * rank gets all shards) and the per-unit step figure.
 *   full_unit[k*S_u + j] = shard_bf16[k][unit->shard_offset + j]
 *   for k < n_ranks, j < S_u = unit->shard_len.
 *   unit        layout from zero_layout (host pointer)
 *   shard_bf16  n_ranks device pointers: rank k's bf16 shard storage of ALL
 *               units (unit u at shard_offset)
 *   full_unit   device pointer, unit->n_padded bf16 (written)
 * A bit copy.  ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero3_gather_unit(const zero_unit_t* unit, int32_t n_ranks,
                      const uint16_t* const* shard_bf16, uint16_t* full_unit,
                      cudaStream_t stream);

/* zero3_reduce_scatter_unit -- ZeRO-3 gradient reduce-scatter of one unit,
 * fused with each owner's AdamW and the write of its new bf16 shard.
 * [DZF] "How FSDP implements ZeRO-3", steps 3-4; Theorem, proof step 7 (no
 * all-gather follows the update).  Per element i < unit->n_padded with owner
 * k = i / S_u and position p = unit->shard_offset + i - k*S_u: the same
 * reduce-scatter mean and AdamW as zero_step_stage12, on master[k][p],
 * m[k][p], v[k][p], then shard_bf16[k][p] = bf16_rne(new master).
 *   unit_grads     n_ranks device pointers, each unit->n_padded bf16
 *   master, m, v   n_ranks device pointers to each rank's fp32 shard storage
 *   shard_bf16     n_ranks device pointers to each rank's bf16 shard storage
 * ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero3_reduce_scatter_unit(const zero_unit_t* unit, int32_t n_ranks,
                              const uint16_t* const* unit_grads,
                              float* const* master, float* const* m,
                              float* const* v, uint16_t* const* shard_bf16,
                              const zero_hparams_t* hp, cudaStream_t stream);

/* zero_state_bytes -- host only.  [DZF] Theorem (table and proof); [DDF]
 * "Memory accounting" (state_bytes raises on params <= 0 or ranks < 1) and
 * "Communication and a roofline sanity check" (ring bytes).
 *   stage 0 = DDP, 1..3 = ZeRO-1..3; K = optimizer bytes per parameter (12
 *   for mixed-precision AdamW).  Model states per rank: (4+K)P, 4P+KP/N,
 *   2P+(2+K)P/N, (4+K)P/N.
 * ZERO_EINVAL on n_params <= 0, n_ranks < 1, stage outside [0,3], K < 0 or a
 * null out. */
int zero_state_bytes(int64_t n_params, int32_t n_ranks, int32_t stage, int32_t K,
                     zero_bytes_t* out);

/* ---------------------------------------------------------------------
 * fp32-gradient reduce-scatter.  [DZF] "Proposition (tokens that hide the
 * all-reduce)" (fp32 gradient reduction doubles the bytes) and "6. Where it
 * shows up" (Llama 3 reduce-scattered its gradients in fp32).  The rank
 * gradients are fp32 (4 bytes each, 26 + 4N bytes per parameter per step);
 * the mean is the same rank-order fp32 sum times (float)(1/N) and the
 * update, the bf16 write and every other argument are those of the bf16
 * calls.
 * ------------------------------------------------------------------- */
int zero_step_stage12_f32grads(int32_t stage, int32_t n_ranks, int64_t n_padded,
                               const float* const* grads, float* const* master, float* const* m,
                               float* const* v, uint16_t* params_bf16, const zero_hparams_t* hp,
                               int64_t bucket_elems, cudaStream_t stream);
int zero3_reduce_scatter_unit_f32grads(const zero_unit_t* unit, int32_t n_ranks,
                                       const float* const* unit_grads, float* const* master,
                                       float* const* m, float* const* v,
                                       uint16_t* const* shard_bf16, const zero_hparams_t* hp,
                                       cudaStream_t stream);

/* ---------------------------------------------------------------------
 * ZeRO-2 gradient accumulation.  [DZF] "Gradient accumulation": m
 * micro-batches run one after the other and their gradients are added before
 * one optimizer step; ZeRO-2 keeps no full gradient, so it reduce-scatters
 * after every micro-batch (m*P + P elements per step).  Each owner k keeps an
 * fp32 accumulator of its slice (S floats, caller memory).  Per element, with
 * mean_mu the reduce-scatter mean of micro-batch mu:
 *   acc = +0;  acc = acc + mean_mu  for mu = 1..m-1      (zero2_accumulate)
 *   g = (acc + mean_m) * (float)(1/m), then AdamW and the bf16 write, as in
 *   zero_step_stage12                               (zero2_step_accumulated)
 * ------------------------------------------------------------------- */

/* zero2_accumulate -- one earlier micro-batch: grad_acc[k] (n_ranks device
 * pointers, S fp32 each) = (first ? +0 : grad_acc[k]) + the mean of this
 * micro-batch's n_ranks bf16 gradients over rank k's slice.  Reads 2N bytes
 * per parameter (+4 unless first), writes 4.  ZERO_EINVAL / ZERO_EALIGN /
 * ZERO_ECUDA. */
int zero2_accumulate(int32_t n_ranks, int64_t n_padded, const uint16_t* const* grads,
                     float* const* grad_acc, int32_t first, cudaStream_t stream);

/* zero2_step_accumulated -- the last micro-batch fused with the step ([DZF]
 * "Gradient accumulation": one optimizer step per m micro-batches): the
 * fused kernel of zero_step_stage12 with g = (grad_acc + mean) * (1/m).
 * micro_batches = m >= 1; with m = 1 it is zero_step_stage12 (stage 2) and
 * grad_acc is not read.  Other arguments as zero_step_stage12. */
int zero2_step_accumulated(int32_t n_ranks, int64_t n_padded, const uint16_t* const* grads,
                           float* const* grad_acc, int32_t micro_batches, float* const* master,
                           float* const* m, float* const* v, uint16_t* params_bf16,
                           const zero_hparams_t* hp, cudaStream_t stream);

/* The same accumulation per ZeRO-3 unit (FSDP with m micro-batches: every
 * micro-batch gathers and reduce-scatters each unit, the 3mP volume of [DZF]
 * "Gradient accumulation"; the update runs once, with the last one).
 *
 * zero3_accumulate_unit -- zero2_accumulate over one unit.
 *   unit         a unit of zero_layout
 *   unit_grads   n_ranks device pointers, each the unit's n_padded bf16
 *                gradients of this micro-batch (read only)
 *   grad_acc     n_ranks device pointers to each rank's fp32 accumulator
 *                storage of all units (laid out like master: this unit at
 *                unit->shard_offset)
 *   first        1 for the step's first micro-batch (the accumulator is not
 *                read), else 0
 *
 * zero3_reduce_scatter_unit_accumulated -- the unit's last micro-batch fused
 * with its update: zero3_reduce_scatter_unit with g = (grad_acc + mean) *
 * (1/m), m = micro_batches >= 1 (m = 1: zero3_reduce_scatter_unit, grad_acc
 * not read).  Other arguments as zero3_reduce_scatter_unit.  Each unit gives
 * the bits zero2_accumulate / zero2_step_accumulated give on that unit as a
 * flat buffer (rank k's shard = slice k of the replicated buffer).
 * ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero3_accumulate_unit(const zero_unit_t* unit, int32_t n_ranks,
                          const uint16_t* const* unit_grads, float* const* grad_acc,
                          int32_t first, cudaStream_t stream);
int zero3_reduce_scatter_unit_accumulated(const zero_unit_t* unit, int32_t n_ranks,
                                          const uint16_t* const* unit_grads,
                                          float* const* grad_acc, int32_t micro_batches,
                                          float* const* master, float* const* m,
                                          float* const* v, uint16_t* const* shard_bf16,
                                          const zero_hparams_t* hp, cudaStream_t stream);

/* zero_reshard_f32 -- one unit's per-rank fp32 state (master, m or v; one
 * call each) re-laid from n_from to n_to ranks, for a run restarted on
 * another N_d ([DZF] "6. Where it shows up", checkpoints: sharded optimizer
 * state needs resharding).  Element i of the unit's flat order (i <
 * n_params) moves from rank i / S_from, position i % S_from, to rank
 * i / S_to, position i % S_to; the new layout's padding is written +0.
 *   from_unit, n_from   the unit's layout at the old rank count (zero_layout)
 *   src          n_from device pointers to each old rank's fp32 storage
 *                (this unit at from_unit->shard_offset), read only
 *   to_unit, n_to       the same unit (same n_params) at the new rank count
 *   dst          n_to device pointers (this unit at to_unit->shard_offset),
 *                written; dst must not overlap src
 * The bf16 shards of the new layout are the bf16 rounding of the new master
 * (zero_cast_bf16).  8 bytes per parameter.
 * ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero_reshard_f32(const zero_unit_t* from_unit, int32_t n_from, const float* const* src,
                     const zero_unit_t* to_unit, int32_t n_to, float* const* dst,
                     cudaStream_t stream);

/* ---------------------------------------------------------------------
 * Global gradient-norm clipping across the shards.  [DZF] "7. Common
 * mistakes" (local gradient clipping: with sharded gradients the global norm
 * needs an all-reduce of the squared shard norms); the rule of the
 * clip_grad_norm_ call in [DDF]'s DDP reference: norm = ||g||_2 of the whole
 * averaged gradient g, coef = max_norm / (norm + 1e-6), at most 1, and the
 * update uses g * coef.  Sequence per step: zero_grad_sqnorm over every
 * flat buffer or unit (accumulate = 0 for the first, 1 for the rest), then
 * zero_clip_coef, then the *_clip step calls, all on one stream; nothing
 * returns to the host.
 * ------------------------------------------------------------------- */

/* Bytes of device scratch the norm pass needs (1216 doubles, 9,728 B). */
int64_t zero_clip_scratch_bytes(void);

/* zero_grad_sqnorm -- adds the squared L2 norm of the averaged gradient of
 * one buffer (g[i] = fp32 rank-order mean of grads[r][i], exactly as the
 * fused step forms it) into per-block fp64 partials in scratch: the squared
 * shard norms whose sum is the global norm ([DZF] "7. Common mistakes").
 *   n_elems      length of each rank's buffer (multiple of 8)
 *   grads        n_ranks device pointers (read only)
 *   accumulate   0: overwrite the partials (first buffer of the step);
 *                1: add to them (further units)
 *   scratch      device, >= zero_clip_scratch_bytes(), 16-byte aligned; the
 *                caller owns it; calls that share it must be ordered
 * The partials and their summation order are fixed, so results repeat bit
 * for bit.  ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero_grad_sqnorm(int32_t n_ranks, int64_t n_elems, const uint16_t* const* grads,
                     int32_t accumulate, double* scratch, int64_t scratch_bytes,
                     cudaStream_t stream);

/* zero_clip_coef -- sums the partials (fp64, fixed order) and writes
 * norm_coef[0] = (float)norm and norm_coef[1] = (float)coef on the device,
 * coef = min(1, max_norm / (norm + 1e-6)): the rule of the clip_grad_norm_
 * call in [DDF]'s "A complete rank-aware DDP reference".
 *   max_norm   > 0, finite
 *   norm_coef  device float[2], 16-byte aligned */
int zero_clip_coef(const double* scratch, int64_t scratch_bytes, double max_norm,
                   float* norm_coef, cudaStream_t stream);

/* zero_step_stage12_clip / zero3_reduce_scatter_unit_clip -- the two fused
 * steps with the mean gradient multiplied (one fp32 multiply) by
 * norm_coef[1] before AdamW (clipping before the optimizer step, as in
 * [DDF]'s "A complete rank-aware DDP reference").  norm_coef: device float[2] written by
 * zero_clip_coef earlier on the same stream.  Other arguments as the
 * unclipped calls. */
int zero_step_stage12_clip(int32_t stage, int32_t n_ranks, int64_t n_padded,
                           const uint16_t* const* grads, float* const* master,
                           float* const* m, float* const* v, uint16_t* params_bf16,
                           const zero_hparams_t* hp, int64_t bucket_elems,
                           const float* norm_coef, cudaStream_t stream);
int zero3_reduce_scatter_unit_clip(const zero_unit_t* unit, int32_t n_ranks,
                                   const uint16_t* const* unit_grads, float* const* master,
                                   float* const* m, float* const* v,
                                   uint16_t* const* shard_bf16, const zero_hparams_t* hp,
                                   const float* norm_coef, cudaStream_t stream);

/* zero3_update_unit_reduced -- zero3_reduce_scatter_unit (or, with norm_coef,
 * its clipped form) reading the unit's mean gradient from the fp32 gradient
 * shard that zero_grad_reduce_sqnorm wrote ([DZF] "How FSDP implements
 * ZeRO-3", step 1: each rank keeps the fp32 shard of its gradient), instead of
 * reducing the rank gradients: the same bits.
 *   grad_shard   n_ranks device pointers to each rank's fp32 gradient shard
 *                storage of all units (laid out like master: this unit at
 *                unit->shard_offset), read only
 *   norm_coef    NULL or the device float[2] of zero_clip_coef
 *   other arguments as zero3_reduce_scatter_unit
 * 30 bytes per parameter.  When every fp32 pointer (master, m, v and
 * grad_shard, at this unit's offset) is 32-byte aligned the kernel moves 32
 * bytes per access, else 16; the bits are the same.
 * ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero3_update_unit_reduced(const zero_unit_t* unit, int32_t n_ranks,
                              const float* const* grad_shard, float* const* master,
                              float* const* m, float* const* v, uint16_t* const* shard_bf16,
                              const zero_hparams_t* hp, const float* norm_coef,
                              cudaStream_t stream);

/* The clipped ZeRO-1/2 step in two passes that keep the reduce-scatter's
 * output, FSDP's fp32 gradient shard ([DZF] "How FSDP implements ZeRO-3",
 * step 1: each rank keeps an fp32 shard of the gradient; [DZF] "7. Common
 * mistakes": the global norm needs every shard before any update).
 *
 * zero_grad_reduce_sqnorm -- zero_grad_sqnorm that also stores each element's
 * mean gradient g[i] = fp32 rank-order mean of grads[r][i] (the fused step's
 * own g) to its owner's shard: grad_shard[k][i - k*S], k = i / S.  The
 * partials equal zero_grad_sqnorm's bit for bit.
 *   n_elems      multiple of 8*n_ranks; S = n_elems / n_ranks
 *   grad_shard   n_ranks device pointers, each S fp32 (written)
 *   other arguments as zero_grad_sqnorm
 *
 * zero_step_stage12_reduced -- zero_step_stage12 (or, with norm_coef, the
 * clipped step) that reads g from grad_shard instead of reducing the rank
 * gradients: the same bits as zero_step_stage12 / zero_step_stage12_clip on
 * the gradients that filled the shard.
 *   grad_shard   n_ranks device pointers, each S fp32 (read only)
 *   norm_coef    NULL (no clipping) or the device float[2] of zero_clip_coef
 *
 * HBM bytes per parameter of a clipped step: 2N + 4 for the norm pass and
 * 30 for the update = 2N + 34, against 4N + 26 for zero_grad_sqnorm +
 * zero_step_stage12_clip (50 against 58 at N = 8).  The price is the fp32
 * shard: 4 bytes per parameter of device memory.  The update moves 32 bytes
 * per access when every fp32 pointer (master, m, v, grad_shard) is 32-byte
 * aligned, else 16; the bits are the same.
 * ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero_grad_reduce_sqnorm(int32_t n_ranks, int64_t n_elems, const uint16_t* const* grads,
                            float* const* grad_shard, int32_t accumulate, double* scratch,
                            int64_t scratch_bytes, cudaStream_t stream);
int zero_step_stage12_reduced(int32_t stage, int32_t n_ranks, int64_t n_padded,
                              const float* const* grad_shard, float* const* master,
                              float* const* m, float* const* v, uint16_t* params_bf16,
                              const zero_hparams_t* hp, int64_t bucket_elems,
                              const float* norm_coef, cudaStream_t stream);

/* zero_clip_coef_units_noalloc -- the same global-norm clip coefficient as
 * zero_grad_sqnorm over each unit followed by zero_clip_coef, for callers that
 * cannot allocate device memory (code running inside another framework whose
 * memory pool owns the GPU, a monitoring thread that must not touch the
 * training loop's allocator, a runtime held to a fixed memory budget).  The
 * pages have no counterpart: this is a library convenience.
 * The scratch is a fixed array inside the library (17,920 bytes of device
 * memory, held on every GPU that loads the library until the process exits);
 * no memory is allocated.  The caller passes inputs and outputs only:
 *   units[n_units]  layouts (host array); unit u's gradients of rank r start
 *                   at grads[r] + units[u].offset and span units[u].n_padded
 *   n_units         1 .. ZERO_NOALLOC_MAX_UNITS (more: ZERO_EINVAL, the
 *                   array's capacity)
 *   grads           n_ranks device pointers (read only)
 *   norm_coef       device float[2], 16-byte aligned: global norm, coefficient
 *   unit_norms      NULL or device float[n_units], 16-byte aligned: each
 *                   unit's gradient norm
 * Each unit's norm in unit_norms equals, bit for bit, norm_coef[0] of
 * zero_grad_sqnorm over that unit alone followed by zero_clip_coef (the same
 * block partials summed in the same order).  The global norm sums the units'
 * squared norms in a different association than zero_clip_coef does over
 * accumulated partials, so the two agree within fp32 rounding, not bit for bit.
 * The first call on a device looks up the array's device address with that
 * device current and keeps it for the process; make it before any stream
 * capture.  cudaDeviceReset rebuilds the device's context and may move the
 * array, so after a reset this entry point must not be called on that device
 * again in the same process.  All calls share the array: calls whose GPU work
 * overlaps (two streams, two threads) race; order them on one stream. */
#define ZERO_NOALLOC_MAX_UNITS 1024
int zero_clip_coef_units_noalloc(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                                 const uint16_t* const* grads, double max_norm,
                                 float* norm_coef, float* unit_norms, cudaStream_t stream);

/* ---------------------------------------------------------------------
 * ZeRO-3 step scheduler: the per-unit order of [DZF] "How FSDP implements
 * ZeRO-3", steps 2-5 (and [COL]'s per-unit step figure), issued natively.
 * ------------------------------------------------------------------- */

/* One operation of a ZeRO-3 step plan.  stream: 0 = main (reduce-scatter,
 * regeneration, unit use), 1 = side (gathers), 2 = the library's second
 * compute stream (the backward units of full buffer 1 when resharding
 * without regeneration: their use, reduce-scatter and buffer release), 3 =
 * the library's second side stream (the gathers into full buffer 1, or of
 * the units of odd positions without resharding).
 * RECORD/WAIT name one of the plan's seven reusable events in `arg` (0 = step
 * start, 1..2 = "unit gathered", 3..4 = "full buffer released", 5 = "the
 * second compute stream may start", 6 = "the second compute stream is
 * done"); GATHER names the unit and in `arg` the full buffer (0 or 1) it
 * fills; USE names the unit and in `arg` the full buffer it reads: it marks
 * where the unit's forward or backward compute would run (no work here);
 * REDUCE_SCATTER and REGEN name the unit. */
typedef struct {
    int32_t kind;
    int32_t stream;
    int32_t unit;
    int32_t arg;
} zero_op_t;

#define ZERO_OP_RECORD 1
#define ZERO_OP_WAIT 2
#define ZERO_OP_GATHER 3
#define ZERO_OP_REDUCE_SCATTER 4
#define ZERO_OP_REGEN 5
#define ZERO_OP_USE 6
#define ZERO_OP_NORM 7      /* unit's squared norm into the clip partials; arg = accumulate */
#define ZERO_OP_CLIP_COEF 8 /* global norm and clip coefficient */
#define ZERO_OP_ACCUMULATE 9 /* unit's micro-batch mean into the fp32 accumulator; arg = 1 first */

/* zero3_plan -- host only.  The operations of one ZeRO-3 step over n_units
 * units, in issue order: record "start" on main and make side wait for it;
 * forward over units 0..U-1 and backward over U-1..0, each pass gathering
 * unit p+1 into the other full buffer on the side stream (after the side
 * stream waits for that buffer's release) before the main stream waits for
 * unit p, uses it, and -- in the backward pass -- (optionally regenerates
 * and) reduce-scatters it, then records the buffer's release.  Two gathers
 * and one reduce-scatter per unit; at most two units gathered at a time.
 * With resharding and without regeneration (and more than one unit) the
 * backward units of full buffer 1 run on stream 2 instead of the main stream,
 * which records event 5 before the backward pass for stream 2 to wait on and
 * waits for stream 2's event 6 after it, so that consecutive units'
 * reduce-scatters overlap at their boundary instead of being separated by an
 * event wait and record on one stream (Llama-1.1B shapes on GB300: 7.94 ->
 * 7.77 ms a step).  With more than one unit the gathers into full buffer 1
 * (without resharding: of the units at odd positions) run on stream 3, which
 * also waits for event 0, so that consecutive gathers overlap as well (7.77
 * -> 7.68 ms).
 *   regen      non-zero: a REGEN op precedes each REDUCE_SCATTER (and each
 *              NORM)
 *   reshard_after_forward  0: [DZF] "How FSDP implements ZeRO-3", step 6 --
 *              the forward pass gathers every unit once into its own region
 *              (GATHER/USE arg = 2) and the backward pass uses the kept
 *              weights: one gather and one reduce-scatter per unit (2P)
 *   clip       non-zero: right after the start, NORM for every unit and one
 *              CLIP_COEF on the main stream, and REDUCE_SCATTER ops carry
 *              arg = 1 (scale by the coefficient)
 *   ops        caller array of max_ops entries; *n_ops receives the count
 *              (13*n_units + 7, plus n_units with regen, plus n_units + 1
 *              with clip, plus n_units with both, at most)
 * ZERO_EINVAL on n_units < 1, null pointers or max_ops too small. */
int zero3_plan(int32_t n_units, int32_t regen, int32_t clip, int32_t reshard_after_forward,
               zero_op_t* ops, int32_t max_ops, int32_t* n_ops);

/* zero3_plan_microbatch -- host only.  The plan of one micro-batch of a
 * ZeRO-3 step with gradient accumulation over micro_batches = m micro-batches
 * ([DZF] "Gradient accumulation": ZeRO-3 gathers twice and reduce-scatters in
 * every micro-batch, 3mP).  The plan of zero3_plan (no regeneration, no
 * clipping), except for what each backward unit does with its gradients:
 * ACCUMULATE (arg 1 for micro_batch 0) while micro_batch < m - 1, and in the
 * last micro-batch REDUCE_SCATTER with arg 2: added to the accumulator and
 * fused with the update.  m = 1 is zero3_plan's plan.
 * ZERO_EINVAL as zero3_plan, and unless 0 <= micro_batch < micro_batches. */
int zero3_plan_microbatch(int32_t n_units, int32_t reshard_after_forward, int32_t micro_batch,
                          int32_t micro_batches, zero_op_t* ops, int32_t max_ops,
                          int32_t* n_ops);

/* Harness regeneration of a unit's gradients inside zero3_step (the
 * stand-in for the backward compute that would produce them). */
typedef struct {
    uint64_t seed;
    double sigma;
    int32_t outliers;
} zero_regen_t;

/* Global-norm clipping inside zero3_step: the buffers of the clipping calls.
 * grad_shard: NULL, or n_ranks device pointers to each rank's fp32 gradient
 * shard storage of all units (laid out like master, S_total fp32 each).
 * With it the norm pre-pass is zero_grad_reduce_sqnorm, storing each unit's
 * mean gradient there, and each unit's update is zero3_update_unit_reduced,
 * reading it: 2N + 4 + 30 instead of 2N + 26 + 2N bytes per parameter of
 * norm pass and update, the same bits. */
typedef struct {
    double max_norm;
    double* scratch;       /* device, >= zero_clip_scratch_bytes() */
    int64_t scratch_bytes;
    float* norm_coef;      /* device float[2]: norm and coefficient of this step */
    float* const* grad_shard; /* host table of n_ranks device pointers, or NULL */
} zero_clip_t;

/* zero3_step -- one whole ZeRO-3 step ([DZF] "How FSDP implements ZeRO-3",
 * steps 2-5, and step 6 without resharding): executes zero3_plan's operations
 * with zero3_gather_unit, zero3_reduce_scatter_unit and (if regen != NULL)
 * zero_gen_grads_unit, on main_stream and side_stream, which must differ.
 *   units[n_units]   layouts from one zero_layout call (host array)
 *   grads            n_ranks device pointers.  grads_resident != 0: rank r's
 *                    gradients of every unit, concatenated (unit u at
 *                    units[u].offset, total padded length); == 0: one
 *                    buffer of the largest unit's n_padded, reused per unit
 *                    (requires regen, which fills it before each unit's
 *                    reduce-scatter)
 *   master, m, v, shard_bf16   as zero3_reduce_scatter_unit
 *   full_a, full_b   reshard_after_forward != 0: two device buffers of the
 *                    largest unit's n_padded bf16 (the double buffer);
 *                    == 0: full_a holds every unit's full weights (the total
 *                    padded length, unit u at units[u].offset, kept from the
 *                    forward to the backward pass), full_b is not used
 *   hp               the step's hyper-parameters (the same t for all units)
 *   clip             NULL, or global-norm clipping over all units (the norm
 *                    pre-pass reads every unit's gradients once more; with
 *                    clip->grad_shard it also keeps their mean, which the
 *                    updates then read instead of the gradients)
 * The library keeps seven timing-free CUDA events and two non-blocking CUDA
 * streams (streams 2 and 3 of zero3_plan) per host thread and device, created on
 * first use and kept for the thread's life (a cudaDeviceReset invalidates
 * them, so zero3_step must not be called on that device from that thread
 * again); no device memory is allocated.  While main_stream is being
 * captured the step keeps to main_stream and side_stream (zero3_graph_create
 * joins consecutive units and gathers with programmatic edges instead).  Work is queued
 * asynchronously; on return main_stream carries the end of the step.  Kernels
 * that follow one another on the main stream with nothing else between them
 * are chained with programmatic dependent launch (each may start while the
 * one before drains, and completes after it): the units' norm passes, and,
 * unless main_stream is being captured, the unit updates of the backward pass
 * without resharding (zero3_graph_create joins those in the graph itself).
 * ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero3_step(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
               const uint16_t* const* grads, int32_t grads_resident,
               float* const* master, float* const* m, float* const* v,
               uint16_t* const* shard_bf16, uint16_t* full_a, uint16_t* full_b,
               const zero_hparams_t* hp, const zero_regen_t* regen,
               const zero_clip_t* clip, int32_t reshard_after_forward,
               cudaStream_t main_stream, cudaStream_t side_stream);

/* zero3_step_f32grads -- zero3_step with fp32 rank gradients ([DZF] "6. Where
 * it shows up": Llama 3 reduce-scatters fp32 gradients): each unit's
 * reduce-scatter is zero3_reduce_scatter_unit_f32grads.  grads holds n_ranks
 * device pointers, each rank's fp32 gradients of every unit concatenated
 * (unit u at units[u].offset); no regeneration, no clipping.  Other
 * arguments as zero3_step.  26 + 4N bytes per parameter for the updates.
 * ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero3_step_f32grads(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                        const float* const* grads, float* const* master, float* const* m,
                        float* const* v, uint16_t* const* shard_bf16, uint16_t* full_a,
                        uint16_t* full_b, const zero_hparams_t* hp,
                        int32_t reshard_after_forward, cudaStream_t main_stream,
                        cudaStream_t side_stream);

/* zero3_step_checked -- zero3_step (without clipping) whose per-unit
 * reduce-scatters carry the fused pre-reduction finite check of
 * zero_step_stage12_checked ([DDF] "Failure investigation and recovery"):
 * bit r of nonfinite_ranks (device uint32[2], 8-byte aligned, zeroed by the
 * caller) is OR-ed in when rank r's gradient of any unit holds an infinity or
 * a NaN.  The results are zero3_step's bit for bit.  Arguments as zero3_step;
 * ZERO_EINVAL also for a null nonfinite_ranks, ZERO_EALIGN when it is not
 * 8-byte aligned (both before anything is issued). */
int zero3_step_checked(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                       const uint16_t* const* grads, int32_t grads_resident,
                       float* const* master, float* const* m, float* const* v,
                       uint16_t* const* shard_bf16, uint16_t* full_a, uint16_t* full_b,
                       const zero_hparams_t* hp, const zero_regen_t* regen,
                       int32_t reshard_after_forward, uint32_t* nonfinite_ranks,
                       cudaStream_t main_stream, cudaStream_t side_stream);

/* zero3_step_microbatch -- one micro-batch of a ZeRO-3 step with gradient
 * accumulation ([DZF] "Gradient accumulation", the 3mP row: both gathers and
 * the reduce-scatter in every micro-batch): zero3_plan_microbatch's
 * operations, issued like zero3_step's
 * (every unit's bf16 gradients of this micro-batch resident; no regeneration,
 * no clipping).  Call it for micro_batch = 0 .. m-1 in order, refilling the
 * gradients between calls; the update happens in the last call, with
 * g = (accumulator + mean) * (1/m) as zero3_reduce_scatter_unit_accumulated.
 *   grad_acc     n_ranks device pointers to each rank's fp32 accumulator
 *                storage of all units (laid out like master); not read when
 *                micro_batches = 1
 *   other arguments as zero3_step
 * ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero3_step_microbatch(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                          const uint16_t* const* grads, float* const* grad_acc,
                          int32_t micro_batch, int32_t micro_batches, float* const* master,
                          float* const* m, float* const* v, uint16_t* const* shard_bf16,
                          uint16_t* full_a, uint16_t* full_b, const zero_hparams_t* hp,
                          int32_t reshard_after_forward, cudaStream_t main_stream,
                          cudaStream_t side_stream);

/* zero3_graph -- the zero3_step of one fixed set of buffers captured once as a
 * CUDA graph and replayed once per step.  The operations, their order and
 * their results are zero3_step's; a replay gives the GPU the step's whole
 * dependency structure at once (event records and waits become graph edges).
 * That saves the launch and event latency between the kernels of models with
 * many small units.  The pages have no counterpart: it is how this library
 * issues [DZF] "How FSDP implements ZeRO-3", steps 2-5, on one GPU.
 *
 * zero3_graph_create -- captures one step.
 *   units .. full_b, clip, reshard_after_forward   as zero3_step, with the
 *                    gradients resident (grads_resident = 1; no regeneration)
 *   hp               any valid hyper-parameters (checked; the step's own come
 *                    with each launch)
 *   capture_stream   a stream created by the caller (not the legacy default
 *                    stream, and not being captured already); the step is
 *                    captured from it
 *   side_stream      a second stream, != capture_stream, idle during the call
 *   out              receives the graph handle
 * The call captures and instantiates; it runs no kernel and changes no
 * buffer.  The buffers must stay allocated, at the same addresses, until
 * zero3_graph_destroy.  This call and the graph, unlike the others, hold
 * host memory and the driver's resources for the graph.  Arguments
 * zero3_step would reject give its code, and nothing is created.
 * ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA (a capture or instantiation error).
 *
 * zero3_graph_launch -- queues one step on `stream` (any stream of the device
 * the graph was created on; ZERO_EINVAL on another device or invalid hp).
 * The AdamW scalars of every unit's fused kernel are set from *hp before the
 * replay, so t, lr, betas, eps and weight decay may change from launch to
 * launch; a replay already queued keeps the scalars it was launched with.
 * Launches of one graph must be made from one host thread at a time.
 *
 * zero3_graph_create_f32grads -- the same for zero3_step_f32grads: grads
 * holds each rank's fp32 gradients of every unit (resident), there is no
 * clipping; the other arguments, the graph and its launches as above.
 *
 * zero3_graph_destroy -- releases the graph (NULL: no-op).  Call it after
 * the last launch has completed. */
typedef struct zero3_graph zero3_graph_t;
int zero3_graph_create(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                       const uint16_t* const* grads, float* const* master, float* const* m,
                       float* const* v, uint16_t* const* shard_bf16, uint16_t* full_a,
                       uint16_t* full_b, const zero_hparams_t* hp, const zero_clip_t* clip,
                       int32_t reshard_after_forward, cudaStream_t capture_stream,
                       cudaStream_t side_stream, zero3_graph_t** out);
int zero3_graph_create_f32grads(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                                const float* const* grads, float* const* master,
                                float* const* m, float* const* v, uint16_t* const* shard_bf16,
                                uint16_t* full_a, uint16_t* full_b, const zero_hparams_t* hp,
                                int32_t reshard_after_forward, cudaStream_t capture_stream,
                                cudaStream_t side_stream, zero3_graph_t** out);
int zero3_graph_launch(zero3_graph_t* graph, const zero_hparams_t* hp, cudaStream_t stream);
int zero3_graph_destroy(zero3_graph_t* graph);

/* zero_grad_nonfinite -- pre-reduction finite check ([DDF] "Failure
 * investigation and recovery": record per-rank finite checks before the
 * reduction, so that it does not conceal where a NaN came from).  Adds to
 * counts[r] the number of rank r's bf16 gradients that are infinite or NaN.
 *   n_elems  length of each rank's buffer (multiple of 8)
 *   counts   device uint32[n_ranks], 16-byte aligned; reset != 0 zeroes it
 *            first (on the stream), otherwise counts accumulate over calls
 * Exact integer counts, independent of order.  Reads 2N bytes per
 * parameter.  ZERO_EINVAL / ZERO_EALIGN / ZERO_ECUDA. */
int zero_grad_nonfinite(int32_t n_ranks, int64_t n_elems, const uint16_t* const* grads,
                        uint32_t* counts, int32_t reset, cudaStream_t stream);

/* zero_step_stage12_checked / zero3_reduce_scatter_unit_checked -- the fused
 * ZeRO-1/2 step and the ZeRO-3 unit reduce-scatter + AdamW with the same
 * pre-reduction finite check done on the gradient values the reduction loads
 * anyway, so it adds no memory traffic ([DDF] "Failure investigation and
 * recovery": which rank a NaN came from).  The results are those of
 * zero_step_stage12 / zero3_reduce_scatter_unit bit for bit (a non-finite
 * gradient propagates by IEEE arithmetic as there; nothing is skipped).
 *   nonfinite_ranks  device uint32[2], 8-byte aligned: bit r % 32 of word
 *                    r / 32 is set (OR-ed in) when rank r's gradient of this
 *                    call holds an infinity or a NaN; bits are never cleared,
 *                    so the caller zeroes the words (e.g. before each step)
 *   other arguments as zero_step_stage12 / zero3_reduce_scatter_unit
 * Only the presence per rank is recorded; zero_grad_nonfinite counts.
 * ZERO_EINVAL (also for a null nonfinite_ranks) / ZERO_EALIGN / ZERO_ECUDA. */
int zero_step_stage12_checked(int32_t stage, int32_t n_ranks, int64_t n_padded,
                              const uint16_t* const* grads, float* const* master,
                              float* const* m, float* const* v, uint16_t* params_bf16,
                              const zero_hparams_t* hp, int64_t bucket_elems,
                              uint32_t* nonfinite_ranks, cudaStream_t stream);
int zero3_reduce_scatter_unit_checked(const zero_unit_t* unit, int32_t n_ranks,
                                      const uint16_t* const* unit_grads, float* const* master,
                                      float* const* m, float* const* v,
                                      uint16_t* const* shard_bf16, const zero_hparams_t* hp,
                                      uint32_t* nonfinite_ranks, cudaStream_t stream);

/* ---------------------------------------------------------------------
 * Harness calls: seeded synthetic inputs and helpers.  They are not part
 * of the method; the benchmark and the tests use them to fill device
 * buffers without a host round trip.
 * ------------------------------------------------------------------- */

/* zero_gen_grads_unit -- rank r's bf16 gradient of one unit at step t (a
 * harness input; no page defines it: SplitMix64, Steele, Lea and Flood 2014).
 * Element j < unit->n_params holds bf16_rne(z), z drawn by a SplitMix64
 * counter stream keyed by (seed, stream 1, step, r) at the true parameter
 * index unit->param_offset + j (an approximately normal value of standard
 * deviation sigma; with outliers != 0 one value in a hundred is scaled by
 * 100).  Padding elements are +0.
 *   unit_grads  n_ranks device pointers, each unit->n_padded bf16 (written) */
int zero_gen_grads_unit(uint64_t seed, int64_t step, double sigma, int32_t outliers,
                        const zero_unit_t* unit, int32_t n_ranks,
                        uint16_t* const* unit_grads, cudaStream_t stream);

/* zero_gen_grads_unit_f32 -- the same draws as zero_gen_grads_unit kept in
 * fp32 (no bf16 rounding): inputs of the fp32-gradient calls (harness; the
 * fp32 gradients of [DZF] "6. Where it shows up").
 *   unit_grads  n_ranks device pointers, each unit->n_padded fp32 (written) */
int zero_gen_grads_unit_f32(uint64_t seed, int64_t step, double sigma, int32_t outliers,
                            const zero_unit_t* unit, int32_t n_ranks, float* const* unit_grads,
                            cudaStream_t stream);

/* zero_gen_master -- initial fp32 master weights of every unit (harness: the
 * fp32 master copy of [DDF] "Memory accounting", filled with synthetic
 * values), written into each owner's shard storage: true parameter p draws from (seed, stream 0,
 * step 0, rank 0) at index p with standard deviation sigma; padding is +0.
 *   units[n_units]  layout from zero_layout (host array)
 *   master          n_ranks device pointers to fp32 shard storage */
int zero_gen_master(uint64_t seed, double sigma, const zero_unit_t* units,
                    int32_t n_units, int32_t n_ranks, float* const* master,
                    cudaStream_t stream);

/* zero_cast_bf16 -- dst[i] = bf16_rne(src[i]) for i < n (n a multiple of 8):
 * the initial bf16 replica or shard of fp32 master weights (the bf16
 * parameters beside the fp32 master of [DDF] "Memory accounting"). */
int zero_cast_bf16(const float* src, uint16_t* dst, int64_t n, cudaStream_t stream);

/* zero_stream_wait -- host wait for all work on a stream, polling with a
 * wall-clock limit instead of blocking forever, so that a stuck step is seen
 * and rank progress can be compared ([DDF] "Failure investigation and
 * recovery", a collective hang).  ZERO_ETIMEOUT if the work
 * has not finished after timeout_ms milliseconds (the work is left running),
 * ZERO_ECUDA if the stream reports an error. */
int zero_stream_wait(cudaStream_t stream, int64_t timeout_ms);

/* zero_strerror -- a static string naming a return code (no page defines
 * it). */
const char* zero_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* ZERO_H */
