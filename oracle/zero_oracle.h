/*
 * zero_oracle.h -- the CPU oracle of the sharded ZeRO/FSDP optimizer step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the package's
 * smoke check and the benchmark's CPU-baseline / reference legs load this
 * library.  It shares no code, header, table or helper with the CUDA path.
 *
 * Plain, single-threaded C.  Build with -O2 -ffp-contract=off and without
 * -ffast-math so that every + - * / sqrt below is exactly one IEEE-754
 * binary32 (or binary64) operation rounded to nearest-even, never fused.
 *
 * Sources (page title, section):
 *  [DZF]  "Data parallelism, ZeRO and FSDP" (ML Systems, lesson 8)
 *         - "2. The picture" (two GPUs, one batch; what is redundant;
 *           the communication is already there)
 *         - "3. Definitions and main results" (Proposition: DDP is exact;
 *           Theorem: ZeRO memory and communication; gradient accumulation;
 *           how FSDP implements ZeRO-3)
 *         - "5. In code", first block (the NumPy ZeRO-1 simulator and its
 *           AdamW update), third block (FSDP2 gloo check)
 *  [DDF]  "Distributed Training Basics -- DDP and FSDP"
 *         - "Memory accounting: derive the table from bytes"
 *         - "Communication and a roofline sanity check"
 *  [COL]  "Data parallelism, collectives and ZeRO/FSDP"
 *         - "Collectives", "ZeRO and FSDP" (table and the per-unit figure)
 *
 * Parity status: every function below is pinned by a test in tests/ against
 * values the pages print, closed forms or brute force, except where its
 * comment says "parity unpinned".
 */
#ifndef ZERO_ORACLE_H
#define ZERO_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OR_OK 0
#define OR_EINVAL (-1)
#define OR_EMISMATCH (-2) /* a literal simulator found replicas that disagree */

/* AdamW hyper-parameters; step is the 1-based step counter t. */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    int64_t step;
} or_hparams_t;

/* Layout of one FSDP unit (one communication group, [DZF] "How FSDP
 * implements ZeRO-3", step 1).  The unit's parameters are flattened and padded
 * to a multiple of n_ranks*align, then cut into n_ranks equal chunks. */
typedef struct {
    int64_t n_params;     /* true parameters of the unit */
    int64_t n_padded;     /* n_params rounded up to a multiple of n_ranks*align */
    int64_t shard_len;    /* n_padded / n_ranks: the chunk each rank owns */
    int64_t offset;       /* start of the unit in the concatenated padded buffer */
    int64_t shard_offset; /* start of the unit inside each rank's shard storage */
    int64_t param_offset; /* start of the unit's true parameters in the model */
    int64_t pad;          /* n_padded - n_params */
} or_unit_t;

/* The fp32 scalars of one step, each computed in double and rounded once. */
typedef struct {
    float b1, b2, omb1, omb2, bc1, bc2, lr, eps, wd, inv_n;
} or_scalars_t;

/* Per-rank byte/element accounting ([DZF] Theorem; [DDF] memory accounting
 * and ring byte counts).  All quantities are per rank. */
typedef struct {
    double weight_bytes;    /* bf16 weights kept by one rank */
    double grad_bytes;      /* bf16 gradients kept by one rank */
    double optim_bytes;     /* optimizer state (K bytes/param) kept by one rank */
    double state_bytes;     /* the sum: the theorem's "model states per GPU" */
    double comm_volume;     /* the theorem's volume in elements: 2P or 3P */
    double comm_sent_elems; /* ring elements sent: volume * (N-1)/N */
    double comm_sent_bytes; /* the same in bytes at 2 bytes per element */
    double hbm_bytes;       /* algorithmic HBM bytes of the one-GPU emulated step */
} or_bytes_t;

/* ---------------------------------------------------------------- layout */
int or_layout(const int64_t* unit_sizes, int32_t n_units, int32_t n_ranks,
              int32_t align, or_unit_t* out_units, int64_t* out_total_padded);

/* -------------------------------------------------------- elementwise math */
uint16_t or_bf16_rne(float x);
void or_bf16_rne_array(const float* x, int64_t n, uint16_t* out);
float or_bf16_to_f32(uint16_t b);
void or_scalars(const or_hparams_t* hp, int32_t n_ranks, or_scalars_t* out);
float or_reduce_mean(const uint16_t* const* grads, int32_t n_ranks, int64_t i,
                     float inv_n);
void or_adamw(float g, float* w, float* m, float* v, const or_scalars_t* s);
void or_adamw_f64(double g, double* w, double* m, double* v,
                  const or_hparams_t* hp);

/* ------------------------------------------------------- whole-buffer steps */
int or_zero12_step(int32_t stage, int32_t n_ranks, int64_t n_padded,
                   const uint16_t* const* grads, float* const* master,
                   float* const* m, float* const* v, uint16_t* params_bf16,
                   const or_hparams_t* hp, int64_t bucket_elems);
int or_zero3_gather_unit(const or_unit_t* unit, int32_t n_ranks,
                         const uint16_t* const* shard_bf16, uint16_t* full_unit);
int or_zero3_reduce_scatter_unit(const or_unit_t* unit, int32_t n_ranks,
                                 const uint16_t* const* unit_grads,
                                 float* const* master, float* const* m,
                                 float* const* v, uint16_t* const* shard_bf16,
                                 const or_hparams_t* hp);

/* Re-lays one unit's per-rank fp32 state from n_from to n_to ranks (a
 * restart on another N_d, [DZF] "6. Where it shows up", checkpoints). */
int or_reshard_f32(const or_unit_t* from, int32_t n_from, const float* const* src,
                   const or_unit_t* to, int32_t n_to, float* const* dst);

/* ------------------------------------------------ global grad-norm clipping */
double or_grad_sumsq(int32_t n_ranks, int64_t n, const uint16_t* const* grads);
float or_clip_coef(double sumsq, double max_norm, double* out_norm);
int or_zero12_step_clip(int32_t stage, int32_t n_ranks, int64_t n_padded,
                        const uint16_t* const* grads, float* const* master,
                        float* const* m, float* const* v, uint16_t* params_bf16,
                        const or_hparams_t* hp, int64_t bucket_elems, double max_norm,
                        double* out_norm, float* out_coef);
int or_zero3_reduce_scatter_unit_coef(const or_unit_t* unit, int32_t n_ranks,
                                      const uint16_t* const* unit_grads,
                                      float* const* master, float* const* m,
                                      float* const* v, uint16_t* const* shard_bf16,
                                      const or_hparams_t* hp, float coef);

/* ------------------------------------------------ ZeRO-2 gradient accumulation */
int or_zero2_accumulate(int32_t n_ranks, int64_t n_padded, const uint16_t* const* grads,
                        float* const* grad_acc, int32_t first);
int or_zero2_step_accumulated(int32_t n_ranks, int64_t n_padded, const uint16_t* const* grads,
                              const float* const* grad_acc, int32_t micro_batches,
                              float* const* master, float* const* m, float* const* v,
                              uint16_t* params_bf16, const or_hparams_t* hp);
double or_comm_volume(int32_t stage, int32_t micro_batches, int32_t reshard_after_forward,
                      double n_params);

/* ------------------------------------------------ fp32-gradient reduce-scatter */
float or_reduce_mean_f32(const float* const* grads, int32_t n_ranks, int64_t i, float inv_n);
int or_zero12_step_f32grads(int32_t stage, int32_t n_ranks, int64_t n_padded,
                            const float* const* grads, float* const* master, float* const* m,
                            float* const* v, uint16_t* params_bf16, const or_hparams_t* hp,
                            int64_t bucket_elems);
int or_zero3_reduce_scatter_unit_f32grads(const or_unit_t* unit, int32_t n_ranks,
                                          const float* const* unit_grads, float* const* master,
                                          float* const* m, float* const* v,
                                          uint16_t* const* shard_bf16, const or_hparams_t* hp);
void or_gen_grads_unit_f32(uint64_t seed, int64_t step, double sigma, int32_t outliers,
                           const or_unit_t* unit, int32_t n_ranks, float* const* unit_grads);

/* ------------------------------------------ pre-reduction finite check */
void or_grad_nonfinite(int32_t n_ranks, int64_t n, const uint16_t* const* grads,
                       uint32_t* counts);

/* ------------------------------------------------------------- accounting */
int or_state_bytes(int64_t n_params, int32_t n_ranks, int32_t stage, int32_t K,
                   or_bytes_t* out);
double or_ring_sent_bytes(double payload_bytes, int32_t n_ranks, int32_t kind);

/* ------------------------------------------------- seeded synthetic inputs */
uint64_t or_splitmix64_next(uint64_t* state);
uint64_t or_gen_key(uint64_t seed, uint64_t stream, uint64_t step, uint64_t rank);
float or_gen_value(uint64_t key, uint64_t index, float scale, int32_t outliers);
float or_gen_scale(double sigma);
void or_gen_master(uint64_t seed, double sigma, const or_unit_t* units,
                   int32_t n_units, int32_t n_ranks, float* const* master);
void or_gen_grads_unit(uint64_t seed, int64_t step, double sigma, int32_t outliers,
                       const or_unit_t* unit, int32_t n_ranks,
                       uint16_t* const* unit_grads);

/* --------------------------------------------- literal rank simulators */
int or_sim_ddp(int32_t n_ranks, int64_t n_params, uint64_t seed, double sigma_w,
               double sigma_g, int32_t outliers, const or_hparams_t* hp0,
               int32_t n_steps, uint16_t* out_params, float* out_master,
               float* out_m, float* out_v);
int or_sim_zero(int32_t stage, int32_t n_ranks, const int64_t* unit_sizes,
                int32_t n_units, int32_t align, uint64_t seed, double sigma_w,
                double sigma_g, int32_t outliers, const or_hparams_t* hp0,
                int32_t n_steps, int64_t bucket_elems, uint16_t* out_params,
                float* out_master, float* out_m, float* out_v,
                int64_t* out_counts);

/* ---------------------------------------------- sampled element parity */
void or_sample(int32_t n_ranks, uint64_t seed, double sigma_w, double sigma_g,
               int32_t outliers, const or_hparams_t* hp0, int32_t n_steps,
               const int64_t* param_index, int64_t n_index, uint16_t* out_params,
               float* out_master, float* out_m, float* out_v);
/* The same under global-norm clipping: the mean gradient of step t (0-based,
 * step hp0->step + t) is multiplied by coef[t] before AdamW. */
void or_sample_coef(int32_t n_ranks, uint64_t seed, double sigma_w, double sigma_g,
                    int32_t outliers, const or_hparams_t* hp0, int32_t n_steps,
                    const float* coef, const int64_t* param_index, int64_t n_index,
                    uint16_t* out_params, float* out_master, float* out_m, float* out_v);
/* The same with gradient accumulation over micro_batches identical
 * micro-batches (or_zero2_accumulate for the first micro_batches - 1, then
 * or_zero2_step_accumulated, every micro-batch carrying the step's gradients). */
void or_sample_accum(int32_t n_ranks, uint64_t seed, double sigma_w, double sigma_g,
                     int32_t outliers, const or_hparams_t* hp0, int32_t n_steps,
                     int32_t micro_batches, const int64_t* param_index, int64_t n_index,
                     uint16_t* out_params, float* out_master, float* out_m, float* out_v);
/* The same as or_sample with one gradient set for every step: the generated
 * rank gradients of step grad_step (>= 1), applied at AdamW steps hp0->step,
 * hp0->step + 1, ... (a job that keeps its gradients resident). */
void or_sample_fixed_grads(int32_t n_ranks, uint64_t seed, double sigma_w, double sigma_g,
                           int32_t outliers, const or_hparams_t* hp0, int32_t n_steps,
                           int64_t grad_step, const int64_t* param_index, int64_t n_index,
                           uint16_t* out_params, float* out_master, float* out_m, float* out_v);

#ifdef __cplusplus
}
#endif
#endif
