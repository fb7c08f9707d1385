/*
 * zero_oracle.c -- the CPU oracle of the sharded ZeRO/FSDP optimizer step.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE (see zero_oracle.h).  Plain,
 * single-threaded, slow on purpose: each function is the definition written
 * out, in the order the pages state it, with no blocking, fusion or
 * reordering beyond that definition.
 *
 * Readings where the pages leave a step open (each one is listed with its
 * reason in the design notes of the repository):
 *  - scalars: every fp32 constant of a step is computed in double from the
 *    double hyper-parameters and rounded to fp32 once; b^t uses libm pow;
 *  - the mean of the reduce-scatter is a multiply by (float)(1/N) after an
 *    fp32 sum that starts at +0 and adds ranks 0..N-1 in order;
 *  - the AdamW update keeps the page's operand order, including
 *    ((1-b2)*g)*g for the second moment and w - lr*(mh/(sqrt(vh)+eps) + wd*w)
 *    with the pre-update w on the right;
 *  - the split is into N equal chunks of a buffer padded to a multiple of
 *    N*align (the FlatParameter reading), not NumPy's uneven array_split;
 *  - padding carries +0 gradients and +0 state, and so stays +0;
 *  - bf16 rounding is to nearest, ties to even; NaN becomes 0x7FC0.
 */
#include "zero_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================
 * Layout: [DZF] "What is redundant" (GPU k owns slice k) and "How FSDP
 * implements ZeRO-3", step 1 (a unit's FlatParameter is split into N_d
 * equal chunks).  Units are padded one by one and concatenated.
 * ==================================================================== */
int or_layout(const int64_t* unit_sizes, int32_t n_units, int32_t n_ranks,
              int32_t align, or_unit_t* out_units, int64_t* out_total_padded)
{
    if (!unit_sizes || !out_units || !out_total_padded || n_units < 1 ||
        n_ranks < 1 || align < 1)
        return OR_EINVAL;
    int64_t chunk = (int64_t)n_ranks * (int64_t)align;
    int64_t offset = 0, param_offset = 0;
    for (int32_t u = 0; u < n_units; ++u) {
        int64_t p = unit_sizes[u];
        if (p <= 0)
            return OR_EINVAL;
        int64_t n_chunks = p / chunk;
        if (n_chunks * chunk < p)
            n_chunks += 1;
        or_unit_t U;
        U.n_params = p;
        U.n_padded = n_chunks * chunk;
        U.shard_len = U.n_padded / n_ranks;
        U.offset = offset;
        U.shard_offset = offset / n_ranks;
        U.param_offset = param_offset;
        U.pad = U.n_padded - p;
        out_units[u] = U;
        offset += U.n_padded;
        param_offset += p;
    }
    *out_total_padded = offset;
    return OR_OK;
}

/* ======================================================================
 * bf16 <-> fp32.  bf16 is the upper half of a binary32.  Rounding keeps the
 * nearer of the two neighbouring bf16 values; on a tie, the one whose last
 * kept bit is 0.
 * ==================================================================== */
uint16_t or_bf16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u)
        return 0x7FC0; /* NaN */
    uint32_t below = u >> 16;        /* truncation toward zero in magnitude */
    uint32_t rest = u & 0xFFFFu;     /* the discarded half */
    uint32_t keep;
    if (rest > 0x8000u)
        keep = below + 1u;
    else if (rest < 0x8000u)
        keep = below;
    else
        keep = (below & 1u) ? below + 1u : below;
    return (uint16_t)keep;
}

void or_bf16_rne_array(const float* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = or_bf16_rne(x[i]);
}

float or_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ======================================================================
 * The scalars of step t.  The pages' update is [DZF] "5. In code", first
 * block: m = b1 m + (1-b1) g; v = b2 v + (1-b2) g g; mh = m/(1-b1^t);
 * vh = v/(1-b2^t); w = w - lr (mh/(sqrt(vh)+eps) + wd w).
 * ==================================================================== */
void or_scalars(const or_hparams_t* hp, int32_t n_ranks, or_scalars_t* s)
{
    double t = (double)hp->step;
    s->b1 = (float)hp->beta1;
    s->b2 = (float)hp->beta2;
    s->omb1 = (float)(1.0 - hp->beta1);
    s->omb2 = (float)(1.0 - hp->beta2);
    s->bc1 = (float)(1.0 - pow(hp->beta1, t));
    s->bc2 = (float)(1.0 - pow(hp->beta2, t));
    s->lr = (float)hp->lr;
    s->eps = (float)hp->eps;
    s->wd = (float)hp->weight_decay;
    s->inv_n = (float)(1.0 / (double)n_ranks);
}

/* The reduce-scatter with a mean: GPU k receives slice k of the average of
 * the N_d rank gradients ([DZF] "The communication is already there";
 * Proposition "DDP is exact", step 3; simulator: np.mean over ranks).
 * fp32 sum from +0 in rank order, then one multiply by 1/N. */
float or_reduce_mean(const uint16_t* const* grads, int32_t n_ranks, int64_t i,
                     float inv_n)
{
    float g = 0.0f;
    for (int32_t r = 0; r < n_ranks; ++r)
        g = g + or_bf16_to_f32(grads[r][i]);
    return g * inv_n;
}

/* AdamW on one element in fp32, in the page's operand order. */
void or_adamw(float g, float* w, float* m, float* v, const or_scalars_t* s)
{
    float w0 = *w;
    float m1 = s->b1 * *m + s->omb1 * g;
    float v1 = s->b2 * *v + s->omb2 * g * g;
    float mh = m1 / s->bc1;
    float vh = v1 / s->bc2;
    float w1 = w0 - s->lr * (mh / (sqrtf(vh) + s->eps) + s->wd * w0);
    *w = w1;
    *m = m1;
    *v = v1;
}

/* The same update in binary64 with binary64 scalars: the page's NumPy
 * arithmetic, used to bound the fp32 rounding error of or_adamw. */
void or_adamw_f64(double g, double* w, double* m, double* v,
                  const or_hparams_t* hp)
{
    double t = (double)hp->step;
    double w0 = *w;
    double m1 = hp->beta1 * *m + (1.0 - hp->beta1) * g;
    double v1 = hp->beta2 * *v + (1.0 - hp->beta2) * g * g;
    double mh = m1 / (1.0 - pow(hp->beta1, t));
    double vh = v1 / (1.0 - pow(hp->beta2, t));
    *w = w0 - hp->lr * (mh / (sqrt(vh) + hp->eps) + hp->weight_decay * w0);
    *m = m1;
    *v = v1;
}

static int bad_hp(const or_hparams_t* hp)
{
    return !hp || hp->step < 1;
}

/* ======================================================================
 * ZeRO-1 / ZeRO-2 step on one flat padded buffer ([DZF] Theorem, proof
 * steps 2, 3 and 6): reduce-scatter the gradients, GPU k updates slice k,
 * all-gather the new weights.  The all-gathered replicas are identical, so
 * one replicated bf16 buffer stands for all of them.  ZeRO-2 reduces bucket
 * by bucket ([DZF] Theorem, proof step 3); the arithmetic per element is the
 * same, so the two stages give the same bits.
 * ==================================================================== */
int or_zero12_step(int32_t stage, int32_t n_ranks, int64_t n_padded,
                   const uint16_t* const* grads, float* const* master,
                   float* const* m, float* const* v, uint16_t* params_bf16,
                   const or_hparams_t* hp, int64_t bucket_elems)
{
    if ((stage != 1 && stage != 2) || n_ranks < 1 || n_padded <= 0 ||
        n_padded % n_ranks != 0 || !grads || !master || !m || !v ||
        !params_bf16 || bad_hp(hp) || bucket_elems < 0)
        return OR_EINVAL;
    int64_t S = n_padded / n_ranks;
    or_scalars_t s;
    or_scalars(hp, n_ranks, &s);
    int64_t bucket = (stage == 2 && bucket_elems > 0) ? bucket_elems : n_padded;
    for (int64_t b0 = 0; b0 < n_padded; b0 += bucket) {
        int64_t b1 = b0 + bucket < n_padded ? b0 + bucket : n_padded;
        for (int64_t i = b0; i < b1; ++i) {
            int64_t k = i / S;      /* owner */
            int64_t j = i - k * S;  /* position inside the owner's slice */
            float g = or_reduce_mean(grads, n_ranks, i, s.inv_n);
            or_adamw(g, &master[k][j], &m[k][j], &v[k][j], &s);
            params_bf16[i] = or_bf16_rne(master[k][j]);
        }
    }
    return OR_OK;
}

/* ======================================================================
 * ZeRO-3 unit all-gather ([DZF] "How FSDP implements ZeRO-3", steps 2-3;
 * [COL] "Collectives": every rank gets all shards): chunk k of the full
 * unit is rank k's bf16 shard of that unit.
 * ==================================================================== */
int or_zero3_gather_unit(const or_unit_t* unit, int32_t n_ranks,
                         const uint16_t* const* shard_bf16, uint16_t* full_unit)
{
    if (!unit || n_ranks < 1 || !shard_bf16 || !full_unit ||
        unit->shard_len * n_ranks != unit->n_padded)
        return OR_EINVAL;
    for (int32_t k = 0; k < n_ranks; ++k)
        for (int64_t j = 0; j < unit->shard_len; ++j)
            full_unit[(int64_t)k * unit->shard_len + j] =
                shard_bf16[k][unit->shard_offset + j];
    return OR_OK;
}

/* A restart on another N_d ([DZF] "6. Where it shows up", checkpoints: sharded
 * optimizer state must be resharded).  Element i of the unit's flat order
 * (i < n_params) sits at rank i / S_from, position i % S_from, and moves to
 * rank i / S_to, position i % S_to; the new layout's padding is +0. */
int or_reshard_f32(const or_unit_t* from, int32_t n_from, const float* const* src,
                   const or_unit_t* to, int32_t n_to, float* const* dst)
{
    if (!from || !to || n_from < 1 || n_to < 1 || !src || !dst ||
        from->n_params != to->n_params || from->shard_len * n_from != from->n_padded ||
        to->shard_len * n_to != to->n_padded)
        return OR_EINVAL;
    for (int32_t k = 0; k < n_to; ++k)
        for (int64_t j = 0; j < to->shard_len; ++j) {
            const int64_t i = (int64_t)k * to->shard_len + j;
            float x = 0.0f;
            if (i < to->n_params)
                x = src[i / from->shard_len][from->shard_offset + i % from->shard_len];
            dst[k][to->shard_offset + j] = x;
        }
    return OR_OK;
}

/* ZeRO-3 unit reduce-scatter followed by the owner's AdamW ([DZF] "How FSDP
 * implements ZeRO-3", steps 3-4; Theorem proof step 7: no all-gather follows
 * the update).  Rank k keeps the new fp32 state and its new bf16 shard. */
int or_zero3_reduce_scatter_unit(const or_unit_t* unit, int32_t n_ranks,
                                 const uint16_t* const* unit_grads,
                                 float* const* master, float* const* m,
                                 float* const* v, uint16_t* const* shard_bf16,
                                 const or_hparams_t* hp)
{
    if (!unit || n_ranks < 1 || !unit_grads || !master || !m || !v ||
        !shard_bf16 || bad_hp(hp) || unit->shard_len * n_ranks != unit->n_padded)
        return OR_EINVAL;
    or_scalars_t s;
    or_scalars(hp, n_ranks, &s);
    int64_t S = unit->shard_len;
    for (int64_t i = 0; i < unit->n_padded; ++i) {
        int64_t k = i / S;
        int64_t j = unit->shard_offset + (i - k * S);
        float g = or_reduce_mean(unit_grads, n_ranks, i, s.inv_n);
        or_adamw(g, &master[k][j], &m[k][j], &v[k][j], &s);
        shard_bf16[k][j] = or_bf16_rne(master[k][j]);
    }
    return OR_OK;
}

/* ======================================================================
 * Global gradient-norm clipping.  [DZF] "7. Common mistakes" (local
 * gradient clipping): with sharded gradients the global norm needs an
 * all-reduce of the squared shard norms.  [DDF] "A complete rank-aware DDP
 * reference" clips with torch's clip_grad_norm_(params, 1.) before the
 * optimizer step; its rule is used: norm = ||g||_2 over the whole averaged
 * gradient, coef = max_norm / (norm + 1e-6) clamped to at most 1, and the
 * gradient is multiplied by coef.  The norm is accumulated in double
 * (each g is an fp32 value, so g*g is exact in double); coef is computed in
 * double and rounded once to fp32; the scaled gradient is one fp32 multiply.
 * ==================================================================== */
double or_grad_sumsq(int32_t n_ranks, int64_t n, const uint16_t* const* grads)
{
    float inv_n = (float)(1.0 / (double)n_ranks);
    double sum = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double g = (double)or_reduce_mean(grads, n_ranks, i, inv_n);
        sum = sum + g * g;
    }
    return sum;
}

float or_clip_coef(double sumsq, double max_norm, double* out_norm)
{
    double norm = sqrt(sumsq);
    double c = max_norm / (norm + 1e-6);
    if (c > 1.0)
        c = 1.0;
    if (out_norm)
        *out_norm = norm;
    return (float)c;
}

int or_zero12_step_clip(int32_t stage, int32_t n_ranks, int64_t n_padded,
                        const uint16_t* const* grads, float* const* master,
                        float* const* m, float* const* v, uint16_t* params_bf16,
                        const or_hparams_t* hp, int64_t bucket_elems, double max_norm,
                        double* out_norm, float* out_coef)
{
    if ((stage != 1 && stage != 2) || n_ranks < 1 || n_padded <= 0 ||
        n_padded % n_ranks != 0 || !grads || !master || !m || !v ||
        !params_bf16 || bad_hp(hp) || bucket_elems < 0 || !(max_norm > 0))
        return OR_EINVAL;
    /* every owner's squared shard norm, summed over the owners: the global norm */
    double coef_norm;
    float coef = or_clip_coef(or_grad_sumsq(n_ranks, n_padded, grads), max_norm, &coef_norm);
    if (out_norm)
        *out_norm = coef_norm;
    if (out_coef)
        *out_coef = coef;
    int64_t S = n_padded / n_ranks;
    or_scalars_t s;
    or_scalars(hp, n_ranks, &s);
    int64_t bucket = (stage == 2 && bucket_elems > 0) ? bucket_elems : n_padded;
    for (int64_t b0 = 0; b0 < n_padded; b0 += bucket) {
        int64_t b1 = b0 + bucket < n_padded ? b0 + bucket : n_padded;
        for (int64_t i = b0; i < b1; ++i) {
            int64_t k = i / S;
            int64_t j = i - k * S;
            float g = or_reduce_mean(grads, n_ranks, i, s.inv_n) * coef;
            or_adamw(g, &master[k][j], &m[k][j], &v[k][j], &s);
            params_bf16[i] = or_bf16_rne(master[k][j]);
        }
    }
    return OR_OK;
}

int or_zero3_reduce_scatter_unit_coef(const or_unit_t* unit, int32_t n_ranks,
                                      const uint16_t* const* unit_grads,
                                      float* const* master, float* const* m,
                                      float* const* v, uint16_t* const* shard_bf16,
                                      const or_hparams_t* hp, float coef)
{
    if (!unit || n_ranks < 1 || !unit_grads || !master || !m || !v ||
        !shard_bf16 || bad_hp(hp) || unit->shard_len * n_ranks != unit->n_padded)
        return OR_EINVAL;
    or_scalars_t s;
    or_scalars(hp, n_ranks, &s);
    int64_t S = unit->shard_len;
    for (int64_t i = 0; i < unit->n_padded; ++i) {
        int64_t k = i / S;
        int64_t j = unit->shard_offset + (i - k * S);
        float g = or_reduce_mean(unit_grads, n_ranks, i, s.inv_n) * coef;
        or_adamw(g, &master[k][j], &m[k][j], &v[k][j], &s);
        shard_bf16[k][j] = or_bf16_rne(master[k][j]);
    }
    return OR_OK;
}

/* ======================================================================
 * ZeRO-2 gradient accumulation.  [DZF] "Gradient accumulation": m
 * micro-batches run one after the other and their gradients are added before
 * one optimizer step; ZeRO-2 keeps no full gradient, so it reduce-scatters
 * after every micro-batch (m*P + P elements per step).  Each owner keeps an
 * fp32 accumulator of its slice: acc = +0, then acc = acc + mean_mu for every
 * micro-batch mu (mean_mu = the reduce-scatter mean of that micro-batch); the
 * step uses g = acc * (float)(1/m), the mean over the micro-batches (each
 * micro-batch's gradient is that of its own mean loss, so the accumulated
 * gradient is the gradient of the mean loss over all m*N micro-batches).
 * or_zero2_accumulate handles micro-batches 1..m-1; the last micro-batch's
 * reduce-scatter is folded into or_zero2_step_accumulated.
 * ==================================================================== */
int or_zero2_accumulate(int32_t n_ranks, int64_t n_padded, const uint16_t* const* grads,
                        float* const* grad_acc, int32_t first)
{
    if (n_ranks < 1 || n_padded <= 0 || n_padded % n_ranks != 0 || !grads || !grad_acc)
        return OR_EINVAL;
    int64_t S = n_padded / n_ranks;
    float inv_n = (float)(1.0 / (double)n_ranks);
    for (int64_t i = 0; i < n_padded; ++i) {
        int64_t k = i / S, j = i - k * S;
        float a = first ? 0.0f : grad_acc[k][j];
        grad_acc[k][j] = a + or_reduce_mean(grads, n_ranks, i, inv_n);
    }
    return OR_OK;
}

int or_zero2_step_accumulated(int32_t n_ranks, int64_t n_padded, const uint16_t* const* grads,
                              const float* const* grad_acc, int32_t micro_batches,
                              float* const* master, float* const* m, float* const* v,
                              uint16_t* params_bf16, const or_hparams_t* hp)
{
    if (n_ranks < 1 || n_padded <= 0 || n_padded % n_ranks != 0 || !grads ||
        (micro_batches > 1 && !grad_acc) || micro_batches < 1 || !master || !m || !v ||
        !params_bf16 || bad_hp(hp))
        return OR_EINVAL;
    int64_t S = n_padded / n_ranks;
    or_scalars_t s;
    or_scalars(hp, n_ranks, &s);
    float inv_m = (float)(1.0 / (double)micro_batches);
    for (int64_t i = 0; i < n_padded; ++i) {
        int64_t k = i / S, j = i - k * S;
        float a = micro_batches > 1 ? grad_acc[k][j] : 0.0f;
        float g = (a + or_reduce_mean(grads, n_ranks, i, s.inv_n)) * inv_m;
        or_adamw(g, &master[k][j], &m[k][j], &v[k][j], &s);
        params_bf16[i] = or_bf16_rne(master[k][j]);
    }
    return OR_OK;
}

/* Elements sent per rank per optimizer step with m micro-batches ([DZF]
 * "Gradient accumulation" table; "How FSDP implements ZeRO-3", step 6, for
 * reshard_after_forward = 0: the backward all-gather disappears): DDP 2P,
 * ZeRO-1 2P, ZeRO-2 mP + P, ZeRO-3 3mP (2mP without resharding). */
double or_comm_volume(int32_t stage, int32_t micro_batches, int32_t reshard_after_forward,
                      double n_params)
{
    double m = (double)micro_batches, P = n_params;
    switch (stage) {
    case 0:
    case 1: return 2.0 * P;
    case 2: return m * P + P;
    case 3: return (reshard_after_forward ? 3.0 : 2.0) * m * P;
    default: return -1.0;
    }
}

/* ======================================================================
 * fp32-gradient reduce-scatter.  [DZF] "Proposition (tokens that hide the
 * all-reduce)" (fp32 gradient reduction doubles the bytes) and "6. Where it
 * shows up" (Llama 3 reduce-scattered gradients in fp32): the N_d rank
 * gradients arrive in fp32; the mean is the same fp32 sum from +0 in rank
 * order times (float)(1/N), and the update is unchanged.
 * ==================================================================== */
float or_reduce_mean_f32(const float* const* grads, int32_t n_ranks, int64_t i, float inv_n)
{
    float g = 0.0f;
    for (int32_t r = 0; r < n_ranks; ++r)
        g = g + grads[r][i];
    return g * inv_n;
}

int or_zero12_step_f32grads(int32_t stage, int32_t n_ranks, int64_t n_padded,
                            const float* const* grads, float* const* master, float* const* m,
                            float* const* v, uint16_t* params_bf16, const or_hparams_t* hp,
                            int64_t bucket_elems)
{
    if ((stage != 1 && stage != 2) || n_ranks < 1 || n_padded <= 0 ||
        n_padded % n_ranks != 0 || !grads || !master || !m || !v ||
        !params_bf16 || bad_hp(hp) || bucket_elems < 0)
        return OR_EINVAL;
    int64_t S = n_padded / n_ranks;
    or_scalars_t s;
    or_scalars(hp, n_ranks, &s);
    int64_t bucket = (stage == 2 && bucket_elems > 0) ? bucket_elems : n_padded;
    for (int64_t b0 = 0; b0 < n_padded; b0 += bucket) {
        int64_t b1 = b0 + bucket < n_padded ? b0 + bucket : n_padded;
        for (int64_t i = b0; i < b1; ++i) {
            int64_t k = i / S, j = i - k * S;
            float g = or_reduce_mean_f32(grads, n_ranks, i, s.inv_n);
            or_adamw(g, &master[k][j], &m[k][j], &v[k][j], &s);
            params_bf16[i] = or_bf16_rne(master[k][j]);
        }
    }
    return OR_OK;
}

int or_zero3_reduce_scatter_unit_f32grads(const or_unit_t* unit, int32_t n_ranks,
                                          const float* const* unit_grads, float* const* master,
                                          float* const* m, float* const* v,
                                          uint16_t* const* shard_bf16, const or_hparams_t* hp)
{
    if (!unit || n_ranks < 1 || !unit_grads || !master || !m || !v ||
        !shard_bf16 || bad_hp(hp) || unit->shard_len * n_ranks != unit->n_padded)
        return OR_EINVAL;
    or_scalars_t s;
    or_scalars(hp, n_ranks, &s);
    int64_t S = unit->shard_len;
    for (int64_t i = 0; i < unit->n_padded; ++i) {
        int64_t k = i / S;
        int64_t j = unit->shard_offset + (i - k * S);
        float g = or_reduce_mean_f32(unit_grads, n_ranks, i, s.inv_n);
        or_adamw(g, &master[k][j], &m[k][j], &v[k][j], &s);
        shard_bf16[k][j] = or_bf16_rne(master[k][j]);
    }
    return OR_OK;
}

/* ======================================================================
 * Pre-reduction finite check.  [DDF] "Failure investigation and recovery":
 * record pre-reduction per-rank finite checks so that the reduction does not
 * conceal where a NaN came from.  counts[r] = how many of rank r's bf16
 * gradients are infinite or NaN (all exponent bits set).
 * ==================================================================== */
void or_grad_nonfinite(int32_t n_ranks, int64_t n, const uint16_t* const* grads,
                       uint32_t* counts)
{
    for (int32_t r = 0; r < n_ranks; ++r) {
        uint32_t c = 0;
        for (int64_t i = 0; i < n; ++i) {
            float x = or_bf16_to_f32(grads[r][i]);
            if (isnan(x) || isinf(x))
                c += 1;
        }
        counts[r] = c;
    }
}

/* ======================================================================
 * Accounting.  [DZF] Theorem (ZeRO memory and communication), table and
 * proof steps 1-7; [DDF] "Memory accounting" (state_bytes raises on
 * params <= 0 or ranks < 1).  Bytes per parameter: bf16 weight 2, bf16
 * gradient 2, optimizer K; stage s shards the first s of (optimizer,
 * gradients, weights).  Volumes: 2P for DDP and ZeRO-1/2, 3P for ZeRO-3;
 * a ring sends (N-1)/N of each volume at 2 bytes per element.
 * hbm_bytes is the one-GPU emulated step: N bf16 gradient reads, fp32
 * master/m/v read and written, one bf16 weight write (26 + 2N per param),
 * plus, for ZeRO-3, two unit gathers of 2+2 bytes per param.
 * ==================================================================== */
int or_state_bytes(int64_t n_params, int32_t n_ranks, int32_t stage, int32_t K,
                   or_bytes_t* out)
{
    if (n_params <= 0 || n_ranks < 1 || stage < 0 || stage > 3 || K < 0 || !out)
        return OR_EINVAL;
    double P = (double)n_params, N = (double)n_ranks;
    out->optim_bytes = stage >= 1 ? (double)K * P / N : (double)K * P;
    out->grad_bytes = stage >= 2 ? 2.0 * P / N : 2.0 * P;
    out->weight_bytes = stage >= 3 ? 2.0 * P / N : 2.0 * P;
    out->state_bytes = out->weight_bytes + out->grad_bytes + out->optim_bytes;
    out->comm_volume = stage == 3 ? 3.0 * P : 2.0 * P;
    out->comm_sent_elems = out->comm_volume * (N - 1.0) / N;
    out->comm_sent_bytes = 2.0 * out->comm_sent_elems;
    out->hbm_bytes = (26.0 + 2.0 * N) * P + (stage == 3 ? 8.0 * P : 0.0);
    return OR_OK;
}

/* Ring bytes sent per rank ([DDF] "Communication and a roofline sanity
 * check"; [COL] "Collectives"): kind 0 = all-reduce, 2(R-1)/R of the
 * payload; kind 1 = reduce-scatter or all-gather, (R-1)/R of it. */
double or_ring_sent_bytes(double payload_bytes, int32_t n_ranks, int32_t kind)
{
    double R = (double)n_ranks;
    double one = (R - 1.0) / R * payload_bytes;
    return kind == 0 ? 2.0 * one : one;
}

/* ======================================================================
 * Literal simulators, built like the page's NumPy ZeRO-1 simulator
 * ([DZF] "5. In code", first block): explicit rank objects, an explicit
 * reduce-scatter loop and an explicit all-gather loop.  They check the
 * structure (ownership, who sends what where) against the fused oracle
 * above and against plain DDP.
 * ==================================================================== */
static void* xcalloc(size_t n, size_t sz)
{
    void* p = calloc(n ? n : 1, sz);
    if (!p)
        abort();
    return p;
}

/* DDP ([DZF] Proposition "DDP is exact"; "The communication is already
 * there", DDP row): every rank all-reduces the gradients, then updates all
 * parameters with its own full optimizer state. */
int or_sim_ddp(int32_t n_ranks, int64_t n_params, uint64_t seed, double sigma_w,
               double sigma_g, int32_t outliers, const or_hparams_t* hp0,
               int32_t n_steps, uint16_t* out_params, float* out_master,
               float* out_m, float* out_v)
{
    if (n_ranks < 1 || n_params <= 0 || bad_hp(hp0) || n_steps < 0)
        return OR_EINVAL;
    int64_t P = n_params;
    or_unit_t whole = {P, P, P, 0, 0, 0, 0}; /* unsharded: every rank holds all */
    float** W = xcalloc((size_t)n_ranks, sizeof *W);
    float** M = xcalloc((size_t)n_ranks, sizeof *M);
    float** V = xcalloc((size_t)n_ranks, sizeof *V);
    uint16_t** Wb = xcalloc((size_t)n_ranks, sizeof *Wb);
    uint16_t** G = xcalloc((size_t)n_ranks, sizeof *G);
    float* gbar = xcalloc((size_t)P, sizeof *gbar);
    for (int32_t r = 0; r < n_ranks; ++r) {
        W[r] = xcalloc((size_t)P, sizeof(float));
        M[r] = xcalloc((size_t)P, sizeof(float));
        V[r] = xcalloc((size_t)P, sizeof(float));
        Wb[r] = xcalloc((size_t)P, sizeof(uint16_t));
        G[r] = xcalloc((size_t)P, sizeof(uint16_t));
        or_gen_master(seed, sigma_w, &whole, 1, 1, &W[r]);
        /* every replica starts from the bf16 rounding of the same master weights */
        for (int64_t p = 0; p < P; ++p)
            Wb[r][p] = or_bf16_rne(W[r][p]);
    }
    for (int32_t t = 0; t < n_steps; ++t) {
        or_hparams_t hp = *hp0;
        hp.step = hp0->step + t;
        or_scalars_t s;
        or_scalars(&hp, n_ranks, &s);
        /* backward on each rank: its own micro-batch gradient */
        for (int32_t r = 0; r < n_ranks; ++r) {
            uint64_t key = or_gen_key(seed, 1, (uint64_t)hp.step, (uint64_t)r);
            float scale = or_gen_scale(sigma_g);
            for (int64_t p = 0; p < P; ++p)
                G[r][p] = or_bf16_rne(or_gen_value(key, (uint64_t)p, scale, outliers));
        }
        for (int32_t r = 0; r < n_ranks; ++r) {
            /* all-reduce: rank r receives the mean of all ranks' gradients */
            for (int64_t p = 0; p < P; ++p)
                gbar[p] = or_reduce_mean((const uint16_t* const*)G, n_ranks, p, s.inv_n);
            /* every rank updates every parameter */
            for (int64_t p = 0; p < P; ++p) {
                or_adamw(gbar[p], &W[r][p], &M[r][p], &V[r][p], &s);
                Wb[r][p] = or_bf16_rne(W[r][p]);
            }
        }
    }
    int rc = OR_OK;
    for (int32_t r = 1; r < n_ranks; ++r)
        if (memcmp(Wb[r], Wb[0], (size_t)P * sizeof(uint16_t)) ||
            memcmp(W[r], W[0], (size_t)P * sizeof(float)) ||
            memcmp(M[r], M[0], (size_t)P * sizeof(float)) ||
            memcmp(V[r], V[0], (size_t)P * sizeof(float)))
            rc = OR_EMISMATCH;
    for (int64_t p = 0; p < P; ++p) {
        if (out_params) out_params[p] = Wb[0][p];
        if (out_master) out_master[p] = W[0][p];
        if (out_m) out_m[p] = M[0][p];
        if (out_v) out_v[p] = V[0][p];
    }
    for (int32_t r = 0; r < n_ranks; ++r) {
        free(W[r]); free(M[r]); free(V[r]); free(Wb[r]); free(G[r]);
    }
    free(W); free(M); free(V); free(Wb); free(G); free(gbar);
    return rc;
}

/* ZeRO-1, ZeRO-2 and ZeRO-3 with explicit rank objects.
 *  stage 1/2: one flat buffer (all units concatenated, padded once).  Every
 *    rank keeps a full bf16 replica of the weights and the fp32 state of its
 *    slice.  Stage 1 reduce-scatters the whole gradient at once; stage 2
 *    reduce-scatters it bucket by bucket into each owner's fp32 gradient
 *    shard.  Then each owner updates its slice, and the all-gather loop
 *    copies every owner's new slice into every replica.
 *  stage 3: per-unit padding; rank k keeps only its bf16 shard and state.
 *    Forward: all-gather each unit.  Backward in reverse unit order:
 *    all-gather again, compute the unit's gradients, reduce-scatter them to
 *    the owners.  Then each rank updates its shards with no communication.
 * out_counts[0] = all-gathers, [1] = reduce-scatters, [2] = elements rank 0
 * sent (RS: the slices it does not own; AG: its slice to the N-1 others),
 * all summed over the steps.  Outputs are in true-parameter order. */
int or_sim_zero(int32_t stage, int32_t n_ranks, const int64_t* unit_sizes,
                int32_t n_units, int32_t align, uint64_t seed, double sigma_w,
                double sigma_g, int32_t outliers, const or_hparams_t* hp0,
                int32_t n_steps, int64_t bucket_elems, uint16_t* out_params,
                float* out_master, float* out_m, float* out_v,
                int64_t* out_counts)
{
    if (stage < 1 || stage > 3 || n_ranks < 1 || !unit_sizes || n_units < 1 ||
        align < 1 || bad_hp(hp0) || n_steps < 0 || bucket_elems < 0)
        return OR_EINVAL;
    int32_t N = n_ranks;
    int64_t counts[3] = {0, 0, 0};
    int rc = OR_OK;

    /* layout: stage 3 pads unit by unit; stages 1/2 pad the flat model once */
    int64_t P = 0;
    for (int32_t u = 0; u < n_units; ++u) {
        if (unit_sizes[u] <= 0)
            return OR_EINVAL;
        P += unit_sizes[u];
    }
    int32_t nu = stage == 3 ? n_units : 1;
    or_unit_t* L = xcalloc((size_t)nu, sizeof *L);
    int64_t total;
    if (stage == 3)
        rc = or_layout(unit_sizes, n_units, N, align, L, &total);
    else
        rc = or_layout(&P, 1, N, align, L, &total);
    if (rc != OR_OK) {
        free(L);
        return rc;
    }
    int64_t shard_total = total / N;

    /* rank objects */
    float** MW = xcalloc((size_t)N, sizeof *MW); /* fp32 master shard */
    float** MM = xcalloc((size_t)N, sizeof *MM);
    float** MV = xcalloc((size_t)N, sizeof *MV);
    float** GS = xcalloc((size_t)N, sizeof *GS); /* reduced fp32 gradient shard */
    uint16_t** WB = xcalloc((size_t)N, sizeof *WB); /* stage 1/2: full replica; 3: shard */
    uint16_t** G = xcalloc((size_t)N, sizeof *G);   /* local gradients of one unit */
    int64_t max_unit = 0;
    for (int32_t u = 0; u < nu; ++u)
        if (L[u].n_padded > max_unit)
            max_unit = L[u].n_padded;
    for (int32_t k = 0; k < N; ++k) {
        MW[k] = xcalloc((size_t)shard_total, sizeof(float));
        MM[k] = xcalloc((size_t)shard_total, sizeof(float));
        MV[k] = xcalloc((size_t)shard_total, sizeof(float));
        GS[k] = xcalloc((size_t)shard_total, sizeof(float));
        WB[k] = xcalloc((size_t)(stage == 3 ? shard_total : total), sizeof(uint16_t));
        G[k] = xcalloc((size_t)max_unit, sizeof(uint16_t));
    }
    uint16_t* full = xcalloc((size_t)max_unit, sizeof(uint16_t)); /* a gathered unit */
    or_gen_master(seed, sigma_w, L, nu, N, MW);
    for (int32_t k = 0; k < N; ++k) {
        if (stage == 3) {
            for (int64_t j = 0; j < shard_total; ++j)
                WB[k][j] = or_bf16_rne(MW[k][j]);
        } else {
            /* every replica starts from the same weights */
            for (int32_t o = 0; o < N; ++o)
                for (int64_t j = 0; j < L[0].shard_len; ++j)
                    WB[k][(int64_t)o * L[0].shard_len + j] = or_bf16_rne(MW[o][j]);
        }
    }

    for (int32_t t = 0; t < n_steps; ++t) {
        or_hparams_t hp = *hp0;
        hp.step = hp0->step + t;
        or_scalars_t s;
        or_scalars(&hp, N, &s);
        if (stage != 3) {
            const or_unit_t* U = &L[0];
            int64_t S = U->shard_len;
            or_gen_grads_unit(seed, hp.step, sigma_g, outliers, U, N, G);
            int64_t bucket = (stage == 2 && bucket_elems > 0) ? bucket_elems : U->n_padded;
            for (int64_t b0 = 0; b0 < U->n_padded; b0 += bucket) {
                int64_t b1 = b0 + bucket < U->n_padded ? b0 + bucket : U->n_padded;
                /* reduce-scatter of this bucket: owner k receives the mean
                 * of its part of the bucket */
                for (int32_t k = 0; k < N; ++k)
                    for (int64_t j = 0; j < S; ++j) {
                        int64_t i = (int64_t)k * S + j;
                        if (i < b0 || i >= b1)
                            continue;
                        GS[k][j] = or_reduce_mean((const uint16_t* const*)G, N, i, s.inv_n);
                    }
                counts[1] += 1;
                /* rank 0 sends the part of the bucket it does not own */
                for (int64_t i = b0; i < b1; ++i)
                    if (i / S != 0)
                        counts[2] += 1;
            }
            /* each owner updates its slice */
            for (int32_t k = 0; k < N; ++k)
                for (int64_t j = 0; j < S; ++j) {
                    or_adamw(GS[k][j], &MW[k][j], &MM[k][j], &MV[k][j], &s);
                    WB[k][(int64_t)k * S + j] = or_bf16_rne(MW[k][j]);
                }
            /* all-gather: every replica receives every owner's new slice */
            for (int32_t k = 0; k < N; ++k)
                for (int32_t o = 0; o < N; ++o) {
                    if (o == k)
                        continue;
                    memcpy(&WB[k][(int64_t)o * S], &WB[o][(int64_t)o * S],
                           (size_t)S * sizeof(uint16_t));
                }
            counts[0] += 1;
            counts[2] += (int64_t)(N - 1) * S;
        } else {
            /* forward: gather each unit, use it, free it */
            for (int32_t u = 0; u < nu; ++u) {
                or_zero3_gather_unit(&L[u], N, (const uint16_t* const*)WB, full);
                counts[0] += 1;
                counts[2] += (int64_t)(N - 1) * L[u].shard_len;
            }
            /* backward, units in reverse: gather again, gradients,
             * reduce-scatter to the owners' fp32 gradient shards */
            for (int32_t u = nu - 1; u >= 0; --u) {
                const or_unit_t* U = &L[u];
                or_zero3_gather_unit(U, N, (const uint16_t* const*)WB, full);
                counts[0] += 1;
                counts[2] += (int64_t)(N - 1) * U->shard_len;
                or_gen_grads_unit(seed, hp.step, sigma_g, outliers, U, N, G);
                for (int32_t k = 0; k < N; ++k)
                    for (int64_t j = 0; j < U->shard_len; ++j)
                        GS[k][U->shard_offset + j] = or_reduce_mean(
                            (const uint16_t* const*)G, N, (int64_t)k * U->shard_len + j,
                            s.inv_n);
                counts[1] += 1;
                counts[2] += (int64_t)(N - 1) * U->shard_len;
            }
            /* optimizer step on the local shards, no communication */
            for (int32_t k = 0; k < N; ++k)
                for (int64_t j = 0; j < shard_total; ++j) {
                    or_adamw(GS[k][j], &MW[k][j], &MM[k][j], &MV[k][j], &s);
                    WB[k][j] = or_bf16_rne(MW[k][j]);
                }
        }
    }

    /* replicas must agree (stage 1/2) */
    if (stage != 3)
        for (int32_t k = 1; k < N; ++k)
            if (memcmp(WB[k], WB[0], (size_t)total * sizeof(uint16_t)))
                rc = OR_EMISMATCH;

    /* outputs in true-parameter order */
    for (int32_t u = 0; u < nu; ++u) {
        const or_unit_t* U = &L[u];
        for (int64_t loc = 0; loc < U->n_params; ++loc) {
            int64_t k = loc / U->shard_len;
            int64_t j = U->shard_offset + (loc - k * U->shard_len);
            int64_t p = U->param_offset + loc;
            if (out_params)
                out_params[p] = stage == 3 ? WB[k][j] : WB[0][U->offset + loc];
            if (out_master) out_master[p] = MW[k][j];
            if (out_m) out_m[p] = MM[k][j];
            if (out_v) out_v[p] = MV[k][j];
        }
    }
    /* padding must have stayed +0 in every rank's state */
    for (int32_t u = 0; u < nu; ++u) {
        const or_unit_t* U = &L[u];
        for (int64_t loc = U->n_params; loc < U->n_padded; ++loc) {
            int64_t k = loc / U->shard_len;
            int64_t j = U->shard_offset + (loc - k * U->shard_len);
            uint32_t bits[3];
            memcpy(&bits[0], &MW[k][j], 4);
            memcpy(&bits[1], &MM[k][j], 4);
            memcpy(&bits[2], &MV[k][j], 4);
            if (bits[0] || bits[1] || bits[2])
                rc = OR_EMISMATCH;
        }
    }
    if (out_counts)
        memcpy(out_counts, counts, sizeof counts);

    for (int32_t k = 0; k < N; ++k) {
        free(MW[k]); free(MM[k]); free(MV[k]); free(GS[k]); free(WB[k]); free(G[k]);
    }
    free(MW); free(MM); free(MV); free(GS); free(WB); free(G); free(full); free(L);
    return rc;
}

/* ======================================================================
 * Sampled parity: the step is elementwise, so the final state of any true
 * parameter after n_steps can be computed alone from its generated inputs.
 * ==================================================================== */
static void sample_steps(int32_t n_ranks, uint64_t seed, double sigma_w, double sigma_g,
                         int32_t outliers, const or_hparams_t* hp0, int32_t n_steps,
                         const float* coef, int32_t micro_batches, int64_t grad_step,
                         const int64_t* param_index, int64_t n_index, uint16_t* out_params,
                         float* out_master, float* out_m, float* out_v);

void or_sample(int32_t n_ranks, uint64_t seed, double sigma_w, double sigma_g,
               int32_t outliers, const or_hparams_t* hp0, int32_t n_steps,
               const int64_t* param_index, int64_t n_index, uint16_t* out_params,
               float* out_master, float* out_m, float* out_v)
{
    sample_steps(n_ranks, seed, sigma_w, sigma_g, outliers, hp0, n_steps, NULL, 0, 0, param_index,
                 n_index, out_params, out_master, out_m, out_v);
}

/* The same with global-norm clipping: step t (0-based) multiplies the mean
 * gradient by coef[t], as or_zero3_reduce_scatter_unit_coef does.  The
 * coefficients are inputs (the norm of a whole model cannot be formed from a
 * sample of its parameters). */
void or_sample_coef(int32_t n_ranks, uint64_t seed, double sigma_w, double sigma_g,
                    int32_t outliers, const or_hparams_t* hp0, int32_t n_steps,
                    const float* coef, const int64_t* param_index, int64_t n_index,
                    uint16_t* out_params, float* out_master, float* out_m, float* out_v)
{
    sample_steps(n_ranks, seed, sigma_w, sigma_g, outliers, hp0, n_steps, coef, 0, 0, param_index,
                 n_index, out_params, out_master, out_m, out_v);
}

/* The same with gradient accumulation over micro_batches identical
 * micro-batches (each micro-batch's rank gradients are the step's generated
 * ones): the owner accumulator starts at +0 and adds the mean after each of
 * the first micro_batches - 1 micro-batches (or_zero2_accumulate), and the
 * update takes g = (accumulator + mean) * (1/micro_batches)
 * (or_zero2_step_accumulated; accumulator +0 for one micro-batch). */
void or_sample_accum(int32_t n_ranks, uint64_t seed, double sigma_w, double sigma_g,
                     int32_t outliers, const or_hparams_t* hp0, int32_t n_steps,
                     int32_t micro_batches, const int64_t* param_index, int64_t n_index,
                     uint16_t* out_params, float* out_master, float* out_m, float* out_v)
{
    sample_steps(n_ranks, seed, sigma_w, sigma_g, outliers, hp0, n_steps, NULL,
                 micro_batches < 1 ? 1 : micro_batches, 0, param_index, n_index, out_params,
                 out_master, out_m, out_v);
}

/* or_sample with the same rank gradients in every step: those the generator
 * gives for step grad_step (>= 1), while AdamW's step counter still advances
 * from hp0->step.  This is a choice of inputs only: a job that keeps one
 * gradient set resident and applies it again at every step. */
void or_sample_fixed_grads(int32_t n_ranks, uint64_t seed, double sigma_w, double sigma_g,
                           int32_t outliers, const or_hparams_t* hp0, int32_t n_steps,
                           int64_t grad_step, const int64_t* param_index, int64_t n_index,
                           uint16_t* out_params, float* out_master, float* out_m, float* out_v)
{
    sample_steps(n_ranks, seed, sigma_w, sigma_g, outliers, hp0, n_steps, NULL, 0,
                 grad_step < 1 ? 1 : grad_step, param_index, n_index, out_params, out_master,
                 out_m, out_v);
}

static void sample_steps(int32_t n_ranks, uint64_t seed, double sigma_w, double sigma_g,
                         int32_t outliers, const or_hparams_t* hp0, int32_t n_steps,
                         const float* coef, int32_t micro_batches, int64_t grad_step,
                         const int64_t* param_index, int64_t n_index, uint16_t* out_params,
                         float* out_master, float* out_m, float* out_v)
{
    float inv_m = micro_batches > 0 ? (float)(1.0 / (double)micro_batches) : 1.0f;
    uint64_t wkey = or_gen_key(seed, 0, 0, 0);
    float wscale = or_gen_scale(sigma_w);
    float gscale = or_gen_scale(sigma_g);
    uint64_t* keys = xcalloc((size_t)n_steps * (size_t)n_ranks + 1, sizeof *keys);
    or_scalars_t* sc = xcalloc((size_t)n_steps + 1, sizeof *sc);
    for (int32_t t = 0; t < n_steps; ++t) {
        or_hparams_t hp = *hp0;
        hp.step = hp0->step + t;
        or_scalars(&hp, n_ranks, &sc[t]);
        for (int32_t r = 0; r < n_ranks; ++r)
            keys[(size_t)t * n_ranks + r] =
                or_gen_key(seed, 1, (uint64_t)(grad_step > 0 ? grad_step : hp.step), (uint64_t)r);
    }
    uint16_t* g1 = xcalloc((size_t)n_ranks, sizeof *g1);
    const uint16_t** gp = xcalloc((size_t)n_ranks, sizeof *gp);
    for (int32_t r = 0; r < n_ranks; ++r)
        gp[r] = &g1[r];
    for (int64_t q = 0; q < n_index; ++q) {
        uint64_t p = (uint64_t)param_index[q];
        float w = or_gen_value(wkey, p, wscale, 0), m = 0.0f, v = 0.0f;
        for (int32_t t = 0; t < n_steps; ++t) {
            for (int32_t r = 0; r < n_ranks; ++r)
                g1[r] = or_bf16_rne(or_gen_value(keys[(size_t)t * n_ranks + r], p, gscale, outliers));
            float g = or_reduce_mean(gp, n_ranks, 0, sc[t].inv_n);
            if (coef)
                g = g * coef[t];
            if (micro_batches > 0) {
                float a = 0.0f;
                if (micro_batches > 1) {
                    a = 0.0f + g;
                    for (int32_t mu = 1; mu < micro_batches - 1; ++mu)
                        a = a + g;
                }
                g = (a + g) * inv_m;
            }
            or_adamw(g, &w, &m, &v, &sc[t]);
        }
        if (out_params) out_params[q] = or_bf16_rne(w);
        if (out_master) out_master[q] = w;
        if (out_m) out_m[q] = m;
        if (out_v) out_v[q] = v;
    }
    free(keys); free(sc); free(g1); free(gp);
}
