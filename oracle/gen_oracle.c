/*
 * gen_oracle.c -- seeded synthetic inputs for the oracle.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  This module holds none of the
 * method's arithmetic: it only draws the numbers that the method consumes
 * (initial fp32 master weights and per-rank bf16 gradients).  The CUDA side
 * has its own implementation of the same counter-based generator, written
 * separately from the same published definition.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; constants as in Vigna's
 * public-domain splitmix64.c).  The state advances by the golden-ratio
 * increment and every output is the 64-bit finaliser of the new state, so
 * output number i of a stream that starts at state s is mix(s + (i+1)*gamma):
 * any element can be drawn without drawing the ones before it.
 *
 * A value is approximately normal: the four 16-bit lanes of one output are
 * summed (an Irwin-Hall sum of four discrete uniforms, mean 131070, standard
 * deviation sqrt((2^32-1)/3)), centred exactly in integers, converted to fp32
 * (exact: |s| <= 131070) and scaled by one fp32 constant sigma/sd.  Tails are
 * cut at about 3.46 sigma.  With outliers on, one value in a hundred (decided
 * by the next output of the value's own stream) is multiplied by 100.
 */
#include "zero_oracle.h"

#include <math.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static uint64_t finalise(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t or_splitmix64_next(uint64_t* state)
{
    *state += GAMMA;
    return finalise(*state);
}

/* Output number i (0-based) of the stream whose state starts at s. */
static uint64_t output_at(uint64_t s, uint64_t i)
{
    return finalise(s + (i + 1) * GAMMA);
}

/* Stream key of (seed, stream, step, rank): the first output of a stream
 * seeded by the previous key xor the next field. */
uint64_t or_gen_key(uint64_t seed, uint64_t stream, uint64_t step, uint64_t rank)
{
    uint64_t k = output_at(seed, 0);
    k = output_at(k ^ stream, 0);
    k = output_at(k ^ step, 0);
    k = output_at(k ^ rank, 0);
    return k;
}

float or_gen_scale(double sigma)
{
    return (float)(sigma / sqrt(4294967295.0 / 3.0));
}

float or_gen_value(uint64_t key, uint64_t index, float scale, int32_t outliers)
{
    uint64_t h = output_at(key, index);
    int32_t s = (int32_t)(h & 0xFFFFu) + (int32_t)((h >> 16) & 0xFFFFu) +
                (int32_t)((h >> 32) & 0xFFFFu) + (int32_t)(h >> 48) - 131070;
    float z = (float)s * scale;
    if (outliers && output_at(h, 0) % 100u == 0u)
        z = z * 100.0f;
    return z;
}

/* Initial fp32 master weights of every unit, written into each owner's shard
 * storage.  The value of true parameter p is drawn from (seed, stream 0,
 * step 0, rank 0) at index p; padding is +0. */
void or_gen_master(uint64_t seed, double sigma, const or_unit_t* units,
                   int32_t n_units, int32_t n_ranks, float* const* master)
{
    uint64_t key = or_gen_key(seed, 0, 0, 0);
    float scale = or_gen_scale(sigma);
    for (int32_t u = 0; u < n_units; ++u) {
        const or_unit_t* U = &units[u];
        for (int32_t k = 0; k < n_ranks; ++k) {
            for (int64_t j = 0; j < U->shard_len; ++j) {
                int64_t local = (int64_t)k * U->shard_len + j;
                float x = 0.0f;
                if (local < U->n_params)
                    x = or_gen_value(key, (uint64_t)(U->param_offset + local), scale, 0);
                master[k][U->shard_offset + j] = x;
            }
        }
    }
}

/* Rank r's bf16 gradient of one unit at step t: true parameter p is drawn
 * from (seed, stream 1, step t, rank r) at index p and rounded to bf16
 * (nearest-even); padding is +0. */
void or_gen_grads_unit(uint64_t seed, int64_t step, double sigma, int32_t outliers,
                       const or_unit_t* unit, int32_t n_ranks,
                       uint16_t* const* unit_grads)
{
    float scale = or_gen_scale(sigma);
    for (int32_t r = 0; r < n_ranks; ++r) {
        uint64_t key = or_gen_key(seed, 1, (uint64_t)step, (uint64_t)r);
        for (int64_t j = 0; j < unit->n_padded; ++j) {
            uint16_t b = 0;
            if (j < unit->n_params)
                b = or_bf16_rne(or_gen_value(key, (uint64_t)(unit->param_offset + j),
                                             scale, outliers));
            unit_grads[r][j] = b;
        }
    }
}

/* The same gradients kept in fp32 (not rounded to bf16): the inputs of the
 * fp32-gradient reduce-scatter. */
void or_gen_grads_unit_f32(uint64_t seed, int64_t step, double sigma, int32_t outliers,
                           const or_unit_t* unit, int32_t n_ranks, float* const* unit_grads)
{
    float scale = or_gen_scale(sigma);
    for (int32_t r = 0; r < n_ranks; ++r) {
        uint64_t key = or_gen_key(seed, 1, (uint64_t)step, (uint64_t)r);
        for (int64_t j = 0; j < unit->n_padded; ++j)
            unit_grads[r][j] = j < unit->n_params
                                   ? or_gen_value(key, (uint64_t)(unit->param_offset + j), scale,
                                                  outliers)
                                   : 0.0f;
    }
}
