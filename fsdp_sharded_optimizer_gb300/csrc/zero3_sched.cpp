// zero3_sched.cpp -- the native ZeRO-3 step scheduler (zero3_plan, zero3_step).
//
// Order ("Data parallelism, ZeRO and FSDP", "How FSDP implements ZeRO-3",
// steps 2-5; "Data parallelism, collectives and ZeRO/FSDP", the per-unit
// FSDP step figure): a forward pass that gathers every unit, a backward pass
// in reverse unit order that gathers each unit again and reduce-scatters its
// gradients, gathers on a separate stream, and the next unit's gather issued
// before the current unit's work, with at most two units gathered at once.
// Without a backward compute to hide them behind, the boundaries between
// consecutive units' updates, and between consecutive gathers, would be idle
// time on one stream, so the backward units alternate between the caller's
// main stream and a second compute stream of the library's own, and the
// gathers between the caller's side stream and a second side stream
// (PlanBuilder::two_compute, two_side).
//
// The plan is built on the host as a list of operations and then executed,
// so the same plan can be checked on a machine without a GPU.  Executing it
// costs one library call per gather / reduce-scatter and a handful of event
// records and waits per unit -- microseconds of host time per unit, so small
// units stay GPU-bound.
#include <vector>

#include "zero_internal.h"

namespace zero {
namespace {

constexpr int kEvents = 7; // start, gathered[2], released[2], aux start, aux done
constexpr int kMaxDevices = 64;
constexpr int kEvStart = 0, kEvGathered = 1, kEvReleased = 3, kEvAuxStart = 5, kEvAuxDone = 6;
constexpr int32_t kOwnRegion = 2; // GATHER/USE arg: the unit's region of the kept full buffer
// Streams of a plan: the caller's main and side streams, and two of the
// library's own: a second compute stream that takes every other backward unit
// and a second side stream that takes the gathers into full buffer 1.
constexpr int32_t kMain = 0, kSide = 1, kAux = 2, kSide2 = 3;

// What a backward pass does with a unit's gradients of this micro-batch.
enum class Reduce {
    kStep,       // reduce-scatter fused with the update (no accumulation)
    kAccFirst,   // the step's first micro-batch: the accumulator starts at its mean
    kAccLater,   // a later one, not the last: added to the accumulator
    kAccLast,    // the last one: added and fused with the update
};

struct PlanBuilder {
    std::vector<zero_op_t> ops;
    bool released_recorded[2] = {false, false};
    Reduce reduce_mode = Reduce::kStep;
    // The resharding backward pass runs the units of odd positions (those of
    // full buffer 1) on the second compute stream: consecutive units' updates
    // then overlap at their boundary, where one stream would separate them by
    // an event wait and record.  Not with regeneration, whose units share one
    // gradient buffer.
    bool two_compute = false;
    // Likewise the gathers into full buffer 1 (into the units of odd positions
    // without resharding) run on the second side stream, so that consecutive
    // gathers overlap at their boundary too.
    bool two_side = false;

    int32_t side_of(int32_t pos) const { return two_side && pos % 2 == 1 ? kSide2 : kSide; }

    void reduce(int32_t u, bool clip, int32_t stream)
    {
        if (reduce_mode == Reduce::kAccFirst || reduce_mode == Reduce::kAccLater)
            add(ZERO_OP_ACCUMULATE, stream, u, reduce_mode == Reduce::kAccFirst ? 1 : 0);
        else
            add(ZERO_OP_REDUCE_SCATTER, stream, u,
                reduce_mode == Reduce::kAccLast ? 2 : (clip ? 1 : 0));
    }

    void add(int32_t kind, int32_t stream, int32_t unit, int32_t arg)
    {
        ops.push_back(zero_op_t{kind, stream, unit, arg});
    }

    // The buffer's side stream fills full buffer `slot` with unit `u` once the
    // compute stream using it has released it, then marks the unit gathered.
    void gather(int32_t u, int32_t pos, int32_t slot)
    {
        const int32_t ss = side_of(pos); // pos % 2 == slot: a buffer's gathers share a stream
        if (released_recorded[slot]) add(ZERO_OP_WAIT, ss, -1, kEvReleased + slot);
        add(ZERO_OP_GATHER, ss, u, slot);
        add(ZERO_OP_RECORD, ss, -1, kEvGathered + pos % 2);
    }

    void pass(int32_t n_units, bool backward, bool regen, bool clip)
    {
        auto unit_at = [&](int32_t pos) { return backward ? n_units - 1 - pos : pos; };
        gather(unit_at(0), 0, 0);
        for (int32_t pos = 0; pos < n_units; ++pos) {
            const int32_t slot = pos % 2;
            const int32_t u = unit_at(pos);
            if (pos + 1 < n_units) gather(unit_at(pos + 1), pos + 1, 1 - slot); // prefetch
            // a unit's work, and the release of its full buffer, on the
            // compute stream of that buffer
            const int32_t cs = backward && two_compute && slot == 1 ? kAux : kMain;
            add(ZERO_OP_WAIT, cs, -1, kEvGathered + pos % 2);
            add(ZERO_OP_USE, cs, u, slot);
            if (backward) {
                if (regen) add(ZERO_OP_REGEN, cs, u, 0);
                reduce(u, clip, cs);
            }
            add(ZERO_OP_RECORD, cs, -1, kEvReleased + slot);
            released_recorded[slot] = true;
        }
    }

    // reshard_after_forward = false: the forward pass gathers every unit into
    // its own region of one full buffer (arg kOwnRegion) and keeps it; the
    // backward pass uses the kept weights with no second gather.
    void forward_keep(int32_t n_units)
    {
        auto gather_own = [&](int32_t u, int32_t pos) {
            add(ZERO_OP_GATHER, side_of(pos), u, kOwnRegion);
            add(ZERO_OP_RECORD, side_of(pos), -1, kEvGathered + pos % 2);
        };
        gather_own(0, 0);
        for (int32_t pos = 0; pos < n_units; ++pos) {
            if (pos + 1 < n_units) gather_own(pos + 1, pos + 1); // prefetch
            add(ZERO_OP_WAIT, 0, -1, kEvGathered + pos % 2);
            add(ZERO_OP_USE, 0, pos, kOwnRegion);
        }
    }

    void backward_kept(int32_t n_units, bool regen, bool clip)
    {
        for (int32_t u = n_units - 1; u >= 0; --u) {
            add(ZERO_OP_USE, kMain, u, kOwnRegion);
            if (regen) add(ZERO_OP_REGEN, kMain, u, 0);
            reduce(u, clip, kMain);
        }
    }

    void step(int32_t n_units, bool regen, bool clip, bool reshard = true)
    {
        // the step's first gathers must see everything the main stream did before
        two_side = two_side && n_units > 1;
        add(ZERO_OP_RECORD, kMain, -1, kEvStart);
        add(ZERO_OP_WAIT, kSide, -1, kEvStart);
        if (two_side) add(ZERO_OP_WAIT, kSide2, -1, kEvStart);
        if (clip) {
            // the global norm before any unit's update: every unit's squared
            // norm on the main stream (overlapping the forward gathers), then
            // the coefficient
            for (int32_t u = 0; u < n_units; ++u) {
                if (regen) add(ZERO_OP_REGEN, 0, u, 0);
                add(ZERO_OP_NORM, 0, u, u > 0 ? 1 : 0);
            }
            add(ZERO_OP_CLIP_COEF, 0, -1, 0);
        }
        if (reshard) {
            pass(n_units, false, regen, clip);
            // the second compute stream starts after everything the main
            // stream did before the backward pass (the caller's work, the
            // clip coefficient) and hands its end back to the main stream
            const bool aux = two_compute && !regen && n_units > 1;
            two_compute = aux;
            if (aux) {
                add(ZERO_OP_RECORD, kMain, -1, kEvAuxStart);
                add(ZERO_OP_WAIT, kAux, -1, kEvAuxStart);
            }
            pass(n_units, true, regen, clip);
            if (aux) {
                add(ZERO_OP_RECORD, kAux, -1, kEvAuxDone);
                add(ZERO_OP_WAIT, kMain, -1, kEvAuxDone);
            }
        } else {
            forward_keep(n_units);
            backward_kept(n_units, regen, clip);
        }
    }
};

// Gradient accumulation inside a ZeRO-3 step: the fp32 accumulator storage and
// this call's place among the step's micro-batches.
struct AccumArgs {
    float* const* grad_acc;
    int32_t micro_batch;   // 0 .. micro_batches - 1
    int32_t micro_batches; // m >= 1
};

Reduce reduce_mode(const AccumArgs* acc)
{
    if (!acc || acc->micro_batches == 1) return Reduce::kStep;
    if (acc->micro_batch == acc->micro_batches - 1) return Reduce::kAccLast;
    return acc->micro_batch == 0 ? Reduce::kAccFirst : Reduce::kAccLater;
}

// Copies a built plan to the caller's array.
int copy_plan(const PlanBuilder& b, zero_op_t* ops, int32_t max_ops, int32_t* n_ops)
{
    if (static_cast<int64_t>(b.ops.size()) > max_ops) return ZERO_EINVAL;
    for (size_t i = 0; i < b.ops.size(); ++i) ops[i] = b.ops[i];
    *n_ops = static_cast<int32_t>(b.ops.size());
    return ZERO_OK;
}

// Seven timing-free events and the second compute and side streams
// (non-blocking) per host thread and device, created on first use.
struct StepResources {
    int device = -1;
    cudaEvent_t ev[kEvents] = {};
    cudaStream_t aux = nullptr;
    cudaStream_t side2 = nullptr;
};
thread_local StepResources t_res[kMaxDevices];

int resources_for_current_device(StepResources** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ZERO_ECUDA;
    StepResources& c = t_res[dev];
    if (c.device != dev) {
        for (int i = 0; i < kEvents; ++i)
            if (!c.ev[i] && cudaEventCreateWithFlags(&c.ev[i], cudaEventDisableTiming) != cudaSuccess)
                return ZERO_ECUDA;
        if (!c.aux && cudaStreamCreateWithFlags(&c.aux, cudaStreamNonBlocking) != cudaSuccess)
            return ZERO_ECUDA;
        if (!c.side2 && cudaStreamCreateWithFlags(&c.side2, cudaStreamNonBlocking) != cudaSuccess)
            return ZERO_ECUDA;
        c.device = dev;
    }
    *out = &c;
    return ZERO_OK;
}

bool unit_consistent(const zero_unit_t& u, int32_t n_ranks)
{
    return u.n_params > 0 && u.n_params <= u.n_padded && u.shard_len > 0 &&
           u.shard_len % 8 == 0 && u.shard_len * n_ranks == u.n_padded && u.offset >= 0 &&
           u.offset % 8 == 0 && u.shard_offset >= 0 && u.shard_offset % 8 == 0;
}

} // namespace

int preload_step_events()
{
    StepResources* r = nullptr;
    return resources_for_current_device(&r);
}

} // namespace zero

using namespace zero;

extern "C" int zero3_plan_microbatch(int32_t n_units, int32_t reshard_after_forward,
                                     int32_t micro_batch, int32_t micro_batches,
                                     zero_op_t* ops, int32_t max_ops, int32_t* n_ops)
{
    if (n_units < 1 || !ops || !n_ops || max_ops < 0 || micro_batches < 1 || micro_batch < 0 ||
        micro_batch >= micro_batches)
        return ZERO_EINVAL;
    const AccumArgs acc{nullptr, micro_batch, micro_batches};
    PlanBuilder b;
    b.reduce_mode = reduce_mode(&acc);
    b.two_compute = b.two_side = true;
    b.step(n_units, false, false, reshard_after_forward != 0);
    return copy_plan(b, ops, max_ops, n_ops);
}

extern "C" int zero3_plan(int32_t n_units, int32_t regen, int32_t clip,
                          int32_t reshard_after_forward, zero_op_t* ops, int32_t max_ops,
                          int32_t* n_ops)
{
    if (n_units < 1 || !ops || !n_ops || max_ops < 0) return ZERO_EINVAL;
    PlanBuilder b;
    b.two_compute = b.two_side = true;
    b.step(n_units, regen != 0, clip != 0, reshard_after_forward != 0);
    return copy_plan(b, ops, max_ops, n_ops);
}

namespace {

// The step of zero3_step / zero3_step_f32grads.  f32: the rank gradients are
// fp32 (grads holds float pointers; no regeneration, no clipping).
int run_step(const zero_unit_t* units, int32_t n_units, int32_t n_ranks, const void* const* grads,
             bool f32, int32_t grads_resident, float* const* master, float* const* m,
             float* const* v, uint16_t* const* shard_bf16, uint16_t* full_a, uint16_t* full_b,
             const zero_hparams_t* hp, const zero_regen_t* regen, const zero_clip_t* clip,
             int32_t reshard_after_forward, cudaStream_t main_stream, cudaStream_t side_stream,
             const AccumArgs* acc = nullptr, uint32_t* nonfinite = nullptr)
{
    const bool reshard = reshard_after_forward != 0;
    if (!units || n_units < 1 || n_ranks < 1 || n_ranks > ZERO_MAX_RANKS || !valid_hparams(hp) ||
        !full_a || (reshard && (!full_b || full_a == full_b)) || main_stream == side_stream ||
        (!grads_resident && !regen))
        return ZERO_EINVAL;
    for (int32_t u = 0; u < n_units; ++u)
        if (!unit_consistent(units[u], n_ranks)) return ZERO_EINVAL;
    int rc;
    if ((rc = check_table(grads, n_ranks)) != ZERO_OK) return rc;
    if ((rc = check_table(master, n_ranks)) != ZERO_OK) return rc;
    if ((rc = check_table(m, n_ranks)) != ZERO_OK) return rc;
    if ((rc = check_table(v, n_ranks)) != ZERO_OK) return rc;
    if ((rc = check_table(shard_bf16, n_ranks)) != ZERO_OK) return rc;
    if (!aligned16(full_a) || (reshard && !aligned16(full_b))) return ZERO_EALIGN;
    if (clip) {
        if (!clip->scratch || clip->scratch_bytes < kNormScratchBytes || !clip->norm_coef ||
            !(clip->max_norm > 0) || !std::isfinite(clip->max_norm))
            return ZERO_EINVAL;
        if (!aligned16(clip->scratch) || !aligned16(clip->norm_coef)) return ZERO_EALIGN;
        if (clip->grad_shard && (rc = check_table(clip->grad_shard, n_ranks)) != ZERO_OK)
            return rc;
    }

    // the fused finite check: the plain step from bf16 rank gradients only
    if (nonfinite && (f32 || clip || acc)) return ZERO_EINVAL;
    if (acc) {
        // accumulation: bf16 rank gradients, no clipping
        if (f32 || clip || acc->micro_batches < 1 || acc->micro_batch < 0 ||
            acc->micro_batch >= acc->micro_batches)
            return ZERO_EINVAL;
        if (acc->micro_batches > 1 && (rc = check_table(acc->grad_acc, n_ranks)) != ZERO_OK)
            return rc;
    }

    StepResources* res = nullptr;
    if ((rc = resources_for_current_device(&res)) != ZERO_OK) return rc;
    cudaEvent_t* ev = res->ev;
    cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
    if ((rc = cuda_status(cudaStreamIsCapturing(main_stream, &capture))) != ZERO_OK) return rc;
    PlanBuilder plan;
    plan.reduce_mode = reduce_mode(acc);
    // While the main stream is being captured the step keeps one compute and
    // one side stream, and the graph builder joins consecutive units and
    // gathers with programmatic edges instead.
    plan.two_compute = plan.two_side = capture == cudaStreamCaptureStatusNone;
    plan.step(n_units, regen != nullptr, clip != nullptr, reshard);

    const uint16_t* unit_grads[ZERO_MAX_RANKS];
    uint16_t* unit_grads_w[ZERO_MAX_RANKS];
    const float* unit_grads_f32[ZERO_MAX_RANKS];
    auto grads_of = [&](int32_t u) {
        const int64_t off = grads_resident ? units[u].offset : 0;
        for (int32_t r = 0; r < n_ranks; ++r) {
            if (f32) {
                unit_grads_f32[r] = static_cast<const float*>(grads[r]) + off;
            } else {
                unit_grads[r] = static_cast<const uint16_t*>(grads[r]) + off;
                unit_grads_w[r] = const_cast<uint16_t*>(unit_grads[r]);
            }
        }
    };
    // The norm passes of consecutive units are chained (programmatic
    // dependent launch) when nothing else was issued on the main stream
    // between them: each reads other gradients and waits for the one before
    // it to complete only before it adds to the shared partials.
    bool after_norm = false;
    // Likewise consecutive unit updates with nothing between them on the main
    // stream (the backward pass without resharding: no gather, no event).
    // Where an event record or wait separates them (the resharding backward
    // pass) they are not chained: measured on GB300, chaining across the
    // events gained nothing.  While the stream is being captured, the graph
    // builder joins the units itself.
    // (tracked per stream: an update follows an update on its own stream)
    bool after_update[4] = {false, false, false, false};
    for (const zero_op_t& op : plan.ops) {
        cudaStream_t s = op.stream == kMain ? main_stream
                         : op.stream == kSide ? side_stream
                         : op.stream == kAux ? res->aux : res->side2;
        const bool chain_norm = after_norm;
        const bool chain_update =
            after_update[op.stream] && capture == cudaStreamCaptureStatusNone;
        if (op.stream == kMain) after_norm = op.kind == ZERO_OP_NORM;
        if (op.kind != ZERO_OP_USE) // USE issues nothing
            after_update[op.stream] = op.kind == ZERO_OP_REDUCE_SCATTER && op.arg != 2;
        switch (op.kind) {
        case ZERO_OP_RECORD:
            rc = cuda_status(cudaEventRecord(ev[op.arg], s));
            break;
        case ZERO_OP_WAIT:
            rc = cuda_status(cudaStreamWaitEvent(s, ev[op.arg], 0));
            break;
        case ZERO_OP_GATHER:
            rc = zero3_gather_unit(&units[op.unit], n_ranks, shard_bf16,
                                   op.arg == kOwnRegion ? full_a + units[op.unit].offset
                                                        : (op.arg == 0 ? full_a : full_b),
                                   s);
            break;
        case ZERO_OP_REGEN:
            grads_of(op.unit);
            rc = zero_gen_grads_unit(regen->seed, hp->step, regen->sigma, regen->outliers,
                                     &units[op.unit], n_ranks, unit_grads_w, s);
            break;
        case ZERO_OP_ACCUMULATE:
            grads_of(op.unit);
            rc = zero3_accumulate_unit(&units[op.unit], n_ranks, unit_grads, acc->grad_acc,
                                       op.arg, s);
            break;
        case ZERO_OP_REDUCE_SCATTER:
            grads_of(op.unit);
            if (op.arg == 2) { // the last micro-batch, fused with the update
                rc = zero3_reduce_scatter_unit_accumulated(&units[op.unit], n_ranks, unit_grads,
                                                           acc->grad_acc, acc->micro_batches,
                                                           master, m, v, shard_bf16, hp, s);
                break;
            }
            if (f32)
                rc = unit_update(&units[op.unit], n_ranks,
                                 reinterpret_cast<const void* const*>(unit_grads_f32), master, m,
                                 v, shard_bf16, hp, nullptr, s, true, false, chain_update);
            else if (op.arg && clip->grad_shard) // the mean the norm pass kept
                rc = unit_update(&units[op.unit], n_ranks,
                                 reinterpret_cast<const void* const*>(clip->grad_shard), master,
                                 m, v, shard_bf16, hp, clip->norm_coef, s, false, true,
                                 chain_update);
            else
                rc = unit_update(&units[op.unit], n_ranks,
                                 reinterpret_cast<const void* const*>(unit_grads), master, m, v,
                                 shard_bf16, hp, op.arg ? clip->norm_coef : nullptr, s, false,
                                 false, chain_update, nonfinite);
            break;
        case ZERO_OP_NORM:
            grads_of(op.unit);
            if (clip->grad_shard) {
                float* unit_shard[ZERO_MAX_RANKS];
                for (int32_t r = 0; r < n_ranks; ++r)
                    unit_shard[r] = clip->grad_shard[r] + units[op.unit].shard_offset;
                rc = grad_reduce_sqnorm(n_ranks, units[op.unit].n_padded, unit_grads, unit_shard,
                                        op.arg, clip->scratch, clip->scratch_bytes, s,
                                        chain_norm);
            } else {
                rc = grad_sqnorm(n_ranks, units[op.unit].n_padded, unit_grads, op.arg,
                                 clip->scratch, clip->scratch_bytes, s, chain_norm);
            }
            break;
        case ZERO_OP_CLIP_COEF:
            rc = clip_coef(clip->scratch, clip->scratch_bytes, clip->max_norm, clip->norm_coef, s);
            break;
        default: // ZERO_OP_USE: the unit's compute would run here
            rc = ZERO_OK;
            break;
        }
        if (rc != ZERO_OK) return rc;
    }
    return ZERO_OK;
}

} // namespace

extern "C" int zero3_step(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                          const uint16_t* const* grads, int32_t grads_resident,
                          float* const* master, float* const* m, float* const* v,
                          uint16_t* const* shard_bf16, uint16_t* full_a, uint16_t* full_b,
                          const zero_hparams_t* hp, const zero_regen_t* regen,
                          const zero_clip_t* clip, int32_t reshard_after_forward,
                          cudaStream_t main_stream, cudaStream_t side_stream)
{
    return run_step(units, n_units, n_ranks, reinterpret_cast<const void* const*>(grads), false,
                    grads_resident, master, m, v, shard_bf16, full_a, full_b, hp, regen, clip,
                    reshard_after_forward, main_stream, side_stream);
}

extern "C" int zero3_step_checked(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                                  const uint16_t* const* grads, int32_t grads_resident,
                                  float* const* master, float* const* m, float* const* v,
                                  uint16_t* const* shard_bf16, uint16_t* full_a,
                                  uint16_t* full_b, const zero_hparams_t* hp,
                                  const zero_regen_t* regen, int32_t reshard_after_forward,
                                  uint32_t* nonfinite_ranks, cudaStream_t main_stream,
                                  cudaStream_t side_stream)
{
    if (!nonfinite_ranks) return ZERO_EINVAL;
    if (reinterpret_cast<uintptr_t>(nonfinite_ranks) % 8 != 0) return ZERO_EALIGN;
    return run_step(units, n_units, n_ranks, reinterpret_cast<const void* const*>(grads), false,
                    grads_resident, master, m, v, shard_bf16, full_a, full_b, hp, regen, nullptr,
                    reshard_after_forward, main_stream, side_stream, nullptr, nonfinite_ranks);
}

extern "C" int zero3_step_microbatch(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                                     const uint16_t* const* grads, float* const* grad_acc,
                                     int32_t micro_batch, int32_t micro_batches,
                                     float* const* master, float* const* m, float* const* v,
                                     uint16_t* const* shard_bf16, uint16_t* full_a,
                                     uint16_t* full_b, const zero_hparams_t* hp,
                                     int32_t reshard_after_forward, cudaStream_t main_stream,
                                     cudaStream_t side_stream)
{
    const AccumArgs acc{grad_acc, micro_batch, micro_batches};
    return run_step(units, n_units, n_ranks, reinterpret_cast<const void* const*>(grads), false, 1,
                    master, m, v, shard_bf16, full_a, full_b, hp, nullptr, nullptr,
                    reshard_after_forward, main_stream, side_stream, &acc);
}

extern "C" int zero3_step_f32grads(const zero_unit_t* units, int32_t n_units, int32_t n_ranks,
                                   const float* const* grads, float* const* master,
                                   float* const* m, float* const* v, uint16_t* const* shard_bf16,
                                   uint16_t* full_a, uint16_t* full_b, const zero_hparams_t* hp,
                                   int32_t reshard_after_forward, cudaStream_t main_stream,
                                   cudaStream_t side_stream)
{
    return run_step(units, n_units, n_ranks, reinterpret_cast<const void* const*>(grads), true, 1,
                    master, m, v, shard_bf16, full_a, full_b, hp, nullptr, nullptr,
                    reshard_after_forward, main_stream, side_stream);
}
