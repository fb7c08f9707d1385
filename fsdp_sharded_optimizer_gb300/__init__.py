"""GB300-native fused ZeRO/FSDP sharded optimizer step.

The N_d data-parallel ranks of a job are emulated as separate buffers on one
GPU; one CUDA kernel reduce-scatters their bf16 gradients (fixed-order fp32
mean), applies AdamW to each owner's fp32 shard and writes the new bf16
weights (the all-gather).  ZeRO-3 adds the per-unit gather and the per-unit
reduce-scatter, scheduled with next-unit prefetch on a side stream
(``zero3_step``, natively or as a CUDA graph).

The public calls carry the C ABI's names (include/zero.h) and live in
``_binding``.  They are loaded on first use, so that ``build`` can be imported
before the library exists; using any of them without a built library raises
ImportError (there is no fallback).
"""
_PUBLIC = ("ZERO_DEFAULT_ALIGN", "ZERO_CHUNK_ELEMS", "ZERO_EALIGN", "ZERO_ECUDA", "ZERO_EINVAL", "ZERO_ETIMEOUT",
           "ZERO_MAX_RANKS", "ZERO_OK", "LIB_PATH", "ZeroError", "hparams", "strerror",
           "zero3_gather_unit", "zero3_reduce_scatter_unit", "zero_bytes_t", "zero_cast_bf16",
           "zero_gen_grads_unit", "zero_gen_master", "zero_hparams_t", "zero_layout",
           "zero_state_bytes", "zero_step_stage12", "zero_stream_wait", "zero_unit_t",
           "zero3_plan", "zero3_step", "zero_op_t", "zero_regen_t", "zero_clip_scratch_bytes",
           "zero_grad_sqnorm", "zero_clip_coef", "zero_step_stage12_clip",
           "zero3_reduce_scatter_unit_clip", "zero_clip_t", "clip_args",
           "zero2_accumulate", "zero2_step_accumulated", "zero_clip_coef_units_noalloc",
           "zero_step_stage12_f32grads", "zero3_reduce_scatter_unit_f32grads",
           "zero_gen_grads_unit_f32", "zero_grad_nonfinite", "zero3_graph_create",
           "zero3_graph_create_f32grads", "zero3_graph_launch", "zero3_graph_destroy",
           "Zero3Graph", "zero_grad_reduce_sqnorm", "zero_step_stage12_reduced",
           "zero3_update_unit_reduced", "zero3_step_f32grads", "zero3_accumulate_unit",
           "zero3_reduce_scatter_unit_accumulated", "zero_reshard_f32", "zero3_plan_microbatch",
           "zero3_step_microbatch", "zero_step_stage12_checked",
           "zero3_reduce_scatter_unit_checked", "zero3_step_checked")

__all__ = list(_PUBLIC)


def __getattr__(name):
    if name in _PUBLIC:
        from . import _binding
        return getattr(_binding, name)
    raise AttributeError("module %r has no attribute %r" % (__name__, name))
