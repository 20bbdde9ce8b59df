"""GB300 (sm_103a) ZeRO Stage-1 optimizer step.

The M data-parallel replicas' bf16 gradients are reduce-scattered in rank
order and scaled by 1/(B*S); each shard's fp32 master weights and Adam moments
get an AdamW update; the updated bf16 parameters are all-gathered into the
full buffer.  One fused CUDA kernel does all three phases.  The C ABI is in
include/zero1.h; this package is its thin Python binding.
"""
from ._lib import (  # noqa: F401
    ZERO1_DTYPE_BF16,
    ZERO1_DTYPE_F32,
    ZERO1_STAGE_GRADS,
    ZERO1_STAGE_PARAMS,
    ZERO1_STAGE_STATE,
    ZERO1_STAGE_TIMELINE,
    ZERO1_MAX_REPLICAS,
    SCALER_BYTES,
    AdamW,
    FusedStep,
    LossScalePolicy,
    Plan,
    Zero1Error,
    dp_allreduce,
    library_path,
    load,
    new_scaler,
    scaler_state,
    zero1_adamw_update,
    zero1_all_gather,
    zero1_all_gather_shards,
    zero1_overflow_check,
    zero1_plan,
    zero1_plan_memory,
    zero1_plan_segments,
    zero1_reduce_scatter,
    zero1_reduce_scatter_adamw_allgather,
    zero1_scaler_init,
    zero1_step_bucket,
    zero1_step_tma,
    zero1_device_status,
    zero1_bounded_wait_selftest,
    zero1_checksum,
    zero1_step_dynamic,
    zero1_step_dynamic_noalloc,
    zero1_step_dynamic_pingpong,
    zero1_pingpong_bucket,
    zero1_pingpong_finish,
    PingPongBuckets,
    current_state,
    debug_last_launch,
)
from .host_stream import HostStreamedStep  # noqa: E402,F401
