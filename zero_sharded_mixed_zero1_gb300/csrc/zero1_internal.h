// zero1_internal.h - helpers shared by the library's host and CUDA sources
// (library-internal; not part of the C ABI).
#pragma once

#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "zero1.h"

// An NVTX range over one C-ABI call, named after the entry point, so that
// Nsight tools can select a call's kernels and copies (ncu --nvtx-include
// "<name>/").  With no tool attached the range calls do nothing.
struct Z1Trace {
    explicit Z1Trace(const char *name) { nvtxRangePushA(name); }
    ~Z1Trace() { nvtxRangePop(); }
    Z1Trace(const Z1Trace &) = delete;
    Z1Trace &operator=(const Z1Trace &) = delete;
};

// The per-step constants of the AdamW update, evaluated once on the host
// ("CS336 Lecture 7: Parallelism 1" naive DP equation for inv = 1/(B*S);
// "五维并行实战" 4.2 for the AdamW hyperparameters).
struct Z1Consts {
    float inv;    // 1 / (B * S)
    float beta1, omb1;  // beta1, 1 - beta1
    float beta2, omb2;  // beta2, 1 - beta2
    float bc1, bc2;     // 1 - beta1^t, 1 - beta2^t
    float eps;
    float lr;
    float cdec;         // 1 - lr * weight_decay
};

// The element range of shards [shard_begin, shard_end): `base` is its first
// global element, L its length, nv how many of its elements are real (< n).
struct Z1Range {
    int64_t base, L, nv;
};

// Record a one-line reason for the calling thread and return `code`.
int z1_fail(int code, const char *fmt, ...);

// Check a plan for internal consistency (as zero1_plan would build it).
int z1_check_plan(const zero1_plan_t *plan);

// Validate [shard_begin, shard_end) against the plan and fill the range.
int z1_range(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end, Z1Range *out);

// b^t in double by square-and-multiply over the bits of t (least significant
// first), one rounding per multiplication: reproducible on any IEEE-754
// implementation, the device included.
double z1_pow_int(double b, int64_t t);

// Validate hyperparameters and evaluate the constants: double precision,
// rounded once to float, beta^t from z1_pow_int.
int z1_adamw_constants(const zero1_adamw_t *hp, int32_t M, Z1Consts *out);

// Pieces of the staged step with dynamic loss scaling (zero1_dynamic.cu):
//  z1_scaled_range launches the in-place fused step on the element range
//  [elem_begin, elem_end) with S and t read from the device scaler; it returns
//  at once on the device when scaler->overflow is set, which must therefore
//  be final before the launch.  Pointers start at elem_begin, as for
//  zero1_step_bucket.
//  z1_scaler_advance launches the scaler update (the loss-scale rule; the
//  attempt's flag is read and cleared).
//  z1_check_scaler_and_policy validates what both need, without launching.
int z1_scaled_range(const zero1_plan_t *plan, int64_t elem_begin, int64_t elem_end, const void *const *grads,
                    float *master, float *m, float *v, void *params, const zero1_adamw_t *hp,
                    const zero1_scaler_t *scaler, zero1_stream_t stream);
int z1_scaler_advance(zero1_scaler_t *scaler, const zero1_loss_scale_policy_t *policy, const zero1_adamw_t *hp,
                      int32_t M, zero1_stream_t stream);
int z1_check_scaler_and_policy(const zero1_scaler_t *scaler, const zero1_loss_scale_policy_t *policy,
                               const zero1_adamw_t *hp, int32_t M);

// Record a kernel launch for zero1_debug_last_launch (per host thread): the
// kernel, its grid, the resident blocks per SM the grid was sized from, and
// whether the vector body moved fp32 in 32-byte accesses.
void z1_note_launch(const void *kernel, int grid, int blocks_per_sm, int block, int w32);
