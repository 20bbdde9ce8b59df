/*
 * zero1.h - C ABI of libzero1.so, the GB300 (sm_103a) ZeRO Stage-1 optimizer
 * step: reduce-scatter of M data-parallel replicas' bf16 gradients, AdamW on
 * the fp32 shard state, all-gather of the updated bf16 parameters.
 *
 * On one GPU the M replicas are M gradient buffers in device memory, so the
 * "collectives" are device-memory traffic inside the kernels.
 *
 * Conventions for every call:
 *  - Pointers named as device pointers must be addressable by the current
 *    CUDA device: HBM of that device, or pinned (page-locked) host memory,
 *    which the unified address space maps at the same address.  On GB300 the
 *    kernels then read and write host memory directly over NVLink-C2C: the
 *    gradients can stream from host memory without a staging copy, the bf16
 *    parameters can land in host memory, and master/m/v can live in host
 *    memory (optimizer-state offload).  Such accesses run at the host link's
 *    speed instead of HBM's.  Arrays of pointers (grads, outs) are HOST arrays
 *    of M such pointers.  The caller owns all memory; the library allocates
 *    nothing and keeps no state between calls, except a staged-step handle
 *    (zero1_staged_create), which owns its staging memory, streams and
 *    events until zero1_staged_destroy.
 *  - Sizes are in elements.  bf16 buffers hold IEEE binary32 values'
 *    upper 16 bits (bfloat16); fp32 buffers hold IEEE binary32.
 *  - Device pointers must be naturally aligned (2 bytes for bf16, 4 for fp32,
 *    4 for the flag); 16-byte alignment at a common element phase selects the
 *    128-bit vector path, anything else runs a per-element path.
 *  - GPU work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and is asynchronous; nothing synchronises the host.
 *  - Every call validates all arguments before launching anything and
 *    returns ZERO1_OK (0) or a negative code; on error nothing was enqueued.
 *    zero1_last_error() gives a one-line reason (per host thread).
 *
 * Pages cited (title, section):
 *  [DP]   "CS336 Lecture 7: Parallelism 1", 朴素数据并行 (naive data parallelism):
 *         theta_{t+1} = theta_t - eta (1/B) sum_{i<=B} grad L(x_i), the sum
 *         split across M GPUs with B/M samples each.
 *  [COLL] same page, 集合通信原语 (All-Reduce, Reduce-Scatter, All-Gather) and
 *         the identity All-Reduce == Reduce-Scatter + All-Gather.
 *  [MEM]  same page, 训练内存的详细分析: 16 bytes per parameter = bf16 param 2 +
 *         bf16 grad 2 + fp32 master 4 + Adam m 4 + Adam v 4.
 *  [Z1]   same page, ZeRO Stage 1 (优化器状态分片): Reduce-Scatter so GPU i holds
 *         the summed gradient of shard i, local update of shard i with its
 *         optimizer state, All-Gather of the updated parameters.
 *  [PART] "第2章 软件程序与专用硬件的结合" 2.3.4: each of N GPUs keeps 1/N of the
 *         optimizer state.
 *  [OPT]  "五维并行实战" 4.2 (AdamW lr, betas, eps, weight_decay; the fp16 loss
 *         scale block) and 3.2 trap 3 (loss becoming inf under loss scaling).
 *
 * Arithmetic (fixed so that results are reproducible bit for bit):
 *  per element j, all fp32 with one round-to-nearest-even per operation, no
 *  fused multiply-add, IEEE division and square root:
 *    s  = f32(g_0[j]) + f32(g_1[j]) + ... + f32(g_{M-1}[j])   (left to right)
 *    g  = s * inv                                   inv = 1/(B*S)
 *    m' = beta1*m + (1-beta1)*g
 *    v' = beta2*v + (1-beta2)*(g*g)
 *    u  = (m'/(1-beta1^t)) / (sqrt(v'/(1-beta2^t)) + eps)
 *    w' = w*(1-lr*wd) - lr*u
 *    param = bf16_round_nearest_even(w')
 *  The constants inv, 1-beta1, 1-beta2, 1-beta^t and 1-lr*wd are evaluated
 *  in double and rounded once to float; beta^t is square-and-multiply over
 *  the bits of t (least significant first), so the host and the device
 *  produce the same constants.  Padding elements (global index >= n) take
 *  g = +0.
 */
#ifndef ZERO1_H
#define ZERO1_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
/* A cudaStream_t. */
typedef struct CUstream_st *zero1_stream_t;

/* Status codes. */
#define ZERO1_OK 0
#define ZERO1_EINVAL (-1) /* null pointer, empty or out-of-range size, bad hyperparameter */
#define ZERO1_EALIGN (-2) /* a device pointer is not naturally aligned */
#define ZERO1_ERANGE (-3) /* M above ZERO1_MAX_REPLICAS or a size the library does not support */
#define ZERO1_ECUDA (-4)  /* a CUDA runtime call or a kernel launch failed */

/* Largest data-parallel degree M; the M gradient pointers travel by value in
 * the kernel arguments. */
#define ZERO1_MAX_REPLICAS 64

#define ZERO1_DTYPE_BF16 0
#define ZERO1_DTYPE_F32 1

/* Shard plan [PART], [Z1].  n real parameters in one flat buffer, padded to
 * P = ceil(n / (M*align)) * M*align; shard i is [i*s, (i+1)*s), s = P/M.
 * The flat buffer may be the concatenation of n_tensors tensors (a model's
 * parameter list, flattened in order); shard cuts may fall inside a tensor. */
typedef struct zero1_plan {
    int64_t n;         /* |theta|, real parameters, >= 1 */
    int64_t padded_n;  /* P */
    int64_t shard;     /* s = P / M */
    int32_t M;         /* data-parallel degree (replicas), 1..ZERO1_MAX_REPLICAS */
    int32_t align;     /* shard alignment unit in elements, >= 1 */
    int32_t n_tensors; /* tensors in the flat buffer; 0 when built without a list */
} zero1_plan_t;

/* AdamW hyperparameters of one step [OPT], the batch of [DP] and the loss
 * scale: gradients arrive multiplied by loss_scale and summed over the B/M
 * samples of each replica. */
typedef struct zero1_adamw {
    float lr;            /* finite */
    float beta1, beta2;  /* in [0, 1) */
    float eps;           /* >= 0 */
    float weight_decay;  /* finite; decoupled, multiplied by lr */
    float loss_scale;    /* S > 0, finite */
    int64_t global_batch;/* B >= M */
    int64_t step;        /* t >= 1; a skipped step does not advance it */
} zero1_adamw_t;

/* Build a plan [PART], [Z1].  Host only; allocates nothing.
 *  n, M, align:   as in zero1_plan_t;
 *  tensor_numels: NULL (one flat buffer; n_tensors must be 0), or a host
 *                 array of n_tensors >= 1 tensor sizes (each >= 0) that sum
 *                 to n; the plan records n_tensors for zero1_plan_segments.
 * EINVAL if n < 1, align < 1, M < 1 or the tensor list is inconsistent;
 * ERANGE if M > ZERO1_MAX_REPLICAS or P overflows int64. */
int zero1_plan(int64_t n, int32_t M, int32_t align, const int64_t *tensor_numels, int32_t n_tensors,
               zero1_plan_t *out);

/* Per-tensor pieces of shard `shard_index` [PART], [Z1], for a plan built
 * with a tensor list: tensor_numels is that list again (plan->n_tensors host
 * int64 sizes summing to plan->n).  Host only.  Writes up to `cap` pieces, in
 * shard order: the tensor index, the piece's first element inside that
 * tensor (seg_begin) and its length.  The pieces tile the shard's real
 * elements from the shard's first element on, so a piece's offset inside the
 * shard is the sum of the lengths before it; padding belongs to no tensor.
 * *count gets the number of pieces.  EINVAL on bad arguments or a plan built
 * without tensors, ERANGE if more than cap pieces are needed. */
int zero1_plan_segments(const zero1_plan_t *plan, const int64_t *tensor_numels, int32_t shard_index,
                        int64_t *seg_tensor, int64_t *seg_begin, int64_t *seg_len, int32_t cap,
                        int32_t *count);

/* Bytes per rank [MEM], [Z1]: naive data parallelism keeps 16 bytes of every
 * parameter on each rank; ZeRO-1 keeps the bf16 parameters and gradients
 * whole (4 bytes per parameter) and 12 bytes of fp32 state per shard element.
 * Host only. */
int zero1_plan_memory(const zero1_plan_t *plan, int64_t *naive_bytes_per_rank,
                      int64_t *zero1_bytes_per_rank);

/* The fused ZeRO-1 step over shards [shard_begin, shard_end) [Z1], [DP], [MEM]:
 * one kernel reads each replica's bf16 gradient once, sums the replicas in
 * rank order, scales by 1/(B*S), updates the fp32 master/m/v in place and
 * writes the bf16 parameters once.
 *
 * Let L = (shard_end - shard_begin) * s, base = shard_begin * s and
 * nv = clamp(n - base, 0, L) (the real parameters in the range).
 *  grads[r]  (r < M): device bf16, element `base` of replica r's gradient;
 *                      nv elements are read.
 *  master, m, v:      device fp32, the range's state, L elements each, read
 *                      and written in place.
 *  params:            device bf16, element `base` of the full parameter
 *                      buffer; nv elements are written.
 *  overflow_flag:     device uint32 or NULL.  With skip_if_flag == 0 the
 *                      kernel ORs 1 into it if any of the nv sums is inf or
 *                      NaN [OPT] (it never clears it).  With skip_if_flag != 0
 *                      the kernel only reads it, and if it is nonzero on entry
 *                      writes nothing at all (run zero1_overflow_check first
 *                      on the same stream to skip a step globally).
 * Buffers must not overlap, except grads may alias one another.  When the
 * range holds no real parameter (nv == 0: all padding) grads and params are
 * not touched and may be NULL.  Keep master, m and v in the same kind of
 * memory: the kernel is chosen from where master lives (pinned host memory
 * selects the offload kernel, which keeps more state loads in flight and
 * writes whole lines of host memory).
 * EINVAL: NULL pointers, bad range, bad hyperparameters, skip_if_flag with a
 * NULL flag, master/m/v/params overlapping one another or a gradient buffer. */
int zero1_reduce_scatter_adamw_allgather(const zero1_plan_t *plan, int32_t shard_begin,
                                         int32_t shard_end, const void *const *grads,
                                         float *master, float *m, float *v, void *params,
                                         const zero1_adamw_t *hp, uint32_t *overflow_flag,
                                         int32_t skip_if_flag, zero1_stream_t stream);

/* Bucketed step: the fused step on the element range [elem_begin, elem_end)
 * of the padded flat buffer (0 <= elem_begin < elem_end <= P) - one bucket of
 * gradients as it arrives during the backward pass [OPT] (reduce_bucket_size,
 * contiguous_gradients, overlap_comm; "CS336 Lecture 7: Parallelism 1", ZeRO
 * Stage 2: gradients handed off bucket by bucket instead of held whole).
 * The step is element-wise, so calls over disjoint buckets that cover [0, P)
 * give bit for bit one zero1_reduce_scatter_adamw_allgather over all shards,
 * and a bucket's gradient buffers can be reused once its launch has run: the
 * full gradient never has to exist at once.
 *  grads[r]:     device bf16, replica r's gradients of the bucket (the real
 *                elements, below n, are read; nv = clamp(n - elem_begin, 0,
 *                elem_end - elem_begin));
 *  master, m, v: device fp32, element elem_begin of the state holding the
 *                bucket; elem_end - elem_begin elements are updated;
 *  params:       device bf16, element elem_begin of the parameters; nv written;
 *  overflow_flag: device uint32 or NULL, ORed as in the fused step.  A bucket
 *                cannot wait for later buckets' flags: when steps must be
 *                skipped on overflow, use zero1_step_dynamic.
 * EINVAL on a bad range or arguments (as the fused step). */
int zero1_step_bucket(const zero1_plan_t *plan, int64_t elem_begin, int64_t elem_end,
                      const void *const *grads, float *master, float *m, float *v, void *params,
                      const zero1_adamw_t *hp, uint32_t *overflow_flag, zero1_stream_t stream);

/* Staged step: the fused step over buffers in pinned host memory, staged
 * through device memory by the copy engines [Z1], [OPT] (offload_optimizer:
 * the fp32 optimizer state kept in host memory; the update itself runs on
 * the GPU).  The handle's range (shards [shard_begin, shard_end)) is cut into
 * chunks of chunk_elems elements (rounded up to a multiple of 8).  For each
 * chunk an inbound stream copies the staged inputs into one of three device
 * slots, `stream` runs zero1_step_bucket on the slot, and an outbound stream
 * copies the staged outputs back; with three slots the inbound copy of one
 * chunk, the step on the next older one and the outbound copy of the one
 * before overlap.  Results are bit for bit those of
 * zero1_reduce_scatter_adamw_allgather on device buffers (the step is
 * element-wise).
 *
 * `what` selects what is staged (at least one bit):
 *  ZERO1_STAGE_GRADS:  grads[r] are pinned host memory, copied in;
 *  ZERO1_STAGE_STATE:  master, m, v are pinned host memory, copied in and
 *                      the updated values copied back;
 *  ZERO1_STAGE_PARAMS: the updated bf16 parameters are also copied to
 *                      params_host (pinned host memory).
 * Buffers not staged must be device memory; params is always device memory
 * (the kernels write it).  Layouts as zero1_reduce_scatter_adamw_allgather:
 * grads[r] and params hold the range's nv real elements, master/m/v its L
 * elements, params_host nv elements.
 *
 * zero1_staged_create allocates, on the current device, 3 x chunk x (2M
 * bytes if gradients are staged + 12 bytes if state is) of device memory,
 * two non-blocking streams and the events that order them.
 * zero1_staged_step enqueues one step; when `stream` reaches the work
 * enqueued after it, the step's copies back to host memory are complete.
 * Successive calls on one handle may use different streams (each waits for
 * the previous call); calls must not be made concurrently from several host
 * threads, and the call cannot be captured in a CUDA graph (EINVAL while
 * `stream` is capturing).  overflow_flag is ORed as in the fused step; a
 * chunk cannot wait for later chunks' flags, so there is no skip: when steps
 * must be skipped on overflow, check the gradients first
 * (zero1_overflow_check) and do not call the step.
 * zero1_staged_destroy waits for the handle's queued work, then frees it
 * (NULL is accepted).
 * EINVAL: bad range, `what` or chunk size, a NULL or misplaced buffer (host
 * where device memory is required or the reverse), overlapping buffers, the
 * wrong current device, a capturing stream.  All arguments are checked before
 * anything is enqueued; on ZERO1_ECUDA part of the step may have been
 * enqueued. */
#define ZERO1_STAGE_GRADS 1
#define ZERO1_STAGE_STATE 2
#define ZERO1_STAGE_PARAMS 4
/* Tracing: with this bit in `what` the handle also records CUDA timing
 * events around each chunk's copies and kernel (zero1_staged_timeline). */
#define ZERO1_STAGE_TIMELINE 8
typedef struct zero1_staged zero1_staged_t;
int zero1_staged_create(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end, int32_t what,
                        int64_t chunk_elems, zero1_staged_t **out);
int zero1_staged_step(zero1_staged_t *handle, const void *const *grads, float *master, float *m, float *v,
                      void *params, void *params_host, const zero1_adamw_t *hp, uint32_t *overflow_flag,
                      zero1_stream_t stream);
int zero1_staged_destroy(zero1_staged_t *handle);

/* The handle's chunk boundaries: *count = chunks + 1 values 0 = cuts[0] <
 * ... < cuts[chunks] = L, written to cuts (if not NULL; ERANGE if cap is
 * smaller): chunks of chunk_elems (rounded up to a multiple of 8) elements,
 * the last one shorter. */
int zero1_staged_chunks(const zero1_staged_t *handle, int64_t *cuts, int32_t cap, int32_t *count);

/* Timeline of the handle's last step (tracing; the handle must have been
 * created with ZERO1_STAGE_TIMELINE).  *count = chunks; if ms is not NULL it
 * gets 6 floats per chunk, in chunk order, in milliseconds since the step
 * started on the caller's stream: inbound copies start, inbound copies end,
 * kernel start, kernel end, outbound copies start, outbound copies end (the
 * last two -1 when nothing is copied back).  A start is when that stream
 * reached the chunk, after its waits for the previous stage.  Waits for the
 * last step to finish (synchronous).  EINVAL without the bit, before any
 * step, or after a step call that returned an error; ERANGE if cap < 6 x
 * chunks. */
int zero1_staged_timeline(zero1_staged_t *handle, float *ms, int32_t cap, int32_t *count);

/* The fused step with its vector body staged through shared memory by the
 * Tensor Memory Accelerator [Z1], [DP], [MEM]: a producer warp issues 1-D bulk
 * copies (cp.async.bulk, completion counted on mbarriers) of each tile's M
 * gradient slices and master/m/v into a ring of shared-memory stages, and
 * eight consumer warps compute from there.  Same arguments and bit for bit the
 * same results as zero1_reduce_scatter_adamw_allgather; every buffer must be
 * device memory (EINVAL otherwise).  On GB300 this staging measured slower
 * than the direct register loads of the fused step (the stream has no reuse),
 * so the fused step does not use it; it is kept so the comparison can be
 * reproduced.  Its waits are bounded: a wait that runs out (1 s) sets
 * bit 0 of the device status (zero1_device_status) and the kernel returns. */
int zero1_step_tma(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                   const void *const *grads, float *master, float *m, float *v, void *params,
                   const zero1_adamw_t *hp, uint32_t *overflow_flag, int32_t skip_if_flag,
                   zero1_stream_t stream);

/* The library's device status word on the current device: bit 0 set if a
 * bounded wait in a kernel ran out (the kernel then stopped early and its
 * outputs are incomplete).  Copies it to *status (synchronous with the
 * device) and clears it if `clear` is nonzero. */
int zero1_device_status(uint32_t *status, int32_t clear);

/* Failure-detection self-test of the bounded waits (no counterpart in the
 * pages): one thread arms a shared-memory mbarrier that expects two arrivals,
 * arrives once and waits for the phase with the same bounded wait the staged
 * kernel uses, limited to limit_us microseconds (1 .. 1,000,000).  The wait
 * must run out: the kernel writes 1 to *gave_up (device uint32), sets bit 0
 * of the device status word (zero1_device_status) and returns, leaving the
 * context usable.  Nothing else is read or written. */
int zero1_bounded_wait_selftest(uint32_t limit_us, uint32_t *gave_up, zero1_stream_t stream);

/* Overflow check [OPT]: ORs 1 into *flag (device uint32) if the rank order
 * fp32 sum of any real element of shards [shard_begin, shard_end) is inf or
 * NaN.  Reads the same nv elements of grads[r] as the fused step (none, and
 * grads may be NULL, when nv == 0); never clears the flag. */
int zero1_overflow_check(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                         const void *const *grads, uint32_t *flag, zero1_stream_t stream);

/* Naive data-parallel All-Reduce [COLL], [DP] over all n elements: every
 * outs[r] receives (rank order fp32 sum) * scale, as bf16 (round to nearest
 * even) or fp32 per out_dtype.  grads_in[r]: device bf16, n elements;
 * outs[r]: device, n elements of out_dtype.  With ZERO1_DTYPE_BF16 outs may
 * alias grads_in (in place); with ZERO1_DTYPE_F32 they must not overlap. */
int dp_allreduce(const zero1_plan_t *plan, const void *const *grads_in, void *const *outs,
                 float scale, int32_t out_dtype, zero1_stream_t stream);

/* Unfused phases [Z1] (for the All-Reduce identity and for comparison with
 * the fused step).  Same range conventions as the fused step.
 *
 * Reduce-scatter [COLL]: out (device, L elements of out_dtype) gets
 * (rank order fp32 sum) * scale for the nv real elements and +0 for padding;
 * flag (device, may be NULL) as in zero1_overflow_check.  These calls reject
 * (EINVAL) a buffer they write that overlaps another buffer of the call (the
 * gradients may alias one another). */
int zero1_reduce_scatter(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                         const void *const *grads, float scale, int32_t out_dtype, void *out,
                         uint32_t *flag, zero1_stream_t stream);

/* AdamW on L elements of fp32 state given the already scaled fp32 gradient g
 * (device, L elements); hp->global_batch and hp->loss_scale are validated
 * but not applied. */
int zero1_adamw_update(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                       const float *g, float *master, float *m, float *v,
                       const zero1_adamw_t *hp, zero1_stream_t stream);

/* All-gather of the updated shard range [COLL], [Z1]: params (device bf16,
 * element `base` of the full buffer) gets bf16(master) for the nv real
 * elements. */
int zero1_all_gather(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                     const float *master, void *params, zero1_stream_t stream);

/* All-gather of bf16 shards [COLL]: `shards` (device bf16, the P-element
 * concatenation of all M shards) is copied, first n elements, into each of
 * the M outputs outs[r] (device bf16, n elements).  With zero1_reduce_scatter
 * over all shards this is the right-hand side of All-Reduce ==
 * Reduce-Scatter + All-Gather. */
int zero1_all_gather_shards(const zero1_plan_t *plan, const void *shards, void *const *outs,
                            zero1_stream_t stream);

/* ---------------------------------------------------------------------------
 * Dynamic loss scaling with the skip decided on the device [OPT]
 *
 * The fp16 block of [OPT] names the policy's keys: loss_scale 0 (dynamic),
 * initial_scale_power, loss_scale_window, hysteresis, min_loss_scale.  The
 * rule taken from them: an attempt whose summed gradients overflow writes
 * nothing and leaves t unchanged; it uses up one unit of hysteresis, and when
 * none is left S is divided by `factor` (not below min_scale) and the
 * hysteresis is refilled; the clean-attempt count restarts.  A clean attempt
 * applies the step and advances t; after `window` clean attempts in a row S
 * is multiplied by `factor` (unless that overflows fp32), the count restarts
 * and the hysteresis is refilled.
 *
 * S, t and the counters live in device memory (zero1_scaler_t), so a training
 * loop never has to read the flag on the host: the caller scales its loss by
 * the device-resident `scale` and calls zero1_step_dynamic each iteration.
 * ------------------------------------------------------------------------- */

typedef struct zero1_loss_scale_policy {
    float initial_scale; /* S at the first attempt (2^initial_scale_power), finite, > 0 */
    float factor;        /* growth and back-off factor, finite, > 1 */
    int32_t window;      /* loss_scale_window, >= 1 */
    int32_t hysteresis;  /* overflowing attempts tolerated before S shrinks, >= 1 */
    float min_scale;     /* min_loss_scale, finite, > 0 */
} zero1_loss_scale_policy_t;

/* Device-resident scaler state (56 bytes, 8-byte aligned, in device memory). */
typedef struct zero1_scaler {
    float scale;             /* S of the next attempt */
    float inv;               /* 1/(B*S) of the next attempt */
    float bc1, bc2;          /* 1 - beta1^t, 1 - beta2^t of the next attempt */
    int64_t step;            /* t of the next applied step */
    int64_t attempts;        /* attempts so far */
    int64_t skipped;         /* attempts skipped because their gradients overflowed */
    int32_t good_steps;      /* clean attempts in a row since S last changed */
    int32_t hysteresis_left; /* overflowing attempts still tolerated */
    uint32_t overflow;       /* flag of the attempt in progress; 0 between attempts */
    uint32_t current;        /* ping-pong step: copy (0 or 1) of master/m/v holding the current state */
} zero1_scaler_t;

/* Start a scaler (one tiny kernel on `stream`): S = policy->initial_scale,
 * t = hp->step, the derived constants for hp->global_batch and hp->beta1/2.
 * scaler: device pointer to a zero1_scaler_t.  hp->loss_scale is not used. */
int zero1_scaler_init(zero1_scaler_t *scaler, const zero1_loss_scale_policy_t *policy,
                      const zero1_adamw_t *hp, zero1_stream_t stream);

/* One attempt of the dynamically scaled ZeRO-1 step over shards
 * [shard_begin, shard_end) [Z1], [OPT], three kernels on `stream`:
 *  1. reduce-scatter: sums[j] = rank-order fp32 sum of the M replicas for
 *     the nv real elements (+0 on padding), ORing the overflow flag into
 *     scaler->overflow;
 *  2. if scaler->overflow is clear: the AdamW update with g = sums * (1/(B*S))
 *     and the bias corrections of the scaler's t, then the bf16 parameters -
 *     bit for bit the fused step with S and t taken from the scaler; if it is
 *     set: nothing is written;
 *  3. the scaler advances by the rule above and its flag is cleared.
 * The gradients are read once: 2M + 4 + 4 + 24 + 2 bytes per parameter.
 * Arguments as for zero1_reduce_scatter_adamw_allgather, plus:
 *  hp:      lr, betas, eps, weight decay and global batch (its loss_scale and
 *           step are ignored: the scaler's are used);
 *  scaler:  device pointer, started with zero1_scaler_init;
 *  sums:    device fp32 workspace of at least L elements (scratch; its
 *           contents on return are the last attempt's sums).
 * EINVAL as the fused step, also if sums or the scaler overlaps another
 * buffer. */
int zero1_step_dynamic(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                       const void *const *grads, float *master, float *m, float *v, void *params,
                       const zero1_adamw_t *hp, zero1_scaler_t *scaler,
                       const zero1_loss_scale_policy_t *policy, float *sums, zero1_stream_t stream);

/* One attempt of the dynamically scaled step with ping-pong state [Z1], [OPT]:
 * the same rule and bit for bit the same results as zero1_step_dynamic, in a
 * single pass over the data (2M + 26 bytes per parameter, the fused step's
 * traffic) at the cost of a second copy of master/m/v.  master[k], m[k],
 * v[k] (k = 0, 1; host arrays of two device pointers, L fp32 elements each,
 * distinct buffers) are two copies of the state; scaler->current (0 after
 * zero1_scaler_init) names the copy that holds the current state.  Three
 * kernels on `stream`:
 *  1. the fused step reading copy `current` and writing the updated master,
 *     m, v into the other copy and the bf16 parameters into params, ORing the
 *     overflow flag into scaler->overflow;
 *  2. if the flag is set, params is rewritten as bf16(master[current]) - so
 *     a skipped attempt leaves params unchanged provided they held
 *     bf16(master[current]) on entry, as they do after any applied step;
 *  3. the scaler advances by the rule above; a clean attempt also switches
 *     scaler->current to the copy just written.
 * The other copy's contents on entry do not matter.  Both copies must start
 * at the same 16-byte phase for the 128-bit path (else the whole range runs
 * per element).  No workspace is needed; the call can be captured in a CUDA
 * graph (the copy to read is decided on the device).  EINVAL: as
 * zero1_step_dynamic, or any two of the six state buffers, params, the
 * scaler and the gradients overlap (the gradients may alias one another). */
int zero1_step_dynamic_pingpong(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                const void *const *grads, float *const *master, float *const *m,
                                float *const *v, void *params, const zero1_adamw_t *hp, zero1_scaler_t *scaler,
                                const zero1_loss_scale_policy_t *policy, zero1_stream_t stream);

/* The ping-pong attempt in buckets, for gradients that arrive bucket by
 * bucket during the backward pass [Z1], [OPT] (reduce_bucket_size,
 * overlap_comm; "CS336 Lecture 7: Parallelism 1", ZeRO Stage 2).  Because an
 * attempt only writes the non-current copy, each bucket can be updated as
 * soon as its gradients exist, before the attempt's overflow flag is known:
 *  zero1_pingpong_bucket: kernel 1 of zero1_step_dynamic_pingpong on the
 *      element range [elem_begin, elem_end) of the padded flat buffer
 *      (grads[r]: the bucket's gradients; master[k], m[k], v[k], params:
 *      pointers to element elem_begin of each copy and of the parameters, as
 *      zero1_step_bucket); the flag is ORed into scaler->overflow;
 *  zero1_pingpong_finish: kernels 2 and 3 over shards [shard_begin,
 *      shard_end) (master[k] and params at the range's first element).
 * The buckets of one attempt must cover the finish's whole range, each
 * element once, before the finish; then the attempt is bit for bit
 * zero1_step_dynamic_pingpong over that range (the step is element-wise and
 * the copy to read does not change before the finish).  A bucket's gradient
 * buffers can be reused once its launch has run. */
int zero1_pingpong_bucket(const zero1_plan_t *plan, int64_t elem_begin, int64_t elem_end,
                          const void *const *grads, float *const *master, float *const *m, float *const *v,
                          void *params, const zero1_adamw_t *hp, zero1_scaler_t *scaler, zero1_stream_t stream);
int zero1_pingpong_finish(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                          float *const *master, void *params, const zero1_adamw_t *hp, zero1_scaler_t *scaler,
                          const zero1_loss_scale_policy_t *policy, zero1_stream_t stream);

/* The staged step with dynamic loss scaling [OPT] (the fp16 block together
 * with offload_optimizer: the fp32 state in host memory, S and t on the
 * device): an overflow pass over the attempt's gradients ORs the flag into
 * scaler->overflow; every chunk is then staged as in zero1_staged_step, and
 * its kernel takes 1/(B*S) and the bias corrections from the scaler and
 * returns at once when the flag is set, so an overflowing attempt changes no
 * state and no parameter (its copies move unchanged values); the scaler then
 * advances by the loss-scale rule.  Bit for bit zero1_step_dynamic on the
 * same buffers in device memory.  scaler: device zero1_scaler_t started with
 * zero1_scaler_init; hp as for zero1_step_dynamic (loss_scale and step are
 * the scaler's).  Arguments and errors otherwise as zero1_staged_step.  The
 * overflow pass reads the gradients where they are: over the host link when
 * they are staged. */
int zero1_staged_step_dynamic(zero1_staged_t *handle, const void *const *grads, float *master, float *m, float *v,
                              void *params, void *params_host, const zero1_adamw_t *hp, zero1_scaler_t *scaler,
                              const zero1_loss_scale_policy_t *policy, zero1_stream_t stream);

/* ---------------------------------------------------------------------------
 * The dynamically scaled step without any device allocation by the caller.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot call cudaMalloc: programs whose own pool allocator takes the device
 * memory at start-up (a library cudaMalloc then fails or splits that pool),
 * and code that must not allocate or free because cudaMalloc/cudaFree can
 * synchronise the device and stall work on other streams.
 *
 * It is zero1_step_dynamic with the fp32 sums workspace replaced by an array
 * inside the library: ZERO1_NOALLOC_MAX_ELEMS floats (64 MiB) that every GPU
 * loading libzero1.so holds until the process exits.  The caller still
 * passes gradients, state, parameters, scaler and policy.
 *  - One call is one whole attempt: it decides the skip for its whole range
 *    and advances the scaler (t, S, the counters) once.  So the range must
 *    fit: L = (shard_end - shard_begin) * s <= ZERO1_NOALLOC_MAX_ELEMS.  A
 *    longer range returns ZERO1_ERANGE before anything is launched, with the
 *    scaler untouched; it needs zero1_step_dynamic and a caller-provided
 *    workspace (splitting one attempt over several calls would advance the
 *    scaler several times and could skip only part of an overflowing step).
 *  - The first call on a device looks up the array's device address on that
 *    device (cudaGetSymbolAddress, with that device current); make that first
 *    call before any stream capture.  The address is looked up again only if
 *    the device's current context is no longer the one it was looked up in
 *    (after cudaDeviceReset).  No cudaMalloc, cudaFree or other allocating
 *    routine is called.
 *  - All calls share the one array and it keeps the last call's sums; nothing
 *    in it needs to start at zero (each call writes all L sums before reading
 *    them).  Calls that overlap on the GPU (other streams, other threads) race
 *    on it: serialise them.
 * Results are bit for bit those of zero1_step_dynamic. */
#define ZERO1_NOALLOC_MAX_ELEMS (16 * 1024 * 1024)
int zero1_step_dynamic_noalloc(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                               const void *const *grads, float *master, float *m, float *v, void *params,
                               const zero1_adamw_t *hp, zero1_scaler_t *scaler,
                               const zero1_loss_scale_policy_t *policy, zero1_stream_t stream);

/* Consistency checksum of a buffer: the silent-data-corruption guard for the
 * replicated parameters ("CS336 Lecture 7: Parallelism 1" case studies report
 * silent data corruption on large runs; after the all-gather every rank must
 * hold the same parameters, so ranks can compare these two words).  Over the
 * buffer's 16-bit units u_0 .. u_{U-1} (U = nbytes / 2, little-endian):
 *   out[0] = sum u_i mod 2^64,  out[1] = sum (i + 1) * u_i mod 2^64.
 * Exact integer sums: the result does not depend on the order of summation.
 * Any change of one unit changes out[0]; swapping two unequal units changes
 * out[1].  data: device (or pinned host) memory, 2-byte aligned; nbytes even;
 * out: device, two uint64, 8-byte aligned, overwritten (cleared on `stream`
 * first). */
int zero1_checksum(const void *data, int64_t nbytes, uint64_t *out, zero1_stream_t stream);

/* Text of a status code. */
const char *zero1_strerror(int code);

/* One-line reason for the last non-OK status returned on this host thread. */
const char *zero1_last_error(void);

/* ABI version, incremented on any incompatible change. */
int zero1_abi_version(void);

/* Introspection for tests and tuning (no counterpart in the pages): the last
 * streaming kernel that a library call launched on this host thread (every
 * kernel whose grid is sized as one resident wave; not the one-thread scaler
 * kernels, the shared-memory staged kernel or the wait self-test).  *kernel_name
 * gets its (mangled) name, owned by the CUDA runtime; *grid the blocks it was
 * launched with; *blocks_per_sm the resident blocks per SM the grid was
 * sized from (one wave = SMs x blocks_per_sm: the kernel's occupancy, or the
 * smaller count of its launch shape); *block the threads per block; *w32 1 if
 * its vector body moved the fp32 arrays in 32-byte accesses, 0 if in 16-byte
 * ones.  Any pointer may be NULL.  EINVAL if this thread has launched nothing
 * yet; ECUDA if the runtime cannot name the kernel. */
int zero1_debug_last_launch(const char **kernel_name, int32_t *grid, int32_t *blocks_per_sm, int32_t *block,
                            int32_t *w32);

#ifdef __cplusplus
}
#endif

#endif /* ZERO1_H */
