// zero1_staged.cpp - the fused step over buffers in pinned host memory, staged
// through HBM by the copy engines (host code: copies, streams and events
// around the fused kernel's launches).
//
// The range of the handle's shards is cut into chunks.  For each chunk an
// inbound stream copies the host-resident inputs (the M gradient slices,
// the fp32 master/m/v) into one of three device staging slots, the caller's
// stream runs the fused step on the slot (zero1_step_bucket), and an
// outbound stream copies the host-resident outputs back (master/m/v, and
// the bf16 parameters when a host copy is wanted).  With three slots the
// inbound copy of chunk k + 1, the step on chunk k and the outbound copy of
// chunk k - 1 proceed together, so both directions of the host link are
// busy when the optimizer state lives in host memory ("五维并行实战" 4.2,
// offload_optimizer: the fp32 state kept in CPU memory; here the update
// itself still runs on the GPU, next to the state's copies).
#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>
#include <new>
#include <vector>

#include "zero1.h"
#include "zero1_internal.h"

namespace {

constexpr int kSlots = 3;
// Inbound copy streams.  Measured on GB300 (124M parameters, M = 8, same box):
// two streams were no faster for staged gradients and 3 % slower for staged
// state than one.
constexpr int kIn = 1;
constexpr int kTimes = 6;

enum class Kind { kNull, kDevice, kPinnedHost, kOther };

Kind kind_of(const void *p)
{
    if (!p) return Kind::kNull;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return Kind::kOther;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return Kind::kDevice;
    if (a.type == cudaMemoryTypeHost) return Kind::kPinnedHost;
    return Kind::kOther;
}

// A buffer that must be pinned host memory (staged) or device memory (used
// in place), naturally aligned for its element size.
int check_buffer(const void *p, bool staged, int elem, const char *what)
{
    const Kind k = kind_of(p);
    if (k == Kind::kNull) return z1_fail(ZERO1_EINVAL, "staged step: %s is NULL", what);
    if (staged && k != Kind::kPinnedHost)
        return z1_fail(ZERO1_EINVAL, "staged step: %s must be pinned host memory (it is staged)", what);
    if (!staged && k != Kind::kDevice)
        return z1_fail(ZERO1_EINVAL, "staged step: %s must be device memory (it is not staged)", what);
    if ((uintptr_t)p % (uintptr_t)elem != 0)
        return z1_fail(ZERO1_EALIGN, "staged step: %s is not %d-byte aligned", what, elem);
    return ZERO1_OK;
}

// EINVAL if buffers the step writes overlap one another or the gradients
// (the gradients may alias one another).
int check_staged_disjoint(const zero1_staged_t *h, const void *const *grads, const float *master, const float *m,
                          const float *v, const void *params, const void *params_host);

int cuda_fail(cudaError_t e, const char *what)
{
    return z1_fail(ZERO1_ECUDA, "staged step: %s: %s", what, cudaGetErrorString(e));
}

}  // namespace

struct zero1_staged {
    zero1_plan_t plan;
    int32_t shard_begin, shard_end, what, device;
    int64_t base, L, nv, chunk;
    int64_t gsize, ssize;        // staging elements per slot and buffer
    uint16_t *gstage;            // kSlots x M x gsize bf16, or NULL
    float *sstage;               // kSlots x 3 x ssize fp32, or NULL
    cudaStream_t in[kIn], out;
    cudaEvent_t copied_in[kSlots][kIn], computed[kSlots], copied_out[kSlots];
    cudaEvent_t entry, done, last;
    bool last_recorded;
    std::vector<int64_t> cuts;   // chunk boundaries, 0 = cuts[0] < ... < cuts.back() = L
    // ZERO1_STAGE_TIMELINE: timing events of the last step, kTimes per chunk
    // (inbound copies start/end, kernel start/end, outbound copies start/end)
    // after t0, recorded on the caller's stream at the step's start
    bool timeline, timed_step, timed_out;
    cudaEvent_t t0;
    std::vector<cudaEvent_t> tev;
};

namespace {

bool spans_overlap(const void *a, int64_t abytes, const void *b, int64_t bbytes)
{
    if (!a || !b || abytes <= 0 || bbytes <= 0) return false;
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

int check_staged_disjoint(const zero1_staged_t *h, const void *const *grads, const float *master, const float *m,
                          const float *v, const void *params, const void *params_host)
{
    struct Span {
        const void *p;
        int64_t bytes;
        const char *what;
    };
    const Span out[5] = {{master, h->L * 4, "master"},
                         {m, h->L * 4, "m"},
                         {v, h->L * 4, "v"},
                         {params, h->nv * 2, "params"},
                         {params_host, h->nv * 2, "params_host"}};
    for (int a = 0; a < 5; ++a)
        for (int b = a + 1; b < 5; ++b)
            if (spans_overlap(out[a].p, out[a].bytes, out[b].p, out[b].bytes))
                return z1_fail(ZERO1_EINVAL, "staged step: %s and %s overlap", out[a].what, out[b].what);
    for (int r = 0; r < h->plan.M && h->nv > 0 && grads; ++r)
        for (int a = 0; a < 5; ++a)
            if (spans_overlap(grads[r], h->nv * 2, out[a].p, out[a].bytes))
                return z1_fail(ZERO1_EINVAL, "staged step: grads[%d] overlaps %s", r, out[a].what);
    return ZERO1_OK;
}

int64_t round8(int64_t x) { return (x + 7) / 8 * 8; }

// Chunk boundaries over [0, L): chunks of c elements (c a multiple of 8),
// the last one shorter.  Every boundary but L is a multiple of 8, so each
// chunk keeps the 16-byte phase of the whole range.  (Smaller chunks at both
// ends, to shorten the step's pipeline fill and drain, measured no faster.)
std::vector<int64_t> chunk_cuts(int64_t L, int64_t c)
{
    std::vector<int64_t> cuts{0};
    for (int64_t e = c; e < L; e += c) cuts.push_back(e);
    cuts.push_back(L);
    return cuts;
}

void release(zero1_staged_t *h)
{
    if (!h) return;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != h->device) cudaSetDevice(h->device);
    if (h->gstage) cudaFree(h->gstage);
    if (h->sstage) cudaFree(h->sstage);
    for (cudaEvent_t *e : {&h->entry, &h->done, &h->last})
        if (*e) cudaEventDestroy(*e);
    for (int s = 0; s < kSlots; ++s) {
        for (cudaEvent_t e : h->copied_in[s])
            if (e) cudaEventDestroy(e);
        for (cudaEvent_t e : {h->computed[s], h->copied_out[s]})
            if (e) cudaEventDestroy(e);
    }
    if (h->t0) cudaEventDestroy(h->t0);
    for (cudaEvent_t e : h->tev)
        if (e) cudaEventDestroy(e);
    for (cudaStream_t q : h->in)
        if (q) cudaStreamDestroy(q);
    if (h->out) cudaStreamDestroy(h->out);
    if (cur >= 0 && cur != h->device) cudaSetDevice(cur);
    delete h;
}

}  // namespace

extern "C" int zero1_staged_create(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                   int32_t what, int64_t chunk_elems, zero1_staged_t **out)
{
    Z1Trace trace("zero1_staged_create");
    if (!out) return z1_fail(ZERO1_EINVAL, "staged create: out is NULL");
    *out = nullptr;
    int rc;
    Z1Range r;
    if ((rc = z1_range(plan, shard_begin, shard_end, &r)) != ZERO1_OK) return rc;
    const int32_t staging = ZERO1_STAGE_GRADS | ZERO1_STAGE_STATE | ZERO1_STAGE_PARAMS;
    if ((what & staging) == 0 || (what & ~(staging | ZERO1_STAGE_TIMELINE)) != 0)
        return z1_fail(ZERO1_EINVAL, "staged create: what = %d is not a non-empty set of ZERO1_STAGE_* bits", what);
    if (chunk_elems < 1) return z1_fail(ZERO1_EINVAL, "staged create: chunk_elems = %lld", (long long)chunk_elems);
    zero1_staged_t *h = new (std::nothrow) zero1_staged_t{};
    if (!h) return z1_fail(ZERO1_ECUDA, "staged create: out of host memory");
    h->plan = *plan;
    h->shard_begin = shard_begin;
    h->shard_end = shard_end;
    h->what = what & staging;
    h->timeline = (what & ZERO1_STAGE_TIMELINE) != 0;
    h->base = r.base;
    h->L = r.L;
    h->nv = r.nv;
    // chunks start at multiples of 8 elements, so every chunk keeps the
    // 16-byte phase of the whole range
    h->chunk = (chunk_elems + 7) / 8 * 8;
    const int64_t span = h->chunk < h->L ? h->chunk : h->L;
    h->ssize = round8(span);
    h->gsize = h->ssize;
    try {
        h->cuts = chunk_cuts(h->L, h->chunk);
    } catch (...) {
        delete h;
        return z1_fail(ZERO1_ECUDA, "staged create: out of host memory");
    }
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) {
        release(h);
        return cuda_fail(e, "cudaGetDevice");
    }
    if ((what & ZERO1_STAGE_GRADS) && h->nv > 0)
        e = cudaMalloc(&h->gstage, sizeof(uint16_t) * (size_t)(kSlots * plan->M) * (size_t)h->gsize);
    if (e == cudaSuccess && (what & ZERO1_STAGE_STATE))
        e = cudaMalloc(&h->sstage, sizeof(float) * (size_t)(kSlots * 3) * (size_t)h->ssize);
    for (cudaStream_t &q : h->in)
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&q, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h->out, cudaStreamNonBlocking);
    for (cudaEvent_t *ev : {&h->entry, &h->done, &h->last})
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    for (int s = 0; s < kSlots && e == cudaSuccess; ++s) {
        for (cudaEvent_t &ev : h->copied_in[s])
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        for (cudaEvent_t *ev : {&h->computed[s], &h->copied_out[s]})
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    }
    if (e == cudaSuccess && h->timeline) {
        try {
            h->tev.assign((h->cuts.size() - 1) * kTimes, nullptr);
        } catch (...) {
            release(h);
            return z1_fail(ZERO1_ECUDA, "staged create: out of host memory");
        }
        e = cudaEventCreate(&h->t0);
        for (cudaEvent_t &ev : h->tev)
            if (e == cudaSuccess) e = cudaEventCreate(&ev);
    }
    if (e != cudaSuccess) {
        release(h);
        return cuda_fail(e, "allocating staging memory, streams or events");
    }
    *out = h;
    return ZERO1_OK;
}

extern "C" int zero1_staged_destroy(zero1_staged_t *h)
{
    if (!h) return ZERO1_OK;
    // the handle's work may still be queued: let it finish before freeing
    for (cudaStream_t q : h->in) cudaStreamSynchronize(q);
    cudaStreamSynchronize(h->out);
    if (h->last_recorded) cudaEventSynchronize(h->last);
    release(h);
    return ZERO1_OK;
}

namespace {

// One staged step.  With a scaler (dynamic loss scaling) an overflow pass
// over the attempt's gradients sets scaler->overflow first, every chunk runs
// the in-place kernel that takes S and t from the scaler and returns at once
// on overflow, and the scaler advances after the last chunk; without one,
// every chunk runs zero1_step_bucket with the host's constants.
int staged_run(zero1_staged_t *h, const void *const *grads, float *master, float *m, float *v, void *params,
               void *params_host, const zero1_adamw_t *hp, uint32_t *overflow_flag, zero1_scaler_t *scaler,
               const zero1_loss_scale_policy_t *policy, zero1_stream_t stream)
{
    if (!h) return z1_fail(ZERO1_EINVAL, "staged step: handle is NULL");
    int rc;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != h->device)
        return z1_fail(ZERO1_EINVAL, "staged step: current device %d, the handle belongs to device %d", dev,
                       h->device);
    if (scaler) {
        if ((rc = z1_check_scaler_and_policy(scaler, policy, hp, h->plan.M)) != ZERO1_OK) return rc;
        if ((rc = check_buffer(scaler, false, 8, "scaler")) != ZERO1_OK) return rc;
    } else {
        Z1Consts c;
        if ((rc = z1_adamw_constants(hp, h->plan.M, &c)) != ZERO1_OK) return rc;
    }
    const bool sg = h->what & ZERO1_STAGE_GRADS, ss = h->what & ZERO1_STAGE_STATE,
               sp = h->what & ZERO1_STAGE_PARAMS;
    const int M = h->plan.M;
    if (h->nv > 0) {
        if (!grads) return z1_fail(ZERO1_EINVAL, "staged step: grads is NULL");
        for (int k = 0; k < M; ++k)
            if ((rc = check_buffer(grads[k], sg, 2, "a gradient buffer")) != ZERO1_OK) return rc;
        if ((rc = check_buffer(params, false, 2, "params")) != ZERO1_OK) return rc;
        if (sp && (rc = check_buffer(params_host, true, 2, "params_host")) != ZERO1_OK) return rc;
    }
    if (!sp && params_host)
        return z1_fail(ZERO1_EINVAL, "staged step: params_host given but ZERO1_STAGE_PARAMS not set");
    if ((rc = check_buffer(master, ss, 4, "master")) || (rc = check_buffer(m, ss, 4, "m")) ||
        (rc = check_buffer(v, ss, 4, "v")))
        return rc;
    if (overflow_flag && (rc = check_buffer(overflow_flag, false, 4, "overflow_flag")) != ZERO1_OK) return rc;
    if ((rc = check_staged_disjoint(h, grads, master, m, v, params, sp ? params_host : nullptr)) != ZERO1_OK)
        return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if ((e = cudaStreamIsCapturing(st, &cap)) != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    if (cap != cudaStreamCaptureStatusNone)
        return z1_fail(ZERO1_EINVAL, "staged step: the stream is capturing a graph; this call cannot be captured");

    const bool has_out = ss || sp;
    float *state[3] = {master, m, v};
    // inputs are ready once the caller's earlier work is; slots are free once
    // this handle's previous call (on whichever stream) is done with them
#define Z1_CUDA(call)                                    \
    do {                                                 \
        if ((e = (call)) != cudaSuccess) return cuda_fail(e, #call); \
    } while (0)
    // a call that fails part way leaves no timeline to read
    h->timed_step = false;
    Z1_CUDA(cudaEventRecord(h->entry, st));
    if (h->timeline) Z1_CUDA(cudaEventRecord(h->t0, st));
    cudaEvent_t *tk = nullptr;  // this chunk's timing events, or NULL
    // and once this handle's outbound copies are done, including those of a
    // call that failed part way (it did not reach its own join)
    Z1_CUDA(cudaEventRecord(h->done, h->out));
    for (cudaStream_t q : h->in) {
        Z1_CUDA(cudaStreamWaitEvent(q, h->entry, 0));
        Z1_CUDA(cudaStreamWaitEvent(q, h->done, 0));
        if (h->last_recorded) Z1_CUDA(cudaStreamWaitEvent(q, h->last, 0));
    }
    // the attempt's flag is final before any chunk's kernel reads it
    if (scaler && h->nv > 0 &&
        (rc = zero1_overflow_check(&h->plan, h->shard_begin, h->shard_end, grads, &scaler->overflow, stream)) !=
            ZERO1_OK)
        return rc;
    for (size_t k = 0; k + 1 < h->cuts.size(); ++k) {
        const int64_t e0 = h->cuts[k], e1 = h->cuts[k + 1];
        const int64_t len = e1 - e0;
        const int64_t real = h->nv > e0 ? (h->nv < e1 ? h->nv : e1) - e0 : 0;
        const int slot = (int)(k % kSlots);
        if (k >= (size_t)kSlots)
            for (cudaStream_t q : h->in)
                Z1_CUDA(cudaStreamWaitEvent(q, has_out ? h->copied_out[slot] : h->computed[slot], 0));
        tk = h->timeline ? &h->tev[k * kTimes] : nullptr;
        if (tk) Z1_CUDA(cudaEventRecord(tk[0], h->in[0]));
        int next = 0;  // the inbound copies take the inbound streams in turn
        const void *gp[ZERO1_MAX_REPLICAS] = {};
        for (int r = 0; r < M && real > 0; ++r) {
            if (sg) {
                uint16_t *dst = h->gstage + ((int64_t)slot * M + r) * h->gsize;
                Z1_CUDA(cudaMemcpyAsync(dst, static_cast<const uint16_t *>(grads[r]) + e0,
                                        sizeof(uint16_t) * real, cudaMemcpyHostToDevice, h->in[next]));
                next = (next + 1) % kIn;
                gp[r] = dst;
            } else {
                gp[r] = static_cast<const uint16_t *>(grads[r]) + e0;
            }
        }
        float *sp3[3];
        for (int a = 0; a < 3; ++a) {
            if (ss) {
                sp3[a] = h->sstage + ((int64_t)slot * 3 + a) * h->ssize;
                Z1_CUDA(cudaMemcpyAsync(sp3[a], state[a] + e0, sizeof(float) * len, cudaMemcpyHostToDevice,
                                        h->in[next]));
                next = (next + 1) % kIn;
            } else {
                sp3[a] = state[a] + e0;
            }
        }
        if (tk) Z1_CUDA(cudaEventRecord(tk[1], h->in[0]));
        for (int q = 0; q < kIn; ++q) {
            Z1_CUDA(cudaEventRecord(h->copied_in[slot][q], h->in[q]));
            Z1_CUDA(cudaStreamWaitEvent(st, h->copied_in[slot][q], 0));
        }
        if (tk) Z1_CUDA(cudaEventRecord(tk[2], st));
        void *pp = real > 0 ? static_cast<uint16_t *>(params) + e0 : nullptr;
        rc = scaler ? z1_scaled_range(&h->plan, h->base + e0, h->base + e1, real > 0 ? gp : nullptr, sp3[0], sp3[1],
                                      sp3[2], pp, hp, scaler, stream)
                    : zero1_step_bucket(&h->plan, h->base + e0, h->base + e1, real > 0 ? gp : nullptr, sp3[0],
                                        sp3[1], sp3[2], pp, hp, overflow_flag, stream);
        if (rc != ZERO1_OK) return rc;
        Z1_CUDA(cudaEventRecord(h->computed[slot], st));
        if (tk) Z1_CUDA(cudaEventRecord(tk[3], st));
        if (has_out) {
            Z1_CUDA(cudaStreamWaitEvent(h->out, h->computed[slot], 0));
            if (tk) Z1_CUDA(cudaEventRecord(tk[4], h->out));
            for (int a = 0; a < 3 && ss; ++a)
                Z1_CUDA(cudaMemcpyAsync(state[a] + e0, sp3[a], sizeof(float) * len, cudaMemcpyDeviceToHost,
                                        h->out));
            if (sp && real > 0)
                Z1_CUDA(cudaMemcpyAsync(static_cast<uint16_t *>(params_host) + e0,
                                        static_cast<const uint16_t *>(params) + e0, sizeof(uint16_t) * real,
                                        cudaMemcpyDeviceToHost, h->out));
            if (tk) Z1_CUDA(cudaEventRecord(tk[5], h->out));
            Z1_CUDA(cudaEventRecord(h->copied_out[slot], h->out));
        }
    }
    if (has_out) {
        // the copies back are part of the step for later work on the stream
        Z1_CUDA(cudaEventRecord(h->done, h->out));
        Z1_CUDA(cudaStreamWaitEvent(st, h->done, 0));
    }
    if (scaler && (rc = z1_scaler_advance(scaler, policy, hp, M, stream)) != ZERO1_OK) return rc;
    Z1_CUDA(cudaEventRecord(h->last, st));
#undef Z1_CUDA
    h->last_recorded = true;
    h->timed_step = h->timeline;
    h->timed_out = has_out;
    return ZERO1_OK;
}

}  // namespace

extern "C" int zero1_staged_step(zero1_staged_t *h, const void *const *grads, float *master, float *m,
                                 float *v, void *params, void *params_host, const zero1_adamw_t *hp,
                                 uint32_t *overflow_flag, zero1_stream_t stream)
{
    Z1Trace trace("zero1_staged_step");
    return staged_run(h, grads, master, m, v, params, params_host, hp, overflow_flag, nullptr, nullptr, stream);
}

extern "C" int zero1_staged_step_dynamic(zero1_staged_t *h, const void *const *grads, float *master, float *m,
                                         float *v, void *params, void *params_host, const zero1_adamw_t *hp,
                                         zero1_scaler_t *scaler, const zero1_loss_scale_policy_t *policy,
                                         zero1_stream_t stream)
{
    Z1Trace trace("zero1_staged_step_dynamic");
    if (!scaler) return z1_fail(ZERO1_EINVAL, "staged dynamic step: scaler is NULL");
    return staged_run(h, grads, master, m, v, params, params_host, hp, nullptr, scaler, policy, stream);
}

extern "C" int zero1_staged_chunks(const zero1_staged_t *h, int64_t *cuts, int32_t cap, int32_t *count)
{
    if (!h || !count) return z1_fail(ZERO1_EINVAL, "staged chunks: handle or count is NULL");
    const int32_t n = (int32_t)h->cuts.size();
    *count = n;
    if (cuts) {
        if (cap < n) return z1_fail(ZERO1_ERANGE, "staged chunks: %d boundaries, room for %d", n, cap);
        for (int32_t i = 0; i < n; ++i) cuts[i] = h->cuts[i];
    }
    return ZERO1_OK;
}

extern "C" int zero1_staged_timeline(zero1_staged_t *h, float *ms, int32_t cap, int32_t *count)
{
    if (!h || !count) return z1_fail(ZERO1_EINVAL, "staged timeline: handle or count is NULL");
    if (!h->timeline) return z1_fail(ZERO1_EINVAL, "staged timeline: the handle was created without ZERO1_STAGE_TIMELINE");
    if (!h->timed_step) return z1_fail(ZERO1_EINVAL, "staged timeline: no step has been enqueued on the handle");
    const int32_t chunks = (int32_t)(h->cuts.size() - 1);
    *count = chunks;
    if (!ms) return ZERO1_OK;
    if (cap < chunks * kTimes)
        return z1_fail(ZERO1_ERANGE, "staged timeline: %d values needed, room for %d", chunks * kTimes, cap);
    cudaError_t e = cudaEventSynchronize(h->last);
    if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
    for (int32_t k = 0; k < chunks; ++k)
        for (int q = 0; q < kTimes; ++q) {
            float t = -1.0f;
            if (q < 4 || h->timed_out) {
                e = cudaEventElapsedTime(&t, h->t0, h->tev[(size_t)k * kTimes + q]);
                if (e != cudaSuccess) return cuda_fail(e, "cudaEventElapsedTime");
            }
            ms[(size_t)k * kTimes + q] = t;
        }
    return ZERO1_OK;
}
