// zero1_host.cpp - host-only part of libzero1: the shard plan, its per-tensor
// segments, memory accounting, hyperparameter validation and error text.
//
// Plan: "第2章 软件程序与专用硬件的结合" 2.3.4 (each of N GPUs keeps 1/N of the
// optimizer state) and "CS336 Lecture 7: Parallelism 1", ZeRO Stage 1 (GPU i
// receives and updates shard i).  Padding rounds n up to a multiple of
// M*align so that every shard has the same size s = P/M.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include <cuda_runtime.h>

#include "zero1.h"
#include "zero1_internal.h"

static thread_local char g_last_error[256] = "no error";

int z1_fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

extern "C" const char *zero1_last_error(void) { return g_last_error; }

namespace {
struct LastLaunch {
    const void *kernel;
    int grid, blocks_per_sm, block, w32;
};
thread_local LastLaunch g_last_launch = {nullptr, 0, 0, 0, 0};
}  // namespace

void z1_note_launch(const void *kernel, int grid, int blocks_per_sm, int block, int w32)
{
    g_last_launch = {kernel, grid, blocks_per_sm, block, w32};
}

extern "C" int zero1_debug_last_launch(const char **kernel_name, int32_t *grid, int32_t *blocks_per_sm,
                                       int32_t *block, int32_t *w32)
{
    if (!g_last_launch.kernel) return z1_fail(ZERO1_EINVAL, "no kernel launched on this thread yet");
    if (kernel_name) {
        const char *name = nullptr;
        const cudaError_t e = cudaFuncGetName(&name, g_last_launch.kernel);
        if (e != cudaSuccess || !name)
            return z1_fail(ZERO1_ECUDA, "cudaFuncGetName: %s", cudaGetErrorString(e));
        *kernel_name = name;
    }
    if (grid) *grid = g_last_launch.grid;
    if (blocks_per_sm) *blocks_per_sm = g_last_launch.blocks_per_sm;
    if (block) *block = g_last_launch.block;
    if (w32) *w32 = g_last_launch.w32;
    return ZERO1_OK;
}

extern "C" int zero1_abi_version(void) { return 3; }

extern "C" const char *zero1_strerror(int code)
{
    switch (code) {
    case ZERO1_OK: return "ok";
    case ZERO1_EINVAL: return "invalid argument";
    case ZERO1_EALIGN: return "misaligned device pointer";
    case ZERO1_ERANGE: return "size or replica count out of the supported range";
    case ZERO1_ECUDA: return "CUDA runtime error";
    default: return "unknown status";
    }
}

extern "C" int zero1_plan(int64_t n, int32_t M, int32_t align, const int64_t *tensor_numels, int32_t n_tensors,
                          zero1_plan_t *out)
{
    if (!out) return z1_fail(ZERO1_EINVAL, "zero1_plan: out is NULL");
    if (n < 1) return z1_fail(ZERO1_EINVAL, "zero1_plan: n = %lld < 1", (long long)n);
    if (M < 1) return z1_fail(ZERO1_EINVAL, "zero1_plan: M = %d < 1", M);
    if (align < 1) return z1_fail(ZERO1_EINVAL, "zero1_plan: align = %d < 1", align);
    if (M > ZERO1_MAX_REPLICAS)
        return z1_fail(ZERO1_ERANGE, "zero1_plan: M = %d > %d", M, ZERO1_MAX_REPLICAS);
    if (tensor_numels ? n_tensors < 1 : n_tensors != 0)
        return z1_fail(ZERO1_EINVAL, "zero1_plan: n_tensors = %d with a %s tensor list", n_tensors,
                       tensor_numels ? "non-NULL" : "NULL");
    if (tensor_numels) {
        int64_t total = 0;
        for (int32_t k = 0; k < n_tensors; ++k) {
            if (tensor_numels[k] < 0 || tensor_numels[k] > n - total)
                return z1_fail(ZERO1_EINVAL, "zero1_plan: tensor sizes do not sum to n = %lld", (long long)n);
            total += tensor_numels[k];
        }
        if (total != n)
            return z1_fail(ZERO1_EINVAL, "zero1_plan: tensor sizes sum to %lld, not n = %lld", (long long)total,
                           (long long)n);
    }
    const int64_t unit = (int64_t)M * (int64_t)align;
    const int64_t units = n / unit + (n % unit != 0);
    if (units > INT64_MAX / unit) return z1_fail(ZERO1_ERANGE, "zero1_plan: padded length overflows");
    out->n = n;
    out->padded_n = units * unit;
    out->shard = out->padded_n / M;
    out->M = M;
    out->align = align;
    out->n_tensors = n_tensors;
    return ZERO1_OK;
}

int z1_check_plan(const zero1_plan_t *p)
{
    if (!p) return z1_fail(ZERO1_EINVAL, "plan is NULL");
    zero1_plan_t q;
    int rc = zero1_plan(p->n, p->M, p->align, nullptr, 0, &q);
    if (rc != ZERO1_OK) return rc;
    if (q.padded_n != p->padded_n || q.shard != p->shard || p->n_tensors < 0)
        return z1_fail(ZERO1_EINVAL, "plan fields are inconsistent (not built by zero1_plan)");
    return ZERO1_OK;
}

int z1_range(const zero1_plan_t *p, int32_t sb, int32_t se, Z1Range *out)
{
    int rc = z1_check_plan(p);
    if (rc != ZERO1_OK) return rc;
    if (sb < 0 || se > p->M || sb >= se)
        return z1_fail(ZERO1_EINVAL, "shard range [%d, %d) not inside [0, %d)", sb, se, p->M);
    out->base = (int64_t)sb * p->shard;
    out->L = (int64_t)(se - sb) * p->shard;
    int64_t nv = p->n - out->base;
    out->nv = nv < 0 ? 0 : (nv > out->L ? out->L : nv);
    return ZERO1_OK;
}

extern "C" int zero1_plan_segments(const zero1_plan_t *plan, const int64_t *numels, int32_t shard_index,
                                   int64_t *seg_tensor, int64_t *seg_begin, int64_t *seg_len, int32_t cap,
                                   int32_t *count)
{
    int rc = z1_check_plan(plan);
    if (rc != ZERO1_OK) return rc;
    const int32_t n_tensors = plan->n_tensors;
    if (n_tensors < 1) return z1_fail(ZERO1_EINVAL, "zero1_plan_segments: the plan was built without tensors");
    if (!numels || !count || cap < 0 || (cap > 0 && (!seg_tensor || !seg_begin || !seg_len)))
        return z1_fail(ZERO1_EINVAL, "zero1_plan_segments: NULL argument");
    if (shard_index < 0 || shard_index >= plan->M)
        return z1_fail(ZERO1_EINVAL, "zero1_plan_segments: shard %d not in [0, %d)", shard_index, plan->M);
    int64_t total = 0;
    for (int32_t k = 0; k < n_tensors; ++k) {
        if (numels[k] < 0) return z1_fail(ZERO1_EINVAL, "tensor %d has negative size", k);
        total += numels[k];
    }
    if (total != plan->n)
        return z1_fail(ZERO1_EINVAL, "tensor sizes sum to %lld, plan has n = %lld", (long long)total,
                       (long long)plan->n);
    const int64_t lo = (int64_t)shard_index * plan->shard, hi = lo + plan->shard;
    int32_t c = 0;
    int64_t start = 0;
    for (int32_t k = 0; k < n_tensors && start < hi; ++k) {
        const int64_t a = start > lo ? start : lo;
        const int64_t end = start + numels[k];
        const int64_t b = end < hi ? end : hi;
        if (b > a) {
            if (c >= cap) return z1_fail(ZERO1_ERANGE, "zero1_plan_segments: more than %d pieces", cap);
            seg_tensor[c] = k;
            seg_begin[c] = a - start;
            seg_len[c] = b - a;
            ++c;
        }
        start = end;
    }
    *count = c;
    return ZERO1_OK;
}

extern "C" int zero1_plan_memory(const zero1_plan_t *plan, int64_t *naive_bytes, int64_t *zero1_bytes)
{
    int rc = z1_check_plan(plan);
    if (rc != ZERO1_OK) return rc;
    if (!naive_bytes || !zero1_bytes) return z1_fail(ZERO1_EINVAL, "zero1_plan_memory: NULL output");
    // 2 (bf16 param) + 2 (bf16 grad) + 4 (fp32 master) + 4 (m) + 4 (v)
    *naive_bytes = plan->n * (2 + 2 + 4 + 4 + 4);
    *zero1_bytes = plan->n * (2 + 2) + plan->shard * (4 + 4 + 4);
    return ZERO1_OK;
}

double z1_pow_int(double b, int64_t t)
{
    // square-and-multiply over the bits of t, least significant first
    double r = 1.0, x = b;
    for (; t > 0; t >>= 1) {
        if (t & 1) r *= x;
        x *= x;
    }
    return r;
}

int z1_adamw_constants(const zero1_adamw_t *hp, int32_t M, Z1Consts *c)
{
    if (!hp) return z1_fail(ZERO1_EINVAL, "hyperparameters are NULL");
    if (!std::isfinite(hp->lr)) return z1_fail(ZERO1_EINVAL, "lr is not finite");
    if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return z1_fail(ZERO1_EINVAL, "betas must lie in [0, 1)");
    if (!(hp->eps >= 0.0f) || !std::isfinite(hp->eps)) return z1_fail(ZERO1_EINVAL, "eps must be finite and >= 0");
    if (!std::isfinite(hp->weight_decay)) return z1_fail(ZERO1_EINVAL, "weight_decay is not finite");
    if (!(hp->loss_scale > 0.0f) || !std::isfinite(hp->loss_scale))
        return z1_fail(ZERO1_EINVAL, "loss_scale must be finite and > 0");
    if (hp->global_batch < M)
        return z1_fail(ZERO1_EINVAL, "global batch B = %lld is smaller than M = %d", (long long)hp->global_batch, M);
    if (hp->step < 1) return z1_fail(ZERO1_EINVAL, "step t = %lld < 1", (long long)hp->step);
    const double b1 = hp->beta1, b2 = hp->beta2;
    c->inv = (float)(1.0 / ((double)hp->global_batch * (double)hp->loss_scale));
    c->beta1 = hp->beta1;
    c->omb1 = (float)(1.0 - b1);
    c->beta2 = hp->beta2;
    c->omb2 = (float)(1.0 - b2);
    c->bc1 = (float)(1.0 - z1_pow_int(b1, hp->step));
    c->bc2 = (float)(1.0 - z1_pow_int(b2, hp->step));
    c->eps = hp->eps;
    c->lr = hp->lr;
    c->cdec = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
    if (!(c->bc1 > 0.0f) || !(c->bc2 > 0.0f))
        return z1_fail(ZERO1_EINVAL, "bias correction 1 - beta^t rounds to 0");
    return ZERO1_OK;
}
