// zero1_checks.h - host-side argument checks and error reporting shared by
// the library's CUDA sources (library-internal): alignment and overlap of the
// caller's buffers, where a pointer lives, the gradient pointer array, launch
// errors, and the compile-time check of the launch-shape tables.  Nothing
// here changes what a kernel does or how it is launched.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "zero1.h"
#include "zero1_device.cuh"
#include "zero1_internal.h"

namespace {

// A launch shape the kernels support: one or two vectors in flight per
// thread, whole warps, at most kBlock threads per block (the kernels' launch
// bounds), and a non-negative cap on the blocks per SM.
constexpr bool shape_ok(Shape s)
{
    return (s.D == 1 || s.D == 2) && s.per_sm >= 0 && s.block >= 32 && s.block <= kBlock && s.block % 32 == 0;
}

// A buffer's byte extent, for the overlap checks.
struct Extent {
    const void *p;
    int64_t bytes;
    const char *what;
};

bool overlap(const Extent &a, const Extent &b)
{
    if (a.bytes <= 0 || b.bytes <= 0 || !a.p || !b.p) return false;
    const uintptr_t a0 = (uintptr_t)a.p, a1 = a0 + (uintptr_t)a.bytes;
    const uintptr_t b0 = (uintptr_t)b.p, b1 = b0 + (uintptr_t)b.bytes;
    return a0 < b1 && b0 < a1;
}

// EINVAL unless the `nout` buffers a call writes are pairwise disjoint and
// none of the M gradient buffers (`nv` bf16 elements each, read through the
// read-only path; they may alias one another) overlaps one of them.
int check_disjoint(const Extent *out, int nout, const GradPtrs &g, int M, int64_t nv, const char *call)
{
    for (int a = 0; a < nout; ++a)
        for (int b = a + 1; b < nout; ++b)
            if (overlap(out[a], out[b]))
                return z1_fail(ZERO1_EINVAL, "%s: %s and %s overlap", call, out[a].what, out[b].what);
    for (int r = 0; r < M && nv > 0; ++r) {
        const Extent gr{g.p[r], nv * 2, "a gradient buffer"};
        for (int a = 0; a < nout; ++a)
            if (overlap(gr, out[a])) return z1_fail(ZERO1_EINVAL, "%s: grads[%d] overlaps %s", call, r, out[a].what);
    }
    return ZERO1_OK;
}

int check_natural(const void *p, int esize, const char *what)
{
    if (((uintptr_t)p & (uintptr_t)(esize - 1)) != 0)
        return z1_fail(ZERO1_EALIGN, "%s is not %d-byte aligned", what, esize);
    return ZERO1_OK;
}

// True if p is host memory the device reaches over the host link (pinned,
// or plain pageable memory on a system where the GPU can address it).
bool in_host_memory(const void *p)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of an unknown pointer
        return false;
    }
    return a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeUnregistered;
}

int launch_status(const char *what)
{
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return z1_fail(ZERO1_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    return ZERO1_OK;
}

// A failed launch_pdl: clear the runtime's last error and report it.
int pdl_fail(cudaError_t e, const char *what)
{
    cudaGetLastError();
    return z1_fail(ZERO1_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

int load_grads(const zero1_plan_t *plan, const void *const *grads, GradPtrs *g, const char *what)
{
    if (!grads) return z1_fail(ZERO1_EINVAL, "%s: grads array is NULL", what);
    for (int r = 0; r < plan->M; ++r) {
        if (!grads[r]) return z1_fail(ZERO1_EINVAL, "%s: grads[%d] is NULL", what, r);
        int rc = check_natural(grads[r], 2, "a gradient pointer");
        if (rc != ZERO1_OK) return rc;
        g->p[r] = static_cast<const uint16_t *>(grads[r]);
    }
    return ZERO1_OK;
}

}  // namespace
