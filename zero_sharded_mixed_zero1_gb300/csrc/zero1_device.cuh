// zero1_device.cuh - device and launch helpers shared by the library's CUDA
// sources (library-internal).
//
// Everything here sits in an anonymous namespace on purpose: kernels that two
// sources instantiate (the reduce-scatter) must have internal linkage, or the
// merged host stubs of one source would launch the other source's module.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <type_traits>

#include "zero1.h"
#include "zero1_internal.h"

namespace {

constexpr int kVec = 8;      // elements per thread per iteration (16 B of bf16)
constexpr int kBlock = 256;  // threads per block (at most; a launch shape may use fewer)

// This thread's index in the grid and the grid's thread count, whatever the
// block size of the launch.
__device__ __forceinline__ int64_t grid_tid() { return (int64_t)blockIdx.x * blockDim.x + threadIdx.x; }
__device__ __forceinline__ int64_t grid_threads() { return (int64_t)gridDim.x * blockDim.x; }

struct GradPtrs {
    const uint16_t *p[ZERO1_MAX_REPLICAS];
};
struct OutPtrs {
    void *p[ZERO1_MAX_REPLICAS];
};

// How a range of L elements is walked: [0, head) per element, then nvec
// aligned 8-element vectors [head, head + 8*nvec) that are all real
// parameters, then [head + 8*nvec, L) per element (real below nv, padding
// above).  w32 != 0 when every fp32 array is also 32-byte aligned at the
// vectors, so that a vector's 8 floats move in one 32-byte access.
struct Walk {
    int64_t L, nv, head, nvec;
    int32_t w32;
};

// ---------------------------------------------------------------- helpers --

// Programmatic dependent launch.  A kernel launched by launch_pdl may be
// scheduled while the kernel before it on the stream is still finishing (its
// blocks take SMs as the earlier grid's blocks exit), and calls
// wait_prior_grid() before it touches global memory: that returns once the
// earlier grid has completed and its writes are visible.  Used for the
// streaming kernels that follow another kernel: the second and third kernels
// of the multi-kernel entry points, and the fused and ping-pong kernels, which
// run back to back over buckets and chunks.  Measured on GB300: about 5 us per
// step of two or three launches (the dynamic step at M = 8: 0.950 -> 0.956 of
// the copy peak; ping-pong 0.987 -> 0.994), and 0.8 % on the Llama layers in
// 18 buckets; a single launch per step does not change.  Launched without the
// attribute, the wait returns at once.
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <class K, class... Args>
cudaError_t launch_pdl(K kernel, int grid, int block, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}


__device__ __forceinline__ uint4 ld_stream_u4(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const uint16_t *p)
{
    uint16_t r;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// Gradient loads.  NC: through the read-only (non-coherent) path, for
// kernels that write nothing overlapping the gradients; otherwise ordinary
// (coherent) global loads, for an in-place kernel whose outputs alias them.
template <bool NC>
__device__ __forceinline__ uint4 ld_grad_u4(const void *p)
{
    if constexpr (NC) {
        return ld_stream_u4(p);
    } else {
        uint4 r;
        asm("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
            : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
            : "l"(p));
        return r;
    }
}

template <bool NC>
__device__ __forceinline__ uint16_t ld_grad_u16(const uint16_t *p)
{
    if constexpr (NC) {
        return ld_stream_u16(p);
    } else {
        uint16_t r;
        asm("ld.global.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
        return r;
    }
}

// bf16 -> fp32 is exact: the bf16 code is the upper half of the binary32.
__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }
__device__ __forceinline__ float bf_one(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }

__device__ __forceinline__ void unpack8(const uint4 q, float s[kVec])
{
    s[0] = bf_lo(q.x); s[1] = bf_hi(q.x); s[2] = bf_lo(q.y); s[3] = bf_hi(q.y);
    s[4] = bf_lo(q.z); s[5] = bf_hi(q.z); s[6] = bf_lo(q.w); s[7] = bf_hi(q.w);
}

__device__ __forceinline__ void add8(const uint4 q, float s[kVec])
{
    s[0] = __fadd_rn(s[0], bf_lo(q.x)); s[1] = __fadd_rn(s[1], bf_hi(q.x));
    s[2] = __fadd_rn(s[2], bf_lo(q.y)); s[3] = __fadd_rn(s[3], bf_hi(q.y));
    s[4] = __fadd_rn(s[4], bf_lo(q.z)); s[5] = __fadd_rn(s[5], bf_hi(q.z));
    s[6] = __fadd_rn(s[6], bf_lo(q.w)); s[7] = __fadd_rn(s[7], bf_hi(q.w));
}

// fp32 -> bf16, round to nearest even (cvt.rn.bf16x2.f32).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint16_t to_bf16(float x)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Rank-order fp32 sum of 8 consecutive elements starting at j (16-byte
// aligned in every replica).  MT > 0: M == MT known at compile time, all M
// loads issued before the first add.  MT == 0: any M >= 8, in groups of 8.
template <int MT, bool NC = true>
__device__ __forceinline__ void sum8(const GradPtrs &g, int M, int64_t j, float s[kVec])
{
    if constexpr (MT > 0) {
        uint4 q[MT];
#pragma unroll
        for (int r = 0; r < MT; ++r) q[r] = ld_grad_u4<NC>(g.p[r] + j);
        unpack8(q[0], s);
#pragma unroll
        for (int r = 1; r < MT; ++r) add8(q[r], s);
    } else {
        uint4 q[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) q[r] = ld_grad_u4<NC>(g.p[r] + j);
        unpack8(q[0], s);
#pragma unroll
        for (int r = 1; r < 8; ++r) add8(q[r], s);
        for (int r0 = 8; r0 < M; r0 += 8) {
            const int cnt = M - r0 < 8 ? M - r0 : 8;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < cnt) q[k] = ld_grad_u4<NC>(g.p[r0 + k] + j);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < cnt) add8(q[k], s);
        }
    }
}

template <bool NC = true>
__device__ __forceinline__ float sum1(const GradPtrs &g, int M, int64_t j)
{
    float s = bf_one(ld_grad_u16<NC>(g.p[0] + j));
    for (int r = 1; r < M; ++r) s = __fadd_rn(s, bf_one(ld_grad_u16<NC>(g.p[r] + j)));
    return s;
}

// One AdamW update in fp32, one rounding per operation
// ("五维并行实战" 4.2 names the optimizer and its hyperparameters):
//   m' = beta1*m + (1-beta1)*g ; v' = beta2*v + (1-beta2)*(g*g)
//   u = (m'/bc1) / (sqrt(v'/bc2) + eps) ; w' = w*(1-lr*wd) - lr*u
__device__ __forceinline__ void adamw1(float g, const Z1Consts &c, float &w, float &m, float &v)
{
    const float m1 = __fadd_rn(__fmul_rn(c.beta1, m), __fmul_rn(c.omb1, g));
    const float v1 = __fadd_rn(__fmul_rn(c.beta2, v), __fmul_rn(c.omb2, __fmul_rn(g, g)));
    const float mh = __fdiv_rn(m1, c.bc1);
    const float vh = __fdiv_rn(v1, c.bc2);
    const float u = __fdiv_rn(mh, __fadd_rn(__fsqrt_rn(vh), c.eps));
    w = __fsub_rn(__fmul_rn(w, c.cdec), __fmul_rn(c.lr, u));
    m = m1;
    v = v1;
}

__device__ __forceinline__ bool finite(float x) { return isfinite(x); }

// Set *flag |= 1 if any thread of the warp saw a non-finite sum: one vote and
// at most one atomic per warp.  Called by all threads of every warp.
__device__ __forceinline__ void warp_flag(uint32_t *flag, bool bad)
{
    const unsigned any = __ballot_sync(0xffffffffu, bad);
    if (any && (threadIdx.x & 31) == 0) atomicOr(flag, 1u);
}

__device__ __forceinline__ int64_t scalar_index(const Walk &w, int64_t q)
{
    return q < w.head ? q : q + w.nvec * kVec;
}

// The vector body [0, nvec) with a grid stride, D vectors of loads in
// flight per thread.  D = 2: the loads of vector i + nthr are issued before
// vector i is computed.  D = 1: one vector at a time, for grids with more
// resident warps instead.  Which is faster depends on the kernel and on M
// (measured; each launch site names its shape table).
template <class Loads, int D = 2, class LoadF, class ComputeF>
__device__ __forceinline__ void pipelined(int64_t nvec, int64_t tid, int64_t nthr, LoadF &&load, ComputeF &&compute)
{
    static_assert(D == 1 || D == 2, "one or two vectors in flight");
    if constexpr (D == 1) {
        for (int64_t i = tid; i < nvec; i += nthr) {
            Loads cur;
            load(cur, i);
            compute(cur, i);
        }
    } else {
        Loads cur, nxt;
        int64_t i = tid;
        if (i < nvec) load(cur, i);
        for (; i < nvec; i += nthr) {
            const bool more = i + nthr < nvec;
            if (more) load(nxt, i + nthr);
            compute(cur, i);
            if (more) cur = nxt;
        }
    }
}

template <int MT>
struct GradLoads {
    uint4 q[MT > 0 ? MT : 1];
};

// Resident blocks per SM requested from the compiler: one for the two-deep
// M <= 8 paths (room for two vectors of loads per thread), four for the
// one-vector paths (at most 64 registers; the grid may use fewer), three for
// the grouped M > 8 paths.
#define Z1_BOUNDS(MT, D) __launch_bounds__(kBlock, (MT) == 0 ? 3 : ((D) == 1 ? 4 : 1))

// How a streaming kernel is launched over a large range: D vectors of loads
// in flight per thread (1 or 2), a grid of at most per_sm resident blocks per
// SM (0: as many as fit), blocks of `block` threads (at most kBlock).
struct Shape {
    int D, per_sm;
    int block = kBlock;
};

// Launch shape of the in-place fused update for M = MT on a large range
// (k_fused_step and k_fused_step_scaled, one vector of loads per thread;
// MT = 0: M > 8, replicas in groups of 8, where the shape is not used).
// Measured on GB300 (fused step, 124M elements, one box, fraction of the
// measured copy bandwidth), by warps per SM: 20 (five blocks of 128) for
// M = 1 and 6..8: 0.984 and 1.017 1.027 1.029; 18 (three blocks of 192) for
// M = 2, 3: 0.995 1.001, where 20 gave 0.977 0.973 and 16 0.978 0.993; 16
// (two blocks of 256) for M = 4, 5: 1.015 1.020, where 18 gave 0.991 0.971
// and 20 0.955 0.939.  12 warps gave 0.79-0.93 and 24 warps 0.85-0.97 for
// every M.  The two-deep pipeline this replaced (two vectors in flight per
// thread, 8 warps per SM) reached 0.995 1.007 1.019 at M = 6..8 and
// 0.93-0.98 at M <= 5.
constexpr Shape fused_shape(int MT)
{
    switch (MT) {
    case 2: case 3: return Shape{1, 3, 192};
    case 4: case 5: return Shape{1, 2};
    case 0: return Shape{2, 0};
    default: return Shape{1, 5, 128};
    }
}

// fp32 state loads that do not allocate in L1 (each line is read once) and
// streaming stores (.cs: the written lines are not read again by this kernel).
__device__ __forceinline__ float4 ld_state(const float *p)
{
    float4 r;
    asm("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ void st_stream(float *p, float a, float b, float c, float d)
{
    __stcs(reinterpret_cast<float4 *>(p), make_float4(a, b, c, d));
}

// The 8 fp32 values of one vector.  With w32 (the walk found every fp32
// array 32-byte aligned) they move in one 256-bit access per thread, so a
// warp's access covers 1 KiB of consecutive bytes and uses every 32-byte
// sector it touches in full; otherwise in two 128-bit accesses, where each
// warp instruction touches 32 sectors and uses half of each.  w32 is the
// same for every thread of the grid (a kernel argument), so the branch never
// diverges.
struct F8 {
    float4 lo, hi;
};

#define Z1_LD8(op, p, r)                                                                              \
    asm(op " {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"                                                  \
        : "=f"((r).lo.x), "=f"((r).lo.y), "=f"((r).lo.z), "=f"((r).lo.w), "=f"((r).hi.x), "=f"((r).hi.y), \
          "=f"((r).hi.z), "=f"((r).hi.w)                                                               \
        : "l"(p))

// L1::no_allocate, as ld_state.
__device__ __forceinline__ F8 ld_state8(const float *p, bool w32)
{
    F8 r;
    if (w32) {
        Z1_LD8("ld.global.L1::no_allocate.v8.f32", p, r);
    } else {
        r.lo = ld_state(p);
        r.hi = ld_state(p + 4);
    }
    return r;
}

// Evict-first (.cs): a stream read once.
__device__ __forceinline__ F8 ld_cs8(const float *p, bool w32)
{
    F8 r;
    if (w32) {
        Z1_LD8("ld.global.cs.v8.f32", p, r);
    } else {
        r.lo = __ldcs(reinterpret_cast<const float4 *>(p));
        r.hi = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
    }
    return r;
}

// The default cache policy.
__device__ __forceinline__ F8 ld_plain8(const float *p, bool w32)
{
    F8 r;
    if (w32) {
        Z1_LD8("ld.global.v8.f32", p, r);
    } else {
        r.lo = reinterpret_cast<const float4 *>(p)[0];
        r.hi = reinterpret_cast<const float4 *>(p)[1];
    }
    return r;
}

// Which kernels store fp32 in 32-byte accesses (each passes w32, or false,
// as st_stream8's flag).  Measured on GB300 with CUDA events, every other
// choice equal: 32-byte loads never lost, but 32-byte stores pay only where
// the writes go to a separate buffer (ping-pong copies, reduce-scatter and
// all-reduce outputs) or make up about half of an in-place update's traffic
// (the dynamic step's update from sums, AdamW); the in-place fused step (and
// k_fused_step_scaled) stores in 16-byte accesses: with 32-byte ones it ran
// 1-9 % slower from M = 3 (7 % at M = 64) and within 0.4 % at M = 1, 2.
constexpr bool kWideStoresInPlace = false;

// Streaming (.cs) store of 8 floats: one 32-byte access if w32, else two
// 16-byte ones.
__device__ __forceinline__ void st_stream8(float *p, const float x[kVec], bool w32)
{
    if (w32) {
        asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     :
                     : "l"(p), "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
                       "f"(x[7])
                     : "memory");
    } else {
        st_stream(p, x[0], x[1], x[2], x[3]);
        st_stream(p + 4, x[4], x[5], x[6], x[7]);
    }
}

__device__ __forceinline__ void unpack_f8(const F8 &x, float a[kVec])
{
    a[0] = x.lo.x; a[1] = x.lo.y; a[2] = x.lo.z; a[3] = x.lo.w;
    a[4] = x.hi.x; a[5] = x.hi.y; a[6] = x.hi.z; a[7] = x.hi.w;
}

// AdamW on one 8-element vector whose replica sums are in s, then the
// streaming stores of master/m/v (32-byte accesses if ws) and the bf16
// parameters.
__device__ __forceinline__ void store_vec(const float s[kVec], const F8 &w, const F8 &m, const F8 &v, float *pw,
                                          float *pm, float *pv, uint16_t *pp, const Z1Consts &c, bool &bad,
                                          bool ws)
{
    float ww[kVec], mm[kVec], vv[kVec];
    unpack_f8(w, ww);
    unpack_f8(m, mm);
    unpack_f8(v, vv);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
        bad |= !finite(s[k]);
        adamw1(__fmul_rn(s[k], c.inv), c, ww[k], mm[k], vv[k]);
    }
    st_stream8(pw, ww, ws);
    st_stream8(pm, mm, ws);
    st_stream8(pv, vv, ws);
    __stcs(reinterpret_cast<uint4 *>(pp),
           make_uint4(pack_bf16x2(ww[0], ww[1]), pack_bf16x2(ww[2], ww[3]), pack_bf16x2(ww[4], ww[5]),
                      pack_bf16x2(ww[6], ww[7])));
}

// The loads of one 8-element vector for M <= 8: every replica's gradient
// vector, then the fp32 state.
template <int MT>
struct VecLoads {
    uint4 q[MT];
    F8 w, m, v;
    __device__ __forceinline__ void load(const GradPtrs &g, const float *master, const float *mom,
                                         const float *var, int64_t j, bool w32)
    {
#pragma unroll
        for (int r = 0; r < MT; ++r) q[r] = ld_stream_u4(g.p[r] + j);
        w = ld_state8(master + j, w32);
        m = ld_state8(mom + j, w32);
        v = ld_state8(var + j, w32);
    }
};

// Per-element remainder of the fused step: [0, head) and the tail after the
// vector body (real elements below nv, padding above).
__device__ __forceinline__ void fused_scalar_rest(const GradPtrs &g, int M, float *master, float *mom,
                                                  float *var, uint16_t *params, const Walk &w,
                                                  const Z1Consts &c, int64_t tid, int64_t nthr, bool &bad)
{
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        float s = 0.0f;
        if (j < w.nv) {
            s = sum1(g, M, j);
            bad |= !finite(s);
        }
        float ww = master[j], mm = mom[j], vv = var[j];
        adamw1(__fmul_rn(s, c.inv), c, ww, mm, vv);
        master[j] = ww;
        mom[j] = mm;
        var[j] = vv;
        if (j < w.nv) params[j] = to_bf16(ww);
    }
}

// AdamW on fp32 state given the scaled fp32 gradient.
struct StateLoads {
    F8 g, w, m, v;
};

__device__ __forceinline__ void load_state_vec(StateLoads &x, const float *gin, const float *master,
                                               const float *mom, const float *var, int64_t j, bool w32)
{
    x.g = ld_cs8(gin + j, w32);
    x.w = ld_state8(master + j, w32);
    x.m = ld_state8(mom + j, w32);
    x.v = ld_state8(var + j, w32);
}

// Reduce-scatter: out[j] = sum * scale (fp32 or bf16), +0 on padding.
template <bool BF16>
__device__ __forceinline__ void rs_store(void *out, int64_t j, float s[kVec], float scale, bool w32)
{
#pragma unroll
    for (int k = 0; k < kVec; ++k) s[k] = __fmul_rn(s[k], scale);
    if constexpr (BF16) {
        __stcs(reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + j),
               make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]),
                          pack_bf16x2(s[6], s[7])));
    } else {
        st_stream8(static_cast<float *>(out) + j, s, w32);
    }
}

template <int MT, bool BF16, int D>
__global__ void Z1_BOUNDS(MT, D)
k_reduce_scatter(const __grid_constant__ GradPtrs g, int M, const Walk w, float scale, void *out,
                 uint32_t *flag)
{
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    bool bad = false;
    if constexpr (MT > 0) {
        pipelined<GradLoads<MT>, D>(
            w.nvec, tid, nthr,
            [&](GradLoads<MT> &x, int64_t i) {
                const int64_t j = w.head + i * kVec;
#pragma unroll
                for (int r = 0; r < MT; ++r) x.q[r] = ld_stream_u4(g.p[r] + j);
            },
            [&](const GradLoads<MT> &x, int64_t i) {
                float s[kVec];
                unpack8(x.q[0], s);
#pragma unroll
                for (int r = 1; r < MT; ++r) add8(x.q[r], s);
#pragma unroll
                for (int k = 0; k < kVec; ++k) bad |= !finite(s[k]);
                rs_store<BF16>(out, w.head + i * kVec, s, scale, w.w32);
            });
    } else {
        for (int64_t i = tid; i < w.nvec; i += nthr) {
            const int64_t j = w.head + i * kVec;
            float s[kVec];
            sum8<0>(g, M, j, s);
#pragma unroll
            for (int k = 0; k < kVec; ++k) bad |= !finite(s[k]);
            rs_store<BF16>(out, j, s, scale, w.w32);
        }
    }
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        float s = 0.0f;
        if (j < w.nv) {
            s = sum1(g, M, j);
            bad |= !finite(s);
        }
        s = __fmul_rn(s, scale);
        if constexpr (BF16) static_cast<uint16_t *>(out)[j] = to_bf16(s);
        else static_cast<float *>(out)[j] = s;
    }
    if (flag) warp_flag(flag, bad);
}

// Launch shape of k_reduce_scatter for M = MT (MT = 0: M > 8, replicas in
// groups of 8, where D is not used).  Measured on GB300, fp32 output, 124M
// elements, fraction of the measured copy bandwidth: two-deep at full
// occupancy 0.937 0.949 0.972 0.979 1.000 1.010 0.990 0.995 for M = 1..8;
// one vector at three blocks of 256 per SM 0.987 1.001 1.011 1.010 for
// M = 4..7; one vector at 20 warps per SM (five blocks of 128) 0.964 and
// 1.006 for M = 2 and 8.  This table: 0.931 0.963 0.976 0.990 1.007 1.016
// 1.016 1.013.  In the dynamic step (followed by k_apply_sums) it measured
// within 0.1 % of the best of the uniform shapes for every M.
constexpr Shape rs_shape(int MT)
{
    switch (MT) {
    case 2: case 8: return Shape{1, 5, 128};
    case 4: case 5: case 6: case 7: return Shape{1, 3};
    default: return Shape{2, 0};
    }
}

// ------------------------------------------------------------ host side ----

struct ArrayRef {
    const void *p;
    int esize;
};

// Choose the per-element head h in [0, 8) at which every array is 16-byte
// aligned; if there is none, the whole range runs per element.  An h at
// which the 4-byte arrays are 32-byte aligned as well is preferred: it sets
// w32 (8 floats per 32-byte access).
Walk make_walk(int64_t L, int64_t nv, const ArrayRef *a, int count)
{
    Walk w{L, nv, 0, 0, 0};
    for (int pass = 0; pass < 2; ++pass) {
        for (int h = 0; h < kVec; ++h) {
            bool ok = true;
            for (int k = 0; k < count && ok; ++k) {
                const uintptr_t mask = (pass == 0 && a[k].esize == 4) ? 31u : 15u;
                ok = (((uintptr_t)a[k].p + (uintptr_t)h * a[k].esize) & mask) == 0;
            }
            if (ok) {
                w.head = h < nv ? h : nv;
                w.nvec = nv > h ? (nv - h) / kVec : 0;
                w.w32 = pass == 0 ? 1 : 0;
                return w;
            }
        }
    }
    return w;
}

int sm_count()
{
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 64) {
        int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

int64_t work_of(const Walk &w)
{
    const int64_t ns = w.L - w.nvec * kVec;
    return w.nvec > ns ? w.nvec : ns;
}

// Resident blocks per SM of one kernel launched with `block` threads per
// block on the current device, from the occupancy API on first use and then
// from a small table keyed by the kernel's address, the block size and the
// device (kernels of the same signature each get their own entry).
int blocks_per_sm(const void *kernel, int block)
{
    struct Entry {
        const void *kernel;
        int block, dev, per_sm;
    };
    static std::mutex mu;
    static Entry table[256];
    static int used = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (int k = 0; k < used; ++k)
            if (table[k].kernel == kernel && table[k].block == block && table[k].dev == dev) return table[k].per_sm;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, block, 0) != cudaSuccess || per_sm <= 0) {
        cudaGetLastError();
        per_sm = 1;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (used < 256) table[used++] = {kernel, block, dev, per_sm};
    return per_sm;
}

// One resident wave for a walk: SMs x this kernel's resident blocks of
// `block` threads (at most max_per_sm of them when that is positive), capped
// by the work.  The launch is noted for zero1_debug_last_launch.
template <class K>
int grid_for(K kernel, const Walk &w, int max_per_sm = 0, int block = kBlock)
{
    const void *k = reinterpret_cast<const void *>(kernel);
    int per_sm = blocks_per_sm(k, block);
    if (max_per_sm > 0 && max_per_sm < per_sm) per_sm = max_per_sm;
    const int64_t wave = (int64_t)sm_count() * per_sm;
    const int64_t work = work_of(w);
    int64_t need = (work + block - 1) / block;
    if (need < 1) need = 1;
    const int grid = (int)(need < wave ? need : (wave > 0 ? wave : 1));
    z1_note_launch(k, grid, per_sm, block, w.w32);
    return grid;
}

// Call f with std::integral_constant<int, MT>: MT = M for 1..8 (all loads of
// an 8-element vector issued at once), MT = 0 for M > 8 (groups of 8).
template <class F>
void dispatch_m(int M, F &&f)
{
    switch (M) {
    case 1: f(std::integral_constant<int, 1>{}); break;
    case 2: f(std::integral_constant<int, 2>{}); break;
    case 3: f(std::integral_constant<int, 3>{}); break;
    case 4: f(std::integral_constant<int, 4>{}); break;
    case 5: f(std::integral_constant<int, 5>{}); break;
    case 6: f(std::integral_constant<int, 6>{}); break;
    case 7: f(std::integral_constant<int, 7>{}); break;
    case 8: f(std::integral_constant<int, 8>{}); break;
    default: f(std::integral_constant<int, 0>{}); break;
    }
}

}  // namespace
