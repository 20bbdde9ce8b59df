// zero1_kernels.cu - sm_103a kernels of the ZeRO Stage-1 optimizer step and
// the C-ABI entry points that launch them.
//
// The step ("CS336 Lecture 7: Parallelism 1", ZeRO Stage 1: Reduce-Scatter of
// the gradients so GPU i holds the summed shard i, local update of shard i,
// All-Gather of the parameters; naive-DP equation for the 1/B mean; the
// 16 bytes/parameter table for the dtypes) is one streaming pass per element:
//
//   M x 2 B bf16 gradient reads  ->  fp32 rank-order sum  ->  x 1/(B*S)
//   12 B fp32 master/m/v read    ->  AdamW in registers   ->  12 B written
//                                ->  bf16 parameter, 2 B written once
//
// 2M + 26 bytes per parameter and ~60 instructions, so the kernel is bound
// by HBM bandwidth.  Each thread owns 8 consecutive elements per iteration:
// one 128-bit load per replica, two per fp32 state array, one 128-bit bf16
// store.  Gradients go through the non-coherent path without L1 allocation
// (they are read exactly once).  All loads of an iteration are issued before
// any arithmetic so each thread keeps (M*16 + 96) bytes in flight; the grid
// is one resident wave (SMs x resident blocks) walking the range with a
// grid stride.
//
// Arithmetic uses the explicit round-to-nearest intrinsics (__fadd_rn,
// __fmul_rn, __fdiv_rn, __fsqrt_rn) so no multiply-add is ever contracted and
// division and square root are IEEE: the results are reproducible bit for bit
// against any IEEE-754 binary32 evaluation of the same operation sequence.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cmath>
#include <type_traits>

#include "zero1.h"
#include "zero1_internal.h"

namespace {

constexpr int kVec = 8;      // elements per thread per iteration (16 B of bf16)
constexpr int kBlock = 256;  // threads per block

struct GradPtrs {
    const uint16_t *p[ZERO1_MAX_REPLICAS];
};
struct OutPtrs {
    void *p[ZERO1_MAX_REPLICAS];
};

// How a range of L elements is walked: [0, head) per element, then nvec
// aligned 8-element vectors [head, head + 8*nvec) that are all real
// parameters, then [head + 8*nvec, L) per element (real below nv, padding
// above).
struct Walk {
    int64_t L, nv, head, nvec;
};

// ---------------------------------------------------------------- helpers --

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
template <int MT>
__device__ __forceinline__ void sum8(const GradPtrs &g, int M, int64_t j, float s[kVec])
{
    if constexpr (MT > 0) {
        uint4 q[MT];
#pragma unroll
        for (int r = 0; r < MT; ++r) q[r] = ld_stream_u4(g.p[r] + j);
        unpack8(q[0], s);
#pragma unroll
        for (int r = 1; r < MT; ++r) add8(q[r], s);
    } else {
        uint4 q[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) q[r] = ld_stream_u4(g.p[r] + j);
        unpack8(q[0], s);
#pragma unroll
        for (int r = 1; r < 8; ++r) add8(q[r], s);
        for (int r0 = 8; r0 < M; r0 += 8) {
            const int cnt = M - r0 < 8 ? M - r0 : 8;
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < cnt) q[k] = ld_stream_u4(g.p[r0 + k] + j);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (k < cnt) add8(q[k], s);
        }
    }
}

__device__ __forceinline__ float sum1(const GradPtrs &g, int M, int64_t j)
{
    float s = bf_one(ld_stream_u16(g.p[0] + j));
    for (int r = 1; r < M; ++r) s = __fadd_rn(s, bf_one(ld_stream_u16(g.p[r] + j)));
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


// Two-deep software pipeline over the vector body [0, nvec) with a grid
// stride: the loads of vector i + nthr are issued before vector i is
// computed, so each thread keeps two vectors of loads in flight.  (Measured
// on the fused step: this beat higher occupancy with one vector in flight.)
template <class Loads, class LoadF, class ComputeF>
__device__ __forceinline__ void pipelined(int64_t nvec, int64_t tid, int64_t nthr, LoadF &&load, ComputeF &&compute)
{
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

template <int MT>
struct GradLoads {
    uint4 q[MT > 0 ? MT : 1];
};

// Resident blocks per SM requested from the compiler: one for the pipelined
// M <= 8 paths (room for two vectors of loads per thread), three for the
// grouped M > 8 paths.
#define Z1_BOUNDS(MT) __launch_bounds__(kBlock, (MT) > 0 ? 1 : 3)

// ---------------------------------------------------------------- kernels --

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

// AdamW on one 8-element vector whose replica sums are in s, then the
// streaming stores of master/m/v and the bf16 parameters.
__device__ __forceinline__ void store_vec(const float s[kVec], float4 w0, float4 w1, float4 m0, float4 m1,
                                          float4 v0, float4 v1, float *pw, float *pm, float *pv, uint16_t *pp,
                                          const Z1Consts &c, bool &bad)
{
    float ww[kVec] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
    float mm[kVec] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    float vv[kVec] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
        bad |= !finite(s[k]);
        adamw1(__fmul_rn(s[k], c.inv), c, ww[k], mm[k], vv[k]);
    }
    st_stream(pw, ww[0], ww[1], ww[2], ww[3]);
    st_stream(pw + 4, ww[4], ww[5], ww[6], ww[7]);
    st_stream(pm, mm[0], mm[1], mm[2], mm[3]);
    st_stream(pm + 4, mm[4], mm[5], mm[6], mm[7]);
    st_stream(pv, vv[0], vv[1], vv[2], vv[3]);
    st_stream(pv + 4, vv[4], vv[5], vv[6], vv[7]);
    __stcs(reinterpret_cast<uint4 *>(pp),
           make_uint4(pack_bf16x2(ww[0], ww[1]), pack_bf16x2(ww[2], ww[3]), pack_bf16x2(ww[4], ww[5]),
                      pack_bf16x2(ww[6], ww[7])));
}

// One 8-element vector of the fused step for M = MT <= 8 whose loads are in q
// and the six state registers.
template <int MT>
__device__ __forceinline__ void fused_vec(int64_t j, const uint4 *q, float4 w0, float4 w1, float4 m0, float4 m1,
                                          float4 v0, float4 v1, float *master, float *mom, float *var,
                                          uint16_t *params, const Z1Consts &c, bool &bad)
{
    float s[kVec];
    unpack8(q[0], s);
#pragma unroll
    for (int r = 1; r < MT; ++r) add8(q[r], s);
    store_vec(s, w0, w1, m0, m1, v0, v1, master + j, mom + j, var + j, params + j, c, bad);
}

// The loads of one 8-element vector for M <= 8: every replica's gradient
// vector, then the fp32 state.
template <int MT>
struct VecLoads {
    uint4 q[MT];
    float4 w0, w1, m0, m1, v0, v1;
    __device__ __forceinline__ void load(const GradPtrs &g, const float *master, const float *mom,
                                         const float *var, int64_t j)
    {
#pragma unroll
        for (int r = 0; r < MT; ++r) q[r] = ld_stream_u4(g.p[r] + j);
        w0 = ld_state(master + j);
        w1 = ld_state(master + j + 4);
        m0 = ld_state(mom + j);
        m1 = ld_state(mom + j + 4);
        v0 = ld_state(var + j);
        v1 = ld_state(var + j + 4);
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

// The fused reduce-scatter + AdamW + all-gather for M <= 8 (M = MT known at
// compile time).
//
// Shape chosen by measurement on GB300 (CUDA events through this entry point
// on the 124M-parameter M = 8 workload): each thread issues all loads of its
// next vector before computing the current one, so two vectors - 2 x
// (16M + 96) bytes - are in flight per thread; the register budget this needs
// (launch bounds of one block per SM) beat higher occupancy with one vector
// in flight.  fp32 state is read with L1::no_allocate and every store is .cs.
template <int MT>
__global__ void __launch_bounds__(kBlock, MT <= 2 ? 2 : 1)
k_fused_step(const __grid_constant__ GradPtrs g, int M, float *__restrict__ master,
             float *__restrict__ mom, float *__restrict__ var, uint16_t *__restrict__ params,
             const Walk w, const Z1Consts c, uint32_t *flag, int skip)
{
    if (skip && *reinterpret_cast<volatile uint32_t *>(flag) != 0u) return;
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    bool bad = false;
    VecLoads<MT> cur, nxt;
    int64_t i = tid;
    if (i < w.nvec) cur.load(g, master, mom, var, w.head + i * kVec);
    for (; i < w.nvec; i += nthr) {
        const int64_t j = w.head + i * kVec;
        const bool more = i + nthr < w.nvec;
        if (more) nxt.load(g, master, mom, var, j + nthr * kVec);
        fused_vec<MT>(j, cur.q, cur.w0, cur.w1, cur.m0, cur.m1, cur.v0, cur.v1, master, mom, var,
                      params, c, bad);
        if (more) cur = nxt;
    }
    fused_scalar_rest(g, M, master, mom, var, params, w, c, tid, nthr, bad);
    if (flag && !skip) warp_flag(flag, bad);
}

// The fused step for M <= 8 on small ranges (at most kWideMaxVec vectors):
// one vector per thread and iteration at up to four blocks per SM.  Few
// vectors per thread means the two-deep pipeline has nothing to overlap, and
// the chain of dependent iterations per thread, not bandwidth, sets the time;
// four times the threads shortens that chain.
constexpr int64_t kWideMaxVec = 1 << 18;  // 2M elements

template <int MT>
__global__ void __launch_bounds__(kBlock, 4)
k_fused_step_wide(const __grid_constant__ GradPtrs g, int M, float *__restrict__ master,
                  float *__restrict__ mom, float *__restrict__ var, uint16_t *__restrict__ params,
                  const Walk w, const Z1Consts c, uint32_t *flag, int skip)
{
    if (skip && *reinterpret_cast<volatile uint32_t *>(flag) != 0u) return;
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    bool bad = false;
    for (int64_t i = tid; i < w.nvec; i += nthr) {
        const int64_t j = w.head + i * kVec;
        VecLoads<MT> x;
        x.load(g, master, mom, var, j);
        fused_vec<MT>(j, x.q, x.w0, x.w1, x.m0, x.m1, x.v0, x.v1, master, mom, var, params, c, bad);
    }
    fused_scalar_rest(g, M, master, mom, var, params, w, c, tid, nthr, bad);
    if (flag && !skip) warp_flag(flag, bad);
}

// The fused step for M > 8: the state is read first with the default
// policy, then the replicas in groups of 8 into the same registers; stores
// are .cs.  Three resident blocks per SM (at most 85 registers).  Measured on
// the 64-replica shard: this shape beat deeper pipelining, fewer resident
// blocks and L1::no_allocate state loads.
__global__ void __launch_bounds__(kBlock, 3)
k_fused_step_grouped(const __grid_constant__ GradPtrs g, int M, float *__restrict__ master,
                     float *__restrict__ mom, float *__restrict__ var, uint16_t *__restrict__ params,
                     const Walk w, const Z1Consts c, uint32_t *flag, int skip)
{
    if (skip && *reinterpret_cast<volatile uint32_t *>(flag) != 0u) return;
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    bool bad = false;
    for (int64_t i = tid; i < w.nvec; i += nthr) {
        const int64_t j = w.head + i * kVec;
        const float4 *pw = reinterpret_cast<const float4 *>(master + j);
        const float4 *pm = reinterpret_cast<const float4 *>(mom + j);
        const float4 *pv = reinterpret_cast<const float4 *>(var + j);
        const float4 w0 = pw[0], w1 = pw[1], m0 = pm[0], m1 = pm[1], v0 = pv[0], v1 = pv[1];
        float s[kVec];
        uint4 q[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) q[r] = ld_stream_u4(g.p[r] + j);
        unpack8(q[0], s);
#pragma unroll
        for (int r = 1; r < 8; ++r) add8(q[r], s);
        for (int r0 = 8; r0 < M; r0 += 8) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (r0 + k < M) q[k] = ld_stream_u4(g.p[r0 + k] + j);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                if (r0 + k < M) add8(q[k], s);
        }
        store_vec(s, w0, w1, m0, m1, v0, v1, master + j, mom + j, var + j, params + j, c, bad);
    }
    fused_scalar_rest(g, M, master, mom, var, params, w, c, tid, nthr, bad);
    if (flag && !skip) warp_flag(flag, bad);
}

// The fused step when master/m/v live in host memory (optimizer-state
// offload over NVLink-C2C).  The host link needs many bytes in flight: each
// thread issues the state loads of kOffloadDepth vectors (grid-strided)
// before computing any of them, and the gradients (in HBM) are loaded per
// vector.  Measured on GB300: the link sustains about 340 GB/s of combined
// reads and writes with four vectors in flight per thread and 285 GB/s with
// one.
constexpr int kOffloadDepth = 4;

template <int MT>
__global__ void __launch_bounds__(kBlock, 1)
k_fused_step_offload(const __grid_constant__ GradPtrs g, int M, float *__restrict__ master,
                     float *__restrict__ mom, float *__restrict__ var, uint16_t *__restrict__ params,
                     const Walk w, const Z1Consts c, uint32_t *flag, int skip)
{
    if (skip && *reinterpret_cast<volatile uint32_t *>(flag) != 0u) return;
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    bool bad = false;
    for (int64_t i0 = tid; i0 < w.nvec; i0 += kOffloadDepth * nthr) {
        float4 st[kOffloadDepth][6];
#pragma unroll
        for (int u = 0; u < kOffloadDepth; ++u) {
            const int64_t i = i0 + u * nthr;
            if (i < w.nvec) {
                const int64_t j = w.head + i * kVec;
                st[u][0] = ld_state(master + j);
                st[u][1] = ld_state(master + j + 4);
                st[u][2] = ld_state(mom + j);
                st[u][3] = ld_state(mom + j + 4);
                st[u][4] = ld_state(var + j);
                st[u][5] = ld_state(var + j + 4);
            }
        }
#pragma unroll
        for (int u = 0; u < kOffloadDepth; ++u) {
            const int64_t i = i0 + u * nthr;
            if (i < w.nvec) {
                const int64_t j = w.head + i * kVec;
                float s[kVec];
                sum8<MT>(g, M, j, s);
                store_vec(s, st[u][0], st[u][1], st[u][2], st[u][3], st[u][4], st[u][5], master + j, mom + j,
                          var + j, params + j, c, bad);
            }
        }
    }
    fused_scalar_rest(g, M, master, mom, var, params, w, c, tid, nthr, bad);
    if (flag && !skip) warp_flag(flag, bad);
}

// ----------------------------------------- shared-memory staged variant ------
//
// The fused step with its vector body staged through shared memory by the
// Tensor Memory Accelerator: a producer warp issues 1-D bulk copies
// (cp.async.bulk, completion counted on an mbarrier) of each tile's M gradient
// slices and master/m/v into a ring of stages; eight consumer warps compute
// from shared memory and store the results directly.  Every wait is bounded
// (kWaitNs of %globaltimer); a wait that runs out records an error in
// g_zero1_status and the kernel drains and returns instead of hanging.
//
// Measured on GB300 against the register-pipelined direct loads of
// k_fused_step: slower on this access pattern (a pure stream with no reuse
// gains nothing from the extra pass through shared memory), so the fused step
// does not use it; it is kept so the comparison can be reproduced.

__device__ uint32_t g_zero1_status;  // bit 0: a bounded wait ran out

constexpr uint64_t kWaitNs = 1000000000ull;  // 1 s
constexpr int kTmaConsumers = 256;           // 8 consumer warps
constexpr int kTmaThreads = kTmaConsumers + 32;

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of the given parity; false (and the status bit set)
// if it has not completed within kWaitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity)
{
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try(b, parity)) {
        if (global_ns() - t0 > kWaitNs) {
            atomicOr(&g_zero1_status, 1u);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Tile of T elements (E = T / 256 per consumer thread); S stages in the ring.
// MT = M for M <= 8, 0 for M > 8 (runtime M).
template <int MT, int T>
__global__ void __launch_bounds__(kTmaThreads, 1)
k_fused_step_tma(const __grid_constant__ GradPtrs g, int M, int S, float *__restrict__ master,
                 float *__restrict__ mom, float *__restrict__ var, uint16_t *__restrict__ params,
                 const Walk w, const Z1Consts c, uint32_t *flag, int skip)
{
    constexpr int E = T / kTmaConsumers;
    static_assert(E == 1 || E == 2 || E == 4, "tile must give 1, 2 or 4 elements per consumer thread");
    if (skip && *reinterpret_cast<volatile uint32_t *>(flag) != 0u) return;
    extern __shared__ __align__(128) unsigned char smem[];
    const int64_t gbytes = (int64_t)T * 2, sbytes = (int64_t)T * 4;
    const int64_t stage_bytes = M * gbytes + 3 * sbytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * stage_bytes);
    uint64_t *empty = full + S;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int k = 0; k < S; ++k) {
            mbar_init(&full[k], 1);
            mbar_init(&empty[k], kTmaConsumers / 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const int64_t nbody = w.nvec * kVec;
    const int64_t ntiles = (nbody + T - 1) / T;
    if (warp == kTmaConsumers / 32) {  // producer warp: one thread issues the copies
        if (lane == 0) {
            int64_t k = 0;
            for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
                const int st = (int)(k % S);
                if (k >= S && !mbar_wait(&empty[st], (uint32_t)((k / S - 1) & 1))) break;
                const int64_t off = w.head + tile * T;
                const uint32_t elems = (uint32_t)(nbody - tile * T < T ? nbody - tile * T : T);
                unsigned char *base = smem + st * stage_bytes;
                mbar_expect_tx(&full[st], elems * (uint32_t)(2 * M + 12));
                for (int r = 0; r < M; ++r) bulk_load(base + r * gbytes, g.p[r] + off, elems * 2, &full[st]);
                bulk_load(base + M * gbytes, master + off, elems * 4, &full[st]);
                bulk_load(base + M * gbytes + sbytes, mom + off, elems * 4, &full[st]);
                bulk_load(base + M * gbytes + 2 * sbytes, var + off, elems * 4, &full[st]);
            }
            // drain: the copies of the last stages issued must land before exit
            for (int64_t q = k > S ? k - S : 0; q < k; ++q) mbar_wait(&full[q % S], (uint32_t)((q / S) & 1));
        }
        return;
    }
    // consumers
    bool bad = false;
    const int t = threadIdx.x;
    int64_t k = 0;
    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k) {
        const int st = (int)(k % S);
        if (!mbar_wait(&full[st], (uint32_t)((k / S) & 1))) break;
        const int64_t off = w.head + tile * T;
        const int elems = (int)(nbody - tile * T < T ? nbody - tile * T : T);
        const unsigned char *base = smem + st * stage_bytes;
        const int e0 = t * E;
        float sum[E], ww[E], mm[E], vv[E];
        const bool mine = e0 < elems;  // elems is a multiple of 8, so E elements at e0 are all in
        if (mine) {
            const int mt = MT > 0 ? MT : M;
            const float *sw = reinterpret_cast<const float *>(base + M * gbytes) + e0;
            const float *sm = reinterpret_cast<const float *>(base + M * gbytes + sbytes) + e0;
            const float *sv = reinterpret_cast<const float *>(base + M * gbytes + 2 * sbytes) + e0;
            if constexpr (E == 4) {
                uint2 q = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(base) + e0);
                sum[0] = bf_lo(q.x); sum[1] = bf_hi(q.x); sum[2] = bf_lo(q.y); sum[3] = bf_hi(q.y);
#pragma unroll(MT > 0 ? MT : 1)
                for (int r = 1; r < mt; ++r) {
                    q = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint16_t *>(base + r * gbytes) + e0);
                    sum[0] = __fadd_rn(sum[0], bf_lo(q.x)); sum[1] = __fadd_rn(sum[1], bf_hi(q.x));
                    sum[2] = __fadd_rn(sum[2], bf_lo(q.y)); sum[3] = __fadd_rn(sum[3], bf_hi(q.y));
                }
                const float4 a4 = *reinterpret_cast<const float4 *>(sw);
                const float4 b4 = *reinterpret_cast<const float4 *>(sm);
                const float4 d4 = *reinterpret_cast<const float4 *>(sv);
                ww[0] = a4.x; ww[1] = a4.y; ww[2] = a4.z; ww[3] = a4.w;
                mm[0] = b4.x; mm[1] = b4.y; mm[2] = b4.z; mm[3] = b4.w;
                vv[0] = d4.x; vv[1] = d4.y; vv[2] = d4.z; vv[3] = d4.w;
            } else if constexpr (E == 2) {
                uint32_t q = *reinterpret_cast<const uint32_t *>(reinterpret_cast<const uint16_t *>(base) + e0);
                sum[0] = bf_lo(q); sum[1] = bf_hi(q);
                for (int r = 1; r < mt; ++r) {
                    q = *reinterpret_cast<const uint32_t *>(reinterpret_cast<const uint16_t *>(base + r * gbytes) + e0);
                    sum[0] = __fadd_rn(sum[0], bf_lo(q)); sum[1] = __fadd_rn(sum[1], bf_hi(q));
                }
                const float2 a2 = *reinterpret_cast<const float2 *>(sw);
                const float2 b2 = *reinterpret_cast<const float2 *>(sm);
                const float2 d2 = *reinterpret_cast<const float2 *>(sv);
                ww[0] = a2.x; ww[1] = a2.y; mm[0] = b2.x; mm[1] = b2.y; vv[0] = d2.x; vv[1] = d2.y;
            } else {
                sum[0] = bf_one(reinterpret_cast<const uint16_t *>(base)[e0]);
                for (int r = 1; r < mt; ++r)
                    sum[0] = __fadd_rn(sum[0], bf_one(reinterpret_cast<const uint16_t *>(base + r * gbytes)[e0]));
                ww[0] = sw[0]; mm[0] = sm[0]; vv[0] = sv[0];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);  // this warp is done with the stage's shared memory
        if (mine) {
            const int64_t j = off + e0;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                bad |= !finite(sum[e]);
                adamw1(__fmul_rn(sum[e], c.inv), c, ww[e], mm[e], vv[e]);
            }
            if constexpr (E == 4) {
                st_stream(master + j, ww[0], ww[1], ww[2], ww[3]);
                st_stream(mom + j, mm[0], mm[1], mm[2], mm[3]);
                st_stream(var + j, vv[0], vv[1], vv[2], vv[3]);
                *reinterpret_cast<uint2 *>(params + j) = make_uint2(pack_bf16x2(ww[0], ww[1]), pack_bf16x2(ww[2], ww[3]));
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    master[j + e] = ww[e];
                    mom[j + e] = mm[e];
                    var[j + e] = vv[e];
                    params[j + e] = to_bf16(ww[e]);
                }
            }
        }
    }
    fused_scalar_rest(g, M, master, mom, var, params, w, c, (int64_t)blockIdx.x * kTmaConsumers + t,
                      (int64_t)gridDim.x * kTmaConsumers, bad);
    if (flag && !skip) warp_flag(flag, bad);
}

// Overflow check: flag |= any non-finite rank-order sum over real elements.
// A pure read stream: one vector in flight per thread at the compiler's
// register budget (5 blocks per SM) measured faster here than the two-deep
// pipeline (7196 vs 6952 GB/s at M = 8); the M > 8 grouped path keeps three
// blocks per SM (7422 GB/s at M = 64).
template <int MT>
__global__ void __launch_bounds__(kBlock, (MT) > 0 ? 5 : 3)
k_overflow(const __grid_constant__ GradPtrs g, int M, const Walk w, uint32_t *flag)
{
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    bool bad = false;
    for (int64_t i = tid; i < w.nvec; i += nthr) {
        float s[kVec];
        sum8<MT>(g, M, w.head + i * kVec, s);
#pragma unroll
        for (int k = 0; k < kVec; ++k) bad |= !finite(s[k]);
    }
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        if (j < w.nv) bad |= !finite(sum1(g, M, j));
    }
    warp_flag(flag, bad);
}

// Reduce-scatter: out[j] = sum * scale (fp32 or bf16), +0 on padding.
template <bool BF16>
__device__ __forceinline__ void rs_store(void *out, int64_t j, float s[kVec], float scale)
{
#pragma unroll
    for (int k = 0; k < kVec; ++k) s[k] = __fmul_rn(s[k], scale);
    if constexpr (BF16) {
        __stcs(reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + j),
               make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]),
                          pack_bf16x2(s[6], s[7])));
    } else {
        st_stream(static_cast<float *>(out) + j, s[0], s[1], s[2], s[3]);
        st_stream(static_cast<float *>(out) + j + 4, s[4], s[5], s[6], s[7]);
    }
}

template <int MT, bool BF16>
__global__ void Z1_BOUNDS(MT)
k_reduce_scatter(const __grid_constant__ GradPtrs g, int M, const Walk w, float scale, void *out,
                 uint32_t *flag)
{
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    bool bad = false;
    if constexpr (MT > 0) {
        pipelined<GradLoads<MT>>(
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
                rs_store<BF16>(out, w.head + i * kVec, s, scale);
            });
    } else {
        for (int64_t i = tid; i < w.nvec; i += nthr) {
            const int64_t j = w.head + i * kVec;
            float s[kVec];
            sum8<0>(g, M, j, s);
#pragma unroll
            for (int k = 0; k < kVec; ++k) bad |= !finite(s[k]);
            rs_store<BF16>(out, j, s, scale);
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

// AdamW on fp32 state given the scaled fp32 gradient.
struct StateLoads {
    float4 g0, g1, w0, w1, m0, m1, v0, v1;
};

__device__ __forceinline__ void load_state_vec(StateLoads &x, const float *gin, const float *master,
                                               const float *mom, const float *var, int64_t j)
{
    x.g0 = __ldcs(reinterpret_cast<const float4 *>(gin + j));
    x.g1 = __ldcs(reinterpret_cast<const float4 *>(gin + j + 4));
    x.w0 = ld_state(master + j);
    x.w1 = ld_state(master + j + 4);
    x.m0 = ld_state(mom + j);
    x.m1 = ld_state(mom + j + 4);
    x.v0 = ld_state(var + j);
    x.v1 = ld_state(var + j + 4);
}

__global__ void __launch_bounds__(kBlock, 1)
k_adamw(const float *__restrict__ gin, float *__restrict__ master, float *__restrict__ mom,
        float *__restrict__ var, const Walk w, const Z1Consts c)
{
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    pipelined<StateLoads>(
        w.nvec, tid, nthr,
        [&](StateLoads &x, int64_t i) { load_state_vec(x, gin, master, mom, var, w.head + i * kVec); },
        [&](const StateLoads &x, int64_t i) {
            const int64_t j = w.head + i * kVec;
            float gg[kVec] = {x.g0.x, x.g0.y, x.g0.z, x.g0.w, x.g1.x, x.g1.y, x.g1.z, x.g1.w};
            float ww[kVec] = {x.w0.x, x.w0.y, x.w0.z, x.w0.w, x.w1.x, x.w1.y, x.w1.z, x.w1.w};
            float mm[kVec] = {x.m0.x, x.m0.y, x.m0.z, x.m0.w, x.m1.x, x.m1.y, x.m1.z, x.m1.w};
            float vv[kVec] = {x.v0.x, x.v0.y, x.v0.z, x.v0.w, x.v1.x, x.v1.y, x.v1.z, x.v1.w};
#pragma unroll
            for (int k = 0; k < kVec; ++k) adamw1(gg[k], c, ww[k], mm[k], vv[k]);
            st_stream(master + j, ww[0], ww[1], ww[2], ww[3]);
            st_stream(master + j + 4, ww[4], ww[5], ww[6], ww[7]);
            st_stream(mom + j, mm[0], mm[1], mm[2], mm[3]);
            st_stream(mom + j + 4, mm[4], mm[5], mm[6], mm[7]);
            st_stream(var + j, vv[0], vv[1], vv[2], vv[3]);
            st_stream(var + j + 4, vv[4], vv[5], vv[6], vv[7]);
        });
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        float ww = master[j], mm = mom[j], vv = var[j];
        adamw1(gin[j], c, ww, mm, vv);
        master[j] = ww;
        mom[j] = mm;
        var[j] = vv;
    }
}

// All-gather of the updated shard: params[j] = bf16(master[j]), real only.
struct MasterLoads {
    float4 a, b;
};

__global__ void __launch_bounds__(kBlock, 1)
k_all_gather(const float *__restrict__ master, uint16_t *__restrict__ params, const Walk w)
{
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    pipelined<MasterLoads>(
        w.nvec, tid, nthr,
        [&](MasterLoads &x, int64_t i) {
            const float4 *pw = reinterpret_cast<const float4 *>(master + w.head + i * kVec);
            x.a = __ldcs(pw);
            x.b = __ldcs(pw + 1);
        },
        [&](const MasterLoads &x, int64_t i) {
            __stcs(reinterpret_cast<uint4 *>(params + w.head + i * kVec),
                   make_uint4(pack_bf16x2(x.a.x, x.a.y), pack_bf16x2(x.a.z, x.a.w), pack_bf16x2(x.b.x, x.b.y),
                              pack_bf16x2(x.b.z, x.b.w)));
        });
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        if (j < w.nv) params[j] = to_bf16(master[j]);
    }
}

// All-gather of bf16 shards into M outputs (real elements only).
__global__ void __launch_bounds__(kBlock)
k_all_gather_shards(const uint16_t *__restrict__ shards, const __grid_constant__ OutPtrs o, int M,
                    const Walk w)
{
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    for (int64_t i = tid; i < w.nvec; i += nthr) {
        const int64_t j = w.head + i * kVec;
        const uint4 q = ld_stream_u4(shards + j);
        for (int r = 0; r < M; ++r) *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(o.p[r]) + j) = q;
    }
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        if (j < w.nv) {
            const uint16_t x = shards[j];
            for (int r = 0; r < M; ++r) static_cast<uint16_t *>(o.p[r])[j] = x;
        }
    }
}

// Naive All-Reduce: every output gets sum * scale.  Element j's inputs are
// all read before any output of j is written (outputs may alias inputs).
template <bool BF16>
__device__ __forceinline__ void ar_store(const OutPtrs &o, int M, int64_t j, float s[kVec], float scale)
{
#pragma unroll
    for (int k = 0; k < kVec; ++k) s[k] = __fmul_rn(s[k], scale);
    if constexpr (BF16) {
        const uint4 q = make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]),
                                   pack_bf16x2(s[6], s[7]));
        for (int r = 0; r < M; ++r) __stcs(reinterpret_cast<uint4 *>(static_cast<uint16_t *>(o.p[r]) + j), q);
    } else {
        for (int r = 0; r < M; ++r) {
            st_stream(static_cast<float *>(o.p[r]) + j, s[0], s[1], s[2], s[3]);
            st_stream(static_cast<float *>(o.p[r]) + j + 4, s[4], s[5], s[6], s[7]);
        }
    }
}

template <int MT, bool BF16>
__global__ void Z1_BOUNDS(MT)
k_allreduce(const __grid_constant__ GradPtrs g, const __grid_constant__ OutPtrs o, int M,
            const Walk w, float scale)
{
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    if constexpr (MT > 0) {
        // in place, the next vector's loads touch other elements than the
        // current vector's stores, so prefetching them stays correct
        pipelined<GradLoads<MT>>(
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
                ar_store<BF16>(o, MT, w.head + i * kVec, s, scale);
            });
    } else {
        for (int64_t i = tid; i < w.nvec; i += nthr) {
            const int64_t j = w.head + i * kVec;
            float s[kVec];
            sum8<0>(g, M, j, s);
            ar_store<BF16>(o, M, j, s, scale);
        }
    }
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        const float s = __fmul_rn(sum1(g, M, j), scale);
        for (int r = 0; r < M; ++r) {
            if constexpr (BF16) static_cast<uint16_t *>(o.p[r])[j] = to_bf16(s);
            else static_cast<float *>(o.p[r])[j] = s;
        }
    }
}

// ------------------------------------------------ dynamic loss scaling ------
//
// "五维并行实战" 4.2 (fp16 block) names the policy's keys; the rule is stated in
// zero1.h.  S, t and the derived constants live in a zero1_scaler_t in device
// memory so the host never waits for the overflow flag.

struct ScalePolicy {
    float factor;
    int32_t window, hysteresis;
    float min_scale;
};

// b^t in double, square-and-multiply over the bits of t (least significant
// first), the same operation sequence as the host's z1_pow_int.
__device__ double pow_int_dev(double b, int64_t t)
{
    double r = 1.0, x = b;
    for (; t > 0; t >>= 1) {
        if (t & 1) r = __dmul_rn(r, x);
        x = __dmul_rn(x, x);
    }
    return r;
}

// 1/(B*S), 1 - beta1^t, 1 - beta2^t: double arithmetic rounded once to
// float, as the host evaluates them.
__device__ void derive_constants(zero1_scaler_t *sc, int64_t B, float beta1, float beta2)
{
    sc->inv = __double2float_rn(__ddiv_rn(1.0, __dmul_rn((double)B, (double)sc->scale)));
    sc->bc1 = __double2float_rn(__dsub_rn(1.0, pow_int_dev((double)beta1, sc->step)));
    sc->bc2 = __double2float_rn(__dsub_rn(1.0, pow_int_dev((double)beta2, sc->step)));
}

__global__ void k_scaler_init(zero1_scaler_t *sc, float initial_scale, int32_t hysteresis, int64_t first_step,
                              int64_t B, float beta1, float beta2)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    sc->scale = initial_scale;
    sc->step = first_step;
    sc->attempts = 0;
    sc->skipped = 0;
    sc->good_steps = 0;
    sc->hysteresis_left = hysteresis;
    sc->overflow = 0u;
    sc->reserved = 0u;
    derive_constants(sc, B, beta1, beta2);
}

// Advance the scaler after an attempt (reads the attempt's flag, clears it).
__global__ void k_scaler_update(zero1_scaler_t *sc, const ScalePolicy pol, int64_t B, float beta1, float beta2)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    sc->attempts += 1;
    if (*reinterpret_cast<volatile uint32_t *>(&sc->overflow) != 0u) {
        sc->skipped += 1;
        sc->good_steps = 0;
        sc->hysteresis_left -= 1;
        if (sc->hysteresis_left <= 0) {
            const float down = __fdiv_rn(sc->scale, pol.factor);
            sc->scale = down < pol.min_scale ? pol.min_scale : down;
            sc->hysteresis_left = pol.hysteresis;
        }
    } else {
        sc->step += 1;
        sc->good_steps += 1;
        if (sc->good_steps >= pol.window) {
            const float up = __fmul_rn(sc->scale, pol.factor);
            if (isfinite(up)) sc->scale = up;
            sc->good_steps = 0;
            sc->hysteresis_left = pol.hysteresis;
        }
    }
    sc->overflow = 0u;
    derive_constants(sc, B, beta1, beta2);
}

// AdamW + all-gather from fp32 replica sums (written by the reduce-scatter
// kernel just before on the same stream), with 1/(B*S) and the bias
// corrections read from the scaler; nothing is written if the attempt's flag
// is set.  The arithmetic is the fused step's, operation for operation.
__global__ void __launch_bounds__(kBlock, 1)
k_apply_sums(const float *__restrict__ sums, float *__restrict__ master, float *__restrict__ mom,
             float *__restrict__ var, uint16_t *__restrict__ params, const Walk w, Z1Consts c,
             const zero1_scaler_t *sc)
{
    if (*reinterpret_cast<const volatile uint32_t *>(&sc->overflow) != 0u) return;
    c.inv = sc->inv;
    c.bc1 = sc->bc1;
    c.bc2 = sc->bc2;
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    bool bad = false;  // the flag was already taken by the reduce-scatter
    pipelined<StateLoads>(
        w.nvec, tid, nthr,
        [&](StateLoads &x, int64_t i) { load_state_vec(x, sums, master, mom, var, w.head + i * kVec); },
        [&](const StateLoads &x, int64_t i) {
            const int64_t j = w.head + i * kVec;
            const float s[kVec] = {x.g0.x, x.g0.y, x.g0.z, x.g0.w, x.g1.x, x.g1.y, x.g1.z, x.g1.w};
            store_vec(s, x.w0, x.w1, x.m0, x.m1, x.v0, x.v1, master + j, mom + j, var + j, params + j, c, bad);
        });
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        float ww = master[j], mm = mom[j], vv = var[j];
        adamw1(__fmul_rn(sums[j], c.inv), c, ww, mm, vv);
        master[j] = ww;
        mom[j] = mm;
        var[j] = vv;
        if (j < w.nv) params[j] = to_bf16(ww);
    }
}

// ----------------------------------------------- consistency checksum -----
//
// Silent-data-corruption guard for the replicated parameters ("CS336 Lecture
// 7: Parallelism 1" case studies): over a buffer's 16-bit units u_i,
// out[0] = sum u_i and out[1] = sum (i + 1) u_i, both mod 2^64.  Integer sums
// are exact, so the per-thread partial sums, the warp reduction and the
// atomicAdd of each warp's partials give the same words in any order.

__device__ __forceinline__ void warp_sum_u64(uint64_t &x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
}

__global__ void __launch_bounds__(kBlock)
k_checksum16(const uint16_t *__restrict__ u, const Walk w, unsigned long long *out)
{
    const int64_t tid = (int64_t)blockIdx.x * kBlock + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * kBlock;
    uint64_t s1 = 0, s2 = 0;
    for (int64_t i = tid; i < w.nvec; i += nthr) {
        const int64_t j = w.head + i * kVec;
        const uint4 q = ld_stream_u4(u + j);
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint64_t lo = words[k] & 0xffffu, hi = words[k] >> 16;
            s1 += lo + hi;
            s2 += (uint64_t)(j + 2 * k + 1) * lo + (uint64_t)(j + 2 * k + 2) * hi;
        }
    }
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        const uint64_t x = ld_stream_u16(u + j);
        s1 += x;
        s2 += (uint64_t)(j + 1) * x;
    }
    warp_sum_u64(s1);
    warp_sum_u64(s2);
    if ((threadIdx.x & 31) == 0 && (s1 | s2)) {
        atomicAdd(out, (unsigned long long)s1);
        atomicAdd(out + 1, (unsigned long long)s2);
    }
}

// ------------------------------------------------------------ host side ----

struct ArrayRef {
    const void *p;
    int esize;
};

// Choose the per-element head h in [0, 8) at which every array is 16-byte
// aligned; if there is none, the whole range runs per element.
Walk make_walk(int64_t L, int64_t nv, const ArrayRef *a, int count)
{
    Walk w{L, nv, 0, 0};
    for (int h = 0; h < kVec; ++h) {
        bool ok = true;
        for (int k = 0; k < count && ok; ++k)
            ok = (((uintptr_t)a[k].p + (uintptr_t)h * a[k].esize) & 15u) == 0;
        if (ok) {
            w.head = h < nv ? h : nv;
            w.nvec = nv > h ? (nv - h) / kVec : 0;
            return w;
        }
    }
    return w;
}

int check_natural(const void *p, int esize, const char *what)
{
    if (((uintptr_t)p & (uintptr_t)(esize - 1)) != 0)
        return z1_fail(ZERO1_EALIGN, "%s is not %d-byte aligned", what, esize);
    return ZERO1_OK;
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

// One resident wave: SMs x resident blocks of this kernel (cached per kernel
// and device), capped by the work.
template <class K>
int grid_for(K kernel, int64_t work_items)
{
    static std::atomic<int> cache[64];
    int dev = 0;
    cudaGetDevice(&dev);
    int per_sm = dev < 64 ? cache[dev].load(std::memory_order_relaxed) : 0;
    if (per_sm <= 0) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBlock, 0) != cudaSuccess ||
            per_sm <= 0)
            per_sm = 1;
        if (dev < 64) cache[dev].store(per_sm, std::memory_order_relaxed);
    }
    const int64_t wave = (int64_t)sm_count() * per_sm;
    int64_t need = (work_items + kBlock - 1) / kBlock;
    if (need < 1) need = 1;
    return (int)(need < wave ? need : (wave > 0 ? wave : 1));
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

int64_t work_of(const Walk &w)
{
    const int64_t ns = w.L - w.nvec * kVec;
    return w.nvec > ns ? w.nvec : ns;
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

// ------------------------------------------------------------ C ABI -------

namespace {

// Validate and launch the fused step over one range of L elements whose
// first nv are real parameters (the pointers are at the range's start).
int launch_fused_range(const zero1_plan_t *plan, int64_t L, int64_t nv, const void *const *grads, float *master,
                       float *m, float *v, void *params, const zero1_adamw_t *hp, uint32_t *overflow_flag,
                       int32_t skip_if_flag, zero1_stream_t stream, const char *what)
{
    Z1Consts c;
    int rc;
    if ((rc = z1_adamw_constants(hp, plan->M, &c)) != ZERO1_OK) return rc;
    if (!master || !m || !v)
        return z1_fail(ZERO1_EINVAL, "%s: master, m and v must be non-NULL", what);
    if (nv > 0 && !params)
        return z1_fail(ZERO1_EINVAL, "%s: params must be non-NULL when the range holds parameters", what);
    if (skip_if_flag && !overflow_flag)
        return z1_fail(ZERO1_EINVAL, "%s: skip_if_flag needs an overflow flag", what);
    GradPtrs g{};
    if (nv > 0 && (rc = load_grads(plan, grads, &g, what)) != ZERO1_OK) return rc;
    if ((rc = check_natural(master, 4, "master")) || (rc = check_natural(m, 4, "m")) ||
        (rc = check_natural(v, 4, "v")) || (rc = check_natural(params, 2, "params")) ||
        (overflow_flag && (rc = check_natural(overflow_flag, 4, "overflow_flag"))))
        return rc;
    ArrayRef arr[ZERO1_MAX_REPLICAS + 4] = {{master, 4}, {m, 4}, {v, 4}, {params, 2}};
    for (int k = 0; k < plan->M; ++k) arr[4 + k] = {g.p[k], 2};
    const Walk w = make_walk(L, nv, arr, 4 + plan->M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint16_t *pp = static_cast<uint16_t *>(params);
    const int M = plan->M;
    const int skip = skip_if_flag ? 1 : 0;
    if (in_host_memory(master)) {
        dispatch_m(M, [&](auto mt) {
            constexpr int MT = decltype(mt)::value;
            const int grid = grid_for(k_fused_step_offload<MT>, work_of(w));
            k_fused_step_offload<MT><<<grid, kBlock, 0, st>>>(g, M, master, m, v, pp, w, c, overflow_flag, skip);
        });
    } else if (M > 8) {
        const int grid = grid_for(k_fused_step_grouped, work_of(w));
        k_fused_step_grouped<<<grid, kBlock, 0, st>>>(g, M, master, m, v, pp, w, c, overflow_flag, skip);
    } else {
        dispatch_m(M, [&](auto mt) {
            constexpr int MT = decltype(mt)::value;
            if constexpr (MT > 0) {
                if (w.nvec <= kWideMaxVec) {
                    const int grid = grid_for(k_fused_step_wide<MT>, work_of(w));
                    k_fused_step_wide<MT><<<grid, kBlock, 0, st>>>(g, M, master, m, v, pp, w, c, overflow_flag,
                                                                   skip);
                } else {
                    const int grid = grid_for(k_fused_step<MT>, work_of(w));
                    k_fused_step<MT><<<grid, kBlock, 0, st>>>(g, M, master, m, v, pp, w, c, overflow_flag, skip);
                }
            }
        });
    }
    return launch_status(what);
}

}  // namespace

extern "C" int zero1_reduce_scatter_adamw_allgather(const zero1_plan_t *plan, int32_t shard_begin,
                                                    int32_t shard_end, const void *const *grads,
                                                    float *master, float *m, float *v, void *params,
                                                    const zero1_adamw_t *hp, uint32_t *overflow_flag,
                                                    int32_t skip_if_flag, zero1_stream_t stream)
{
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    return launch_fused_range(plan, r.L, r.nv, grads, master, m, v, params, hp, overflow_flag, skip_if_flag,
                              stream, "fused step");
}

extern "C" int zero1_step_bucket(const zero1_plan_t *plan, int64_t elem_begin, int64_t elem_end,
                                 const void *const *grads, float *master, float *m, float *v, void *params,
                                 const zero1_adamw_t *hp, uint32_t *overflow_flag, zero1_stream_t stream)
{
    int rc = z1_check_plan(plan);
    if (rc != ZERO1_OK) return rc;
    if (elem_begin < 0 || elem_end > plan->padded_n || elem_begin >= elem_end)
        return z1_fail(ZERO1_EINVAL, "bucket [%lld, %lld) not inside [0, %lld)", (long long)elem_begin,
                       (long long)elem_end, (long long)plan->padded_n);
    const int64_t L = elem_end - elem_begin;
    int64_t nv = plan->n - elem_begin;
    nv = nv < 0 ? 0 : (nv > L ? L : nv);
    return launch_fused_range(plan, L, nv, grads, master, m, v, params, hp, overflow_flag, 0, stream,
                              "bucketed step");
}

extern "C" int zero1_overflow_check(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                    const void *const *grads, uint32_t *flag, zero1_stream_t stream)
{
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    if (!flag) return z1_fail(ZERO1_EINVAL, "overflow check: flag is NULL");
    if ((rc = check_natural(flag, 4, "flag")) != ZERO1_OK) return rc;
    if (r.nv == 0) return ZERO1_OK;
    GradPtrs g{};
    if ((rc = load_grads(plan, grads, &g, "overflow check")) != ZERO1_OK) return rc;
    ArrayRef arr[ZERO1_MAX_REPLICAS];
    for (int k = 0; k < plan->M; ++k) arr[k] = {grads[k], 2};
    const Walk w = make_walk(r.nv, r.nv, arr, plan->M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int M = plan->M;
    dispatch_m(M, [&](auto mt) {
        constexpr int MT = decltype(mt)::value;
        const int grid = grid_for(k_overflow<MT>, work_of(w));
        k_overflow<MT><<<grid, kBlock, 0, st>>>(g, M, w, flag);
    });
    return launch_status("overflow check launch");
}

extern "C" int dp_allreduce(const zero1_plan_t *plan, const void *const *grads_in, void *const *outs,
                            float scale, int32_t out_dtype, zero1_stream_t stream)
{
    int rc = z1_check_plan(plan);
    if (rc != ZERO1_OK) return rc;
    if (out_dtype != ZERO1_DTYPE_BF16 && out_dtype != ZERO1_DTYPE_F32)
        return z1_fail(ZERO1_EINVAL, "all-reduce: unknown output dtype %d", out_dtype);
    if (!std::isfinite(scale)) return z1_fail(ZERO1_EINVAL, "all-reduce: scale is not finite");
    GradPtrs g{};
    if ((rc = load_grads(plan, grads_in, &g, "all-reduce")) != ZERO1_OK) return rc;
    if (!outs) return z1_fail(ZERO1_EINVAL, "all-reduce: outs is NULL");
    const int M = plan->M;
    const int osz = out_dtype == ZERO1_DTYPE_BF16 ? 2 : 4;
    OutPtrs o{};
    ArrayRef arr[2 * ZERO1_MAX_REPLICAS];
    for (int k = 0; k < M; ++k) {
        if (!outs[k]) return z1_fail(ZERO1_EINVAL, "all-reduce: outs[%d] is NULL", k);
        if ((rc = check_natural(outs[k], osz, "an all-reduce output")) != ZERO1_OK) return rc;
        if (osz == 4) {
            const uintptr_t a = (uintptr_t)outs[k], b = a + (uintptr_t)plan->n * 4;
            for (int q = 0; q < M; ++q) {
                const uintptr_t c0 = (uintptr_t)grads_in[q], c1 = c0 + (uintptr_t)plan->n * 2;
                if (a < c1 && c0 < b)
                    return z1_fail(ZERO1_EINVAL, "all-reduce: fp32 output %d overlaps input %d", k, q);
            }
        }
        o.p[k] = outs[k];
        arr[k] = {grads_in[k], 2};
        arr[M + k] = {outs[k], osz};
    }
    const Walk w = make_walk(plan->n, plan->n, arr, 2 * M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    dispatch_m(M, [&](auto mt) {
        constexpr int MT = decltype(mt)::value;
        if (osz == 2) {
            const int grid = grid_for(k_allreduce<MT, true>, work_of(w));
            k_allreduce<MT, true><<<grid, kBlock, 0, st>>>(g, o, M, w, scale);
        } else {
            const int grid = grid_for(k_allreduce<MT, false>, work_of(w));
            k_allreduce<MT, false><<<grid, kBlock, 0, st>>>(g, o, M, w, scale);
        }
    });
    return launch_status("all-reduce launch");
}

extern "C" int zero1_reduce_scatter(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                    const void *const *grads, float scale, int32_t out_dtype, void *out,
                                    uint32_t *flag, zero1_stream_t stream)
{
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    if (out_dtype != ZERO1_DTYPE_BF16 && out_dtype != ZERO1_DTYPE_F32)
        return z1_fail(ZERO1_EINVAL, "reduce-scatter: unknown output dtype %d", out_dtype);
    if (!std::isfinite(scale)) return z1_fail(ZERO1_EINVAL, "reduce-scatter: scale is not finite");
    if (!out) return z1_fail(ZERO1_EINVAL, "reduce-scatter: out is NULL");
    const int osz = out_dtype == ZERO1_DTYPE_BF16 ? 2 : 4;
    if ((rc = check_natural(out, osz, "reduce-scatter output")) != ZERO1_OK) return rc;
    if (flag && (rc = check_natural(flag, 4, "flag")) != ZERO1_OK) return rc;
    GradPtrs g{};
    if (r.nv > 0 && (rc = load_grads(plan, grads, &g, "reduce-scatter")) != ZERO1_OK) return rc;
    ArrayRef arr[ZERO1_MAX_REPLICAS + 1] = {{out, osz}};
    for (int k = 0; k < plan->M; ++k) arr[1 + k] = {g.p[k], 2};
    const Walk w = make_walk(r.L, r.nv, arr, 1 + plan->M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int M = plan->M;
    dispatch_m(M, [&](auto mt) {
        constexpr int MT = decltype(mt)::value;
        if (osz == 2) {
            const int grid = grid_for(k_reduce_scatter<MT, true>, work_of(w));
            k_reduce_scatter<MT, true><<<grid, kBlock, 0, st>>>(g, M, w, scale, out, flag);
        } else {
            const int grid = grid_for(k_reduce_scatter<MT, false>, work_of(w));
            k_reduce_scatter<MT, false><<<grid, kBlock, 0, st>>>(g, M, w, scale, out, flag);
        }
    });
    return launch_status("reduce-scatter launch");
}

extern "C" int zero1_adamw_update(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                  const float *gin, float *master, float *m, float *v,
                                  const zero1_adamw_t *hp, zero1_stream_t stream)
{
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    Z1Consts c;
    if ((rc = z1_adamw_constants(hp, plan->M, &c)) != ZERO1_OK) return rc;
    if (!gin || !master || !m || !v) return z1_fail(ZERO1_EINVAL, "adamw: NULL array");
    if ((rc = check_natural(gin, 4, "g")) || (rc = check_natural(master, 4, "master")) ||
        (rc = check_natural(m, 4, "m")) || (rc = check_natural(v, 4, "v")))
        return rc;
    const ArrayRef arr[4] = {{gin, 4}, {master, 4}, {m, 4}, {v, 4}};
    // every element of the range is updated: walk it as if all were real
    const Walk w = make_walk(r.L, r.L, arr, 4);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int grid = grid_for(k_adamw, work_of(w));
    k_adamw<<<grid, kBlock, 0, st>>>(gin, master, m, v, w, c);
    return launch_status("adamw launch");
}

extern "C" int zero1_all_gather(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                const float *master, void *params, zero1_stream_t stream)
{
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    if (r.nv == 0) return ZERO1_OK;
    if (!master || !params) return z1_fail(ZERO1_EINVAL, "all-gather: NULL array");
    if ((rc = check_natural(master, 4, "master")) || (rc = check_natural(params, 2, "params"))) return rc;
    const ArrayRef arr[2] = {{master, 4}, {params, 2}};
    const Walk w = make_walk(r.nv, r.nv, arr, 2);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int grid = grid_for(k_all_gather, work_of(w));
    k_all_gather<<<grid, kBlock, 0, st>>>(master, static_cast<uint16_t *>(params), w);
    return launch_status("all-gather launch");
}

extern "C" int zero1_all_gather_shards(const zero1_plan_t *plan, const void *shards, void *const *outs,
                                       zero1_stream_t stream)
{
    int rc = z1_check_plan(plan);
    if (rc != ZERO1_OK) return rc;
    if (!shards || !outs) return z1_fail(ZERO1_EINVAL, "all-gather shards: NULL argument");
    if ((rc = check_natural(shards, 2, "shards")) != ZERO1_OK) return rc;
    OutPtrs o{};
    ArrayRef arr[ZERO1_MAX_REPLICAS + 1] = {{shards, 2}};
    for (int k = 0; k < plan->M; ++k) {
        if (!outs[k]) return z1_fail(ZERO1_EINVAL, "all-gather shards: outs[%d] is NULL", k);
        if ((rc = check_natural(outs[k], 2, "an all-gather output")) != ZERO1_OK) return rc;
        o.p[k] = outs[k];
        arr[1 + k] = {outs[k], 2};
    }
    const Walk w = make_walk(plan->n, plan->n, arr, 1 + plan->M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int grid = grid_for(k_all_gather_shards, work_of(w));
    k_all_gather_shards<<<grid, kBlock, 0, st>>>(static_cast<const uint16_t *>(shards), o, plan->M, w);
    return launch_status("all-gather shards launch");
}

namespace {

int check_policy(const zero1_loss_scale_policy_t *p)
{
    if (!p) return z1_fail(ZERO1_EINVAL, "loss-scale policy is NULL");
    if (!(p->initial_scale > 0.0f) || !std::isfinite(p->initial_scale))
        return z1_fail(ZERO1_EINVAL, "initial_scale must be finite and > 0");
    if (!(p->factor > 1.0f) || !std::isfinite(p->factor)) return z1_fail(ZERO1_EINVAL, "factor must be finite and > 1");
    if (p->window < 1) return z1_fail(ZERO1_EINVAL, "window must be >= 1");
    if (p->hysteresis < 1) return z1_fail(ZERO1_EINVAL, "hysteresis must be >= 1");
    if (!(p->min_scale > 0.0f) || !std::isfinite(p->min_scale))
        return z1_fail(ZERO1_EINVAL, "min_scale must be finite and > 0");
    return ZERO1_OK;
}

// Validate the hyperparameters a dynamic step uses (its own S and t come
// from the scaler) and evaluate the host constants.
int dynamic_constants(const zero1_adamw_t *hp, int32_t M, Z1Consts *c)
{
    if (!hp) return z1_fail(ZERO1_EINVAL, "hyperparameters are NULL");
    zero1_adamw_t h = *hp;
    h.loss_scale = 1.0f;
    h.step = 1;
    return z1_adamw_constants(&h, M, c);
}

int check_scaler_ptr(const zero1_scaler_t *sc)
{
    if (!sc) return z1_fail(ZERO1_EINVAL, "scaler is NULL");
    if (((uintptr_t)sc & 7u) != 0) return z1_fail(ZERO1_EALIGN, "scaler is not 8-byte aligned");
    return ZERO1_OK;
}

}  // namespace

extern "C" int zero1_scaler_init(zero1_scaler_t *scaler, const zero1_loss_scale_policy_t *policy,
                                 const zero1_adamw_t *hp, zero1_stream_t stream)
{
    int rc;
    if ((rc = check_scaler_ptr(scaler)) != ZERO1_OK || (rc = check_policy(policy)) != ZERO1_OK) return rc;
    if (!hp) return z1_fail(ZERO1_EINVAL, "hyperparameters are NULL");
    if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return z1_fail(ZERO1_EINVAL, "betas must lie in [0, 1)");
    if (hp->global_batch < 1) return z1_fail(ZERO1_EINVAL, "global batch must be >= 1");
    if (hp->step < 1) return z1_fail(ZERO1_EINVAL, "step t = %lld < 1", (long long)hp->step);
    k_scaler_init<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        scaler, policy->initial_scale, policy->hysteresis, hp->step, hp->global_batch, hp->beta1, hp->beta2);
    return launch_status("scaler init launch");
}

extern "C" int zero1_step_dynamic(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                  const void *const *grads, float *master, float *m, float *v, void *params,
                                  const zero1_adamw_t *hp, zero1_scaler_t *scaler,
                                  const zero1_loss_scale_policy_t *policy, float *sums, zero1_stream_t stream)
{
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    Z1Consts c;
    if ((rc = dynamic_constants(hp, plan->M, &c)) != ZERO1_OK) return rc;
    if ((rc = check_scaler_ptr(scaler)) != ZERO1_OK || (rc = check_policy(policy)) != ZERO1_OK) return rc;
    if (!master || !m || !v || !sums)
        return z1_fail(ZERO1_EINVAL, "dynamic step: master, m, v and sums must be non-NULL");
    if (r.nv > 0 && !params)
        return z1_fail(ZERO1_EINVAL, "dynamic step: params must be non-NULL when the range holds parameters");
    GradPtrs g{};
    if (r.nv > 0 && (rc = load_grads(plan, grads, &g, "dynamic step")) != ZERO1_OK) return rc;
    if ((rc = check_natural(master, 4, "master")) || (rc = check_natural(m, 4, "m")) ||
        (rc = check_natural(v, 4, "v")) || (rc = check_natural(params, 2, "params")) ||
        (rc = check_natural(sums, 4, "sums")))
        return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int M = plan->M;
    // 1. reduce-scatter into the fp32 sums, flag into the scaler
    ArrayRef ra[ZERO1_MAX_REPLICAS + 1] = {{sums, 4}};
    for (int k = 0; k < M; ++k) ra[1 + k] = {g.p[k], 2};
    const Walk wr = make_walk(r.L, r.nv, ra, 1 + M);
    uint32_t *flag = &scaler->overflow;
    dispatch_m(M, [&](auto mt) {
        constexpr int MT = decltype(mt)::value;
        const int grid = grid_for(k_reduce_scatter<MT, false>, work_of(wr));
        k_reduce_scatter<MT, false><<<grid, kBlock, 0, st>>>(g, M, wr, 1.0f, sums, flag);
    });
    // 2. the update from the sums (skipped on overflow)
    const ArrayRef ua[5] = {{sums, 4}, {master, 4}, {m, 4}, {v, 4}, {params, 2}};
    const Walk wu = make_walk(r.L, r.nv, ua, 5);
    const int grid = grid_for(k_apply_sums, work_of(wu));
    k_apply_sums<<<grid, kBlock, 0, st>>>(sums, master, m, v, static_cast<uint16_t *>(params), wu, c, scaler);
    // 3. the scaler advances
    const ScalePolicy pol{policy->factor, policy->window, policy->hysteresis, policy->min_scale};
    k_scaler_update<<<1, 32, 0, st>>>(scaler, pol, hp->global_batch, hp->beta1, hp->beta2);
    return launch_status("dynamic step launch");
}

// ------------------------------------------- step without caller allocation --
//
// For callers that cannot call cudaMalloc (their pool allocator owns the
// device memory, or allocation would synchronise the device): the sums
// workspace of zero1_step_dynamic is this file-scope array, which exists on
// every device that loads the library until the process exits.  Its name is a
// host-side stand-in in host code; the device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
static __device__ __align__(256) float g_noalloc_sums[ZERO1_NOALLOC_MAX_ELEMS];

namespace {

std::atomic<float *> g_noalloc_addr[64];

// Device address of g_noalloc_sums on the current device (looked up on the
// first call on each device).
int noalloc_sums(float **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return z1_fail(ZERO1_ECUDA, "no-alloc step: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return z1_fail(ZERO1_ERANGE, "no-alloc step: device %d beyond 64 devices", dev);
    float *p = g_noalloc_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        void *addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_noalloc_sums);
        if (e != cudaSuccess || !addr)
            return z1_fail(ZERO1_ECUDA, "no-alloc step: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        p = static_cast<float *>(addr);
        g_noalloc_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return ZERO1_OK;
}

}  // namespace

extern "C" int zero1_step_dynamic_noalloc(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                          const void *const *grads, float *master, float *m, float *v,
                                          void *params, const zero1_adamw_t *hp, zero1_scaler_t *scaler,
                                          const zero1_loss_scale_policy_t *policy, zero1_stream_t stream)
{
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    if (r.L > (int64_t)ZERO1_NOALLOC_MAX_ELEMS)
        return z1_fail(ZERO1_ERANGE,
                       "no-alloc step: range of %lld elements exceeds the built-in workspace of %d elements "
                       "(64 MiB); split the call by shards",
                       (long long)r.L, ZERO1_NOALLOC_MAX_ELEMS);
    float *sums = nullptr;
    if ((rc = noalloc_sums(&sums)) != ZERO1_OK) return rc;
    return zero1_step_dynamic(plan, shard_begin, shard_end, grads, master, m, v, params, hp, scaler, policy,
                              sums, stream);
}

// ----------------------------------------------------- staged variant: ABI --

namespace {

template <int MT, int T>
int launch_tma(const GradPtrs &g, int M, float *master, float *m, float *v, uint16_t *params, const Walk &w,
               const Z1Consts &c, uint32_t *flag, int skip, cudaStream_t st)
{
    int dev = 0, smem_max = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return z1_fail(ZERO1_ECUDA, "staged step: device query: %s", cudaGetErrorString(e));
    const int64_t stage_bytes = (int64_t)M * T * 2 + 3 * (int64_t)T * 4;
    int S = (int)((smem_max - 7 * 16) / stage_bytes);
    if (S > 7) S = 7;
    if (S < 1) return z1_fail(ZERO1_ERANGE, "staged step: one stage of %lld bytes does not fit", (long long)stage_bytes);
    const int smem = (int)(S * stage_bytes + 2 * S * 8);
    auto kernel = k_fused_step_tma<MT, T>;
    if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
        return z1_fail(ZERO1_ECUDA, "staged step: shared memory %d bytes: %s", smem, cudaGetErrorString(e));
    int per_sm = 0;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kTmaThreads, smem)) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    const int64_t ntiles = (w.nvec * kVec + T - 1) / T;
    int64_t grid = (int64_t)sms * per_sm;
    if (ntiles < grid) grid = ntiles;
    if (grid < 1) grid = 1;
    kernel<<<(int)grid, kTmaThreads, smem, st>>>(g, M, S, master, m, v, params, w, c, flag, skip);
    return launch_status("staged step launch");
}

}  // namespace

extern "C" int zero1_step_tma(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                              const void *const *grads, float *master, float *m, float *v, void *params,
                              const zero1_adamw_t *hp, uint32_t *overflow_flag, int32_t skip_if_flag,
                              zero1_stream_t stream)
{
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    Z1Consts c;
    if ((rc = z1_adamw_constants(hp, plan->M, &c)) != ZERO1_OK) return rc;
    if (!master || !m || !v) return z1_fail(ZERO1_EINVAL, "staged step: master, m and v must be non-NULL");
    if (r.nv > 0 && !params)
        return z1_fail(ZERO1_EINVAL, "staged step: params must be non-NULL when the range holds parameters");
    if (skip_if_flag && !overflow_flag) return z1_fail(ZERO1_EINVAL, "staged step: skip_if_flag needs a flag");
    GradPtrs g{};
    if (r.nv > 0 && (rc = load_grads(plan, grads, &g, "staged step")) != ZERO1_OK) return rc;
    if ((rc = check_natural(master, 4, "master")) || (rc = check_natural(m, 4, "m")) ||
        (rc = check_natural(v, 4, "v")) || (rc = check_natural(params, 2, "params")) ||
        (overflow_flag && (rc = check_natural(overflow_flag, 4, "overflow_flag"))))
        return rc;
    bool host = in_host_memory(master) || in_host_memory(m) || in_host_memory(v) ||
                (params && in_host_memory(params));
    for (int k = 0; k < plan->M && !host && r.nv > 0; ++k) host = in_host_memory(g.p[k]);
    if (host) return z1_fail(ZERO1_EINVAL, "staged step: every buffer must be device memory");
    ArrayRef arr[ZERO1_MAX_REPLICAS + 4] = {{master, 4}, {m, 4}, {v, 4}, {params, 2}};
    for (int k = 0; k < plan->M; ++k) arr[4 + k] = {g.p[k], 2};
    const Walk w = make_walk(r.L, r.nv, arr, 4 + plan->M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint16_t *pp = static_cast<uint16_t *>(params);
    const int M = plan->M;
    const int skip = skip_if_flag ? 1 : 0;
    if (M > 8) return launch_tma<0, 512>(g, M, master, m, v, pp, w, c, overflow_flag, skip, st);
    int out = ZERO1_OK;
    dispatch_m(M, [&](auto mt) {
        constexpr int MT = decltype(mt)::value;
        if constexpr (MT > 0) out = launch_tma<MT, 1024>(g, M, master, m, v, pp, w, c, overflow_flag, skip, st);
    });
    return out;
}

extern "C" int zero1_device_status(uint32_t *status, int32_t clear)
{
    if (!status) return z1_fail(ZERO1_EINVAL, "device status: out is NULL");
    cudaError_t e = cudaMemcpyFromSymbol(status, g_zero1_status, sizeof(uint32_t));
    if (e == cudaSuccess && clear) {
        const uint32_t zero = 0;
        e = cudaMemcpyToSymbol(g_zero1_status, &zero, sizeof(uint32_t));
    }
    if (e != cudaSuccess) return z1_fail(ZERO1_ECUDA, "device status: %s", cudaGetErrorString(e));
    return ZERO1_OK;
}

extern "C" int zero1_checksum(const void *data, int64_t nbytes, uint64_t *out, zero1_stream_t stream)
{
    if (!out) return z1_fail(ZERO1_EINVAL, "checksum: out is NULL");
    if (((uintptr_t)out & 7u) != 0) return z1_fail(ZERO1_EALIGN, "checksum: out is not 8-byte aligned");
    if (nbytes < 0 || (nbytes & 1)) return z1_fail(ZERO1_EINVAL, "checksum: %lld bytes is not a whole number of "
                                                   "16-bit units", (long long)nbytes);
    if (nbytes > 0 && !data) return z1_fail(ZERO1_EINVAL, "checksum: data is NULL");
    int rc;
    if ((rc = check_natural(data, 2, "checksum data")) != ZERO1_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(out, 0, 2 * sizeof(uint64_t), st);
    if (e != cudaSuccess) return z1_fail(ZERO1_ECUDA, "checksum: clearing out: %s", cudaGetErrorString(e));
    const int64_t U = nbytes / 2;
    if (U == 0) return ZERO1_OK;
    const ArrayRef arr[1] = {{data, 2}};
    const Walk w = make_walk(U, U, arr, 1);
    const int grid = grid_for(k_checksum16, work_of(w));
    k_checksum16<<<grid, kBlock, 0, st>>>(static_cast<const uint16_t *>(data), w,
                                         reinterpret_cast<unsigned long long *>(out));
    return launch_status("checksum launch");
}
