// zero1_fused.cu - the fused ZeRO-1 step: reduce-scatter of the M replicas'
// gradients, AdamW on the shard and all-gather of the bf16 parameters in one
// pass ("CS336 Lecture 7: Parallelism 1", ZeRO Stage 1; naive-DP equation for
// the 1/B mean; 16 bytes/parameter table for the dtypes).
//
//   M x 2 B bf16 gradient reads  ->  fp32 rank-order sum  ->  x 1/(B*S)
//   12 B fp32 master/m/v read    ->  AdamW in registers   ->  12 B written
//                                ->  bf16 parameter, 2 B written once
//
// 2M + 26 bytes per parameter, bound by HBM bandwidth.  Three kernels, chosen
// per call: for M <= 8 one vector of loads per thread, in the launch shape
// fused_shape gives for M (at full occupancy on small ranges); replicas in
// groups of 8 for M > 8; and four vectors of state loads in flight when
// master/m/v live in host memory.  Arithmetic uses the explicit
// round-to-nearest intrinsics (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn):
// no contraction, IEEE division and square root, so the results are
// reproducible bit for bit.

#include "zero1_device.cuh"
#include "zero1_checks.h"

namespace {

// One 8-element vector of the fused step for M = MT <= 8 whose gradient and
// state loads are in x.
template <int MT>
__device__ __forceinline__ void fused_vec(int64_t j, const VecLoads<MT> &x, float *master, float *mom, float *var,
                                          uint16_t *params, const Z1Consts &c, bool &bad, bool w32)
{
    float s[kVec];
    unpack8(x.q[0], s);
#pragma unroll
    for (int r = 1; r < MT; ++r) add8(x.q[r], s);
    store_vec(s, x.w, x.m, x.v, master + j, mom + j, var + j, params + j, c, bad, w32 && kWideStoresInPlace);
}

// The fused reduce-scatter + AdamW + all-gather for M <= 8 (M = MT known at
// compile time): one vector of loads per thread and iteration, at most 64
// registers.  On a large range the grid has the shape fused_shape gives for
// M (warps per SM and block size, measured); on a small range (at most
// kSmallMaxVec vectors) it runs at its full occupancy, where the chain of
// dependent iterations per thread, not bandwidth, sets the time.  fp32 state
// is read with L1::no_allocate and every store is .cs.
constexpr int64_t kSmallMaxVec = 1 << 18;  // 2M elements

template <int MT>
__global__ void __launch_bounds__(kBlock, 4)
k_fused_step(const __grid_constant__ GradPtrs g, int M, float *__restrict__ master,
             float *__restrict__ mom, float *__restrict__ var, uint16_t *__restrict__ params,
             const Walk w, const Z1Consts c, uint32_t *flag, int skip)
{
    wait_prior_grid();
    if (skip && *reinterpret_cast<volatile uint32_t *>(flag) != 0u) return;
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    bool bad = false;
    const bool w32 = w.w32 != 0;
    for (int64_t i = tid; i < w.nvec; i += nthr) {
        const int64_t j = w.head + i * kVec;
        VecLoads<MT> x;
        x.load(g, master, mom, var, j, w32);
        fused_vec<MT>(j, x, master, mom, var, params, c, bad, w32);
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
    wait_prior_grid();
    if (skip && *reinterpret_cast<volatile uint32_t *>(flag) != 0u) return;
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    bool bad = false;
    const bool w32 = w.w32 != 0;
    for (int64_t i = tid; i < w.nvec; i += nthr) {
        const int64_t j = w.head + i * kVec;
        const F8 sw = ld_plain8(master + j, w32), sm = ld_plain8(mom + j, w32), sv = ld_plain8(var + j, w32);
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
        store_vec(s, sw, sm, sv, master + j, mom + j, var + j, params + j, c, bad, w32 && kWideStoresInPlace);
    }
    fused_scalar_rest(g, M, master, mom, var, params, w, c, tid, nthr, bad);
    if (flag && !skip) warp_flag(flag, bad);
}

// The fused step when master/m/v live in host memory (optimizer-state
// offload over NVLink-C2C, read and written by the kernel itself).  The host
// link needs many bytes in flight: each thread issues the state loads of
// kOffloadDepth vectors (grid-strided) before computing any of them, and the
// gradients (in HBM) are loaded per vector.  The state goes back in 32-byte
// stores, so that each warp store writes whole 128-byte lines of host memory.
// Measured on GB300 (one box each, 124M parameters, M = 8): 16.2 ms per step
// with four vectors in flight against 21-24 ms with one (six: 14.0 against
// 13.6 ms); 16-byte stores 13.6 ms, 32-byte stores 8.9 ms, 0.98 of the host
// link's bound, ahead of the copy-engine staged step (9.6 ms).
constexpr int kOffloadDepth = 4;

template <int MT>
__global__ void __launch_bounds__(kBlock, 1)
k_fused_step_offload(const __grid_constant__ GradPtrs g, int M, float *__restrict__ master,
                     float *__restrict__ mom, float *__restrict__ var, uint16_t *__restrict__ params,
                     const Walk w, const Z1Consts c, uint32_t *flag, int skip)
{
    wait_prior_grid();
    if (skip && *reinterpret_cast<volatile uint32_t *>(flag) != 0u) return;
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    bool bad = false;
    const bool w32 = w.w32 != 0;
    for (int64_t i0 = tid; i0 < w.nvec; i0 += kOffloadDepth * nthr) {
        F8 st[kOffloadDepth][3];
#pragma unroll
        for (int u = 0; u < kOffloadDepth; ++u) {
            const int64_t i = i0 + u * nthr;
            if (i < w.nvec) {
                const int64_t j = w.head + i * kVec;
                st[u][0] = ld_state8(master + j, w32);
                st[u][1] = ld_state8(mom + j, w32);
                st[u][2] = ld_state8(var + j, w32);
            }
        }
#pragma unroll
        for (int u = 0; u < kOffloadDepth; ++u) {
            const int64_t i = i0 + u * nthr;
            if (i < w.nvec) {
                const int64_t j = w.head + i * kVec;
                float s[kVec];
                sum8<MT>(g, M, j, s);
                store_vec(s, st[u][0], st[u][1], st[u][2], master + j, mom + j, var + j, params + j, c, bad, w32);
            }
        }
    }
    fused_scalar_rest(g, M, master, mom, var, params, w, c, tid, nthr, bad);
    if (flag && !skip) warp_flag(flag, bad);
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
    const Extent out[4] = {{master, L * 4, "master"}, {m, L * 4, "m"}, {v, L * 4, "v"}, {params, nv * 2, "params"}};
    if ((rc = check_disjoint(out, 4, g, plan->M, nv, what)) != ZERO1_OK) return rc;
    ArrayRef arr[ZERO1_MAX_REPLICAS + 4] = {{master, 4}, {m, 4}, {v, 4}, {params, 2}};
    for (int k = 0; k < plan->M; ++k) arr[4 + k] = {g.p[k], 2};
    const Walk w = make_walk(L, nv, arr, 4 + plan->M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint16_t *pp = static_cast<uint16_t *>(params);
    const int M = plan->M;
    const int skip = skip_if_flag ? 1 : 0;
    // programmatic dependent launch: consecutive calls (buckets, chunks)
    // overlap each launch with the end of the kernel before it
    cudaError_t e = cudaSuccess;
    if (in_host_memory(master)) {
        dispatch_m(M, [&](auto mt) {
            constexpr int MT = decltype(mt)::value;
            const int grid = grid_for(k_fused_step_offload<MT>, w);
            e = launch_pdl(k_fused_step_offload<MT>, grid, kBlock, st, g, M, master, m, v, pp, w, c, overflow_flag,
                           skip);
        });
    } else if (M > 8) {
        const int grid = grid_for(k_fused_step_grouped, w);
        e = launch_pdl(k_fused_step_grouped, grid, kBlock, st, g, M, master, m, v, pp, w, c, overflow_flag, skip);
    } else {
        dispatch_m(M, [&](auto mt) {
            constexpr int MT = decltype(mt)::value;
            if constexpr (MT > 0) {
                // small ranges: the kernel's full occupancy; large ones: fused_shape
                constexpr Shape sh = fused_shape(MT);
                static_assert(sh.D == 1, "the fused kernel keeps one vector per thread");
                const bool small = w.nvec <= kSmallMaxVec;
                const int block = small ? kBlock : sh.block;
                const int grid = grid_for(k_fused_step<MT>, w, small ? 0 : sh.per_sm, block);
                e = launch_pdl(k_fused_step<MT>, grid, block, st, g, M, master, m, v, pp, w, c, overflow_flag, skip);
            }
        });
    }
    if (e != cudaSuccess) return pdl_fail(e, what);
    return launch_status(what);
}

}  // namespace

extern "C" int zero1_reduce_scatter_adamw_allgather(const zero1_plan_t *plan, int32_t shard_begin,
                                                    int32_t shard_end, const void *const *grads,
                                                    float *master, float *m, float *v, void *params,
                                                    const zero1_adamw_t *hp, uint32_t *overflow_flag,
                                                    int32_t skip_if_flag, zero1_stream_t stream)
{
    Z1Trace trace("zero1_reduce_scatter_adamw_allgather");
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
    Z1Trace trace("zero1_step_bucket");
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

