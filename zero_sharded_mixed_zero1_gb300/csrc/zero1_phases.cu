// zero1_phases.cu - the step's phases as separate kernels, and the naive
// data-parallel All-Reduce ("CS336 Lecture 7: Parallelism 1": the five
// collectives and All-Reduce == Reduce-Scatter + All-Gather): the overflow
// check, AdamW from a scaled fp32 gradient, the all-gather of the updated
// shard, the all-gather of bf16 shards into M outputs and the All-Reduce.
// (The reduce-scatter kernel itself is in zero1_device.cuh: the dynamic step
// uses it too.)

#include "zero1_device.cuh"
#include "zero1_checks.h"

namespace {

// Overflow check: flag |= any non-finite rank-order sum over real elements.
// A pure read stream: one vector in flight per thread at the compiler's
// register budget (5 blocks per SM) measured faster here than the two-deep
// pipeline (7196 vs 6952 GB/s at M = 8); the M > 8 grouped path keeps three
// blocks per SM (7422 GB/s at M = 64).
template <int MT>
__global__ void __launch_bounds__(kBlock, (MT) > 0 ? 5 : 3)
k_overflow(const __grid_constant__ GradPtrs g, int M, const Walk w, uint32_t *flag)
{
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
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

// Blocks per SM of k_overflow's grid for M = MT (0: as many as fit, five for
// M <= 8).  Measured on GB300, 124M elements, fraction of the measured copy
// bandwidth at the full occupancy against this cap: M = 6 1.066 against 1.080
// (four), M = 7 1.066 against 1.079 (three), M = 8 1.066 against 1.087
// (three); for M <= 5 and M > 8 the full occupancy was fastest.
constexpr int overflow_per_sm(int MT)
{
    return MT == 6 ? 4 : (MT == 7 || MT == 8 ? 3 : 0);
}

// D = 2: two resident blocks per SM (at most 128 registers), measured 1.5 %
// faster for the unfused chain than one block of 138 registers; D = 1: one
// vector per thread at most 64 registers.
template <int D>
__global__ void __launch_bounds__(kBlock, D == 1 ? 4 : 2)
k_adamw(const float *__restrict__ gin, float *__restrict__ master, float *__restrict__ mom,
        float *__restrict__ var, const Walk w, const Z1Consts c)
{
    wait_prior_grid();
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    const bool w32 = w.w32 != 0;
    pipelined<StateLoads, D>(
        w.nvec, tid, nthr,
        [&](StateLoads &x, int64_t i) { load_state_vec(x, gin, master, mom, var, w.head + i * kVec, w32); },
        [&](const StateLoads &x, int64_t i) {
            const int64_t j = w.head + i * kVec;
            float gg[kVec], ww[kVec], mm[kVec], vv[kVec];
            unpack_f8(x.g, gg);
            unpack_f8(x.w, ww);
            unpack_f8(x.m, mm);
            unpack_f8(x.v, vv);
#pragma unroll
            for (int k = 0; k < kVec; ++k) adamw1(gg[k], c, ww[k], mm[k], vv[k]);
            st_stream8(master + j, ww, w32);
            st_stream8(mom + j, mm, w32);
            st_stream8(var + j, vv, w32);
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
template <int D>
__global__ void __launch_bounds__(kBlock, D == 1 ? 4 : 1)
k_all_gather(const float *__restrict__ master, uint16_t *__restrict__ params, const Walk w)
{
    wait_prior_grid();
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    const bool w32 = w.w32 != 0;
    pipelined<F8, D>(
        w.nvec, tid, nthr, [&](F8 &x, int64_t i) { x = ld_cs8(master + w.head + i * kVec, w32); },
        [&](const F8 &x, int64_t i) {
            __stcs(reinterpret_cast<uint4 *>(params + w.head + i * kVec),
                   make_uint4(pack_bf16x2(x.lo.x, x.lo.y), pack_bf16x2(x.lo.z, x.lo.w),
                              pack_bf16x2(x.hi.x, x.hi.y), pack_bf16x2(x.hi.z, x.hi.w)));
        });
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        if (j < w.nv) params[j] = to_bf16(master[j]);
    }
}

// Launch shapes of k_adamw and k_all_gather.  Measured on GB300, 124M
// elements, fraction of the measured copy bandwidth: k_adamw two-deep at two
// blocks of 256 per SM 0.952, one vector at 12, 16, 18, 20, 24, 32 warps per
// SM 0.845, 0.973, 1.007, 1.000, 0.949, 0.921 (18: three blocks of 192, 20:
// five blocks of 128); k_all_gather two-deep at its full occupancy 0.998,
// one vector at 12-32 warps per SM 0.62-0.98.
constexpr Shape kAdamwShape{1, 3, 192};
constexpr Shape kAllGatherShape{2, 0};

// All-gather of bf16 shards into M outputs (real elements only).
__global__ void __launch_bounds__(kBlock)
k_all_gather_shards(const uint16_t *__restrict__ shards, const __grid_constant__ OutPtrs o, int M,
                    const Walk w)
{
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
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
__device__ __forceinline__ void ar_store(const OutPtrs &o, int M, int64_t j, float s[kVec], float scale, bool w32)
{
#pragma unroll
    for (int k = 0; k < kVec; ++k) s[k] = __fmul_rn(s[k], scale);
    if constexpr (BF16) {
        const uint4 q = make_uint4(pack_bf16x2(s[0], s[1]), pack_bf16x2(s[2], s[3]), pack_bf16x2(s[4], s[5]),
                                   pack_bf16x2(s[6], s[7]));
        for (int r = 0; r < M; ++r) __stcs(reinterpret_cast<uint4 *>(static_cast<uint16_t *>(o.p[r]) + j), q);
    } else {
        for (int r = 0; r < M; ++r) st_stream8(static_cast<float *>(o.p[r]) + j, s, w32);
    }
}

// The all-reduce body.  NC: the gradients are read through the read-only
// (non-coherent) path, which is allowed only while no buffer this kernel
// writes overlaps them; an in-place call (an output aliasing an input) runs
// the coherent instance, which reads them with ordinary global loads.
template <int MT, bool BF16, bool NC, int D>
__device__ __forceinline__ void allreduce_body(const GradPtrs &g, const OutPtrs &o, int M, const Walk &w,
                                               float scale)
{
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    const bool w32 = w.w32 != 0;
    if constexpr (MT > 0) {
        // in place, the next vector's loads touch other elements than the
        // current vector's stores, so prefetching them stays correct
        pipelined<GradLoads<MT>, D>(
            w.nvec, tid, nthr,
            [&](GradLoads<MT> &x, int64_t i) {
                const int64_t j = w.head + i * kVec;
#pragma unroll
                for (int r = 0; r < MT; ++r) x.q[r] = ld_grad_u4<NC>(g.p[r] + j);
            },
            [&](const GradLoads<MT> &x, int64_t i) {
                float s[kVec];
                unpack8(x.q[0], s);
#pragma unroll
                for (int r = 1; r < MT; ++r) add8(x.q[r], s);
                ar_store<BF16>(o, MT, w.head + i * kVec, s, scale, w32);
            });
    } else {
        for (int64_t i = tid; i < w.nvec; i += nthr) {
            const int64_t j = w.head + i * kVec;
            float s[kVec];
            sum8<0, NC>(g, M, j, s);
            ar_store<BF16>(o, M, j, s, scale, w32);
        }
    }
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        const float s = __fmul_rn(sum1<NC>(g, M, j), scale);
        for (int r = 0; r < M; ++r) {
            if constexpr (BF16) static_cast<uint16_t *>(o.p[r])[j] = to_bf16(s);
            else static_cast<float *>(o.p[r])[j] = s;
        }
    }
}

// Separate outputs: gradients through the read-only path.
template <int MT, bool BF16, int D>
__global__ void Z1_BOUNDS(MT, D)
k_allreduce(const __grid_constant__ GradPtrs g, const __grid_constant__ OutPtrs o, int M,
            const Walk w, float scale)
{
    allreduce_body<MT, BF16, true, D>(g, o, M, w, scale);
}

// In place (bf16 outputs overlapping the inputs): coherent loads.
template <int MT, int D>
__global__ void Z1_BOUNDS(MT, D)
k_allreduce_inplace(const __grid_constant__ GradPtrs g, const __grid_constant__ OutPtrs o, int M,
                    const Walk w, float scale)
{
    allreduce_body<MT, true, false, D>(g, o, M, w, scale);
}

// Launch shapes of the all-reduce kernels for M = MT (MT = 0: M > 8, where D
// is not used), with separate outputs and in place.  Measured on GB300, bf16
// outputs, 124M elements, M = 1..8, fraction of the measured copy bandwidth:
// separate outputs two-deep 0.761 0.951 0.948 0.940 0.933 0.944 0.941 0.952,
// this table 0.924 0.957 0.970 0.971 0.967 0.976 0.961 0.979; in place
// two-deep 0.788 0.963 0.954 0.942 0.939 0.944 0.935 0.956, this table 0.777
// 0.960 0.966 0.977 0.974 0.982 0.967 0.984.  The one-vector grids tried were
// 12, 16, 18, 20, 24 and 32 warps per SM (blocks of 128, 192 or 256); the
// best differs by M, reproducibly across boxes (at M = 5, 18 warps measured
// 0.8 % and, in place, 0.5 % above 16).  M > 8 (16M elements): two blocks of 256
// per SM 0.942 at M = 16 and 0.948 at M = 64, against 0.922 and 0.929 at the
// kernel's occupancy of three.
constexpr Shape allreduce_shape(int MT)
{
    switch (MT) {
    case 1: return Shape{1, 3};
    case 2: case 4: return Shape{1, 5, 128};
    case 3: case 6: return Shape{1, 2};
    case 5: return Shape{1, 3, 192};
    case 7: case 8: return Shape{1, 3, 128};
    case 0: return Shape{2, 2};
    default: return Shape{2, 0};
    }
}

constexpr Shape allreduce_inplace_shape(int MT)
{
    switch (MT) {
    case 3: return Shape{1, 3};
    case 4: return Shape{1, 5, 128};
    case 5: return Shape{1, 3, 192};
    case 6: return Shape{1, 2};
    case 7: case 8: return Shape{1, 3, 128};
    case 0: return Shape{2, 2};
    default: return Shape{2, 0};
    }
}

}  // namespace

extern "C" int zero1_overflow_check(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                    const void *const *grads, uint32_t *flag, zero1_stream_t stream)
{
    Z1Trace trace("zero1_overflow_check");
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    if (!flag) return z1_fail(ZERO1_EINVAL, "overflow check: flag is NULL");
    if ((rc = check_natural(flag, 4, "flag")) != ZERO1_OK) return rc;
    if (r.nv == 0) return ZERO1_OK;
    GradPtrs g{};
    if ((rc = load_grads(plan, grads, &g, "overflow check")) != ZERO1_OK) return rc;
    ArrayRef arr[ZERO1_MAX_REPLICAS] = {};
    for (int k = 0; k < plan->M; ++k) arr[k] = {grads[k], 2};
    const Walk w = make_walk(r.nv, r.nv, arr, plan->M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int M = plan->M;
    dispatch_m(M, [&](auto mt) {
        constexpr int MT = decltype(mt)::value;
        const int grid = grid_for(k_overflow<MT>, w, overflow_per_sm(MT));
        k_overflow<MT><<<grid, kBlock, 0, st>>>(g, M, w, flag);
    });
    return launch_status("overflow check launch");
}

extern "C" int dp_allreduce(const zero1_plan_t *plan, const void *const *grads_in, void *const *outs,
                            float scale, int32_t out_dtype, zero1_stream_t stream)
{
    Z1Trace trace("dp_allreduce");
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
    ArrayRef arr[2 * ZERO1_MAX_REPLICAS] = {};
    bool overlap = false;  // some output overlaps some input
    for (int k = 0; k < M; ++k) {
        if (!outs[k]) return z1_fail(ZERO1_EINVAL, "all-reduce: outs[%d] is NULL", k);
        if ((rc = check_natural(outs[k], osz, "an all-reduce output")) != ZERO1_OK) return rc;
        const uintptr_t a = (uintptr_t)outs[k], b = a + (uintptr_t)plan->n * osz;
        for (int q = 0; q < M; ++q) {
            const uintptr_t c0 = (uintptr_t)grads_in[q], c1 = c0 + (uintptr_t)plan->n * 2;
            if (a < c1 && c0 < b) {
                if (osz == 4) return z1_fail(ZERO1_EINVAL, "all-reduce: fp32 output %d overlaps input %d", k, q);
                overlap = true;
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
        constexpr Shape sh = allreduce_shape(MT), ish = allreduce_inplace_shape(MT);
        static_assert(shape_ok(sh) && shape_ok(ish), "all-reduce shapes");
        if (osz == 2 && overlap) {
            const int grid = grid_for(k_allreduce_inplace<MT, ish.D>, w, ish.per_sm, ish.block);
            k_allreduce_inplace<MT, ish.D><<<grid, ish.block, 0, st>>>(g, o, M, w, scale);
        } else if (osz == 2) {
            const int grid = grid_for(k_allreduce<MT, true, sh.D>, w, sh.per_sm, sh.block);
            k_allreduce<MT, true, sh.D><<<grid, sh.block, 0, st>>>(g, o, M, w, scale);
        } else {
            const int grid = grid_for(k_allreduce<MT, false, sh.D>, w, sh.per_sm, sh.block);
            k_allreduce<MT, false, sh.D><<<grid, sh.block, 0, st>>>(g, o, M, w, scale);
        }
    });
    return launch_status("all-reduce launch");
}

extern "C" int zero1_reduce_scatter(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                    const void *const *grads, float scale, int32_t out_dtype, void *out,
                                    uint32_t *flag, zero1_stream_t stream)
{
    Z1Trace trace("zero1_reduce_scatter");
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
    const Extent outs[2] = {{out, r.L * osz, "out"}, {flag, 4, "flag"}};
    if ((rc = check_disjoint(outs, 2, g, plan->M, r.nv, "reduce-scatter")) != ZERO1_OK) return rc;
    ArrayRef arr[ZERO1_MAX_REPLICAS + 1] = {{out, osz}};
    for (int k = 0; k < plan->M; ++k) arr[1 + k] = {g.p[k], 2};
    const Walk w = make_walk(r.L, r.nv, arr, 1 + plan->M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int M = plan->M;
    dispatch_m(M, [&](auto mt) {
        constexpr int MT = decltype(mt)::value;
        constexpr Shape sh = rs_shape(MT);
        static_assert(shape_ok(sh), "reduce-scatter shape");
        if (osz == 2) {
            const int grid = grid_for(k_reduce_scatter<MT, true, sh.D>, w, sh.per_sm, sh.block);
            k_reduce_scatter<MT, true, sh.D><<<grid, sh.block, 0, st>>>(g, M, w, scale, out, flag);
        } else {
            const int grid = grid_for(k_reduce_scatter<MT, false, sh.D>, w, sh.per_sm, sh.block);
            k_reduce_scatter<MT, false, sh.D><<<grid, sh.block, 0, st>>>(g, M, w, scale, out, flag);
        }
    });
    return launch_status("reduce-scatter launch");
}

extern "C" int zero1_adamw_update(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                  const float *gin, float *master, float *m, float *v,
                                  const zero1_adamw_t *hp, zero1_stream_t stream)
{
    Z1Trace trace("zero1_adamw_update");
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    Z1Consts c;
    if ((rc = z1_adamw_constants(hp, plan->M, &c)) != ZERO1_OK) return rc;
    if (!gin || !master || !m || !v) return z1_fail(ZERO1_EINVAL, "adamw: NULL array");
    if ((rc = check_natural(gin, 4, "g")) || (rc = check_natural(master, 4, "master")) ||
        (rc = check_natural(m, 4, "m")) || (rc = check_natural(v, 4, "v")))
        return rc;
    const Extent bufs[4] = {{gin, r.L * 4, "g"}, {master, r.L * 4, "master"}, {m, r.L * 4, "m"}, {v, r.L * 4, "v"}};
    if ((rc = check_disjoint(bufs, 4, GradPtrs{}, 0, 0, "adamw")) != ZERO1_OK) return rc;
    const ArrayRef arr[4] = {{gin, 4}, {master, 4}, {m, 4}, {v, 4}};
    // every element of the range is updated: walk it as if all were real
    const Walk w = make_walk(r.L, r.L, arr, 4);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    static_assert(shape_ok(kAdamwShape), "AdamW shape");
    const int grid = grid_for(k_adamw<kAdamwShape.D>, w, kAdamwShape.per_sm, kAdamwShape.block);
    const cudaError_t e = launch_pdl(k_adamw<kAdamwShape.D>, grid, kAdamwShape.block, st, gin, master, m, v, w, c);
    if (e != cudaSuccess) return pdl_fail(e, "adamw launch");
    return launch_status("adamw launch");
}

extern "C" int zero1_all_gather(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                const float *master, void *params, zero1_stream_t stream)
{
    Z1Trace trace("zero1_all_gather");
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    if (r.nv == 0) return ZERO1_OK;
    if (!master || !params) return z1_fail(ZERO1_EINVAL, "all-gather: NULL array");
    if ((rc = check_natural(master, 4, "master")) || (rc = check_natural(params, 2, "params"))) return rc;
    const Extent bufs[2] = {{master, r.nv * 4, "master"}, {params, r.nv * 2, "params"}};
    if ((rc = check_disjoint(bufs, 2, GradPtrs{}, 0, 0, "all-gather")) != ZERO1_OK) return rc;
    const ArrayRef arr[2] = {{master, 4}, {params, 2}};
    const Walk w = make_walk(r.nv, r.nv, arr, 2);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    static_assert(shape_ok(kAllGatherShape), "all-gather shape");
    const int grid = grid_for(k_all_gather<kAllGatherShape.D>, w, kAllGatherShape.per_sm, kAllGatherShape.block);
    const cudaError_t e = launch_pdl(k_all_gather<kAllGatherShape.D>, grid, kAllGatherShape.block, st, master,
                                     static_cast<uint16_t *>(params), w);
    if (e != cudaSuccess) return pdl_fail(e, "all-gather launch");
    return launch_status("all-gather launch");
}

extern "C" int zero1_all_gather_shards(const zero1_plan_t *plan, const void *shards, void *const *outs,
                                       zero1_stream_t stream)
{
    Z1Trace trace("zero1_all_gather_shards");
    int rc = z1_check_plan(plan);
    if (rc != ZERO1_OK) return rc;
    if (!shards || !outs) return z1_fail(ZERO1_EINVAL, "all-gather shards: NULL argument");
    if ((rc = check_natural(shards, 2, "shards")) != ZERO1_OK) return rc;
    OutPtrs o{};
    ArrayRef arr[ZERO1_MAX_REPLICAS + 1] = {{shards, 2}};
    for (int k = 0; k < plan->M; ++k) {
        if (!outs[k]) return z1_fail(ZERO1_EINVAL, "all-gather shards: outs[%d] is NULL", k);
        if ((rc = check_natural(outs[k], 2, "an all-gather output")) != ZERO1_OK) return rc;
        if (overlap({shards, plan->padded_n * 2, "shards"}, {outs[k], plan->n * 2, "an output"}))
            return z1_fail(ZERO1_EINVAL, "all-gather shards: outs[%d] overlaps the shards", k);
        o.p[k] = outs[k];
        arr[1 + k] = {outs[k], 2};
    }
    const Walk w = make_walk(plan->n, plan->n, arr, 1 + plan->M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int grid = grid_for(k_all_gather_shards, w);
    k_all_gather_shards<<<grid, kBlock, 0, st>>>(static_cast<const uint16_t *>(shards), o, plan->M, w);
    return launch_status("all-gather shards launch");
}

