// zero1_tma.cu - the fused step staged through shared memory by the Tensor
// Memory Accelerator (bulk copies counted on mbarriers), kept to reproduce
// the design comparison with the direct loads of zero1_fused.cu.

#include "zero1_device.cuh"
#include "zero1_checks.h"

namespace {

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
// if it has not completed within limit_ns of %globaltimer, or within
// kWaitPolls polls should the timer not advance.
constexpr uint64_t kWaitPolls = 1ull << 24;

__device__ __forceinline__ bool mbar_wait(uint64_t *b, uint32_t parity, uint64_t limit_ns = kWaitNs)
{
    if (mbar_try(b, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint64_t polls = 1; !mbar_try(b, parity); ++polls) {
        if (global_ns() - t0 > limit_ns || polls >= kWaitPolls) {
            atomicOr(&g_zero1_status, 1u);
            return false;
        }
    }
    return true;
}

// Self-test of the bounded wait: a barrier that expects two arrivals gets
// one, so its phase never completes; the wait must give up after limit_ns,
// set bit 0 of g_zero1_status and return.  Only shared memory and the status
// word are touched.
__global__ void k_wait_selftest(uint64_t limit_ns, uint32_t *gave_up)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 2);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    mbar_arrive(&bar);
    *gave_up = mbar_wait(&bar, 0, limit_ns) ? 0u : 1u;
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

}  // namespace

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
    Z1Trace trace("zero1_step_tma");
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


extern "C" int zero1_bounded_wait_selftest(uint32_t limit_us, uint32_t *gave_up, zero1_stream_t stream)
{
    Z1Trace trace("zero1_bounded_wait_selftest");
    if (limit_us < 1 || limit_us > 1000000)
        return z1_fail(ZERO1_EINVAL, "wait self-test: limit of %u us not in [1, 1000000]", limit_us);
    if (!gave_up) return z1_fail(ZERO1_EINVAL, "wait self-test: gave_up is NULL");
    int rc;
    if ((rc = check_natural(gave_up, 4, "gave_up")) != ZERO1_OK) return rc;
    k_wait_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>((uint64_t)limit_us * 1000ull, gave_up);
    return launch_status("wait self-test launch");
}
