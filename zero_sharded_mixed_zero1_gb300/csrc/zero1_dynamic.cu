// zero1_dynamic.cu - dynamic loss scaling with the step's skip decided on the
// device ("五维并行实战" 4.2: the fp16 block's loss_scale 0, initial_scale_power,
// loss_scale_window, hysteresis, min_loss_scale; 3.2 trap 3), and the same
// step for callers that cannot allocate device memory.

#include <mutex>

#include "zero1_device.cuh"
#include "zero1_checks.h"

namespace {

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
    sc->current = 0u;
    derive_constants(sc, B, beta1, beta2);
}

// Advance the scaler after an attempt (reads the attempt's flag, clears it).
// With ping-pong state a clean attempt also makes the buffer it wrote the
// current one.
__global__ void k_scaler_update(zero1_scaler_t *sc, const ScalePolicy pol, int64_t B, float beta1, float beta2,
                                int pingpong)
{
    wait_prior_grid();
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    sc->attempts += 1;
    const bool overflow = *reinterpret_cast<volatile uint32_t *>(&sc->overflow) != 0u;
    if (pingpong && !overflow) sc->current ^= 1u;
    if (overflow) {
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
// D = 2: two resident blocks per SM (at most 128 registers), measured
// 0.8-1.4 % faster for the whole dynamic step than one block with 144
// registers; D = 1: one vector per thread at most 64 registers.
template <int D>
__global__ void __launch_bounds__(kBlock, D == 1 ? 4 : 2)
k_apply_sums(const float *__restrict__ sums, float *__restrict__ master, float *__restrict__ mom,
             float *__restrict__ var, uint16_t *__restrict__ params, const Walk w, Z1Consts c,
             const zero1_scaler_t *sc)
{
    wait_prior_grid();
    if (*reinterpret_cast<const volatile uint32_t *>(&sc->overflow) != 0u) return;
    c.inv = sc->inv;
    c.bc1 = sc->bc1;
    c.bc2 = sc->bc2;
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    bool bad = false;  // the flag was already taken by the reduce-scatter
    const bool w32 = w.w32 != 0;
    pipelined<StateLoads, D>(
        w.nvec, tid, nthr,
        [&](StateLoads &x, int64_t i) { load_state_vec(x, sums, master, mom, var, w.head + i * kVec, w32); },
        [&](const StateLoads &x, int64_t i) {
            const int64_t j = w.head + i * kVec;
            float s[kVec];
            unpack_f8(x.g, s);
            store_vec(s, x.w, x.m, x.v, master + j, mom + j, var + j, params + j, c, bad, w32);
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

// Launch shape of k_apply_sums (which reads no gradients).  Measured on
// GB300, the whole dynamic step on 124M elements, M = 1..8, fraction of the
// measured copy bandwidth: 0.928-0.953 with both of its kernels two-deep,
// 0.982-0.998 with this shape (and rs_shape's), 0.915-0.952 with both one
// vector per thread at three or four blocks per SM.
constexpr Shape kApplyShape{1, 2};

// k_apply_sums when master/m/v live in host memory: two vectors in flight per
// thread at the kernel's occupancy.  Measured on GB300 against kApplyShape on
// one box (the dynamic step on host-resident state, M = 8, two runs each):
// 9.16-9.18 against 9.28-9.29 ms at 124M elements, 64.5-64.8 against
// 64.9-65.1 ms on the Llama layers.
constexpr Shape kApplyHostShape{2, 0};

// --------------------------------------------------- ping-pong state ------
//
// The dynamic step in one pass over the data: master/m/v exist twice, and
// scaler->current says which copy holds the current state.  An attempt reads
// the current copy and writes the updated state into the other one, so an
// attempt whose gradients overflow has changed nothing that is current: the
// scaler update simply does not switch copies.  The bf16 parameters (one
// copy) are written by the attempt and, if it overflowed, rewritten from the
// current master by k_restore_params.  Traffic per element is the fused
// step's 2M + 26 bytes instead of the two-pass 2M + 34.

struct PingPong {
    float *master[2], *mom[2], *var[2];
};

// One attempt for M <= 8 (MT = M, D vectors of loads in flight per thread,
// pingpong_shape) or M > 8 (MT = 0, replicas in groups of 8).  For M > 8, measured on the
// 64-replica shard: state read with the default policy at two blocks per SM
// (107 registers) beat three blocks per SM, whose 85-register cap spilled
// (2.64 against 2.75-2.85 ms).
// The body for a copy index known at compile time: every pointer is then a
// kernel parameter, which the compiler can reload instead of holding it in a
// register (169 registers at M = 8 against 179 with the copy picked at run
// time; the same speed on the same box).
template <int MT, int CUR, int D>
__device__ __forceinline__ void pingpong_body(const GradPtrs &g, int M, const PingPong &s,
                                              uint16_t *__restrict__ params, const Walk &w, const Z1Consts &c,
                                              zero1_scaler_t *sc)
{
    const float *__restrict__ sw = s.master[CUR];
    const float *__restrict__ sm = s.mom[CUR];
    const float *__restrict__ sv = s.var[CUR];
    float *__restrict__ dw = s.master[CUR ^ 1];
    float *__restrict__ dm = s.mom[CUR ^ 1];
    float *__restrict__ dv = s.var[CUR ^ 1];
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    bool bad = false;
    const bool w32 = w.w32 != 0;
    if constexpr (MT > 0) {
        pipelined<VecLoads<MT>, D>(
            w.nvec, tid, nthr,
            [&](VecLoads<MT> &x, int64_t i) { x.load(g, sw, sm, sv, w.head + i * kVec, w32); },
            [&](const VecLoads<MT> &x, int64_t i) {
                const int64_t j = w.head + i * kVec;
                float sum[kVec];
                unpack8(x.q[0], sum);
#pragma unroll
                for (int r = 1; r < MT; ++r) add8(x.q[r], sum);
                store_vec(sum, x.w, x.m, x.v, dw + j, dm + j, dv + j, params + j, c, bad, w32);
            });
    } else {
        for (int64_t i = tid; i < w.nvec; i += nthr) {
            const int64_t j = w.head + i * kVec;
            const F8 xw = ld_plain8(sw + j, w32), xm = ld_plain8(sm + j, w32), xv = ld_plain8(sv + j, w32);
            float sum[kVec];
            sum8<0>(g, M, j, sum);
            store_vec(sum, xw, xm, xv, dw + j, dm + j, dv + j, params + j, c, bad, w32);
        }
    }
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        float gs = 0.0f;
        if (j < w.nv) {
            gs = sum1(g, M, j);
            bad |= !finite(gs);
        }
        float ww = sw[j], mm = sm[j], vv = sv[j];
        adamw1(__fmul_rn(gs, c.inv), c, ww, mm, vv);
        dw[j] = ww;
        dm[j] = mm;
        dv[j] = vv;
        if (j < w.nv) params[j] = to_bf16(ww);
    }
    warp_flag(&sc->overflow, bad);
}

template <int MT, int D>
__global__ void __launch_bounds__(kBlock, MT == 0 ? 2 : (D == 1 ? 4 : (MT <= 2 ? 2 : 1)))
k_fused_step_pingpong(const __grid_constant__ GradPtrs g, int M, const __grid_constant__ PingPong s,
                      uint16_t *__restrict__ params, const Walk w, Z1Consts c, zero1_scaler_t *sc)
{
    wait_prior_grid();
    const uint32_t cur = *reinterpret_cast<const volatile uint32_t *>(&sc->current) & 1u;
    c.inv = sc->inv;
    c.bc1 = sc->bc1;
    c.bc2 = sc->bc2;
    if (cur)
        pingpong_body<MT, 1, D>(g, M, s, params, w, c, sc);
    else
        pingpong_body<MT, 0, D>(g, M, s, params, w, c, sc);
}

// Launch shape of k_fused_step_pingpong for M = MT (MT = 0: M > 8, replicas
// in groups of 8, where D is not used).  Measured on GB300, the ping-pong
// step on 124M elements, fraction of the measured copy bandwidth: two-deep
// 0.909 0.915 0.932 0.951 0.967 0.981 0.992 1.002 for M = 1..8; one vector
// at 18 warps per SM (three blocks of 192) 0.989 0.991 for M = 1, 2 (20
// warps: 0.966 0.955); at 16 warps per SM 0.995 1.006 for M = 3, 4 and, at
// M = 5, 1.003 in blocks of 128 but 0.91 in blocks of 256; at 20 warps per
// SM (five blocks of 128) 1.009 1.014 1.016 for M = 6..8.
constexpr Shape pingpong_shape(int MT)
{
    switch (MT) {
    case 1: case 2: return Shape{1, 3, 192};
    case 3: case 4: return Shape{1, 2};
    case 5: return Shape{1, 4, 128};
    case 0: return Shape{2, 0};
    default: return Shape{1, 5, 128};
    }
}

// The ping-pong kernel's shape when both state copies live in host memory:
// two vectors in flight per thread at the kernel's occupancy.  Measured on
// GB300 against the HBM table's shape on one box (M = 8, three runs each,
// median step): 8.94-8.97 against 9.06-9.15 ms at 124M elements, 94.3-94.4
// against 94.6-95.6 ms at 1.3B, 63.2-63.4 against 63.6-64.0 ms on the Llama
// layers.
constexpr Shape kPingPongHostShape{2, 0};

// The fused step in place, with S and t taken from the scaler, for a range
// whose overflow flag is already final (an overflow pass over all of the
// attempt's gradients ran before it): the kernel returns at once when
// scaler->overflow is set, so an overflowing attempt writes nothing.  The
// staged step with dynamic loss scaling uses it on its HBM slots: there the
// state lives in host memory, where a second copy would cost host memory and
// twice the link traffic.
template <int MT, int D>
__global__ void __launch_bounds__(kBlock, MT == 0 ? 2 : (D == 1 ? 4 : (MT <= 2 ? 2 : 1)))
k_fused_step_scaled(const __grid_constant__ GradPtrs g, int M, float *__restrict__ master,
                    float *__restrict__ mom, float *__restrict__ var, uint16_t *__restrict__ params, const Walk w,
                    Z1Consts c, const zero1_scaler_t *sc)
{
    if (*reinterpret_cast<const volatile uint32_t *>(&sc->overflow) != 0u) return;
    c.inv = sc->inv;
    c.bc1 = sc->bc1;
    c.bc2 = sc->bc2;
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    bool bad = false;  // the flag is final already; nothing is reported
    const bool w32 = w.w32 != 0;
    if constexpr (MT > 0) {
        pipelined<VecLoads<MT>, D>(
            w.nvec, tid, nthr,
            [&](VecLoads<MT> &x, int64_t i) { x.load(g, master, mom, var, w.head + i * kVec, w32); },
            [&](const VecLoads<MT> &x, int64_t i) {
                const int64_t j = w.head + i * kVec;
                float sum[kVec];
                unpack8(x.q[0], sum);
#pragma unroll
                for (int r = 1; r < MT; ++r) add8(x.q[r], sum);
                store_vec(sum, x.w, x.m, x.v, master + j, mom + j, var + j, params + j, c, bad,
                          w32 && kWideStoresInPlace);
            });
    } else {
        for (int64_t i = tid; i < w.nvec; i += nthr) {
            const int64_t j = w.head + i * kVec;
            const F8 xw = ld_plain8(master + j, w32), xm = ld_plain8(mom + j, w32), xv = ld_plain8(var + j, w32);
            float sum[kVec];
            sum8<0>(g, M, j, sum);
            store_vec(sum, xw, xm, xv, master + j, mom + j, var + j, params + j, c, bad, w32 && kWideStoresInPlace);
        }
    }
    fused_scalar_rest(g, M, master, mom, var, params, w, c, tid, nthr, bad);
}

// After an attempt that overflowed, put back params = bf16(current master);
// after a clean attempt, return at once.  Its grid is four blocks per SM:
// the blocks of a clean attempt only start and return, and fewer of them
// cost less, while an overflowing attempt needs enough of them to stream
// the restore.  Measured on GB300, the ping-pong step on 124M elements at
// M = 8 (fraction of the measured copy bandwidth, clean / every attempt
// overflowing): full occupancy 1.002 / 1.001, four blocks per SM 1.003 /
// 1.003, one block per SM 1.006 / 0.875.
constexpr int kRestorePerSm = 4;

__global__ void __launch_bounds__(kBlock)
k_restore_params(const PingPong s, uint16_t *__restrict__ params, const Walk w, const zero1_scaler_t *sc)
{
    wait_prior_grid();
    if (*reinterpret_cast<const volatile uint32_t *>(&sc->overflow) == 0u) return;
    const float *__restrict__ master =
        (*reinterpret_cast<const volatile uint32_t *>(&sc->current) & 1u) ? s.master[1] : s.master[0];
    const int64_t tid = grid_tid();
    const int64_t nthr = grid_threads();
    const bool w32 = w.w32 != 0;
    for (int64_t i = tid; i < w.nvec; i += nthr) {
        const int64_t j = w.head + i * kVec;
        const F8 x = ld_state8(master + j, w32);
        __stcs(reinterpret_cast<uint4 *>(params + j),
               make_uint4(pack_bf16x2(x.lo.x, x.lo.y), pack_bf16x2(x.lo.z, x.lo.w), pack_bf16x2(x.hi.x, x.hi.y),
                          pack_bf16x2(x.hi.z, x.hi.w)));
    }
    const int64_t ns = w.L - w.nvec * kVec;
    for (int64_t q = tid; q < ns; q += nthr) {
        const int64_t j = scalar_index(w, q);
        if (j < w.nv) params[j] = to_bf16(master[j]);
    }
}

}  // namespace

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
    Z1Trace trace("zero1_scaler_init");
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
    Z1Trace trace("zero1_step_dynamic");
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
    const Extent out[6] = {{master, r.L * 4, "master"}, {m, r.L * 4, "m"},   {v, r.L * 4, "v"},
                           {params, r.nv * 2, "params"},  {sums, r.L * 4, "sums"}, {scaler, (int64_t)sizeof(zero1_scaler_t), "the scaler"}};
    if ((rc = check_disjoint(out, 6, g, plan->M, r.nv, "dynamic step")) != ZERO1_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int M = plan->M;
    // 1. reduce-scatter into the fp32 sums, flag into the scaler
    ArrayRef ra[ZERO1_MAX_REPLICAS + 1] = {{sums, 4}};
    for (int k = 0; k < M; ++k) ra[1 + k] = {g.p[k], 2};
    const Walk wr = make_walk(r.L, r.nv, ra, 1 + M);
    uint32_t *flag = &scaler->overflow;
    dispatch_m(M, [&](auto mt) {
        constexpr int MT = decltype(mt)::value;
        constexpr Shape sh = rs_shape(MT);
        static_assert(shape_ok(sh), "reduce-scatter shape");
        const int grid = grid_for(k_reduce_scatter<MT, false, sh.D>, wr, sh.per_sm, sh.block);
        k_reduce_scatter<MT, false, sh.D><<<grid, sh.block, 0, st>>>(g, M, wr, 1.0f, sums, flag);
    });
    // 2. the update from the sums (skipped on overflow)
    const ArrayRef ua[5] = {{sums, 4}, {master, 4}, {m, 4}, {v, 4}, {params, 2}};
    const Walk wu = make_walk(r.L, r.nv, ua, 5);
    static_assert(shape_ok(kApplyShape) && shape_ok(kApplyHostShape), "update-from-sums shapes");
    if ((rc = launch_status("dynamic step: reduce-scatter launch")) != ZERO1_OK) return rc;
    cudaError_t e;
    if (in_host_memory(master)) {
        // the state crosses the host link: the two-deep kernel at its occupancy
        const int grid = grid_for(k_apply_sums<kApplyHostShape.D>, wu, kApplyHostShape.per_sm, kApplyHostShape.block);
        e = launch_pdl(k_apply_sums<kApplyHostShape.D>, grid, kApplyHostShape.block, st, (const float *)sums, master,
                       m, v, static_cast<uint16_t *>(params), wu, c, (const zero1_scaler_t *)scaler);
    } else {
        const int grid = grid_for(k_apply_sums<kApplyShape.D>, wu, kApplyShape.per_sm, kApplyShape.block);
        e = launch_pdl(k_apply_sums<kApplyShape.D>, grid, kApplyShape.block, st, (const float *)sums, master, m, v,
                       static_cast<uint16_t *>(params), wu, c, (const zero1_scaler_t *)scaler);
    }
    if (e != cudaSuccess) return pdl_fail(e, "dynamic step: update launch");
    // 3. the scaler advances (only once the update is enqueued)
    const ScalePolicy pol{policy->factor, policy->window, policy->hysteresis, policy->min_scale};
    const cudaError_t e2 =
        launch_pdl(k_scaler_update, 1, 32, st, scaler, pol, (int64_t)hp->global_batch, hp->beta1, hp->beta2, 0);
    if (e2 != cudaSuccess) return pdl_fail(e2, "dynamic step: scaler launch");
    return launch_status("dynamic step launch");
}

namespace {

// The two copies of master/m/v (host arrays of two device pointers each).
int load_pingpong(float *const *master, float *const *m, float *const *v, PingPong *s, const char *what)
{
    if (!master || !m || !v) return z1_fail(ZERO1_EINVAL, "%s: master, m and v arrays are NULL", what);
    int rc;
    for (int k = 0; k < 2; ++k) {
        if (!master[k] || !m[k] || !v[k])
            return z1_fail(ZERO1_EINVAL, "%s: copy %d of master, m or v is NULL", what, k);
        if ((rc = check_natural(master[k], 4, "master")) || (rc = check_natural(m[k], 4, "m")) ||
            (rc = check_natural(v[k], 4, "v")))
            return rc;
        s->master[k] = master[k];
        s->mom[k] = m[k];
        s->var[k] = v[k];
    }
    if (s->master[0] == s->master[1] || s->mom[0] == s->mom[1] || s->var[0] == s->var[1])
        return z1_fail(ZERO1_EINVAL, "%s: the two copies of master, m or v are the same buffer", what);
    return ZERO1_OK;
}

// Validate and launch the ping-pong kernel over L elements (nv real) whose
// pointers all start at the range's first element.
int launch_pingpong_range(const zero1_plan_t *plan, int64_t L, int64_t nv, const void *const *grads,
                          float *const *master, float *const *m, float *const *v, void *params,
                          const zero1_adamw_t *hp, zero1_scaler_t *scaler, cudaStream_t st, const char *what)
{
    int rc;
    Z1Consts c;
    if ((rc = dynamic_constants(hp, plan->M, &c)) != ZERO1_OK) return rc;
    if ((rc = check_scaler_ptr(scaler)) != ZERO1_OK) return rc;
    PingPong s{};
    if ((rc = load_pingpong(master, m, v, &s, what)) != ZERO1_OK) return rc;
    if (nv > 0 && !params)
        return z1_fail(ZERO1_EINVAL, "%s: params must be non-NULL when the range holds parameters", what);
    if ((rc = check_natural(params, 2, "params")) != ZERO1_OK) return rc;
    GradPtrs g{};
    if (nv > 0 && (rc = load_grads(plan, grads, &g, what)) != ZERO1_OK) return rc;
    const Extent out[8] = {{s.master[0], L * 4, "master[0]"}, {s.mom[0], L * 4, "m[0]"}, {s.var[0], L * 4, "v[0]"},
                           {s.master[1], L * 4, "master[1]"}, {s.mom[1], L * 4, "m[1]"}, {s.var[1], L * 4, "v[1]"},
                           {params, nv * 2, "params"},        {scaler, (int64_t)sizeof(zero1_scaler_t), "the scaler"}};
    if ((rc = check_disjoint(out, 8, g, plan->M, nv, what)) != ZERO1_OK) return rc;
    // one walk serves both copies: they must share the 16-byte phase
    ArrayRef arr[ZERO1_MAX_REPLICAS + 7] = {{s.master[0], 4}, {s.mom[0], 4}, {s.var[0], 4}, {s.master[1], 4},
                                            {s.mom[1], 4},    {s.var[1], 4}, {params, 2}};
    const int M = plan->M;
    for (int k = 0; k < M; ++k) arr[7 + k] = {g.p[k], 2};
    const Walk w = make_walk(L, nv, arr, 7 + M);
    uint16_t *pp = static_cast<uint16_t *>(params);
    cudaError_t e = cudaSuccess;
    // state copies in host memory: the link, not HBM, sets the pace
    const bool host = in_host_memory(s.master[0]);
    dispatch_m(M, [&](auto mt) {
        constexpr int MT = decltype(mt)::value;
        constexpr Shape sh = pingpong_shape(MT);
        static_assert(shape_ok(sh) && shape_ok(kPingPongHostShape), "ping-pong shapes");
        if (host) {
            const int grid = grid_for(k_fused_step_pingpong<MT, kPingPongHostShape.D>, w, kPingPongHostShape.per_sm,
                                      kPingPongHostShape.block);
            e = launch_pdl(k_fused_step_pingpong<MT, kPingPongHostShape.D>, grid, kPingPongHostShape.block, st, g, M,
                           s, pp, w, c, scaler);
        } else {
            const int grid = grid_for(k_fused_step_pingpong<MT, sh.D>, w, sh.per_sm, sh.block);
            e = launch_pdl(k_fused_step_pingpong<MT, sh.D>, grid, sh.block, st, g, M, s, pp, w, c, scaler);
        }
    });
    if (e != cudaSuccess) return pdl_fail(e, what);
    return launch_status(what);
}

// Validate and launch the end of a ping-pong attempt over L elements (nv
// real): params restored after an overflow, then the scaler update.
int launch_pingpong_finish(const zero1_plan_t *plan, int64_t L, int64_t nv, float *const *master, void *params,
                           const zero1_adamw_t *hp, zero1_scaler_t *scaler, const zero1_loss_scale_policy_t *policy,
                           cudaStream_t st, const char *what)
{
    int rc;
    Z1Consts c;  // validates the betas and the global batch the scaler update uses
    if ((rc = dynamic_constants(hp, plan->M, &c)) != ZERO1_OK) return rc;
    if ((rc = check_scaler_ptr(scaler)) != ZERO1_OK || (rc = check_policy(policy)) != ZERO1_OK) return rc;
    if (!master || !master[0] || !master[1])
        return z1_fail(ZERO1_EINVAL, "%s: the master copies are NULL", what);
    if (master[0] == master[1]) return z1_fail(ZERO1_EINVAL, "%s: the two master copies are the same buffer", what);
    if ((rc = check_natural(master[0], 4, "master")) || (rc = check_natural(master[1], 4, "master")))
        return rc;
    if (nv > 0 && !params)
        return z1_fail(ZERO1_EINVAL, "%s: params must be non-NULL when the range holds parameters", what);
    if ((rc = check_natural(params, 2, "params")) != ZERO1_OK) return rc;
    PingPong s{};
    s.master[0] = master[0];
    s.master[1] = master[1];
    const ArrayRef arr[3] = {{master[0], 4}, {master[1], 4}, {params, 2}};
    const Walk w = make_walk(L, nv, arr, 3);
    const int grid = grid_for(k_restore_params, w, kRestorePerSm);
    const cudaError_t e =
        launch_pdl(k_restore_params, grid, kBlock, st, s, static_cast<uint16_t *>(params), w, (const zero1_scaler_t *)scaler);
    if (e != cudaSuccess) return pdl_fail(e, what);
    const ScalePolicy pol{policy->factor, policy->window, policy->hysteresis, policy->min_scale};
    const cudaError_t e2 =
        launch_pdl(k_scaler_update, 1, 32, st, scaler, pol, (int64_t)hp->global_batch, hp->beta1, hp->beta2, 1);
    if (e2 != cudaSuccess) return pdl_fail(e2, what);
    return launch_status(what);
}

}  // namespace

extern "C" int zero1_step_dynamic_pingpong(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                           const void *const *grads, float *const *master, float *const *m,
                                           float *const *v, void *params, const zero1_adamw_t *hp,
                                           zero1_scaler_t *scaler, const zero1_loss_scale_policy_t *policy,
                                           zero1_stream_t stream)
{
    Z1Trace trace("zero1_step_dynamic_pingpong");
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    if ((rc = check_policy(policy)) != ZERO1_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((rc = launch_pingpong_range(plan, r.L, r.nv, grads, master, m, v, params, hp, scaler, st,
                                    "ping-pong step")) != ZERO1_OK)
        return rc;
    return launch_pingpong_finish(plan, r.L, r.nv, master, params, hp, scaler, policy, st, "ping-pong step");
}

extern "C" int zero1_pingpong_bucket(const zero1_plan_t *plan, int64_t elem_begin, int64_t elem_end,
                                     const void *const *grads, float *const *master, float *const *m,
                                     float *const *v, void *params, const zero1_adamw_t *hp,
                                     zero1_scaler_t *scaler, zero1_stream_t stream)
{
    Z1Trace trace("zero1_pingpong_bucket");
    int rc = z1_check_plan(plan);
    if (rc != ZERO1_OK) return rc;
    if (elem_begin < 0 || elem_end > plan->padded_n || elem_begin >= elem_end)
        return z1_fail(ZERO1_EINVAL, "bucket [%lld, %lld) not inside [0, %lld)", (long long)elem_begin,
                       (long long)elem_end, (long long)plan->padded_n);
    const int64_t L = elem_end - elem_begin;
    int64_t nv = plan->n - elem_begin;
    nv = nv < 0 ? 0 : (nv > L ? L : nv);
    return launch_pingpong_range(plan, L, nv, grads, master, m, v, params, hp, scaler,
                                 reinterpret_cast<cudaStream_t>(stream), "ping-pong bucket");
}

extern "C" int zero1_pingpong_finish(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                     float *const *master, void *params, const zero1_adamw_t *hp,
                                     zero1_scaler_t *scaler, const zero1_loss_scale_policy_t *policy,
                                     zero1_stream_t stream)
{
    Z1Trace trace("zero1_pingpong_finish");
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    return launch_pingpong_finish(plan, r.L, r.nv, master, params, hp, scaler, policy,
                                  reinterpret_cast<cudaStream_t>(stream), "ping-pong finish");
}

// ------------------------------------- pieces of the staged dynamic step --

int z1_scaled_range(const zero1_plan_t *plan, int64_t elem_begin, int64_t elem_end, const void *const *grads,
                    float *master, float *m, float *v, void *params, const zero1_adamw_t *hp,
                    const zero1_scaler_t *scaler, zero1_stream_t stream)
{
    int rc = z1_check_plan(plan);
    if (rc != ZERO1_OK) return rc;
    if (elem_begin < 0 || elem_end > plan->padded_n || elem_begin >= elem_end)
        return z1_fail(ZERO1_EINVAL, "scaled range [%lld, %lld) not inside [0, %lld)", (long long)elem_begin,
                       (long long)elem_end, (long long)plan->padded_n);
    const int64_t L = elem_end - elem_begin;
    int64_t nv = plan->n - elem_begin;
    nv = nv < 0 ? 0 : (nv > L ? L : nv);
    Z1Consts c;
    if ((rc = dynamic_constants(hp, plan->M, &c)) != ZERO1_OK) return rc;
    if ((rc = check_scaler_ptr(scaler)) != ZERO1_OK) return rc;
    if (!master || !m || !v) return z1_fail(ZERO1_EINVAL, "scaled range: master, m and v must be non-NULL");
    if (nv > 0 && !params)
        return z1_fail(ZERO1_EINVAL, "scaled range: params must be non-NULL when the range holds parameters");
    GradPtrs g{};
    if (nv > 0 && (rc = load_grads(plan, grads, &g, "scaled range")) != ZERO1_OK) return rc;
    if ((rc = check_natural(master, 4, "master")) || (rc = check_natural(m, 4, "m")) ||
        (rc = check_natural(v, 4, "v")) || (rc = check_natural(params, 2, "params")))
        return rc;
    const Extent out[4] = {{master, L * 4, "master"}, {m, L * 4, "m"}, {v, L * 4, "v"}, {params, nv * 2, "params"}};
    if ((rc = check_disjoint(out, 4, g, plan->M, nv, "scaled range")) != ZERO1_OK) return rc;
    ArrayRef arr[ZERO1_MAX_REPLICAS + 4] = {{master, 4}, {m, 4}, {v, 4}, {params, 2}};
    const int M = plan->M;
    for (int k = 0; k < M; ++k) arr[4 + k] = {g.p[k], 2};
    const Walk w = make_walk(L, nv, arr, 4 + M);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint16_t *pp = static_cast<uint16_t *>(params);
    dispatch_m(M, [&](auto mt) {
        constexpr int MT = decltype(mt)::value;
        constexpr Shape sh = fused_shape(MT);
        static_assert(shape_ok(sh), "fused shape");
        const int grid = grid_for(k_fused_step_scaled<MT, sh.D>, w, sh.per_sm, sh.block);
        k_fused_step_scaled<MT, sh.D><<<grid, sh.block, 0, st>>>(g, M, master, m, v, pp, w, c, scaler);
    });
    return launch_status("scaled range launch");
}

int z1_scaler_advance(zero1_scaler_t *scaler, const zero1_loss_scale_policy_t *policy, const zero1_adamw_t *hp,
                      int32_t M, zero1_stream_t stream)
{
    int rc;
    Z1Consts c;
    if ((rc = dynamic_constants(hp, M, &c)) != ZERO1_OK) return rc;
    if ((rc = check_scaler_ptr(scaler)) != ZERO1_OK || (rc = check_policy(policy)) != ZERO1_OK) return rc;
    const ScalePolicy pol{policy->factor, policy->window, policy->hysteresis, policy->min_scale};
    k_scaler_update<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(scaler, pol, hp->global_batch, hp->beta1,
                                                                          hp->beta2, 0);
    return launch_status("scaler update launch");
}

int z1_check_scaler_and_policy(const zero1_scaler_t *scaler, const zero1_loss_scale_policy_t *policy,
                               const zero1_adamw_t *hp, int32_t M)
{
    int rc;
    Z1Consts c;
    if ((rc = dynamic_constants(hp, M, &c)) != ZERO1_OK) return rc;
    if ((rc = check_scaler_ptr(scaler)) != ZERO1_OK) return rc;
    return check_policy(policy);
}

// ------------------------------------------- step without caller allocation --
//
// For callers that cannot call cudaMalloc (their pool allocator owns the
// device memory, or allocation would synchronise the device): the sums
// workspace of zero1_step_dynamic is this file-scope array, which exists on
// every device that loads the library until the process exits.  Its name is a
// host-side stand-in in host code; the device address comes from
// cudaGetSymbolAddress, looked up with the device current on the first call
// on each device, and again whenever the device's current context is not
// the one the address was looked up in (after cudaDeviceReset the array
// lives in a new context).
static __device__ __align__(256) float g_noalloc_sums[ZERO1_NOALLOC_MAX_ELEMS];

namespace {

// cuCtxGetCurrent, reached through the runtime (no link to the driver
// library); NULL if the runtime cannot provide it.
typedef int (*CtxGetCurrentFn)(void **ctx);

CtxGetCurrentFn ctx_get_current()
{
    static std::once_flag once;
    static CtxGetCurrentFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        cudaGetLastError();
    });
    return fn;
}

void *current_context()
{
    void *ctx = nullptr;
    const CtxGetCurrentFn fn = ctx_get_current();
    if (fn && fn(&ctx) != 0) ctx = nullptr;
    return ctx;
}

struct NoallocAddr {
    void *ctx;
    float *addr;
};
std::mutex g_noalloc_mu;
NoallocAddr g_noalloc_addr[64];

// Device address of g_noalloc_sums in the current device's current context.
int noalloc_sums(float **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return z1_fail(ZERO1_ECUDA, "no-alloc step: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return z1_fail(ZERO1_ERANGE, "no-alloc step: device %d beyond 64 devices", dev);
    void *ctx = current_context();
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocAddr &c = g_noalloc_addr[dev];
    if (ctx && c.addr && c.ctx == ctx) {
        *out = c.addr;
        return ZERO1_OK;
    }
    void *addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_noalloc_sums);
    if (e != cudaSuccess || !addr)
        return z1_fail(ZERO1_ECUDA, "no-alloc step: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    // the lookup makes the device's primary context current if none was
    c.ctx = ctx ? ctx : current_context();
    c.addr = static_cast<float *>(addr);
    *out = c.addr;
    return ZERO1_OK;
}

}  // namespace

extern "C" int zero1_step_dynamic_noalloc(const zero1_plan_t *plan, int32_t shard_begin, int32_t shard_end,
                                          const void *const *grads, float *master, float *m, float *v,
                                          void *params, const zero1_adamw_t *hp, zero1_scaler_t *scaler,
                                          const zero1_loss_scale_policy_t *policy, zero1_stream_t stream)
{
    Z1Trace trace("zero1_step_dynamic_noalloc");
    Z1Range r;
    int rc = z1_range(plan, shard_begin, shard_end, &r);
    if (rc != ZERO1_OK) return rc;
    if (r.L > (int64_t)ZERO1_NOALLOC_MAX_ELEMS)
        return z1_fail(ZERO1_ERANGE,
                       "no-alloc step: range of %lld elements exceeds the built-in workspace of %d elements "
                       "(64 MiB); one call is one whole attempt, so a longer range needs zero1_step_dynamic "
                       "with a caller-provided workspace",
                       (long long)r.L, ZERO1_NOALLOC_MAX_ELEMS);
    float *sums = nullptr;
    if ((rc = noalloc_sums(&sums)) != ZERO1_OK) return rc;
    return zero1_step_dynamic(plan, shard_begin, shard_end, grads, master, m, v, params, hp, scaler, policy,
                              sums, stream);
}
