/*
 * zero1_oracle.c - plain, slow, single-threaded CPU oracle of the ZeRO Stage-1
 * optimizer step (reduce-scatter of M replicas' bf16 gradients, AdamW on the
 * fp32 shard, all-gather of the bf16 parameters).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant generator
 * with the CUDA library; it is written from the pages' statement of the
 * method, not from the kernels.
 *
 * Build: cc -std=c99 -O2 -ffp-contract=off -fno-fast-math -shared -fPIC
 * (-ffp-contract=off matters: every product and sum below is a separate
 * IEEE-754 binary32 operation rounded to nearest-even; a fused multiply-add
 * would round once instead of twice).
 *
 * Sources (page title, section):
 *  [DP]   "CS336 Lecture 7: Parallelism 1", section "朴素数据并行" (naive data
 *         parallelism), the SGD equation theta_{t+1} = theta_t - eta (1/B) sum_i grad L(x_i)
 *         with the sum split over M GPUs holding B/M samples each.
 *  [COLL] same page, "集合通信原语" (the five collectives) and the identity
 *         All-Reduce == Reduce-Scatter + All-Gather.
 *  [MEM]  same page, "训练内存的详细分析", the 16 bytes/parameter table
 *         (bf16 param 2, bf16 grad 2, fp32 master 4, Adam m 4, Adam v 4).
 *  [Z1]   same page, "ZeRO Stage 1：优化器状态分片", its four steps: full
 *         local gradient; Reduce-Scatter so GPU i holds the summed gradient of
 *         shard i; GPU i updates shard i with its optimizer state; All-Gather.
 *  [PART] "第2章 软件程序与专用硬件的结合", section 2.3.4 (ZeRO): on N GPUs each
 *         one keeps 1/N of the optimizer state.
 *  [ADAMW] "五维并行实战", section 4.2 (the DeepSpeed config: AdamW with lr,
 *         betas, eps, weight_decay; the fp16 loss-scale block) and section 3.2
 *         (trap 3: a loss that becomes inf under AMP loss scaling).
 *
 * Readings where the pages are silent (each one is a stated choice):
 *  - AdamW update: decoupled weight decay multiplied by lr, bias correction on,
 *    eps added after the square root of v-hat; exact fp32 operation order in
 *    orc_adamw below.
 *  - The replica sum is a left fold in rank order 0..M-1 starting from rank 0's
 *    value, in fp32; unscaling by 1/(B*S) follows the sum.
 *  - Host constants are evaluated in double and rounded once to float; the
 *    power beta^t is evaluated in double by square-and-multiply over the bits
 *    of t, least significant first (orc_pow_int), so that any IEEE-754
 *    implementation - the GPU included - reproduces it exactly.
 *  - Padding elements (global index >= n) have gradient +0 and are updated
 *    like any other element.
 *  - The overflow flag is the OR over real elements of !isfinite(sum).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32.  bf16 is the upper half of an IEEE binary32 word.          */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

float orc_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Round a binary32 value to the nearest bfloat16, ties to the even mantissa,
 * written from the definition: take the two bf16 neighbours of |x| (the value
 * truncated toward zero and the next one up in magnitude), compare the exact
 * distances in double, break ties on the low mantissa bit.  Values past the
 * largest finite bf16 by at least half an ulp become inf.  NaN stays NaN
 * (sign kept, quiet bit set). */
uint16_t orc_f32_to_bf16(float x)
{
    uint32_t u = f32_bits(x);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    if (isnan(x)) return (uint16_t)((u >> 16) | 0x0040u);
    if (isinf(x)) return (uint16_t)(u >> 16);
    uint16_t lo = (uint16_t)((u >> 16) & 0x7fffu);       /* |x| truncated  */
    uint16_t hi = (uint16_t)(lo + 1u);                    /* next magnitude */
    int e = (lo >> 7) & 0xff;                             /* biased exponent */
    double ulp = ldexp(1.0, (e == 0 ? 1 : e) - 127 - 7);  /* spacing at lo  */
    double a = fabs((double)x);
    double dlo = (double)orc_bf16_to_f32(lo);
    double dhi = dlo + ulp;             /* exact even when hi is inf's code */
    double below = a - dlo, above = dhi - a;
    uint16_t mag;
    if (below < above) mag = lo;
    else if (above < below) mag = hi;
    else mag = (lo & 1u) ? hi : lo;
    return (uint16_t)(sign | mag);
}

void orc_bf16_to_f32_array(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f32(in[i]);
}

void orc_f32_to_bf16_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Shard plan [PART], [Z1]: n parameters, M ranks, padded length P a        */
/* multiple of M*align, shard size s = P/M, shard i = [i*s, (i+1)*s).        */
/* ------------------------------------------------------------------------ */

int orc_plan(int64_t n, int32_t M, int32_t align, int64_t *padded_n, int64_t *shard)
{
    if (n < 1 || M < 1 || align < 1) return -1;
    int64_t unit = (int64_t)M * (int64_t)align;
    int64_t P = ((n + unit - 1) / unit) * unit;
    *padded_n = P;
    *shard = P / M;
    return 0;
}

/* The pieces of a flat concatenation of tensors (numels[0], numels[1], ...)
 * that fall in shard `idx` of size `shard` (only real elements, < n).  For each
 * piece: tensor index, offset inside the tensor, offset inside the shard,
 * length.  Returns the number of pieces, or -1 if more than cap. */
int orc_segments(const int64_t *numels, int32_t n_tensors, int64_t shard, int32_t idx,
                 int32_t cap, int64_t *seg_tensor, int64_t *seg_tensor_off,
                 int64_t *seg_shard_off, int64_t *seg_len)
{
    int64_t lo = (int64_t)idx * shard, hi = lo + shard;
    int64_t base = 0;
    int count = 0;
    for (int32_t k = 0; k < n_tensors; ++k) {
        int64_t a = base, b = base + numels[k];
        int64_t x0 = a > lo ? a : lo, x1 = b < hi ? b : hi;
        if (x1 > x0) {
            if (count >= cap) return -1;
            seg_tensor[count] = k;
            seg_tensor_off[count] = x0 - a;
            seg_shard_off[count] = x0 - lo;
            seg_len[count] = x1 - x0;
            ++count;
        }
        base = b;
    }
    return count;
}

/* Memory per rank in bytes [MEM], [Z1]: naive data parallelism keeps all 16
 * bytes of every parameter on every rank; ZeRO-1 keeps the bf16 parameters and
 * gradients whole (2+2 bytes each) and 12 bytes of fp32 state per shard
 * element. */
void orc_memory(int64_t n, int64_t shard, int64_t *naive_bytes, int64_t *zero1_bytes)
{
    *naive_bytes = 16 * n;
    *zero1_bytes = 2 * n + 2 * n + 12 * shard;
}

/* ------------------------------------------------------------------------ */
/* AdamW host constants, in double, rounded once to float.                   */
/* out: [0] inv = 1/(B*S)  [1] 1-beta1  [2] 1-beta2  [3] 1-beta1^t            */
/*      [4] 1-beta2^t      [5] 1-lr*wd                                        */
/* ------------------------------------------------------------------------ */

/* b^t for t >= 0 in double: square-and-multiply over the bits of t, least
 * significant bit first; one rounding per multiplication. */
double orc_pow_int(double b, int64_t t)
{
    double r = 1.0, x = b;
    while (t > 0) {
        if (t & 1) r = r * x;
        x = x * x;
        t >>= 1;
    }
    return r;
}

void orc_adamw_constants(float lr, float beta1, float beta2, float weight_decay,
                         int64_t B, float S, int64_t t, float *out)
{
    out[0] = (float)(1.0 / ((double)B * (double)S));
    out[1] = (float)(1.0 - (double)beta1);
    out[2] = (float)(1.0 - (double)beta2);
    out[3] = (float)(1.0 - orc_pow_int((double)beta1, t));
    out[4] = (float)(1.0 - orc_pow_int((double)beta2, t));
    out[5] = (float)(1.0 - (double)lr * (double)weight_decay);
}

/* ------------------------------------------------------------------------ */
/* The three phases of [Z1].                                                 */
/* ------------------------------------------------------------------------ */

/* Reduce-scatter [COLL], [DP], [Z1] step 2: for each element j of the shard
 * range, sum the M replicas' bf16 gradients in fp32, rank 0 first, and scale
 * by `scale` (1/(B*S) in the step).  Elements j >= n_valid are padding and
 * get +0.  flag |= 1 if any real sum is not finite. */
void orc_reduce_scatter(int32_t M, const uint16_t *const *grads, int64_t len, int64_t n_valid,
                        float scale, float *g_out, uint32_t *flag)
{
    uint32_t f = 0;
    for (int64_t j = 0; j < len; ++j) {
        float s = 0.0f;
        if (j < n_valid) {
            s = orc_bf16_to_f32(grads[0][j]);
            for (int32_t r = 1; r < M; ++r) s = s + orc_bf16_to_f32(grads[r][j]);
            if (!isfinite(s)) f = 1;
        }
        g_out[j] = s * scale;
    }
    if (flag) *flag |= f;
}

/* AdamW on the shard [ADAMW], [MEM], [Z1] step 3, in fp32, one rounding per
 * operation:
 *   m' = beta1*m + (1-beta1)*g
 *   v' = beta2*v + (1-beta2)*(g*g)
 *   u  = (m'/(1-beta1^t)) / (sqrt(v'/(1-beta2^t)) + eps)
 *   w' = w*(1-lr*wd) - lr*u                                                */
void orc_adamw(int64_t len, const float *g, float *master, float *m, float *v,
               float lr, float beta1, float beta2, float eps, const float *c)
{
    float omb1 = c[1], omb2 = c[2], bc1 = c[3], bc2 = c[4], cdec = c[5];
    for (int64_t j = 0; j < len; ++j) {
        float gj = g[j];
        float m1 = beta1 * m[j] + omb1 * gj;
        float v1 = beta2 * v[j] + omb2 * (gj * gj);
        float mh = m1 / bc1;
        float vh = v1 / bc2;
        float u = mh / (sqrtf(vh) + eps);
        float w = master[j] * cdec - lr * u;
        m[j] = m1;
        v[j] = v1;
        master[j] = w;
    }
}

/* All-gather [COLL], [Z1] step 4: the updated shard, rounded to bf16, lands
 * in its place in the full parameter buffer (real elements only). */
void orc_all_gather(int64_t n_valid, const float *master, uint16_t *params)
{
    for (int64_t j = 0; j < n_valid; ++j) params[j] = orc_f32_to_bf16(master[j]);
}

/* One ZeRO-1 step over a range of `len` shard elements, the first n_valid of
 * which are real parameters.  grads[r], params point at the range's first
 * element; master, m, v hold the range's fp32 state.  If skip_if_flag is set
 * and *flag is already nonzero, nothing is written; if skip_if_flag is set the
 * flag is only read.  Returns 0, or -1 if memory for the gradient runs out. */
int orc_zero1_step(int32_t M, const uint16_t *const *grads, int64_t len, int64_t n_valid,
                   float *master, float *m, float *v, uint16_t *params,
                   float lr, float beta1, float beta2, float eps, float weight_decay,
                   float S, int64_t B, int64_t t, uint32_t *flag, int32_t skip_if_flag)
{
    if (skip_if_flag && flag && *flag) return 0;
    float c[6];
    orc_adamw_constants(lr, beta1, beta2, weight_decay, B, S, t, c);
    float *g = (float *)malloc((size_t)(len > 0 ? len : 1) * sizeof(float));
    if (!g) return -1;
    uint32_t f = 0;
    orc_reduce_scatter(M, grads, len, n_valid, c[0], g, &f);
    orc_adamw(len, g, master, m, v, lr, beta1, beta2, eps, c);
    orc_all_gather(n_valid, master, params);
    free(g);
    if (flag && !skip_if_flag) *flag |= f;
    return 0;
}

/* Naive data-parallel All-Reduce [COLL], [DP]: every output r gets the rank
 * order fp32 sum times `scale`, as bf16 (out_bf16 != 0) or fp32.  All inputs
 * of element j are read before any output of j is written, so outputs may
 * alias inputs. */
void orc_allreduce(int32_t M, const uint16_t *const *in, int64_t n, float scale,
                   int32_t out_bf16, void *const *outs)
{
    for (int64_t j = 0; j < n; ++j) {
        float s = orc_bf16_to_f32(in[0][j]);
        for (int32_t r = 1; r < M; ++r) s = s + orc_bf16_to_f32(in[r][j]);
        float y = s * scale;
        for (int32_t r = 0; r < M; ++r) {
            if (out_bf16) ((uint16_t *)outs[r])[j] = orc_f32_to_bf16(y);
            else ((float *)outs[r])[j] = y;
        }
    }
}

/* Overflow check [ADAMW] (loss scaling): flag |= 1 if the rank order fp32
 * sum of any real element is inf or NaN. */
void orc_overflow_check(int32_t M, const uint16_t *const *grads, int64_t n_valid, uint32_t *flag)
{
    uint32_t f = 0;
    for (int64_t j = 0; j < n_valid; ++j) {
        float s = orc_bf16_to_f32(grads[0][j]);
        for (int32_t r = 1; r < M; ++r) s = s + orc_bf16_to_f32(grads[r][j]);
        if (!isfinite(s)) f = 1;
    }
    *flag |= f;
}

/* ------------------------------------------------------------------------ */
/* Dynamic loss scaling [ADAMW]: the fp16 block of the DeepSpeed config     */
/* ("五维并行实战" 4.2) gives loss_scale 0 (dynamic), initial_scale_power,       */
/* loss_scale_window, hysteresis and min_loss_scale; 3.2 trap 3 gives the     */
/* failure it guards against (a loss that turns inf).  The page names the    */
/* keys, not the rule; the reading taken here:                               */
/*  - S starts at initial_scale (2^initial_scale_power); t starts at the    */
/*    first step.                                                            */
/*  - An attempt whose summed gradients overflow is skipped (nothing is     */
/*    written, t stays); it uses up one unit of hysteresis; when none is     */
/*    left, S is divided by factor (not below min_scale) and the hysteresis  */
/*    is refilled.  The clean-attempt count restarts at 0.                   */
/*  - A clean attempt applies the step (t advances) and counts towards the   */
/*    window; after `window` clean attempts in a row S is multiplied by      */
/*    factor (unless that overflows fp32), the count restarts and the        */
/*    hysteresis is refilled.                                                */
/* ------------------------------------------------------------------------ */

typedef struct {
    float scale;
    int32_t good;
    int32_t hyst_left;
    int64_t step;
    int64_t attempts;
    int64_t skipped;
} orc_scaler;

void orc_scaler_init(orc_scaler *sc, float initial_scale, int32_t hysteresis, int64_t first_step)
{
    sc->scale = initial_scale;
    sc->good = 0;
    sc->hyst_left = hysteresis;
    sc->step = first_step;
    sc->attempts = 0;
    sc->skipped = 0;
}

void orc_scaler_update(orc_scaler *sc, uint32_t overflow, float factor, int32_t window,
                       int32_t hysteresis, float min_scale)
{
    sc->attempts += 1;
    if (overflow) {
        sc->skipped += 1;
        sc->good = 0;
        sc->hyst_left -= 1;
        if (sc->hyst_left <= 0) {
            float down = sc->scale / factor;
            sc->scale = down < min_scale ? min_scale : down;
            sc->hyst_left = hysteresis;
        }
    } else {
        sc->step += 1;
        sc->good += 1;
        if (sc->good >= window) {
            float up = sc->scale * factor;
            if (isfinite(up)) sc->scale = up;
            sc->good = 0;
            sc->hyst_left = hysteresis;
        }
    }
}

/* One attempt of the dynamically scaled step over a whole range: the global
 * overflow flag of this attempt's gradients decides whether the step (with
 * the scaler's S and t) is applied, then the scaler advances. */
int orc_zero1_dynamic_attempt(int32_t M, const uint16_t *const *grads, int64_t len, int64_t n_valid,
                              float *master, float *m, float *v, uint16_t *params,
                              float lr, float beta1, float beta2, float eps, float weight_decay,
                              int64_t B, orc_scaler *sc, float factor, int32_t window,
                              int32_t hysteresis, float min_scale, uint32_t *flag_out)
{
    uint32_t f = 0;
    orc_overflow_check(M, grads, n_valid, &f);
    int rc = orc_zero1_step(M, grads, len, n_valid, master, m, v, params, lr, beta1, beta2, eps,
                            weight_decay, sc->scale, B, sc->step, &f, 1);
    if (rc != 0) return rc;
    orc_scaler_update(sc, f, factor, window, hysteresis, min_scale);
    if (flag_out) *flag_out = f;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Consistency checksum of a buffer (the silent-data-corruption guard of    */
/* the replicated parameters: "CS336 Lecture 7: Parallelism 1" case studies */
/* report silent data corruption on large runs; after the all-gather every  */
/* rank must hold the same parameters).  Over the buffer's 16-bit units      */
/* u_0 .. u_{U-1} (little-endian):                                           */
/*   out[0] = sum u_i            mod 2^64                                    */
/*   out[1] = sum (i + 1) * u_i  mod 2^64                                    */
/* Exact integer sums, so any order of summation gives the same words.       */
/* ------------------------------------------------------------------------ */

void orc_checksum16(const uint16_t *u, int64_t U, uint64_t *out)
{
    uint64_t s1 = 0, s2 = 0;
    for (int64_t i = 0; i < U; ++i) {
        s1 += (uint64_t)u[i];
        s2 += (uint64_t)(i + 1) * (uint64_t)u[i];
    }
    out[0] = s1;
    out[1] = s2;
}
