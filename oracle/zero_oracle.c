/*
 * Oracle for the ZeRO sharded optimizer step -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU restatement of what the data-parallel
 * ZeRO step computes.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this file's library; the product path never does.
 * It shares no code, header or constant with the CUDA library.
 *
 * Sources (web pages on the subject, cited by title and section):
 *   [ZH]  "ZeRO 与 FSDP：切分优化器状态、梯度与参数" (AI-infra handbook),
 *         section "从零实现 ZeRO 的 Adam", class ZeroAdam: flat vector,
 *         shard = ceil(numel / world), zero-padded tail, reduce_scatter (sum),
 *         divide by world, Adam with bias correction, all_gather back.
 *   [PD]  "论文专题讲解：ZeRO" section "显存账": fp32 master / momentum /
 *         variance next to 16-bit params and grads (mixed-precision Adam).
 *   [PP]  "PaddlePaddle ZeRO优化" section "混合精度才是最佳拍档": GradScaler
 *         scale / step (skipped on overflow) / update.
 *
 * Arithmetic: IEEE-754 binary32, round-to-nearest-even, evaluated one
 * operation at a time.  Build with -O2 -ffp-contract=off and never with
 * -ffast-math, so that no multiply-add is fused and no subnormal is flushed.
 * The pages fix the state precision (fp32 master, m and v), so the oracle
 * computes in fp32 in the order written below, not in fp64.
 *
 * Element types are passed as codes: 0 = fp32, 1 = bf16, 2 = fp16; 16-bit
 * buffers hold raw IEEE bit patterns (uint16).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2 };

/* ---------------------------------------------------------------- layout */

/* [ZH] "每个 rank 负责的元素个数（末尾补零对齐）": shard = ceil(numel / world). */
int64_t orc_shard_size(int64_t numel, int32_t world)
{
    if (world <= 0 || numel < 0) return -1;
    return (numel + world - 1) / world;
}

/* Owner rank of flat index i: rank r owns [r*S, r*S + S). */
int32_t orc_owner(int64_t i, int64_t numel, int32_t world)
{
    int64_t S = orc_shard_size(numel, world);
    if (S <= 0 || i < 0 || i >= S * world) return -1;
    return (int32_t)(i / S);
}

/* ------------------------------------------------------- type conversion */

int32_t orc_elem_size(int32_t dtype)
{
    return dtype == ORC_F32 ? 4 : (dtype == ORC_BF16 || dtype == ORC_F16) ? 2 : -1;
}

/* Read element i of a typed buffer as fp32 (both 16-bit widenings are exact). */
static float widen(const void *buf, int32_t dtype, int64_t i)
{
    if (dtype == ORC_F32) return ((const float *)buf)[i];
    uint16_t h = ((const uint16_t *)buf)[i];
    if (dtype == ORC_BF16) {
        /* bf16 is the upper half of a binary32 pattern. */
        uint32_t u = (uint32_t)h << 16;
        float f;
        memcpy(&f, &u, 4);
        return f;
    }
    _Float16 hf;
    memcpy(&hf, &h, 2);
    return (float)hf;
}

/* fp32 -> bf16, round to nearest, ties to even; overflow rounds to inf;
 * NaN stays NaN (quiet bit forced). */
static uint16_t to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t hi = u >> 16;          /* truncated result */
    uint32_t lo = u & 0xffffu;      /* discarded bits */
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u; /* carry may reach inf */
    return (uint16_t)hi;
}

/* fp32 -> fp16 through the compiler's IEEE binary16 conversion (round to
 * nearest even under the default rounding mode, overflow to inf, gradual
 * underflow to subnormals). */
static uint16_t to_f16(float f)
{
    _Float16 h = (_Float16)f;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

static void narrow(float x, int32_t dtype, void *buf, int64_t i)
{
    if (dtype == ORC_F32) ((float *)buf)[i] = x;
    else if (dtype == ORC_BF16) ((uint16_t *)buf)[i] = to_bf16(x);
    else ((uint16_t *)buf)[i] = to_f16(x);
}

/* Exposed so the tests can pin the conversions against other libraries. */
void orc_widen_array(const void *in, int32_t dtype, int64_t n, float *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = widen(in, dtype, i);
}

/* [PD] the fp16/bf16 params used by forward/backward are the rounded fp32 master. */
void orc_cast(const float *x, int64_t n, int32_t dtype, void *out)
{
    for (int64_t i = 0; i < n; ++i) narrow(x[i], dtype, out, i);
}

/* ------------------------------------------------------------ collectives */

/* The sum at the heart of reduce-scatter, over n aligned positions of N
 * rank buffers: acc[j] = g_0[j] + g_1[j] + ... + g_{N-1}[j], added in rank
 * order starting from g_0 (not from 0.0, so a lone -0 keeps its sign).
 * Positions j >= n_valid are padding and read as exactly 0. */
void orc_rank_sum(const void *const *bufs, int32_t dtype, int32_t world,
                  int64_t n, int64_t n_valid, float *acc)
{
    for (int64_t j = 0; j < n; ++j) {
        if (j >= n_valid) { acc[j] = 0.0f; continue; }
        float a = widen(bufs[0], dtype, j);
        for (int32_t k = 1; k < world; ++k) a = a + widen(bufs[k], dtype, j);
        acc[j] = a;
    }
}

/* [ZH] dist.reduce_scatter_tensor(g, grads): rank `rank` receives, for each j
 * in its shard, the sum over all ranks k of rank k's flat (zero-padded) grad
 * at rank*S + j.  grads[k] holds rank k's `numel` unpadded grads.
 * bytes_sent[k] (optional) accumulates what rank k ships to this rank. */
int orc_reduce_scatter_sum(const void *const *grads, int32_t dtype, int64_t numel,
                           int32_t world, int32_t rank, float *out, int64_t *bytes_sent)
{
    int64_t S = orc_shard_size(numel, world);
    if (S < 0 || rank < 0 || rank >= world) return -1;
    int32_t es = orc_elem_size(dtype);
    for (int64_t j = 0; j < S; ++j) {
        int64_t i = (int64_t)rank * S + j;
        if (i >= numel) { out[j] = 0.0f; continue; }
        float a = widen(grads[0], dtype, i);
        for (int32_t k = 1; k < world; ++k) a = a + widen(grads[k], dtype, i);
        out[j] = a;
    }
    if (bytes_sent)
        for (int32_t k = 0; k < world; ++k)
            if (k != rank) bytes_sent[k] += S * es;
    return 0;
}

/* [ZH] "g /= self.world" (average), then, with a loss scale in use, divide by
 * the scale to undo it ([PP] GradScaler).  loss_scale <= 0 means no scaling.
 * Returns how many results are not finite ([PP] the overflow check behind
 * scaler.step). */
int64_t orc_average(const float *acc, int64_t n, int32_t world, float loss_scale, float *g)
{
    int64_t bad = 0;
    float w = (float)world;
    for (int64_t j = 0; j < n; ++j) {
        float x = acc[j] / w;
        if (loss_scale > 0.0f) x = x / loss_scale;
        g[j] = x;
        if (!isfinite(x)) ++bad;
    }
    return bad;
}

/* [ZH] dist.all_gather_into_tensor(full, master): shard r lands at r*S. */
void orc_all_gather(const void *const *shards, int32_t dtype, int64_t S, int32_t world,
                    void *full, int64_t *bytes_sent)
{
    int32_t es = orc_elem_size(dtype);
    for (int32_t r = 0; r < world; ++r) {
        for (int64_t j = 0; j < S; ++j)
            memcpy((char *)full + ((int64_t)r * S + j) * es,
                   (const char *)shards[r] + j * es, (size_t)es);
        if (bytes_sent) bytes_sent[r] += (int64_t)(world - 1) * S * es;
    }
}

/* Plain data parallelism's all-reduce followed by the average: every rank
 * ends with the mean of all ranks' padded grads over the whole vector. */
void orc_all_reduce_mean(const void *const *grads, int32_t dtype, int64_t numel,
                         int32_t world, float *out)
{
    int64_t P = orc_shard_size(numel, world) * world;
    float w = (float)world;
    for (int64_t i = 0; i < P; ++i) {
        if (i >= numel) { out[i] = 0.0f; continue; }
        float a = widen(grads[0], dtype, i);
        for (int32_t k = 1; k < world; ++k) a = a + widen(grads[k], dtype, i);
        out[i] = a / w;
    }
}

/* ------------------------------------------------------------------ Adam */

/* Per-step scalars of Adam.  The hyperparameters are real numbers held in
 * double (Python floats in [ZH]); every scalar the elementwise update uses is
 * evaluated in double from them and rounded once to fp32:
 *   out[0] = 1 - beta1            (weight of the new gradient in m)
 *   out[1] = 1 - beta2            (weight of the squared gradient in v)
 *   out[2] = 1 - beta1^t          (bias correction of m)
 *   out[3] = 1 - beta2^t          (bias correction of v)                   */
void orc_adam_scalars(double beta1, double beta2, int64_t t, float *out)
{
    out[0] = (float)(1.0 - beta1);
    out[1] = (float)(1.0 - beta2);
    out[2] = (float)(1.0 - pow(beta1, (double)t));
    out[3] = (float)(1.0 - pow(beta2, (double)t));
}

/* [ZH] ZeroAdam.step, on one shard of n elements, step t >= 1:
 *   m     = beta1*m + (1-beta1)*g
 *   v     = beta2*v + (1-beta2)*g*g
 *   m_hat = m / (1 - beta1^t)
 *   v_hat = v / (1 - beta2^t)
 *   x     = x - lr*m_hat / (sqrt(v_hat) + eps)       (eps outside the root)
 * With weight_decay != 0 the decay is decoupled from the gradient (AdamW,
 * Loshchilov & Hutter, "Decoupled Weight Decay Regularization", ICLR 2019;
 * the Paddle page names AdamW as the optimizer): the weight is first scaled
 * by 1 - lr*weight_decay (one fp32 scalar, computed in double), then the
 * Adam step is subtracted:  x = x*(1 - lr*wd) - lr*m_hat/(sqrt(v_hat)+eps). */
void orc_adam(float *x, float *m, float *v, const float *g, int64_t n,
              double lr, double beta1, double beta2, double eps, int64_t t,
              double weight_decay)
{
    const float decay = (float)(1.0 - lr * weight_decay);
    float s[4];
    orc_adam_scalars(beta1, beta2, t, s);
    const float c1 = s[0], c2 = s[1], bc1 = s[2], bc2 = s[3];
    const float b1 = (float)beta1, b2 = (float)beta2, lrf = (float)lr, epsf = (float)eps;
    for (int64_t j = 0; j < n; ++j) {
        float gj = g[j];
        float mj = m[j] * b1 + c1 * gj;
        float vj = v[j] * b2 + c2 * (gj * gj);
        float mh = mj / bc1;
        float vh = vj / bc2;
        float den = sqrtf(vh) + epsf;
        float upd = (lrf * mh) / den;
        float xj = x[j];
        if (weight_decay != 0.0) xj = xj * decay;
        m[j] = mj;
        v[j] = vj;
        x[j] = xj - upd;
    }
}

/* Reduce-scatter as above for an explicit shard length S (S*world >= numel):
 * the row-granular layout below rounds shards up to whole rows. */
static void reduce_scatter_s(const void *const *grads, int32_t dtype, int64_t numel,
                             int32_t world, int64_t S, int32_t rank, float *out)
{
    for (int64_t j = 0; j < S; ++j) {
        int64_t i = (int64_t)rank * S + j;
        if (i >= numel) { out[j] = 0.0f; continue; }
        float a = widen(grads[0], dtype, i);
        for (int32_t k = 1; k < world; ++k) a = a + widen(grads[k], dtype, i);
        out[j] = a;
    }
}

/* FSDP2's per-parameter layout ("ZeRO 与 FSDP…", section ZeRO-3 与 FSDP: each
 * parameter is a DTensor sharded along dim 0): a parameter of `rows` rows of
 * `row_elems` elements is cut into chunks of ceil(rows/world) whole rows;
 * rank r holds rows [r*c, r*c + c), padded with zero rows past the end
 * (ranks past the last row hold padding only).  As a flat shard length:
 * S = ceil(rows / world) * row_elems. */
int64_t orc_row_shard_size(int64_t rows, int64_t row_elems, int32_t world)
{
    if (world <= 0 || rows < 0 || row_elems < 0) return -1;
    return (rows + world - 1) / world * row_elems;
}

/* -------------------------------------------------------- the whole step */

/* One ZeRO-2 step with every rank's state held here ("all ranks" layout):
 * master/m/v are the N shards laid end to end (length P = N*S, rank r's at
 * r*S), grads[k] are rank k's `numel` local grads, full is the P-element
 * low-precision parameter buffer every rank ends up holding.
 *
 * Order, after ZeroAdam.step ([ZH]) with the GradScaler skip ([PP]):
 *   1. for each rank r: reduce-scatter (sum) its shard of the grads;
 *   2. average (divide by N), then unscale by loss_scale when it is > 0;
 *   3. overflow check over every rank's shard: with loss scaling on and any
 *      value non-finite, the step is skipped: nothing below happens;
 *   4. for each rank r: Adam on its shard with step t;
 *   5. each rank casts its shard to the param type; all-gather into `full`.
 * Returns 1 when skipped, 0 when applied, -1 on bad arguments.
 * *n_nonfinite (optional) gets the count from step 3.
 * `work` must hold P floats plus P param elements (8*P bytes suffice). */
int orc_zero_step_s(const void *const *grads, int32_t grad_dtype, int64_t numel, int32_t world,
                    int64_t S, float *master, float *m, float *v, void *full, int32_t param_dtype,
                    double lr, double beta1, double beta2, double eps, int64_t t,
                    float loss_scale, float *work, int64_t *n_nonfinite, double weight_decay)
{
    if (S < 0 || S * world < numel || t < 1 || world > 4096) return -1;
    int64_t P = S * world;
    int64_t bad = 0;
    for (int32_t r = 0; r < world; ++r) {
        float *gr = work + (int64_t)r * S;
        reduce_scatter_s(grads, grad_dtype, numel, world, S, r, gr);
        bad += orc_average(gr, S, world, loss_scale, gr);
    }
    if (n_nonfinite) *n_nonfinite = bad;
    if (loss_scale > 0.0f && bad > 0) return 1;
    for (int32_t r = 0; r < world; ++r) {
        int64_t o = (int64_t)r * S;
        orc_adam(master + o, m + o, v + o, work + o, S, lr, beta1, beta2, eps, t, weight_decay);
    }
    int32_t es = orc_elem_size(param_dtype);
    char *lp = (char *)(work + P);            /* rank r's cast shard at lp + r*S*es */
    const void *shards[4096];
    for (int32_t r = 0; r < world; ++r) {
        int64_t o = (int64_t)r * S;
        orc_cast(master + o, S, param_dtype, lp + o * es);
        shards[r] = lp + o * es;
    }
    orc_all_gather(shards, param_dtype, S, world, full, 0);
    return 0;
}

int orc_zero_step(const void *const *grads, int32_t grad_dtype, int64_t numel, int32_t world,
                  float *master, float *m, float *v, void *full, int32_t param_dtype,
                  double lr, double beta1, double beta2, double eps, int64_t t, float loss_scale,
                  float *work, int64_t *n_nonfinite, double weight_decay)
{
    return orc_zero_step_s(grads, grad_dtype, numel, world, orc_shard_size(numel, world), master,
                           m, v, full, param_dtype, lr, beta1, beta2, eps, t, loss_scale, work,
                           n_nonfinite, weight_decay);
}

/* One rank's view of the same step ([ZH] ZeroAdam.step as run by rank
 * `rank`): slices[k] is the S-element piece of rank k's flat grads that
 * belongs to this rank's shard (what reduce-scatter brings in), master/m/v
 * are this rank's S-element shard state, and the cast shard is written to
 * lp_out (S elements: the rank's place in the full buffer, or its own
 * persistent shard when params are sharded too).  Positions of the shard at
 * or past `numel` are padding: their grads read as 0.  With loss scaling on,
 * the step is skipped when this rank's shard or `others_nonfinite` (the other
 * ranks' findings, combined by the caller) has a non-finite value.
 * Returns 1 when skipped, 0 when applied, -1 on bad arguments.  `work` holds
 * S floats. */
int orc_zero_rank_step_s(const void *const *slices, int32_t grad_dtype, int64_t numel,
                         int32_t world, int64_t S, int32_t rank, float *master, float *m,
                         float *v, void *lp_out, int32_t param_dtype, double lr, double beta1,
                         double beta2, double eps, int64_t t, float loss_scale,
                         int64_t others_nonfinite, float *work, int64_t *n_nonfinite,
                         double weight_decay)
{
    if (S < 0 || S * world < numel || t < 1 || rank < 0 || rank >= world) return -1;
    int64_t n_valid = numel - (int64_t)rank * S;
    if (n_valid < 0) n_valid = 0;
    if (n_valid > S) n_valid = S;
    orc_rank_sum(slices, grad_dtype, world, S, n_valid, work);
    int64_t bad = orc_average(work, S, world, loss_scale, work);
    if (n_nonfinite) *n_nonfinite = bad;
    if (loss_scale > 0.0f && bad + others_nonfinite > 0) return 1;
    orc_adam(master, m, v, work, S, lr, beta1, beta2, eps, t, weight_decay);
    orc_cast(master, S, param_dtype, lp_out);
    return 0;
}

int orc_zero_rank_step(const void *const *slices, int32_t grad_dtype, int64_t numel,
                       int32_t world, int32_t rank, float *master, float *m, float *v,
                       void *lp_out, int32_t param_dtype, double lr, double beta1, double beta2,
                       double eps, int64_t t, float loss_scale, int64_t others_nonfinite,
                       float *work, int64_t *n_nonfinite, double weight_decay)
{
    return orc_zero_rank_step_s(slices, grad_dtype, numel, world, orc_shard_size(numel, world),
                                rank, master, m, v, lp_out, param_dtype, lr, beta1, beta2, eps,
                                t, loss_scale, others_nonfinite, work, n_nonfinite,
                                weight_decay);
}

/* GradScaler-style update of the loss scale after a step ([PP]): halve on a
 * skipped step and restart the clean-step count; after `growth_interval`
 * clean steps in a row, double it.  Returns the new scale. */
float orc_scale_update(float scale, int32_t skipped, int64_t *good_steps,
                       int64_t growth_interval)
{
    if (skipped) {
        *good_steps = 0;
        return scale * 0.5f;
    }
    *good_steps += 1;
    if (growth_interval > 0 && *good_steps >= growth_interval) {
        *good_steps = 0;
        /* grow only to a finite scale */
        const float grown = scale * 2.0f;
        return isfinite(grown) ? grown : scale;
    }
    return scale;
}
