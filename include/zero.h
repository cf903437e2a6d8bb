/*
 * zero.h -- C ABI of the GB300 ZeRO sharded optimizer step (libzero.so).
 *
 * The method (ZeRO data parallelism, stages 1/2/3):
 *   - "ZeRO 与 FSDP：切分优化器状态、梯度与参数", section 从零实现 ZeRO 的 Adam:
 *     all parameters form one flat vector, cut into N shards of
 *     S = ceil(numel / N) elements with a zero-padded tail; rank r owns
 *     [r*S, r*S + S).  One step = reduce-scatter (sum) of the grads, divide by
 *     N, Adam with bias correction on the owned shard, all-gather of the
 *     updated shards back into the full parameter vector.
 *   - "论文专题讲解：ZeRO：大模型训练的零冗余状态优化", sections 显存账 and
 *     ZeRO-DP 三阶段: fp32 master weights, momentum and variance beside 16-bit
 *     params and grads; stage 1 shards the optimizer states, stage 2 also the
 *     grads, stage 3 also the params.
 *   - "ZeRO 与 FSDP…", section ZeRO-3 与 FSDP, and guanweilu.cn article 1460,
 *     section Stage 3: with params sharded, each unit (layer) is all-gathered
 *     before its forward and again before its backward, then its grads are
 *     reduce-scattered.
 *   - "PaddlePaddle ZeRO优化", section 混合精度才是最佳拍档: with a loss
 *     scale, a step whose grads hold inf/nan is skipped and the scale halved.
 *
 * On one GPU the N data-parallel ranks are N device buffers, so every
 * "collective" here is a kernel reading those buffers; nothing talks to
 * another GPU.  Three views are supported:
 *   rank = -1  ("all ranks"): the state of every rank lives here.  master, m,
 *              v hold the N shards end to end (P = N*S floats, rank r's at
 *              r*S); grads[k] is rank k's whole local gradient (numel
 *              elements; no padding needed).  One step performs the
 *              reduce-scatter, Adam on every shard, the cast and the
 *              all-gather in one pass over P elements.
 *   rank = r   ("one rank's view"): master, m, v hold rank r's shard (S
 *              floats); grads[k] is the S-element slice of rank k's flat
 *              gradient that belongs to shard r (what reduce-scatter brings to
 *              rank r).  The updated shard is cast into rank r's place of the
 *              full parameter buffer; zero_allgather() places the others.
 *   ranks r..r+k-1 (zero_init_ranks): the k shards of ranks r to r+k-1
 *              laid end to end (k*S floats, rank r+j's at j*S); grads[i] is
 *              the k*S-element piece [r*S, (r+k)*S) of rank i's flat
 *              gradient.  One pass steps all k shards and casts them into
 *              their places of the full buffer: what k one-rank views would
 *              do, in one launch.  k = 1 is rank r's view; r = 0, k = N holds
 *              the same state as the all-ranks view.  Stage 3 likewise per
 *              unit: k*S_u floats and persistent param elements, grads of
 *              k*S_u elements.
 *
 * Numerics (every backend path follows this exactly, element by element):
 *   acc = g_0 + g_1 + ... + g_{N-1}      (fp32, rank order, starting at g_0)
 *   g   = acc / N, then g = g / loss_scale when loss_scale > 0
 *   nonfinite |= !isfinite(g)            (over every element of the step)
 *   m   = b1*m + (1-b1)*g ;  v = b2*v + (1-b2)*(g*g)
 *   x   = x - (lr * (m/(1-b1^t))) / (sqrt(v/(1-b2^t)) + eps)
 *         (AdamW, zero_set_weight_decay: x*(1 - lr*wd) in place of the first x)
 *   param = round-to-nearest-even(x) in the param type
 * each operation a single IEEE binary32 operation (no fused multiply-add, no
 * flush to zero).  lr, b1, b2 and eps arrive as doubles; the fp32 scalars
 * b1, b2, 1-b1, 1-b2, 1-b1^t, 1-b2^t, lr and eps are computed in double on the
 * host and rounded once.  Padding positions (flat index >= numel) take grad 0
 * and therefore stay exactly +0.
 *
 * Conventions:
 *   - Every call returns an int: >= 0 is success (ZERO_OK, or ZERO_SKIPPED
 *     from zero_step_status), < 0 an error code; zero_strerror() names it and
 *     zero_last_error() gives a message for the calling thread.  A call that
 *     fails launches nothing.
 *   - The caller owns every device buffer (allocated by PyTorch or
 *     cudaMalloc).  The library never allocates device memory; the context
 *     itself is a small host object.
 *   - Launching calls are asynchronous on the caller's stream (a
 *     cudaStream_t passed as void*; NULL = legacy default stream).  Only the
 *     calls that read a device word back synchronize: zero_step_status(),
 *     zero_current_state() and zero_gather_timeouts().
 *   - The step kernels and the SM gathers are launched with programmatic
 *     dependent launch: one may be scheduled while the kernel before it in the
 *     stream is finishing, but it touches memory only after that kernel has
 *     completed, so stream order holds as for any launch.
 *   - Device pointers must be aligned to their element size.  16-byte
 *     alignment is not required: unaligned buffers take slower but correct
 *     paths.
 *   - Hyperparameters are checked as torch.optim.Adam checks them: lr >= 0,
 *     0 <= beta1 < 1, 0 <= beta2 < 1, eps >= 0, all finite, t >= 1; a loss
 *     scale must be finite (<= 0 turns scaling off).  Anything else returns
 *     ZERO_EINVAL and launches nothing.
 *   - A context is not thread-safe; use one per host thread.
 *   - Element types: ZERO_F32, ZERO_BF16, ZERO_F16.  master/m/v are fp32.
 */
#ifndef ZERO_GB300_ZERO_H
#define ZERO_GB300_ZERO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct zero_ctx zero_ctx;

enum zero_dtype { ZERO_F32 = 0, ZERO_BF16 = 1, ZERO_F16 = 2 };

enum zero_code {
    ZERO_OK = 0,
    ZERO_SKIPPED = 1,      /* status: the step was skipped (loss-scale overflow) */
    ZERO_EINVAL = -1,      /* bad argument (size, dtype, rank, unit, null pointer) */
    ZERO_ECUDA = -2,       /* a CUDA runtime call failed */
    ZERO_EALIGN = -3,      /* a device pointer is not aligned to its element size */
    ZERO_ESTATE = -4,      /* call not valid in this context's state (e.g. unbound) */
    ZERO_ETIMEOUT = -5     /* a bounded device wait ran out (zero_gather_timeouts) */
};

#define ZERO_MAX_RANKS 256
#define ZERO_HYPER_BYTES 128     /* size of a device block of per-step scalars */

enum zero_gather_mode {
    ZERO_GATHER_FAST = 0,  /* all SMs, many blocks: the fastest placement on an idle GPU */
    ZERO_GATHER_LEAN = 1   /* bulk-copy (TMA) engine, one warp per SM: placement beside compute */
};

/* ------------------------------------------------------------ host only */

/* Shard length S = ceil(numel / world) ("ZeRO 与 FSDP…", 从零实现 ZeRO 的
 * Adam).  Returns -1 when world < 1 or numel < 0. */
int64_t zero_shard_size(int64_t numel, int32_t world);

/* Per-device bytes of model states for `numel` parameters over `world`
 * ranks, mixed-precision Adam (K = 12): stage 0 (plain data parallelism)
 * 16*numel, stage 1 4*numel + 12*numel/world, stage 2 2*numel +
 * 14*numel/world, stage 3 16*numel/world ("论文专题讲解：ZeRO", ZeRO-DP 三阶段;
 * Table 1).  Returns -1.0 on bad arguments. */
double zero_model_state_bytes(int64_t numel, int32_t world, int32_t stage);

/* Loss-scale update after a step, as GradScaler.update does ("PaddlePaddle
 * ZeRO优化", 混合精度才是最佳拍档): a skipped step halves the scale and
 * resets *good_steps; otherwise *good_steps counts up and, on reaching
 * growth_interval (> 0), the scale doubles (unless that would overflow to
 * infinity, when it stays) and the count restarts.
 * Returns the new scale; a NULL good_steps returns the scale unchanged. */
float zero_scale_update(float scale, int32_t skipped, int64_t *good_steps,
                        int64_t growth_interval);

/* Name of a return code.  Never NULL. */
const char *zero_strerror(int code);

/* Message describing the last error returned on the calling thread ("" if
 * none).  Valid until the next failing call on this thread. */
const char *zero_last_error(void);

/* ------------------------------------------------------------- context */

/* Create a context.
 *   numel       parameters in the flat vector (stages 1, 2); ignored for
 *               stage 3, where it must equal the sum of unit_numels.
 *   world       N, data-parallel ranks, 1..ZERO_MAX_RANKS.
 *   stage       1, 2 or 3.  Stages 1 and 2 step identically; stage 1 can
 *               also write the averaged grads (zero_bind_allreduce_out).
 *   grad_dtype, param_dtype  element types of the grads and of the params.
 *   rank        -1 for the all-ranks view, or 0..world-1 for one rank's view.
 *   unit_numels, n_units  stage 3 only: parameter counts of the units
 *               (layers), each sharded on its own with S_u = ceil(numel_u/N).
 *               Must be NULL, 0 for stages 1 and 2.
 * On success *out owns a host allocation released by zero_destroy(). */
int zero_init(zero_ctx **out, int64_t numel, int32_t world, int32_t stage,
              int32_t grad_dtype, int32_t param_dtype, int32_t rank,
              const int64_t *unit_numels, int32_t n_units);

/* A context holding the consecutive ranks [first_rank, first_rank + n_ranks)
 * of `world`: the third view above, for a process that is several
 * data-parallel ranks ("ZeRO 与 FSDP…", 从零实现 ZeRO 的 Adam: each rank owns
 * shard r of S = ceil(numel/world); here one process owns k of them).  The
 * other arguments are zero_init's.  Stages 1 and 2: zero_ctx_state_elems()
 * is n_ranks * S, and every call works as in one rank's view over that
 * longer range (bucket offsets run over [0, n_ranks*S)).  Stage 3: unit u's
 * state, scratch and persistent params are its n_ranks * S_u elements
 * (zero_ctx_unit_state_offset gives where they start), and every unit call
 * works as in one rank's view over them; the gathers still place `world`
 * shards of S_u.  ZERO_EINVAL for ranks not within [0, world) or as
 * zero_init. */
int zero_init_ranks(zero_ctx **out, int64_t numel, int32_t world, int32_t stage,
                    int32_t grad_dtype, int32_t param_dtype, int32_t first_rank,
                    int32_t n_ranks, const int64_t *unit_numels, int32_t n_units);

/* A stage-3 context in FSDP2's per-parameter layout ("ZeRO 与 FSDP…", section
 * ZeRO-3 与 FSDP: each parameter is a DTensor sharded along dim 0, a
 * (256,64) weight over 2 ranks being (128,64) on each).  Unit u is one
 * parameter of rows[u] rows of row_elems[u] elements (the product of its
 * other dimensions); it is cut into chunks of ceil(rows/N) whole rows, rank r
 * holding rows [r*c, r*c + c) and zero rows past the end (ranks past the last
 * row hold padding only).  Its shard length is ceil(rows/N) * row_elems; all
 * stage-3 calls then work as for zero_init's units, and a gather places the
 * N chunks one after another, i.e. the parameter's rows in order followed by
 * the padding rows. */
int zero_init_dim0(zero_ctx **out, int32_t world, int32_t grad_dtype, int32_t param_dtype,
                   int32_t rank, const int64_t *rows, const int64_t *row_elems, int32_t n_units);

int zero_destroy(zero_ctx *ctx);

/* Geometry of a context.  unit = -1 means the whole flat vector (stages 1,
 * 2); for stage 3 pass a unit id.  Return -1 on bad arguments. */
int64_t zero_ctx_shard_size(const zero_ctx *ctx, int32_t unit);
/* floats the caller allocates for each of master, m and v */
int64_t zero_ctx_state_elems(const zero_ctx *ctx);
/* param-type elements of the bound parameter buffer: P for stages 1 and 2
 * (the full vector), and for stage 3 the persistent shards: sum of P_u
 * (all ranks) or sum of S_u (one rank) */
int64_t zero_ctx_param_elems(const zero_ctx *ctx);
/* where unit u starts inside the bound state (and scratch) and param buffers */
int64_t zero_ctx_unit_state_offset(const zero_ctx *ctx, int32_t unit);
int64_t zero_ctx_unit_param_offset(const zero_ctx *ctx, int32_t unit);

/* Bytes of fp32 master + m + v the bound state occupies: 12 *
 * zero_ctx_state_elems (what ZeroAdam.state_bytes() reports per rank in
 * "ZeRO 与 FSDP…", 从零实现 ZeRO 的 Adam, for the one-rank view). */
int64_t zero_state_bytes(const zero_ctx *ctx);

/* ---------------------------------------------------- caller's buffers */

/* Bind the caller's device buffers (the caller keeps ownership).
 *   master, m, v  zero_ctx_state_elems() floats each.  The caller
 *                 initializes master and zeroes m and v before step 1.
 *   params        zero_ctx_param_elems() elements of param_dtype: the full
 *                 parameter buffer every rank holds (stages 1, 2), or the
 *                 persistent parameter shards (stage 3).
 *   g_scratch     zero_ctx_state_elems() floats, or NULL.  Needed only by
 *                 the two-pass loss-scaled path (zero_step with loss_scale >
 *                 0, zero_step_reduce, zero3_reduce_unit): the reduced and
 *                 unscaled grads wait there until the global overflow
 *                 verdict is known.
 *   flag          one 8-byte device word, zeroed by the caller before the
 *                 first step.  Holds the id of the latest step that saw a
 *                 non-finite grad; never needs clearing.
 * May be called again to rebind.
 *
 * Saving and resuming: the whole optimizer state is in the caller's
 * buffers.  To save, copy master, m and v (with two state sets, the current
 * one: zero_current_state) and params, and keep the step count t and the
 * loss-scale state (scale, good steps).  To resume, create a context of the
 * same shape, bind buffers holding those copies (the saved set as the
 * zero_bind set; a second set's cur word zeroed), zero the flag word, and
 * continue with t + 1.  Step ids restart at 1 in a new context, so a flag
 * word kept from another context could name one of them: it must be zeroed
 * ("PaddlePaddle ZeRO优化", sharded checkpoints: each rank saves and restores
 * its own shard of the optimizer state). */
int zero_bind(zero_ctx *ctx, float *master, float *m, float *v, void *params,
              float *g_scratch, uint64_t *flag);

/* Stage 1 only: also write the all-reduced mean grad (acc / N, before
 * unscaling, in grad_dtype) to `grad_avg` (guanweilu.cn article 1460, Stage
 * 1: each rank keeps the full averaged gradient).  All ranks: P elements,
 * every position.  One rank: rank r writes its S positions at r*S of a
 * P-element buffer.  NULL turns it off. */
int zero_bind_allreduce_out(zero_ctx *ctx, void *grad_avg);

/* Bind a second fp32 state set so that every step is one pass, loss-scaled
 * or not (stages 1 and 2; for stage 3 see zero3_begin_step_scaled and
 * zero3_end_step): the step reads the current set, writes the
 * other, and a small finalize kernel then makes the written set current --
 * unless the step is loss-scaled and overflowed, in which case the old set
 * stays current and the params are cast again from it ("PaddlePaddle
 * ZeRO优化", 混合精度才是最佳拍档: the skipped step changes nothing).  This
 * trades zero_ctx_state_elems() * 12 more bytes of memory for the two-pass
 * path's extra scratch write and read (8 bytes per element).
 *   master_b, m_b, v_b  zero_ctx_state_elems() floats each (contents unused
 *               until written).
 *   cur         one 8-byte device word, zeroed by the caller before the first
 *               step: bit 0 clear = the zero_bind set is current, set = this
 *               one.  Read it with zero_current_state().
 * All four NULL unbinds.  With a second set bound, zero_step_apply and
 * zero_step_noalloc update whichever set is current, in place (stages 1 and
 * 2).  ZERO_ESTATE while a stage-3 step is open. */
int zero_bind_shadow(zero_ctx *ctx, float *master_b, float *m_b, float *v_b, uint64_t *cur);

/* Synchronizes the stream of the last step and reports which state set holds
 * the current master/m/v: 0 = the zero_bind buffers, 1 = the second set.
 * Always 0 without a second set. */
int zero_current_state(zero_ctx *ctx, int32_t *which);

/* At most blocks_per_sm resident blocks per SM for this context's step
 * kernels (the fused step, the two passes, the finalize); 0, the default,
 * takes as many as fit (four of 256 threads at 64 registers for 16-bit
 * grads, which is every register of an SM).  A lower number leaves room on
 * every SM for a kernel that runs at the same time -- the step of a bucket
 * during the backward of the next ("论文专题讲解：ZeRO", ZeRO-DP 三阶段: the
 * gradients are reduce-scattered while backward goes on) -- at some cost to
 * the step alone.  Results do not depend on it.  ZERO_EINVAL outside [0, 32]. */
int zero_set_step_occupancy(zero_ctx *ctx, int32_t blocks_per_sm);

/* Decoupled weight decay (AdamW; Loshchilov & Hutter, "Decoupled Weight
 * Decay Regularization", ICLR 2019 -- "PaddlePaddle ZeRO优化" names AdamW as
 * the optimizer whose states are sharded).  From the next step on, every
 * update scales the master weight by fp32(1 - lr*weight_decay) before
 * subtracting the Adam step:  x = x*(1 - lr*wd) - lr*m_hat/(sqrt(v_hat)+eps).
 * 0 (the default) is plain Adam.  Returns ZERO_EINVAL for a negative or
 * non-finite value. */
int zero_set_weight_decay(zero_ctx *ctx, double weight_decay);

/* ------------------------------------------- steps captured in a graph */

/* Bind a device block of ZERO_HYPER_BYTES (16-byte aligned; NULL unbinds)
 * from which every kernel of this context then reads the step's scalars (the
 * Adam scalars, the averaging and loss-scale divisors, the step id) instead of
 * taking them as launch arguments -- so a whole step, however many launches
 * it makes, can be captured once in a CUDA graph and replayed step after
 * step.  With a block bound, a step is:
 *   1. zero_prepare_step(ctx, host_block, ...): starts the step (new step id,
 *      loss scaling on or off) and writes its scalars into host_block
 *      (ZERO_HYPER_BYTES of host memory; pinned, when the copy is captured);
 *   2. a copy of host_block into the device block on the stream (inside the
 *      graph: a memcpy node), before the step's kernels;
 *   3. the step's calls (zero_step, the bucket calls, zero3_begin_step and
 *      the unit calls, ...), or the replay of a graph that captured them.
 *      They no longer start steps; their lr, betas, eps and t arguments are
 *      not used (the block's are), and loss scaling must be on exactly when
 *      the prepared step has it.
 * zero_step_status reads the verdict of the prepared step as usual.
 * A host block must not be refilled before the copy that reads it has run:
 * with steps queued ahead of the GPU, alternate two host blocks (two
 * captured graphs) and wait on an event recorded after the older one.
 * The kernels read the scalars as constant-bank operands: each bound context
 * holds one of 8 constant-memory slots per device (ZERO_ESTATE when all are
 * taken; unbinding or zero_destroy frees it), and the step's first launch
 * copies the device block into the slot on its stream (one small copy per
 * step, captured with the step).  Binding the slot's own address
 * (zero_hyper_slot) as the block removes that copy: step 2 then writes the
 * slot directly.  The device advance (zero_advance_step) needs a block in
 * ordinary device memory, which it rewrites. */
int zero_bind_hyper(zero_ctx *ctx, void *d_hyper);

/* The device address of this context's constant slot (claimed if it holds
 * none yet): a ZERO_HYPER_BYTES block that a host-to-device copy may fill
 * directly, to be bound with zero_bind_hyper. */
int zero_hyper_slot(zero_ctx *ctx, void **d_slot);

/* Step 2 for a context bound to its own constant slot: copy host_block
 * (ZERO_HYPER_BYTES, pinned when captured) into the slot on `stream`. */
int zero_load_hyper(zero_ctx *ctx, const void *host_block, void *stream);
int zero_prepare_step(zero_ctx *ctx, void *host_hyper, double lr, double beta1, double beta2,
                      double eps, int64_t t, float loss_scale);

/* Scalars that advance on the device: asynchronous loss scaling.  With a
 * device scalar block bound, zero_advance_step() launched after a step's
 * kernels does on the GPU what the host otherwise does between steps: it
 * reads the step's overflow verdict, applies the loss-scale policy of
 * zero_scale_update (halve on a skipped step; t advances only on applied
 * steps; double after growth_interval clean steps, never to infinity) and
 * rewrites the block for the next step -- bias corrections 1 - beta^t from
 * a table the host computed (the same values zero_prepare_step derives), the
 * unscale factor from the new scale, the next step id.  No host round trip
 * per step: a loss-scaled training loop, or one CUDA graph of [step,
 * advance] replayed, runs without reading the verdict back.  lr, betas, eps
 * and the weight decay stay as the block has them.
 *
 * zero_advance_table_bytes(t_max): bytes of the table for steps 1..t_max
 *   (8 per step), or -1.
 * zero_fill_advance_table(host_table, t_max, beta1, beta2): fill a host
 *   buffer of that size (two floats per step); the caller copies it to the
 *   device.
 * zero_advance_state(host_state, t, loss_scale, growth_interval): fill the
 *   32-byte state block -- {int64 t; float scale; int32 status; int64
 *   good_steps; int64 growth_interval} -- for the step the block describes
 *   (the one zero_prepare_step prepared); the caller copies it to the device
 *   and may read it back at any time (status 1: the table ran out and the
 *   block stopped advancing).
 * zero_bind_advance(ctx, d_table, t_max, d_state): bind both (NULL, NULL
 *   unbinds); the table 4-byte, the state 8-byte aligned.
 * zero_advance_step(ctx, stream): the advance itself (one small launch).  The
 *   context's host-side step id advances with it, so zero_step_status()
 *   describes the step before the last advance only until that advance is
 *   issued; read the verdict before advancing, or read the state block. */
int64_t zero_advance_table_bytes(int64_t t_max);
int zero_fill_advance_table(void *host_table, int64_t t_max, double beta1, double beta2);
int zero_advance_state(void *host_state, int64_t t, float loss_scale, int64_t growth_interval);
int zero_bind_advance(zero_ctx *ctx, const void *d_table, int64_t t_max, void *d_state);
int zero_advance_step(zero_ctx *ctx, void *stream);

/* ------------------------------------------------------------ the step */

/* One ZeRO step (stages 1, 2) on `stream`.
 *   grads, n_grads  host array of n_grads == world device pointers (see the
 *                   two views above).
 *   lr, beta1, beta2, eps  Adam hyperparameters; t >= 1 is the step count,
 *                   advanced by the caller only for applied steps.
 *   loss_scale      <= 0: no loss scaling, one fused pass (reduce-scatter +
 *                   average + Adam + cast + all-gather placement); a
 *                   non-finite grad is still reported by zero_step_status
 *                   but never skips the step.  > 0: grads are divided by it
 *                   after averaging, and if any element of the step is
 *                   non-finite the step changes nothing.  With a second
 *                   state set bound (zero_bind_shadow) that is still one
 *                   pass; otherwise two passes, zero_step_reduce then
 *                   zero_step_apply (needs g_scratch).
 * The overflow verdict is read with zero_step_status() after the stream
 * reaches it. */
int zero_step(zero_ctx *ctx, const void *const *grads, int32_t n_grads, double lr,
              double beta1, double beta2, double eps, int64_t t, float loss_scale,
              void *stream);

/* First pass of the two-pass step: reduce-scatter sum, average, unscale
 * (loss_scale > 0 divides), write the grads to g_scratch and record a
 * non-finite value in the flag word.  Starts a new step. */
int zero_step_reduce(zero_ctx *ctx, const void *const *grads, int32_t n_grads,
                     float loss_scale, void *stream);

/* Second pass: Adam from g_scratch on every element of the bound state, cast
 * and placement -- unless the flag word names the current step, in which
 * case the kernel returns without writing.  In the one-rank view the flag
 * word may first be combined with the other ranks' words (a MAX
 * all-reduce in a multi-process deployment); for stage 3 call it once after
 * every unit's zero3_reduce_unit.  ZERO_ESTATE while a bucketed step is
 * open. */
int zero_step_apply(zero_ctx *ctx, double lr, double beta1, double beta2, double eps,
                    int64_t t, void *stream);

/* ------------------------------------------------------- bucketed step */

/* The step one bucket at a time, as ZeRO-2 reduce-scatters gradient buckets
 * during backward and frees each full bucket at once ("ZeRO 与 FSDP…", 从零
 * 实现 ZeRO 的 Adam, closing note: real ZeRO-2 reduce-scatters by bucket so
 * resident grads fall to 1/N).  Here a bucket is a range [offset,
 * offset+count) of this context's elements (stages 1 and 2; all ranks: the
 * P-element vector; one rank: its S-element shard), and grads[k] hold only
 * that range of rank k's grads -- constant-size buffers reused bucket after
 * bucket.  A step is zero_bucket_begin, bucket calls covering every element
 * once (any order, any sizes), then zero_bucket_end; the result equals
 * zero_step's bit for bit.
 *   - No loss scaling: each bucket is updated in place at once.
 *   - Loss-scaled with a second state set: each bucket writes the other
 *     set; zero_bucket_end makes it current or, on overflow, keeps the old.
 *   - Loss-scaled with g_scratch only: each bucket is reduced into the
 *     scratch; zero_bucket_end applies Adam to every element, or to none.
 * Bucket offsets that are multiples of 8 elements keep every access on the
 * 16-byte vector path. */
/* With one process per rank (the one-rank view), zero_bucket_end of a
 * loss-scaled step decides from the flag word: combine it with the other
 * ranks' words first (a MAX all-reduce), as before zero_step_apply. */
int zero_bucket_begin(zero_ctx *ctx, float loss_scale);
int zero_bucket_step(zero_ctx *ctx, int64_t offset, int64_t count, const void *const *grads,
                     int32_t n_grads, double lr, double beta1, double beta2, double eps,
                     int64_t t, void *stream);
int zero_bucket_end(zero_ctx *ctx, double lr, double beta1, double beta2, double eps,
                    int64_t t, void *stream);

/* Synchronizes the stream of the context's last step launch (gathers do not
 * count: they never touch the flag) and reads the flag.
 * *nonfinite (may be NULL) = 1 if the step saw an inf/nan; *skipped (may be
 * NULL) = 1 if the step was loss-scaled and therefore skipped.  Returns
 * ZERO_SKIPPED when skipped, ZERO_OK otherwise, < 0 on error. */
int zero_step_status(zero_ctx *ctx, int32_t *nonfinite, int32_t *skipped);

/* The id of the current step (what the flag word holds when it overflowed). */
uint64_t zero_step_id(const zero_ctx *ctx);

/* ------------------------------------------------------------ all-gather */

/* Place the N shards of S = zero_ctx_shard_size(ctx, -1) elements of `dtype`
 * into `full` (N*S elements): shard k lands at k*S ("ZeRO 与 FSDP…",
 * all_gather_into_tensor).  shards is a host array of n_shards == world
 * device pointers; a NULL entry is skipped (e.g. the own shard, already
 * written by zero_step in the one-rank view).  Shard and destination may
 * have any element-aligned addresses. */
int zero_allgather(zero_ctx *ctx, const void *const *shards, int32_t n_shards,
                   void *full, int32_t dtype, void *stream);

/* How this context's gathers (zero_allgather, zero3_gather_unit) run.
 * ZERO_GATHER_FAST (default) fills every SM with copy blocks -- the fastest
 * placement when nothing else runs, but blocks queued first hold the SMs, so
 * a compute kernel launched after it waits.  ZERO_GATHER_LEAN drives the
 * SMs' bulk-copy (TMA) units from one warp per SM through a 128 KB shared
 * ring: nearly as fast alone, and it leaves the SMs' threads and registers to
 * kernels running at the same time -- the ZeRO-3 prefetch of the next unit
 * while this one computes ("ZeRO 与 FSDP…", ZeRO-3 与 FSDP: prefetch hides the
 * all-gather behind the computation).  LEAN needs 16-byte aligned shards and
 * destinations and a shard length that is a multiple of 16 bytes; other
 * gathers fall back to FAST.  Its waits are bounded: see
 * zero_gather_timeouts. */
int zero_set_gather_mode(zero_ctx *ctx, int32_t mode);

/* Number of lean-gather waits that ran out in this process (each one drains
 * its copies in flight and abandons the rest of that gather; the result is
 * then incomplete).  0 in normal operation.  Returns ZERO_OK when the count
 * is 0, ZERO_ETIMEOUT (the count still written) when a wait ran out, and
 * ZERO_ECUDA when the counter cannot be read.  Read it after the gathers'
 * streams are synchronized. */
int zero_gather_timeouts(uint32_t *count);

/* How many times the lean gather polls for each tile's load before it gives
 * up on that gather (the drain of the loads in flight after a give-up always
 * polls for the full default).  polls >= 0 sets the limit -- 0 makes every
 * such wait run out at once, which exercises the timeout path without a
 * fault; polls < 0 restores the default (2^22 polls, seconds at the least).
 * Process-wide; synchronous; call it only while no lean gather is in flight.
 * Returns ZERO_OK, or ZERO_ECUDA when the device variable cannot be set. */
int zero_set_gather_wait_polls(int64_t polls);

/* ------------------------------------------------------------- stage 3 */

/* Begin a stage-3 step: the units' calls until the next begin share one
 * step id and one overflow verdict.  Same as zero3_begin_step_scaled(ctx, 0). */
int zero3_begin_step(zero_ctx *ctx);

/* Begin a stage-3 step with loss scaling (loss_scale > 0: grads divided by
 * it, and the step skipped when any unit's grads hold inf/nan).  Two ways to
 * run it:
 *   - one state set: zero3_reduce_unit (or _group) for every unit, then one
 *     zero_step_apply (the fp32 scratch holds the grads until the verdict);
 *   - a second state set bound (zero_bind_shadow): zero3_step_unit (or
 *     _group) for every unit, each one pass that reads the current set and
 *     writes the other, then zero3_end_step, which makes the written set
 *     current or, when some unit overflowed, keeps the old set and casts
 *     every unit's params again from it -- the skip without a second pass
 *     ("PaddlePaddle ZeRO优化", 混合精度才是最佳拍档).
 * With a second set bound every stage-3 step, scaled or not, runs the second
 * way and must end with zero3_end_step before the next begins (ZERO_ESTATE
 * otherwise); zero3_reduce_unit/_group and zero_step_apply are refused. */
int zero3_begin_step_scaled(zero_ctx *ctx, float loss_scale);

/* End a stage-3 step begun with a second state set bound (the finalize
 * described above, one small launch); without one it does nothing.  In the
 * one-rank view with one process per rank, combine the flag word with the
 * other ranks' words first (a MAX all-reduce of the 8 bytes: every rank runs
 * the same step ids), so that every rank keeps or discards the step alike. */
int zero3_end_step(zero_ctx *ctx, void *stream);

/* Gather unit `unit`'s N parameter shards (S_u elements of param_dtype
 * each) into unit_full (N*S_u elements), before the unit's forward and again
 * before its backward ("ZeRO 与 FSDP…", ZeRO-3 与 FSDP).  NULL shards are
 * skipped. */
int zero3_gather_unit(zero_ctx *ctx, int32_t unit, const void *const *shards,
                      int32_t n_shards, void *unit_full, void *stream);

/* Reduce-scatter + average + Adam + cast for unit `unit` in one fused pass:
 * without loss scaling, or loss-scaled into the second state set (see
 * zero3_begin_step_scaled; with one set a skip would need every unit's
 * verdict first).
 * grads follow the view: all ranks -> numel_u-element local grads of the
 * unit; one rank -> S_u-element slices.  The cast shard is written to the
 * unit's place in the bound param buffer. */
int zero3_step_unit(zero_ctx *ctx, int32_t unit, const void *const *grads,
                    int32_t n_grads, double lr, double beta1, double beta2, double eps,
                    int64_t t, void *stream);

/* One visit of the stage-3 backward in one call: unit `unit`'s step (as
 * zero3_step_unit, same arguments and conditions) and the gather of unit
 * `gather_unit`'s shards into unit_full (as zero3_gather_unit).  In the
 * backward each unit is gathered before its backward and reduce-scattered
 * and updated after it ("ZeRO 与 FSDP…", section ZeRO-3 与 FSDP), so once unit
 * u's backward is done, u's update and the gather of the unit visited next
 * (u - 1) are both due; issuing them together saves one launch per unit,
 * which is most of the cost of small units.  The result equals the two
 * calls in either order, bit for bit.
 *   - gather_unit must differ from unit, and the two halves must touch
 *     disjoint memory: unit_full and the shards may not overlap the stepped
 *     unit's params, state, flag or current-set word, and unit_full may not
 *     overlap its grads (ZERO_EINVAL, nothing launched).
 *   - One launch (a kernel whose first blocks run the unit's fused pass and
 *     whose other blocks place the shards) for the default gather mode;
 *     in the lean mode, with a bound scalar block, with a capped step
 *     occupancy, or for shards of 32 MiB or more it makes the two launches
 *     of the two calls instead. */
int zero3_step_unit_gather(zero_ctx *ctx, int32_t unit, const void *const *grads,
                           int32_t n_grads, double lr, double beta1, double beta2, double eps,
                           int64_t t, int32_t gather_unit, const void *const *shards,
                           int32_t n_shards, void *unit_full, void *stream);

/* A visit of two units in one call: the steps of units [first_unit,
 * first_unit + n_units) (1 or 2 units, each as zero3_step_unit; grads holds
 * n_units * world pointers, unit-major) and the gathers of units
 * [gather_first, gather_first + gather_n) (0 to 2 units, as
 * zero3_gather_unit into unit_fulls[j]; shards holds gather_n * world
 * pointers, unit-major).  With two unit buffers the backward can step two
 * units and gather the two visited next at once ("ZeRO 与 FSDP…", ZeRO-3 与
 * FSDP: the next units' all-gathers issued before the current ones are
 * done), halving the launches of zero3_step_unit_gather.  The result equals
 * the separate calls, bit for bit.
 *   - The gathered units must not be stepped ones, the two unit buffers must
 *     not overlap, and every gather must touch memory disjoint from every
 *     step as for zero3_step_unit_gather (ZERO_EINVAL, nothing launched).
 *   - One launch for the default gather mode when the placed shards number
 *     64 at most and are under 32 MiB each; otherwise (and in the lean mode,
 *     with a bound scalar block or a capped step occupancy) the launches of
 *     the separate calls. */
int zero3_step_units_gather(zero_ctx *ctx, int32_t first_unit, int32_t n_units,
                            const void *const *grads, int32_t n_grads, double lr, double beta1,
                            double beta2, double eps, int64_t t, int32_t gather_first,
                            int32_t gather_n, const void *const *shards, int32_t n_shards,
                            void *const *unit_fulls, void *stream);

/* Loss-scaled stage 3: first pass for one unit (as zero_step_reduce on the
 * unit's range).  After every unit, one zero_step_apply() applies Adam to all
 * units, or to none if any unit overflowed. */
int zero3_reduce_unit(zero_ctx *ctx, int32_t unit, const void *const *grads,
                      int32_t n_grads, float loss_scale, void *stream);

/* Groups of units: FSDP2 shards every parameter tensor on dim 0 and
 * gathers and reduces the parameters of one module together ("ZeRO 与
 * FSDP…", ZeRO-3 与 FSDP: per-parameter dim-0 sharding; a module's
 * parameters form one gather unit).  With one unit per parameter tensor
 * (zero_init_dim0), a group is a run of consecutive units -- a module's
 * parameters -- handled in one launch.
 *
 * zero3_gather_group: units [first_unit, first_unit + n_units) at once.
 *   shards      n_units * N pointers, unit-major: shards[ul*N + k] is shard k
 *               (S_u elements) of unit first_unit + ul; NULL skips it.
 *   unit_fulls  n_units destinations of N*S_u elements each (as
 *               zero3_gather_unit's unit_full).
 * At most 512 shards per call (n_units * N); any element alignment.  In the
 * lean mode (zero_set_gather_mode) a group whose shards and destinations are
 * all 16-byte aligned with lengths that are multiples of 16 bytes runs on the
 * bulk-copy engine; any other group takes the SM placement. */
int zero3_gather_group(zero_ctx *ctx, int32_t first_unit, int32_t n_units,
                       const void *const *shards, int32_t n_shards, void *const *unit_fulls,
                       void *stream);

/* zero3_step_group / zero3_reduce_group: zero3_step_unit / zero3_reduce_unit
 * over units [first_unit, first_unit + n_units) in one launch.  grads[k]
 * holds rank k's grads of every unit of the group end to end, in unit order
 * -- one rank: S_u-element slices; all ranks: numel_u-element local grads --
 * the layout of one flat reduce-scatter buffer per module.  Every unit of the
 * group must be free of padding in this view (one rank: numel_u >= (r+1)*S_u;
 * all ranks: numel_u == N*S_u); otherwise ZERO_EINVAL, and that unit is
 * stepped on its own.  Results are bit-identical to the per-unit calls. */
int zero3_step_group(zero_ctx *ctx, int32_t first_unit, int32_t n_units,
                     const void *const *grads, int32_t n_grads, double lr, double beta1,
                     double beta2, double eps, int64_t t, void *stream);
int zero3_reduce_group(zero_ctx *ctx, int32_t first_unit, int32_t n_units,
                       const void *const *grads, int32_t n_grads, float loss_scale,
                       void *stream);

/* ------------------------------------------------ step without allocation */

/* The pages have no counterpart of this call; it serves callers that can
 * hand the library only their inputs and outputs and cannot call cudaMalloc
 * for a scratch buffer -- for example a plugin whose host framework owns all
 * device memory, or a code path that must not trigger cudaMalloc's implicit
 * device synchronization.
 *
 * Same step as zero_step (stages 1 and 2, either view; loss_scale <= 0 means
 * no unscaling and no skip), always run as the two passes, with the fp32
 * scratch taken from a fixed 16 MiB array inside the library (4,194,304
 * floats) instead of the bound g_scratch, which may be NULL.  Every GPU that
 * loads the library holds that array until the process exits.  The call
 * allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 *   - The rank's range (zero_ctx_state_elems) must be at most 4,194,304
 *     elements; larger ranges return ZERO_EINVAL with a message and launch
 *     nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - All calls in the process share the one array per device, and it keeps
 *     the last call's contents.  Nothing in it needs to start at zero: the
 *     first pass writes every element the second pass reads.  Calls that
 *     overlap on the GPU (different streams, or contexts used concurrently)
 *     race on the array and corrupt each other's results; calls on one
 *     stream are ordered and safe.
 * ZERO_ESTATE while a bucketed step is open.  The verdict is read with
 * zero_step_status() as for zero_step. */
int zero_step_noalloc(zero_ctx *ctx, const void *const *grads, int32_t n_grads, double lr,
                      double beta1, double beta2, double eps, int64_t t, float loss_scale,
                      void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_GB300_ZERO_H */
