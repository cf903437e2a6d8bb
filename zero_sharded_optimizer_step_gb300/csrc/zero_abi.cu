// C ABI of the ZeRO step library: argument checking, geometry of the flat
// sharded vector, the per-step fp32 scalars, and the kernel launches.  The
// declarations and their contracts are in include/zero.h.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/zero.h"
#include "zero_internal.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(ZERO_ECUDA, "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
}

bool valid_dtype(int32_t d) { return d == ZERO_F32 || d == ZERO_BF16 || d == ZERO_F16; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned(const void *p, int64_t a) { return ((uintptr_t)p % (uintptr_t)a) == 0; }

int align_of(const void *p)
{
    const uintptr_t u = (uintptr_t)p;
    return (u & 15) == 0 ? 16 : (u & 7) == 0 ? 8 : (u & 3) == 0 ? 4 : (u & 1) == 0 ? 2 : 1;
}

// A power of two whose reciprocal is a normal binary32 (so multiplying by
// the reciprocal rounds exactly like dividing).
bool pow2_with_normal_inverse(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    const uint32_t exp = (u >> 23) & 0xffu, man = u & 0x7fffffu;
    return (u >> 31) == 0 && man == 0 && exp >= 1 && exp <= 253;
}

}  // namespace

struct zero_ctx {
    int64_t numel = 0;
    int32_t world = 1, stage = 2, gdt = 0, pdt = 0, rank = -1;
    int32_t nranks = 1;          // rank >= 0: the view holds ranks [rank, rank + nranks)
    int64_t S = 0, P = 0;
    std::vector<int64_t> unit_numel, unit_S, unit_state_off;
    int64_t state_elems = 0, param_elems = 0;

    float *master = nullptr, *m = nullptr, *v = nullptr, *g = nullptr;
    float *xb = nullptr, *mb = nullptr, *vb = nullptr;   // second state set
    uint64_t *cur = nullptr;                              // which set is current
    void *params = nullptr, *grad_avg = nullptr;
    uint64_t *flag = nullptr;
    bool bound = false;
    int device = -1, sms = 0;

    double weight_decay = 0.0;   // AdamW's decoupled decay; 0 = Adam
    int32_t gather_mode = 0;     // ZERO_GATHER_FAST or ZERO_GATHER_LEAN
    int32_t step_per_sm = 0;     // > 0: step kernels use at most this many blocks per SM

    void *hyper = nullptr;       // device block of per-step scalars (graph capture)
    int hyper_slot = -1;         // its constant-memory slot on hyper_device
    int hyper_device = -1;
    bool slot_stale = false;     // the step's first launch copies the block into the slot
    bool hyper_direct = false;   // the bound block is the slot itself (no copy)
    const float *adv_table = nullptr;   // zero_bind_advance: bias corrections per t
    int64_t adv_tmax = 0;
    void *adv_state = nullptr;          // 32-byte device step state

    uint64_t step_id = 0;
    bool step_scaled = false;
    bool bucket_open = false;    // between zero_bucket_begin and zero_bucket_end
    float bucket_scale = 0.0f;
    // stage 3 with two state sets: units step into the other set between
    // zero3_begin_step(_scaled) and zero3_end_step, which finalizes once
    bool stage3_open = false;
    float step_scale = 0.0f;     // the loss scale of the open stage-3 step
    cudaStream_t last_stream = nullptr;
};

namespace zgb {

int resident_blocks_per_sm(const void *kernel, int threads)
{
    struct Entry { const void *k; int dev, threads, blocks; };
    static std::mutex mu;
    static std::vector<Entry> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry &e : cache)
        if (e.k == kernel && e.dev == dev && e.threads == threads) return e.blocks;
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, threads, 0) != cudaSuccess || b < 1) {
        cudaGetLastError();
        b = 1;
    }
    cache.push_back({kernel, dev, threads, b});
    return b;
}

}  // namespace zgb

namespace {

using zgb::StepArgs;

int check_ready(zero_ctx *c)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (!c->bound) return fail(ZERO_ESTATE, "no buffers bound (call zero_bind first)");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != c->device)
        return fail(ZERO_ESTATE, "current device %d is not the device %d the buffers were bound on",
                    dev, c->device);
    return ZERO_OK;
}

int check_ptr_array(const void *const *p, int32_t n, int32_t world, int es, bool need,
                    const char *what)
{
    if (n != world) return fail(ZERO_EINVAL, "%s: %d pointers given, world is %d", what, n, world);
    if (!p) return fail(ZERO_EINVAL, "%s: null pointer array", what);
    for (int32_t k = 0; k < n; ++k) {
        if (!p[k]) {
            if (need) return fail(ZERO_EINVAL, "%s[%d] is null", what, k);
            continue;
        }
        if (!aligned(p[k], es))
            return fail(ZERO_EALIGN, "%s[%d] is not aligned to its %d-byte elements", what, k, es);
    }
    return ZERO_OK;
}

zgb::AdamScalars adam_scalars(double lr, double b1, double b2, double eps, int64_t t,
                              double weight_decay)
{
    zgb::AdamScalars s;
    s.decoupled = weight_decay != 0.0;
    s.decay = (float)(1.0 - lr * weight_decay);
    s.lr = (float)lr;
    s.b1 = (float)b1;
    s.b2 = (float)b2;
    s.c1 = (float)(1.0 - b1);
    s.c2 = (float)(1.0 - b2);
    s.bc1 = (float)(1.0 - std::pow(b1, (double)t));
    s.bc2 = (float)(1.0 - std::pow(b2, (double)t));
    s.eps = (float)eps;
    return s;
}

zgb::AverageScalars average_scalars(int32_t world, float loss_scale)
{
    zgb::AverageScalars s{};
    s.world_f = (float)world;
    s.world_pow2 = (world & (world - 1)) == 0;
    s.inv_world = 1.0f / (float)world;
    s.scaled = loss_scale > 0.0f;
    s.scale = s.scaled ? loss_scale : 1.0f;
    s.scale_pow2 = s.scaled && pow2_with_normal_inverse(loss_scale);
    s.inv_scale = 1.0f / s.scale;
    return s;
}

// One contiguous range of the state: [state_off, state_off + n), with the
// first n_valid elements backed by real grads.
struct Range {
    int64_t state_off = 0, n = 0, n_valid = 0;
    char *params = nullptr;     // low-precision destination of element 0
    char *grad_avg = nullptr;   // stage-1 output of element 0, or null
};

// The whole-vector range of stages 1 and 2.
Range vector_range(const zero_ctx *c)
{
    Range r;
    const int es_p = zgb::elem_size(c->pdt), es_g = zgb::elem_size(c->gdt);
    if (c->rank < 0) {
        r.n = c->P;
        r.n_valid = c->numel;
        r.params = static_cast<char *>(c->params);
        r.grad_avg = static_cast<char *>(c->grad_avg);
    } else {
        // the view's consecutive shards, [rank*S, (rank + nranks)*S)
        const int64_t lo = (int64_t)c->rank * c->S;
        r.n = c->S * c->nranks;
        r.n_valid = std::max<int64_t>(0, std::min<int64_t>(r.n, c->numel - lo));
        r.params = static_cast<char *>(c->params) + lo * es_p;
        r.grad_avg = c->grad_avg ? static_cast<char *>(c->grad_avg) + lo * es_g : nullptr;
    }
    return r;
}

// Unit u of stage 3.
Range unit_range(const zero_ctx *c, int32_t u)
{
    Range r;
    const int es_p = zgb::elem_size(c->pdt);
    const int64_t Su = c->unit_S[u];
    r.state_off = c->unit_state_off[u];
    if (c->rank < 0) {
        r.n = Su * c->world;
        r.n_valid = c->unit_numel[u];
    } else {
        // the view's consecutive shards of the unit
        r.n = Su * c->nranks;
        r.n_valid = std::max<int64_t>(0, std::min<int64_t>(r.n, c->unit_numel[u] - (int64_t)c->rank * Su));
    }
    r.params = static_cast<char *>(c->params) + r.state_off * es_p;
    return r;
}

// Constant slots in use, per device.
std::mutex g_slot_mu;
std::vector<std::pair<int, unsigned>> g_slots_used;   // (device, bit mask of slots)

int claim_slot(int dev)
{
    std::lock_guard<std::mutex> lock(g_slot_mu);
    for (auto &e : g_slots_used)
        if (e.first == dev) {
            for (int k = 0; k < zgb::kHyperSlots; ++k)
                if (!(e.second & (1u << k))) {
                    e.second |= 1u << k;
                    return k;
                }
            return -1;
        }
    g_slots_used.push_back({dev, 1u});
    return 0;
}

void release_slot(int dev, int slot)
{
    if (slot < 0) return;
    std::lock_guard<std::mutex> lock(g_slot_mu);
    for (auto &e : g_slots_used)
        if (e.first == dev) e.second &= ~(1u << slot);
}

// The first launch of a step in the graph form copies the context's device
// block into its constant slot, on that launch's stream (so a captured step
// holds the copy too).
int load_slot_if_stale(zero_ctx *c, cudaStream_t s)
{
    if (!c->hyper || !c->slot_stale) return ZERO_OK;
    if (c->hyper_direct) {            // the caller writes the slot itself
        c->slot_stale = false;
        return ZERO_OK;
    }
    const cudaError_t e =
        zgb::load_hyper_slot(c->hyper_slot, static_cast<const zgb::DeviceHyper *>(c->hyper), s);
    if (e != cudaSuccess) return cuda_fail(e, "copying the scalar block to its constant slot");
    c->slot_stale = false;
    return ZERO_OK;
}

StepArgs make_args(const zero_ctx *c, const Range &r, const void *const *grads)
{
    StepArgs a;
    memset(&a, 0, sizeof a);
    a.world = c->world;
    a.n = r.n;
    a.n_valid = r.n_valid;
    a.master = c->master + r.state_off;
    a.m = c->m + r.state_off;
    a.v = c->v + r.state_off;
    a.g = c->g ? c->g + r.state_off : nullptr;
    if (c->cur) {
        a.xb = c->xb + r.state_off;
        a.mb = c->mb + r.state_off;
        a.vb = c->vb + r.state_off;
        a.cur = reinterpret_cast<unsigned long long *>(c->cur);
    }
    a.params = r.params;
    a.grad_avg = r.grad_avg;
    a.param_align = align_of(r.params);
    a.avg_align = r.grad_avg ? align_of(r.grad_avg) : 16;
    a.flag = reinterpret_cast<unsigned long long *>(c->flag);
    a.hyper = static_cast<const zgb::DeviceHyper *>(c->hyper);
    a.slot = c->hyper_slot;
    if (grads)
        for (int32_t k = 0; k < c->world; ++k) a.grads[k] = grads[k];
    a.grad_align = zgb::step_grad_align(a);
    a.vec_ok = zgb::step_vector_path_ok(a) ? 1 : 0;
    return a;
}

// Start a step: a new step id and whether it is loss-scaled.  With a device
// block of scalars bound, zero_prepare_step has started it already (the
// kernels of a captured graph take the id from the block); the call must then
// take the prepared path.
int begin_step(zero_ctx *c, bool scaled)
{
    if (c->hyper) {
        if (c->step_id == 0) return fail(ZERO_ESTATE, "call zero_prepare_step first");
        if (scaled != c->step_scaled)
            return fail(ZERO_EINVAL, "loss scaling differs from the prepared step");
        c->slot_stale = true;
        return ZERO_OK;
    }
    c->step_id += 1;
    c->step_scaled = scaled;
    return ZERO_OK;
}

int finish_launch(zero_ctx *c, cudaError_t e, const char *what, cudaStream_t s)
{
    if (e != cudaSuccess) return cuda_fail(e, what);
    c->last_stream = s;
    return ZERO_OK;
}

int do_reduce(zero_ctx *c, const Range &r, const void *const *grads, float loss_scale,
              cudaStream_t s)
{
    if (r.n == 0) return ZERO_OK;
    if (int rc = load_slot_if_stale(c, s)) return rc;
    StepArgs a = make_args(c, r, grads);
    a.av = average_scalars(c->world, loss_scale);
    a.step_id = c->step_id;
    return finish_launch(c, zgb::launch_reduce(c->gdt, a, c->sms, c->step_per_sm, s),
                         "reduce kernel", s);
}

int do_apply(zero_ctx *c, const Range &r, double lr, double b1, double b2, double eps,
             int64_t t, cudaStream_t s)
{
    if (r.n == 0) return ZERO_OK;
    if (int rc = load_slot_if_stale(c, s)) return rc;
    StepArgs a = make_args(c, r, nullptr);
    a.ad = adam_scalars(lr, b1, b2, eps, t, c->weight_decay);
    // an unscaled step never skips: use an id the flag cannot hold
    a.step_id = c->step_scaled ? c->step_id : ~0ull;
    return finish_launch(c, zgb::launch_apply(c->pdt, a, c->sms, c->step_per_sm, s),
                         "apply kernel", s);
}

int do_finalize(zero_ctx *c, const Range &r, cudaStream_t s)
{
    if (r.n == 0 || !c->cur) return ZERO_OK;
    if (int rc = load_slot_if_stale(c, s)) return rc;
    StepArgs a = make_args(c, r, nullptr);
    a.step_id = c->step_scaled ? c->step_id : ~0ull;
    return finish_launch(c, zgb::launch_finalize(c->pdt, a, c->sms, c->step_per_sm, s),
                         "finalize kernel", s);
}

int do_fused(zero_ctx *c, const Range &r, const void *const *grads, double lr, double b1,
             double b2, double eps, int64_t t, cudaStream_t s, float loss_scale = 0.0f,
             bool finalize = true)
{
    if (r.n == 0) return ZERO_OK;
    if (int rc = load_slot_if_stale(c, s)) return rc;
    StepArgs a = make_args(c, r, grads);
    a.av = average_scalars(c->world, loss_scale);
    a.ad = adam_scalars(lr, b1, b2, eps, t, c->weight_decay);
    a.step_id = c->step_id;
    int rc = finish_launch(
        c, zgb::launch_fused_step(c->gdt, c->pdt, a, c->sms, c->step_per_sm, s), "step kernel", s);
    if (rc || !c->cur || !finalize) return rc;
    // two state sets: the written set becomes current unless the step is
    // loss-scaled and overflowed
    a.step_id = c->step_scaled ? c->step_id : ~0ull;
    return finish_launch(c, zgb::launch_finalize(c->pdt, a, c->sms, c->step_per_sm, s),
                         "finalize kernel", s);
}

// The ranges Adam is defined on (those torch.optim.Adam also enforces):
// lr >= 0, 0 <= beta < 1 (beta2 = 1 would divide by 1 - beta2^t = 0),
// eps >= 0, all finite; t counts from 1.
int check_hyper(double lr, double b1, double b2, double eps, int64_t t)
{
    if (t < 1) return fail(ZERO_EINVAL, "step count t must be >= 1 (got %lld)", (long long)t);
    if (!(lr >= 0.0) || !std::isfinite(lr))
        return fail(ZERO_EINVAL, "lr must be a finite value >= 0 (got %g)", lr);
    if (!(b1 >= 0.0 && b1 < 1.0)) return fail(ZERO_EINVAL, "beta1 must be in [0, 1) (got %g)", b1);
    if (!(b2 >= 0.0 && b2 < 1.0)) return fail(ZERO_EINVAL, "beta2 must be in [0, 1) (got %g)", b2);
    if (!(eps >= 0.0) || !std::isfinite(eps))
        return fail(ZERO_EINVAL, "eps must be a finite value >= 0 (got %g)", eps);
    return ZERO_OK;
}

// A loss scale is finite; <= 0 turns scaling off.
int check_scale(float loss_scale)
{
    if (!std::isfinite(loss_scale))
        return fail(ZERO_EINVAL, "loss_scale must be finite (<= 0 turns loss scaling off)");
    return ZERO_OK;
}

// The apply pass covers every element of the bound state: the whole vector
// range for stages 1 and 2, all units (laid end to end) for stage 3.
Range apply_range(const zero_ctx *c)
{
    if (c->stage < 3) return vector_range(c);
    Range r;
    r.n = c->state_elems;
    r.params = static_cast<char *>(c->params);
    return r;
}

// Units of stage 3: unit u has numel[u] elements sharded into shard[u] per
// rank (shard[u] * world >= numel[u]); state, scratch and param shards lie
// unit after unit.
int init_units(zero_ctx *c, const int64_t *numel, const int64_t *shard, int32_t n, int64_t total)
{
    const int64_t kLimit = (int64_t)1 << 56;
    int64_t sum = 0, off = 0;
    for (int32_t u = 0; u < n; ++u) {
        const int64_t nu = numel[u], su = shard[u];
        if (nu < 0 || nu > kLimit || su < 0 || su > kLimit || su * c->world < nu)
            return fail(ZERO_EINVAL, "unit %d: bad size (%lld elements, shard %lld)", u,
                        (long long)nu, (long long)su);
        c->unit_numel.push_back(nu);
        c->unit_S.push_back(su);
        c->unit_state_off.push_back(off);
        off += c->rank < 0 ? su * c->world : su * c->nranks;
        sum += nu;
        if (sum > kLimit || off > kLimit) return fail(ZERO_EINVAL, "units too large");
    }
    if (total != sum)
        return fail(ZERO_EINVAL, "numel (%lld) must equal the sum of the units (%lld)",
                    (long long)total, (long long)sum);
    c->numel = sum;
    c->S = -1;
    c->P = -1;
    c->state_elems = off;
    c->param_elems = off;
    return ZERO_OK;
}

}  // namespace

extern "C" {

int64_t zero_shard_size(int64_t numel, int32_t world)
{
    if (world < 1 || numel < 0) return -1;
    return ceil_div(numel, world);
}

double zero_model_state_bytes(int64_t numel, int32_t world, int32_t stage)
{
    if (numel < 0 || world < 1) return -1.0;
    const double p = (double)numel, n = (double)world;
    switch (stage) {
    case 0: return 16.0 * p;
    case 1: return 4.0 * p + 12.0 * p / n;
    case 2: return 2.0 * p + 14.0 * p / n;
    case 3: return 16.0 * p / n;
    }
    return -1.0;
}

float zero_scale_update(float scale, int32_t skipped, int64_t *good_steps, int64_t growth_interval)
{
    if (!good_steps) return scale;
    if (skipped) {
        *good_steps = 0;
        return scale * 0.5f;
    }
    if (++*good_steps >= growth_interval && growth_interval > 0) {
        *good_steps = 0;
        const float grown = scale * 2.0f;      // grow only to a finite scale
        return isfinite(grown) ? grown : scale;
    }
    return scale;
}

const char *zero_strerror(int code)
{
    switch (code) {
    case ZERO_OK: return "ZERO_OK";
    case ZERO_SKIPPED: return "ZERO_SKIPPED";
    case ZERO_EINVAL: return "ZERO_EINVAL: invalid argument";
    case ZERO_ECUDA: return "ZERO_ECUDA: CUDA runtime error";
    case ZERO_EALIGN: return "ZERO_EALIGN: misaligned device pointer";
    case ZERO_ESTATE: return "ZERO_ESTATE: call not valid in this state";
    case ZERO_ETIMEOUT: return "ZERO_ETIMEOUT: a bounded device wait ran out";
    }
    return "unknown zero code";
}

const char *zero_last_error(void) { return g_last_error.c_str(); }

// A context of `nranks` consecutive ranks from `rank` (rank -1: all of them).
static int init_ctx(zero_ctx **out, int64_t numel, int32_t world, int32_t stage,
                    int32_t grad_dtype, int32_t param_dtype, int32_t rank, int32_t nranks,
                    const int64_t *unit_numels, int32_t n_units)
{
    if (!out) return fail(ZERO_EINVAL, "out is null");
    *out = nullptr;
    if (world < 1 || world > ZERO_MAX_RANKS)
        return fail(ZERO_EINVAL, "world must be in [1, %d] (got %d)", ZERO_MAX_RANKS, world);
    if (stage < 1 || stage > 3) return fail(ZERO_EINVAL, "stage must be 1, 2 or 3 (got %d)", stage);
    if (!valid_dtype(grad_dtype) || !valid_dtype(param_dtype))
        return fail(ZERO_EINVAL, "unknown dtype code (grad %d, param %d)", grad_dtype, param_dtype);
    if (rank < -1 || rank >= world)
        return fail(ZERO_EINVAL, "rank must be -1 or in [0, %d) (got %d)", world, rank);
    const int64_t kLimit = (int64_t)1 << 56;
    zero_ctx *c = new zero_ctx;
    c->world = world;
    c->stage = stage;
    c->gdt = grad_dtype;
    c->pdt = param_dtype;
    c->rank = rank;
    c->nranks = rank < 0 ? world : nranks;
    if (stage < 3) {
        if (unit_numels || n_units) {
            delete c;
            return fail(ZERO_EINVAL, "units are only for stage 3");
        }
        if (numel < 0 || numel > kLimit) {
            delete c;
            return fail(ZERO_EINVAL, "numel out of range (%lld)", (long long)numel);
        }
        c->numel = numel;
        c->S = ceil_div(numel, world);
        c->P = c->S * world;
        c->state_elems = rank < 0 ? c->P : c->S * nranks;
        c->param_elems = c->P;
    } else {
        if (!unit_numels || n_units < 1) {
            delete c;
            return fail(ZERO_EINVAL, "stage 3 needs unit_numels and n_units >= 1");
        }
        std::vector<int64_t> shards;
        for (int32_t u = 0; u < n_units; ++u)
            shards.push_back(unit_numels[u] < 0 ? -1 : ceil_div(unit_numels[u], world));
        int rc = init_units(c, unit_numels, shards.data(), n_units, numel);
        if (rc) {
            delete c;
            return rc;
        }
    }
    *out = c;
    return ZERO_OK;
}

int zero_init(zero_ctx **out, int64_t numel, int32_t world, int32_t stage, int32_t grad_dtype,
              int32_t param_dtype, int32_t rank, const int64_t *unit_numels, int32_t n_units)
{
    return init_ctx(out, numel, world, stage, grad_dtype, param_dtype, rank, 1, unit_numels,
                    n_units);
}

int zero_init_ranks(zero_ctx **out, int64_t numel, int32_t world, int32_t stage,
                    int32_t grad_dtype, int32_t param_dtype, int32_t first_rank,
                    int32_t n_ranks, const int64_t *unit_numels, int32_t n_units)
{
    if (!out) return fail(ZERO_EINVAL, "out is null");
    *out = nullptr;
    if (world < 1 || world > ZERO_MAX_RANKS)
        return fail(ZERO_EINVAL, "world must be in [1, %d] (got %d)", ZERO_MAX_RANKS, world);
    if (first_rank < 0 || n_ranks < 1 || n_ranks > world - first_rank)
        return fail(ZERO_EINVAL, "ranks [%d, %d + %d) are not within [0, %d)", first_rank,
                    first_rank, n_ranks, world);
    return init_ctx(out, numel, world, stage, grad_dtype, param_dtype, first_rank, n_ranks,
                    unit_numels, n_units);
}

int zero_init_dim0(zero_ctx **out, int32_t world, int32_t grad_dtype, int32_t param_dtype,
                   int32_t rank, const int64_t *rows, const int64_t *row_elems, int32_t n_units)
{
    if (!out) return fail(ZERO_EINVAL, "out is null");
    *out = nullptr;
    if (!rows || !row_elems || n_units < 1)
        return fail(ZERO_EINVAL, "rows and row_elems of n_units >= 1 parameters are needed");
    std::vector<int64_t> numel, shard;
    int64_t total = 0;
    for (int32_t u = 0; u < n_units; ++u) {
        if (rows[u] < 0 || row_elems[u] < 0 || (row_elems[u] && rows[u] > ((int64_t)1 << 56) / row_elems[u]))
            return fail(ZERO_EINVAL, "parameter %d: bad shape (%lld x %lld)", u,
                        (long long)rows[u], (long long)row_elems[u]);
        numel.push_back(rows[u] * row_elems[u]);
        total += numel.back();
    }
    // the shared checks of world, dtypes and rank
    zero_ctx *c = nullptr;
    int rc = zero_init(&c, total, world, 3, grad_dtype, param_dtype, rank, numel.data(), n_units);
    if (rc) return rc;
    c->unit_numel.clear();
    c->unit_S.clear();
    c->unit_state_off.clear();
    for (int32_t u = 0; u < n_units; ++u)
        shard.push_back(ceil_div(rows[u], world) * row_elems[u]);
    rc = init_units(c, numel.data(), shard.data(), n_units, total);
    if (rc) {
        delete c;
        return rc;
    }
    *out = c;
    return ZERO_OK;
}

int zero_destroy(zero_ctx *ctx)
{
    if (ctx) release_slot(ctx->hyper_device, ctx->hyper_slot);
    delete ctx;
    return ZERO_OK;
}

int64_t zero_ctx_shard_size(const zero_ctx *c, int32_t unit)
{
    if (!c) return -1;
    if (unit < 0) return c->stage < 3 ? c->S : -1;
    if (c->stage < 3 || unit >= (int32_t)c->unit_S.size()) return -1;
    return c->unit_S[unit];
}

int64_t zero_ctx_state_elems(const zero_ctx *c) { return c ? c->state_elems : -1; }

int64_t zero_ctx_param_elems(const zero_ctx *c) { return c ? c->param_elems : -1; }

int64_t zero_ctx_unit_state_offset(const zero_ctx *c, int32_t unit)
{
    if (!c) return -1;
    if (c->stage < 3) return unit == -1 ? 0 : -1;
    if (unit < 0 || unit >= (int32_t)c->unit_S.size()) return -1;
    return c->unit_state_off[unit];
}

int64_t zero_ctx_unit_param_offset(const zero_ctx *c, int32_t unit)
{
    return zero_ctx_unit_state_offset(c, unit);
}

int64_t zero_state_bytes(const zero_ctx *c) { return c ? 12 * c->state_elems : -1; }

int zero_bind(zero_ctx *c, float *master, float *m, float *v, void *params, float *g_scratch,
              uint64_t *flag)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (c->state_elems > 0 && (!master || !m || !v || !params))
        return fail(ZERO_EINVAL, "master, m, v and params must not be null");
    if (!flag) return fail(ZERO_EINVAL, "flag must not be null");
    const int es_p = zgb::elem_size(c->pdt);
    if (!aligned(master, 4) || !aligned(m, 4) || !aligned(v, 4) || !aligned(g_scratch, 4))
        return fail(ZERO_EALIGN, "master/m/v/g_scratch must be 4-byte aligned");
    if (!aligned(params, es_p)) return fail(ZERO_EALIGN, "params not aligned to %d bytes", es_p);
    if (!aligned(flag, 8)) return fail(ZERO_EALIGN, "flag must be 8-byte aligned");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    c->master = master;
    c->m = m;
    c->v = v;
    c->params = params;
    c->g = g_scratch;
    c->flag = flag;
    c->device = dev;
    c->sms = sms > 0 ? sms : 1;
    c->bound = true;
    return ZERO_OK;
}

int zero_bind_shadow(zero_ctx *c, float *master_b, float *m_b, float *v_b, uint64_t *cur)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (c->stage3_open) return fail(ZERO_ESTATE, "a stage-3 step is open (zero3_end_step)");
    if (!master_b && !m_b && !v_b && !cur) {
        c->xb = c->mb = c->vb = nullptr;
        c->cur = nullptr;
        return ZERO_OK;
    }
    if (!cur || (c->state_elems > 0 && (!master_b || !m_b || !v_b)))
        return fail(ZERO_EINVAL, "master_b, m_b, v_b and cur must all be given (or all NULL)");
    if (!aligned(master_b, 4) || !aligned(m_b, 4) || !aligned(v_b, 4))
        return fail(ZERO_EALIGN, "the second state set must be 4-byte aligned");
    if (!aligned(cur, 8)) return fail(ZERO_EALIGN, "cur must be 8-byte aligned");
    c->xb = master_b;
    c->mb = m_b;
    c->vb = v_b;
    c->cur = cur;
    return ZERO_OK;
}

int zero_current_state(zero_ctx *c, int32_t *which)
{
    if (!c || !which) return fail(ZERO_EINVAL, "null argument");
    if (!c->cur) {
        *which = 0;
        return ZERO_OK;
    }
    unsigned long long h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, c->cur, sizeof h, cudaMemcpyDeviceToHost, c->last_stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->last_stream);
    if (e != cudaSuccess) return cuda_fail(e, "reading the current-set word");
    *which = (int32_t)(h & 1ull);
    return ZERO_OK;
}

int zero_set_gather_mode(zero_ctx *c, int32_t mode)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (mode != ZERO_GATHER_FAST && mode != ZERO_GATHER_LEAN)
        return fail(ZERO_EINVAL, "unknown gather mode %d", mode);
    c->gather_mode = mode;
    return ZERO_OK;
}

int zero_gather_timeouts(uint32_t *count)
{
    if (!count) return fail(ZERO_EINVAL, "null argument");
    unsigned int h = 0;
    cudaError_t e = zgb::lean_gather_timeouts(&h);
    if (e != cudaSuccess) return cuda_fail(e, "reading the gather timeout counter");
    *count = h;
    return h ? ZERO_ETIMEOUT : ZERO_OK;
}

int zero_set_gather_wait_polls(int64_t polls)
{
    cudaError_t e = zgb::set_lean_first_wait_polls((long long)polls);
    if (e != cudaSuccess) return cuda_fail(e, "setting the lean gather's wait limit");
    return ZERO_OK;
}

int zero_set_step_occupancy(zero_ctx *c, int32_t blocks_per_sm)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (blocks_per_sm < 0 || blocks_per_sm > 32)
        return fail(ZERO_EINVAL, "blocks_per_sm must be in [0, 32] (0: as many as fit)");
    c->step_per_sm = blocks_per_sm;
    return ZERO_OK;
}

int zero_set_weight_decay(zero_ctx *c, double weight_decay)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (!(weight_decay >= 0.0) || weight_decay > 1e6)
        return fail(ZERO_EINVAL, "weight_decay must be a finite value >= 0");
    c->weight_decay = weight_decay;
    return ZERO_OK;
}

int zero_bind_hyper(zero_ctx *c, void *d_hyper)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    static_assert(sizeof(zgb::DeviceHyper) <= ZERO_HYPER_BYTES, "hyper block too large");
    if (!aligned(d_hyper, 16)) return fail(ZERO_EALIGN, "the hyper block must be 16-byte aligned");
    if (c->bucket_open || c->stage3_open) return fail(ZERO_ESTATE, "a step is open");
    if (!d_hyper) {
        release_slot(c->hyper_device, c->hyper_slot);
        c->hyper_slot = -1;
        c->hyper = nullptr;
        c->hyper_direct = false;
        return ZERO_OK;
    }
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (c->hyper_slot < 0 || c->hyper_device != dev) {
        release_slot(c->hyper_device, c->hyper_slot);
        const int slot = claim_slot(dev);
        if (slot < 0)
            return fail(ZERO_ESTATE, "all %d constant slots of this device are bound to other "
                                     "contexts' scalar blocks", zgb::kHyperSlots);
        c->hyper_slot = slot;
        c->hyper_device = dev;
    }
    void *slot_addr = nullptr;
    e = zgb::hyper_slot_address(c->hyper_slot, &slot_addr);
    if (e != cudaSuccess) return cuda_fail(e, "the address of the constant slot");
    c->hyper = d_hyper;
    c->hyper_direct = d_hyper == slot_addr;
    c->slot_stale = true;
    return ZERO_OK;
}

int zero_load_hyper(zero_ctx *c, const void *host_block, void *stream)
{
    if (!c || !host_block) return fail(ZERO_EINVAL, "null argument");
    if (!c->hyper || !c->hyper_direct)
        return fail(ZERO_ESTATE, "bind the constant slot (zero_hyper_slot) as the block first");
    const cudaError_t e = cudaMemcpyAsync(c->hyper, host_block, sizeof(zgb::DeviceHyper),
                                          cudaMemcpyHostToDevice, (cudaStream_t)stream);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e, "copying the scalar block to its slot");
}

int zero_hyper_slot(zero_ctx *c, void **d_slot)
{
    if (!c || !d_slot) return fail(ZERO_EINVAL, "null argument");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (c->hyper_slot < 0 || c->hyper_device != dev) {
        if (c->hyper) return fail(ZERO_ESTATE, "a block is bound on another device");
        const int slot = claim_slot(dev);
        if (slot < 0)
            return fail(ZERO_ESTATE, "all %d constant slots of this device are in use",
                        zgb::kHyperSlots);
        c->hyper_slot = slot;
        c->hyper_device = dev;
    }
    e = zgb::hyper_slot_address(c->hyper_slot, d_slot);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e, "the address of the constant slot");
}

int zero_prepare_step(zero_ctx *c, void *host_hyper, double lr, double b1, double b2,
                      double eps, int64_t t, float loss_scale)
{
    if (!c || !host_hyper) return fail(ZERO_EINVAL, "null argument");
    if (!c->hyper) return fail(ZERO_ESTATE, "no device hyper block bound (zero_bind_hyper)");
    if (c->bucket_open) return fail(ZERO_ESTATE, "a bucketed step is open");
    int rc = check_hyper(lr, b1, b2, eps, t);
    if (rc || (rc = check_scale(loss_scale))) return rc;
    c->step_id += 1;
    c->step_scaled = loss_scale > 0.0f;
    zgb::DeviceHyper h;
    memset(&h, 0, sizeof h);
    h.ad = adam_scalars(lr, b1, b2, eps, t, c->weight_decay);
    h.av = average_scalars(c->world, loss_scale);
    h.flag_id = c->step_id;
    h.skip_id = c->step_scaled ? c->step_id : ~0ull;
    memset(host_hyper, 0, ZERO_HYPER_BYTES);
    memcpy(host_hyper, &h, sizeof h);
    return ZERO_OK;
}

int64_t zero_advance_table_bytes(int64_t t_max)
{
    return t_max >= 1 && t_max <= ((int64_t)1 << 40) ? 8 * t_max : -1;
}

int zero_fill_advance_table(void *host_table, int64_t t_max, double b1, double b2)
{
    if (!host_table || t_max < 1 || t_max > ((int64_t)1 << 40))
        return fail(ZERO_EINVAL, "host_table and 1 <= t_max required");
    float *p = static_cast<float *>(host_table);
    for (int64_t t = 1; t <= t_max; ++t) {
        // exactly the host's derivation of a step's bias corrections
        p[2 * (t - 1)] = (float)(1.0 - std::pow(b1, (double)t));
        p[2 * (t - 1) + 1] = (float)(1.0 - std::pow(b2, (double)t));
    }
    return ZERO_OK;
}

int zero_advance_state(void *host_state, int64_t t, float loss_scale, int64_t growth_interval)
{
    if (!host_state || t < 1) return fail(ZERO_EINVAL, "host_state and t >= 1 required");
    if (int rc = check_scale(loss_scale)) return rc;
    zgb::AdvanceState st{};
    st.t = t;
    st.scale = loss_scale > 0.0f ? loss_scale : 0.0f;
    st.status = 0;
    st.good_steps = 0;
    st.growth_interval = growth_interval;
    memcpy(host_state, &st, sizeof st);
    return ZERO_OK;
}

int zero_bind_advance(zero_ctx *c, const void *d_table, int64_t t_max, void *d_state)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (!d_table && !d_state) {
        c->adv_table = nullptr;
        c->adv_tmax = 0;
        c->adv_state = nullptr;
        return ZERO_OK;
    }
    if (!d_table || !d_state || t_max < 1)
        return fail(ZERO_EINVAL, "d_table, d_state and t_max >= 1 required (or both NULL)");
    if (!aligned(d_table, 4) || !aligned(d_state, 8))
        return fail(ZERO_EALIGN, "the table must be 4-byte and the state 8-byte aligned");
    c->adv_table = static_cast<const float *>(d_table);
    c->adv_tmax = t_max;
    c->adv_state = d_state;
    return ZERO_OK;
}

int zero_advance_step(zero_ctx *c, void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if (!c->hyper) return fail(ZERO_ESTATE, "no device scalar block bound (zero_bind_hyper)");
    if (!c->adv_state) return fail(ZERO_ESTATE, "no device step state bound (zero_bind_advance)");
    if (c->hyper_direct)
        return fail(ZERO_ESTATE, "the device advance rewrites the bound block: bind a block in "
                                 "device memory, not the constant slot");
    if (c->step_id == 0) return fail(ZERO_ESTATE, "prepare the first step (zero_prepare_step)");
    if (c->bucket_open) return fail(ZERO_ESTATE, "a bucketed step is open (zero_bucket_end)");
    if (c->stage3_open) return fail(ZERO_ESTATE, "a stage-3 step is open (zero3_end_step)");
    const cudaError_t e = zgb::launch_advance(
        static_cast<zgb::DeviceHyper *>(c->hyper), reinterpret_cast<const unsigned long long *>(c->flag),
        static_cast<zgb::AdvanceState *>(c->adv_state), c->adv_table, c->adv_tmax,
        (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "advance kernel");
    c->step_id += 1;             // the device block now describes the next step
    return ZERO_OK;
}

int zero_bind_allreduce_out(zero_ctx *c, void *grad_avg)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (c->stage != 1) return fail(ZERO_EINVAL, "the all-reduce output is a stage-1 feature");
    if (!aligned(grad_avg, zgb::elem_size(c->gdt)))
        return fail(ZERO_EALIGN, "grad_avg not aligned to its elements");
    c->grad_avg = grad_avg;
    return ZERO_OK;
}

int zero_step_reduce(zero_ctx *c, const void *const *grads, int32_t n_grads, float loss_scale,
                     void *stream)
{
    int rc = check_ready(c);
    if (rc || (rc = check_scale(loss_scale))) return rc;
    if (c->stage == 3) return fail(ZERO_EINVAL, "stage 3 reduces per unit (zero3_reduce_unit)");
    if (c->bucket_open) return fail(ZERO_ESTATE, "a bucketed step is open (zero_bucket_end)");
    if (!c->g) return fail(ZERO_ESTATE, "the two-pass step needs g_scratch (zero_bind)");
    const Range r = vector_range(c);
    rc = check_ptr_array(grads, n_grads, c->world, zgb::elem_size(c->gdt), r.n_valid > 0, "grads");
    if (rc) return rc;
    if ((rc = begin_step(c, loss_scale > 0.0f))) return rc;
    return do_reduce(c, r, grads, loss_scale, (cudaStream_t)stream);
}

int zero_step_apply(zero_ctx *c, double lr, double b1, double b2, double eps, int64_t t,
                    void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if ((rc = check_hyper(lr, b1, b2, eps, t))) return rc;
    if (c->bucket_open) return fail(ZERO_ESTATE, "a bucketed step is open (zero_bucket_end)");
    if (c->stage == 3 && c->cur)
        return fail(ZERO_ESTATE, "with two state sets, stage-3 steps finish with zero3_end_step");
    if (!c->g) return fail(ZERO_ESTATE, "the two-pass step needs g_scratch (zero_bind)");
    if (c->step_id == 0) return fail(ZERO_ESTATE, "no reduce pass ran before apply");
    return do_apply(c, apply_range(c), lr, b1, b2, eps, t, (cudaStream_t)stream);
}

int zero_step(zero_ctx *c, const void *const *grads, int32_t n_grads, double lr, double b1,
              double b2, double eps, int64_t t, float loss_scale, void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if ((rc = check_hyper(lr, b1, b2, eps, t)) || (rc = check_scale(loss_scale))) return rc;
    if (c->stage == 3) return fail(ZERO_EINVAL, "stage 3 steps per unit (zero3_step_unit)");
    if (c->bucket_open) return fail(ZERO_ESTATE, "a bucketed step is open (zero_bucket_end)");
    const Range r = vector_range(c);
    rc = check_ptr_array(grads, n_grads, c->world, zgb::elem_size(c->gdt), r.n_valid > 0, "grads");
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    if (c->cur) {
        // two state sets: one pass whatever the loss scale
        if ((rc = begin_step(c, loss_scale > 0.0f))) return rc;
        return do_fused(c, r, grads, lr, b1, b2, eps, t, s, loss_scale);
    }
    if (loss_scale > 0.0f) {
        if (!c->g) return fail(ZERO_ESTATE, "a loss-scaled step needs g_scratch (zero_bind)");
        if ((rc = begin_step(c, true))) return rc;
        rc = do_reduce(c, r, grads, loss_scale, s);
        if (rc) return rc;
        return do_apply(c, r, lr, b1, b2, eps, t, s);
    }
    if ((rc = begin_step(c, false))) return rc;
    return do_fused(c, r, grads, lr, b1, b2, eps, t, s);
}

int zero_bucket_begin(zero_ctx *c, float loss_scale)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (c->stage == 3) return fail(ZERO_EINVAL, "buckets cover the flat vector of stages 1 and 2");
    if (c->bucket_open) return fail(ZERO_ESTATE, "a bucketed step is already open");
    if (int rc = check_scale(loss_scale)) return rc;
    if (loss_scale > 0.0f && !c->cur && !c->g)
        return fail(ZERO_ESTATE, "a loss-scaled bucketed step needs g_scratch or a second state set");
    int rc = begin_step(c, loss_scale > 0.0f);
    if (rc) return rc;
    c->bucket_scale = loss_scale;
    c->bucket_open = true;
    return ZERO_OK;
}

int zero_bucket_step(zero_ctx *c, int64_t offset, int64_t count, const void *const *grads,
                     int32_t n_grads, double lr, double b1, double b2, double eps, int64_t t,
                     void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if (!c->bucket_open) return fail(ZERO_ESTATE, "call zero_bucket_begin first");
    if ((rc = check_hyper(lr, b1, b2, eps, t))) return rc;
    const Range whole = vector_range(c);
    if (offset < 0 || count < 0 || offset > whole.n || count > whole.n - offset)
        return fail(ZERO_EINVAL, "bucket [%lld, %lld) outside the range of %lld elements",
                    (long long)offset, (long long)(offset + count), (long long)whole.n);
    Range r;
    r.state_off = whole.state_off + offset;
    r.n = count;
    r.n_valid = std::max<int64_t>(0, std::min<int64_t>(count, whole.n_valid - offset));
    r.params = whole.params + offset * zgb::elem_size(c->pdt);
    r.grad_avg = whole.grad_avg ? whole.grad_avg + offset * zgb::elem_size(c->gdt) : nullptr;
    rc = check_ptr_array(grads, n_grads, c->world, zgb::elem_size(c->gdt), r.n_valid > 0, "grads");
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    if (c->cur)              // one pass into the other set; finalized by zero_bucket_end
        return do_fused(c, r, grads, lr, b1, b2, eps, t, s, c->bucket_scale, false);
    if (c->step_scaled)      // first pass only; zero_bucket_end applies
        return do_reduce(c, r, grads, c->bucket_scale, s);
    return do_fused(c, r, grads, lr, b1, b2, eps, t, s);
}

int zero_bucket_end(zero_ctx *c, double lr, double b1, double b2, double eps, int64_t t,
                    void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if (!c->bucket_open) return fail(ZERO_ESTATE, "no bucketed step is open");
    if ((rc = check_hyper(lr, b1, b2, eps, t))) return rc;
    c->bucket_open = false;
    cudaStream_t s = (cudaStream_t)stream;
    const Range whole = vector_range(c);
    if (c->cur) return do_finalize(c, whole, s);
    if (c->step_scaled) return do_apply(c, whole, lr, b1, b2, eps, t, s);
    return ZERO_OK;
}

int zero_step_status(zero_ctx *c, int32_t *nonfinite, int32_t *skipped)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (!c->bound) return fail(ZERO_ESTATE, "no buffers bound");
    unsigned long long h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, c->flag, sizeof h, cudaMemcpyDeviceToHost, c->last_stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(c->last_stream);
    if (e != cudaSuccess) return cuda_fail(e, "reading the flag word");
    const bool bad = c->step_id > 0 && h == c->step_id;
    const bool skip = bad && c->step_scaled;
    if (nonfinite) *nonfinite = bad ? 1 : 0;
    if (skipped) *skipped = skip ? 1 : 0;
    return skip ? ZERO_SKIPPED : ZERO_OK;
}

uint64_t zero_step_id(const zero_ctx *c) { return c ? c->step_id : 0; }

// Shards at least this long take the row placement (gather_rows_kernel) in
// a ZeRO-3 unit gather: measured on GB300, a Llama-7B-layer unit's 8 shards
// of 50.6 MB in 0.1214 ms against 0.1248 ms with gather_kernel, while 4-11 MB
// shards were faster with gather_kernel (0.0178 against 0.0185 ms) and the
// one-rank placement of 234 MB shards too (4.24 against 4.35 ms).
constexpr int64_t kRowsGatherMinShardBytes = (int64_t)32 << 20;

static int gather(zero_ctx *c, const void *const *shards, int32_t n, void *full, int32_t dtype,
                  int64_t S, cudaStream_t s, bool unit = false)
{
    if (!valid_dtype(dtype)) return fail(ZERO_EINVAL, "unknown dtype %d", dtype);
    const int es = zgb::elem_size(dtype);
    int rc = check_ptr_array(shards, n, c->world, es, false, "shards");
    if (rc) return rc;
    if (!full && S > 0) return fail(ZERO_EINVAL, "full is null");
    if (!aligned(full, es)) return fail(ZERO_EALIGN, "full not aligned to %d bytes", es);
    if (S == 0) return ZERO_OK;
    zgb::GatherArgs a;
    memset(&a, 0, sizeof a);
    for (int32_t k = 0; k < n; ++k) a.src[k] = shards[k];
    a.dst = static_cast<char *>(full);
    a.shard_bytes = S * es;
    a.n = n;
    a.es = es;
    // a gather neither reads nor writes the flag: it does not become the
    // stream zero_step_status waits on
    cudaError_t e;
    if (c->gather_mode == ZERO_GATHER_LEAN && zgb::lean_gather_eligible(a)) {
        e = zgb::launch_gather_lean(a, c->sms, s);
    } else if (unit && a.shard_bytes >= kRowsGatherMinShardBytes) {
        zgb::GatherRowsArgs r;
        memset(&r, 0, sizeof r);
        for (int32_t k = 0; k < n; ++k) {
            r.src[k] = a.src[k];
            r.dst[k] = a.dst + (int64_t)k * a.shard_bytes;
            r.bytes[k] = a.shard_bytes;
        }
        r.n = n;
        r.es = es;
        e = zgb::launch_gather_rows(r, c->sms, s);
    } else {
        e = zgb::launch_gather(a, c->sms, s);
    }
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e, "gather kernel");
}

int zero_allgather(zero_ctx *c, const void *const *shards, int32_t n_shards, void *full,
                   int32_t dtype, void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if (c->stage == 3) return fail(ZERO_EINVAL, "stage 3 gathers per unit (zero3_gather_unit)");
    return gather(c, shards, n_shards, full, dtype, c->S, (cudaStream_t)stream);
}

int zero3_begin_step_scaled(zero_ctx *c, float loss_scale)
{
    if (!c) return fail(ZERO_EINVAL, "null context");
    if (c->stage != 3) return fail(ZERO_EINVAL, "zero3_begin_step is for stage 3");
    if (c->stage3_open) return fail(ZERO_ESTATE, "the last stage-3 step is open (zero3_end_step)");
    if (int rc = check_scale(loss_scale)) return rc;
    const bool scaled = loss_scale > 0.0f;
    if (c->hyper) {
        if (c->step_id == 0) return fail(ZERO_ESTATE, "call zero_prepare_step first");
        if (scaled && !c->step_scaled)
            return fail(ZERO_EINVAL, "loss scaling differs from the prepared step");
        c->slot_stale = true;
    } else {
        c->step_id += 1;
        c->step_scaled = scaled;
    }
    c->step_scale = scaled ? loss_scale : 0.0f;
    c->stage3_open = c->cur != nullptr;
    return ZERO_OK;
}

int zero3_begin_step(zero_ctx *c)
{
    // with a device scalar block the prepared step fixes the loss scaling;
    // the kernels take the scale from the block
    return zero3_begin_step_scaled(c, 0.0f);
}

int zero3_end_step(zero_ctx *c, void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if (c->stage != 3) return fail(ZERO_EINVAL, "zero3_end_step is for stage 3");
    if (!c->cur) return ZERO_OK;     // one state set: every unit call was complete
    if (!c->stage3_open) return fail(ZERO_ESTATE, "no stage-3 step is open");
    c->stage3_open = false;
    // the written set becomes current, or, when some unit overflowed in a
    // loss-scaled step, the old set stays and every unit's params are cast
    // again from it
    return do_finalize(c, apply_range(c), (cudaStream_t)stream);
}

static int check_unit(zero_ctx *c, int32_t unit)
{
    if (c->stage != 3) return fail(ZERO_EINVAL, "unit calls are for stage 3");
    if (unit < 0 || unit >= (int32_t)c->unit_S.size())
        return fail(ZERO_EINVAL, "unit %d out of range [0, %d)", unit, (int)c->unit_S.size());
    if (c->step_id == 0) return fail(ZERO_ESTATE, "call zero3_begin_step first");
    return ZERO_OK;
}

static const char *kTwoSetsStage3 =
    "with two state sets, stage-3 steps run one pass per unit (zero3_step_unit / "
    "zero3_step_group) and finish with zero3_end_step";

// A stage-3 fused pass may run: a loss-scaled step needs the second state
// set (one pass into it, the verdict applied by zero3_end_step), and with
// that set bound the step must have been begun with it.
static int check_stage3_pass(zero_ctx *c)
{
    if (c->cur && !c->stage3_open)
        return fail(ZERO_ESTATE, "no stage-3 step is open (zero3_begin_step)");
    if (c->step_scaled && !c->cur)
        return fail(ZERO_ESTATE, "this step is loss-scaled: bind a second state set "
                                 "(zero_bind_shadow) or use zero3_reduce_unit + zero_step_apply");
    return ZERO_OK;
}

// With two state sets the pass reads the current set and writes the other;
// zero3_end_step finalizes once for every unit of the step.
static int stage3_fused(zero_ctx *c, const Range &r, const void *const *grads, double lr,
                        double b1, double b2, double eps, int64_t t, cudaStream_t s)
{
    if (c->cur) return do_fused(c, r, grads, lr, b1, b2, eps, t, s, c->step_scale, false);
    return do_fused(c, r, grads, lr, b1, b2, eps, t, s);
}

int zero3_gather_unit(zero_ctx *c, int32_t unit, const void *const *shards, int32_t n_shards,
                      void *unit_full, void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if (c->stage != 3) return fail(ZERO_EINVAL, "unit calls are for stage 3");
    if (unit < 0 || unit >= (int32_t)c->unit_S.size())
        return fail(ZERO_EINVAL, "unit %d out of range [0, %d)", unit, (int)c->unit_S.size());
    return gather(c, shards, n_shards, unit_full, c->pdt, c->unit_S[unit], (cudaStream_t)stream,
                  true);
}

int zero3_step_unit(zero_ctx *c, int32_t unit, const void *const *grads, int32_t n_grads,
                    double lr, double b1, double b2, double eps, int64_t t, void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if ((rc = check_unit(c, unit))) return rc;
    if ((rc = check_hyper(lr, b1, b2, eps, t))) return rc;
    if ((rc = check_stage3_pass(c))) return rc;
    const Range r = unit_range(c, unit);
    rc = check_ptr_array(grads, n_grads, c->world, zgb::elem_size(c->gdt), r.n_valid > 0, "grads");
    if (rc) return rc;
    return stage3_fused(c, r, grads, lr, b1, b2, eps, t, (cudaStream_t)stream);
}

// Whether the byte ranges [a, a + na) and [b, b + nb) share a byte.
static bool overlap(const void *a, int64_t na, const void *b, int64_t nb)
{
    if (!a || !b || na <= 0 || nb <= 0) return false;
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
}

// The buffers a unit's step writes (its params and state, the flag and
// current-set words) or reads (its grads), against a gather's destination
// and sources: the two halves of a visit may run at the same time only if
// the gather writes none of the step's buffers and reads none it writes.
static int check_visit_disjoint(const zero_ctx *c, const Range &r, const void *const *grads,
                                const void *const *shards, int64_t shard_bytes,
                                const void *full, int64_t full_bytes)
{
    const int es_p = zgb::elem_size(c->pdt), es_g = zgb::elem_size(c->gdt);
    const int64_t sb = r.n * 4;
    const void *written[] = {r.params, c->master + r.state_off, c->m + r.state_off,
                             c->v + r.state_off, c->cur ? c->xb + r.state_off : nullptr,
                             c->cur ? c->mb + r.state_off : nullptr,
                             c->cur ? c->vb + r.state_off : nullptr, c->flag, c->cur};
    const int64_t wbytes[] = {r.n * es_p, sb, sb, sb, sb, sb, sb, 8, 8};
    for (int i = 0; i < 9; ++i) {
        if (overlap(full, full_bytes, written[i], wbytes[i]))
            return fail(ZERO_EINVAL, "unit_full overlaps a buffer the stepped unit writes");
        for (int32_t k = 0; k < c->world; ++k)
            if (overlap(shards[k], shard_bytes, written[i], wbytes[i]))
                return fail(ZERO_EINVAL, "shards[%d] overlaps a buffer the stepped unit writes", k);
    }
    for (int32_t k = 0; k < c->world; ++k)
        if (overlap(full, full_bytes, grads[k], r.n_valid * es_g))
            return fail(ZERO_EINVAL, "unit_full overlaps grads[%d] of the stepped unit", k);
    return ZERO_OK;
}

int zero3_step_unit_gather(zero_ctx *c, int32_t unit, const void *const *grads, int32_t n_grads,
                           double lr, double b1, double b2, double eps, int64_t t,
                           int32_t gather_unit, const void *const *shards, int32_t n_shards,
                           void *unit_full, void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if ((rc = check_unit(c, unit))) return rc;
    const int32_t U = (int32_t)c->unit_S.size();
    if (gather_unit < 0 || gather_unit >= U)
        return fail(ZERO_EINVAL, "gather_unit %d out of range [0, %d)", gather_unit, U);
    if (gather_unit == unit)
        return fail(ZERO_EINVAL, "a visit steps one unit and gathers another (both are %d)", unit);
    if ((rc = check_hyper(lr, b1, b2, eps, t))) return rc;
    if ((rc = check_stage3_pass(c))) return rc;
    const Range r = unit_range(c, unit);
    rc = check_ptr_array(grads, n_grads, c->world, zgb::elem_size(c->gdt), r.n_valid > 0, "grads");
    if (rc) return rc;
    const int es = zgb::elem_size(c->pdt);
    const int64_t Sg = c->unit_S[gather_unit];
    if ((rc = check_ptr_array(shards, n_shards, c->world, es, false, "shards"))) return rc;
    if (!unit_full && Sg > 0) return fail(ZERO_EINVAL, "unit_full is null");
    if (!aligned(unit_full, es)) return fail(ZERO_EALIGN, "unit_full not aligned to %d bytes", es);
    rc = check_visit_disjoint(c, r, grads, shards, Sg * es, unit_full, Sg * es * c->world);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    // Two launches where one would not pay: a lean gather (it runs beside
    // compute), a bound scalar block (the graph form), a capped step
    // occupancy, or shards of the size the row placement serves better.
    if (c->gather_mode == ZERO_GATHER_LEAN || c->hyper || c->step_per_sm > 0 ||
        Sg * es >= kRowsGatherMinShardBytes) {
        if ((rc = stage3_fused(c, r, grads, lr, b1, b2, eps, t, s))) return rc;
        return gather(c, shards, n_shards, unit_full, c->pdt, Sg, s, true);
    }
    StepArgs a = make_args(c, r, grads);
    // with two state sets the pass writes the other set under the step's
    // loss scale (zero3_end_step decides); with one, the step is unscaled
    a.av = average_scalars(c->world, c->cur ? c->step_scale : 0.0f);
    a.ad = adam_scalars(lr, b1, b2, eps, t, c->weight_decay);
    a.step_id = c->step_id;
    zgb::GatherArgs g;
    memset(&g, 0, sizeof g);
    for (int32_t k = 0; k < c->world; ++k) g.src[k] = Sg > 0 ? shards[k] : nullptr;
    g.dst = static_cast<char *>(unit_full);
    g.shard_bytes = Sg * es;
    g.n = c->world;
    g.es = es;
    const cudaError_t e = zgb::launch_step_gather(c->gdt, c->pdt, a, g, c->sms, 0, s);
    if (r.n > 0) return finish_launch(c, e, "visit kernel", s);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e, "visit kernel");
}

int zero3_step_units_gather(zero_ctx *c, int32_t first_unit, int32_t n_units,
                            const void *const *grads, int32_t n_grads, double lr, double b1,
                            double b2, double eps, int64_t t, int32_t gather_first,
                            int32_t gather_n, const void *const *shards, int32_t n_shards,
                            void *const *unit_fulls, void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if (c->stage != 3) return fail(ZERO_EINVAL, "unit calls are for stage 3");
    const int32_t U = (int32_t)c->unit_S.size();
    const int32_t N = c->world;
    if (n_units < 1 || n_units > zgb::kVisitSteps || first_unit < 0 || first_unit > U - n_units)
        return fail(ZERO_EINVAL, "stepped units [%d, %d + %d) must be 1 or 2 units of [0, %d)",
                    first_unit, first_unit, n_units, U);
    if (gather_n < 0 || gather_n > zgb::kVisitSteps ||
        (gather_n > 0 && (gather_first < 0 || gather_first > U - gather_n)))
        return fail(ZERO_EINVAL, "gathered units [%d, %d + %d) must be 0 to 2 units of [0, %d)",
                    gather_first, gather_first, gather_n, U);
    if (gather_n > 0 && gather_first < first_unit + n_units && first_unit < gather_first + gather_n)
        return fail(ZERO_EINVAL, "a visit gathers units other than those it steps");
    if ((rc = check_hyper(lr, b1, b2, eps, t))) return rc;
    if ((rc = check_stage3_pass(c))) return rc;
    if (!grads || n_grads != n_units * N)
        return fail(ZERO_EINVAL, "grads: %d pointers given, %d units need %d", n_grads, n_units,
                    n_units * N);
    const int es_g = zgb::elem_size(c->gdt), es = zgb::elem_size(c->pdt);
    Range r[zgb::kVisitSteps];
    for (int32_t i = 0; i < n_units; ++i) {
        r[i] = unit_range(c, first_unit + i);
        rc = check_ptr_array(grads + (int64_t)i * N, N, N, es_g, r[i].n_valid > 0, "grads");
        if (rc) return rc;
    }
    if (n_shards != gather_n * N)
        return fail(ZERO_EINVAL, "shards: %d pointers given, %d units need %d", n_shards,
                    gather_n, gather_n * N);
    if (gather_n > 0 && (!shards || !unit_fulls)) return fail(ZERO_EINVAL, "null pointer array");
    int64_t Sg[zgb::kVisitSteps] = {0, 0};
    for (int32_t j = 0; j < gather_n; ++j) {
        Sg[j] = c->unit_S[gather_first + j];
        const void *const *sh = shards + (int64_t)j * N;
        if ((rc = check_ptr_array(sh, N, N, es, false, "shards"))) return rc;
        if (!unit_fulls[j] && Sg[j] > 0) return fail(ZERO_EINVAL, "unit_fulls[%d] is null", j);
        if (!aligned(unit_fulls[j], es))
            return fail(ZERO_EALIGN, "unit_fulls[%d] not aligned to %d bytes", j, es);
        for (int32_t i = 0; i < n_units; ++i) {
            rc = check_visit_disjoint(c, r[i], grads + (int64_t)i * N, sh, Sg[j] * es,
                                      unit_fulls[j], Sg[j] * es * N);
            if (rc) return rc;
        }
    }
    if (gather_n == 2 &&
        overlap(unit_fulls[0], Sg[0] * es * N, unit_fulls[1], Sg[1] * es * N))
        return fail(ZERO_EINVAL, "the two unit buffers overlap");
    cudaStream_t s = (cudaStream_t)stream;
    // The separate calls where one launch would not pay, as for
    // zero3_step_unit_gather, or where the rows would not fit one launch.
    bool separate = c->gather_mode == ZERO_GATHER_LEAN || c->hyper || c->step_per_sm > 0 ||
                    gather_n * N > zgb::kVisitRows;
    for (int32_t j = 0; j < gather_n; ++j) separate |= Sg[j] * es >= kRowsGatherMinShardBytes;
    if (separate) {
        for (int32_t i = 0; i < n_units; ++i)
            if ((rc = stage3_fused(c, r[i], grads + (int64_t)i * N, lr, b1, b2, eps, t, s)))
                return rc;
        for (int32_t j = 0; j < gather_n; ++j)
            if ((rc = gather(c, shards + (int64_t)j * N, N, unit_fulls[j], c->pdt, Sg[j], s, true)))
                return rc;
        return ZERO_OK;
    }
    zgb::VisitArgs v;
    memset(&v, 0, sizeof v);
    v.n_steps = n_units;
    bool steps = false;
    for (int32_t i = 0; i < n_units; ++i) {
        StepArgs a = make_args(c, r[i], grads + (int64_t)i * N);
        // with two state sets the pass writes the other set under the
        // step's loss scale (zero3_end_step decides); with one, unscaled
        a.av = average_scalars(N, c->cur ? c->step_scale : 0.0f);
        a.ad = adam_scalars(lr, b1, b2, eps, t, c->weight_decay);
        a.step_id = c->step_id;
        v.step[i] = a;
        steps |= r[i].n > 0;
    }
    v.n_rows = gather_n * N;
    v.es = es;
    for (int32_t j = 0; j < gather_n; ++j)
        for (int32_t k = 0; k < N; ++k) {
            const int32_t y = j * N + k;
            v.src[y] = Sg[j] > 0 ? shards[(int64_t)j * N + k] : nullptr;
            v.dst[y] = static_cast<char *>(unit_fulls[j]) + (int64_t)k * Sg[j] * es;
            v.bytes[y] = Sg[j] * es;
        }
    const cudaError_t e = zgb::launch_visit(c->gdt, c->pdt, v, c->sms, 0, s);
    if (steps) return finish_launch(c, e, "visit kernel", s);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e, "visit kernel");
}

int zero3_reduce_unit(zero_ctx *c, int32_t unit, const void *const *grads, int32_t n_grads,
                      float loss_scale, void *stream)
{
    int rc = check_ready(c);
    if (rc || (rc = check_scale(loss_scale))) return rc;
    if ((rc = check_unit(c, unit))) return rc;
    if (c->cur) return fail(ZERO_ESTATE, kTwoSetsStage3);
    if (!c->g) return fail(ZERO_ESTATE, "the two-pass step needs g_scratch (zero_bind)");
    const Range r = unit_range(c, unit);
    rc = check_ptr_array(grads, n_grads, c->world, zgb::elem_size(c->gdt), r.n_valid > 0, "grads");
    if (rc) return rc;
    if (c->hyper) {
        if ((loss_scale > 0.0f) != c->step_scaled)
            return fail(ZERO_EINVAL, "loss scaling differs from the prepared step");
    } else if (loss_scale > 0.0f) {
        c->step_scaled = true;
    }
    return do_reduce(c, r, grads, loss_scale, (cudaStream_t)stream);
}

// A run of consecutive units of stage 3 as one range (their state, scratch
// and param shards lie end to end).  A unit with padding in this view cannot
// join a group: the kernels treat only the tail of a range as padding.
static int group_range(zero_ctx *c, int32_t first, int32_t count, Range *out)
{
    const int32_t U = (int32_t)c->unit_S.size();
    if (count < 1 || first < 0 || first > U - count)
        return fail(ZERO_EINVAL, "units [%d, %d) outside [0, %d)", first, first + count, U);
    for (int32_t u = first; u < first + count; ++u) {
        const Range ru = unit_range(c, u);
        if (ru.n_valid != ru.n)
            return fail(ZERO_EINVAL, "unit %d has padding in this view: step it on its own", u);
    }
    Range r = unit_range(c, first);
    const Range last = unit_range(c, first + count - 1);
    r.n = last.state_off + last.n - r.state_off;
    r.n_valid = r.n;
    *out = r;
    return ZERO_OK;
}

int zero3_gather_group(zero_ctx *c, int32_t first_unit, int32_t n_units,
                       const void *const *shards, int32_t n_shards, void *const *unit_fulls,
                       void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if (c->stage != 3) return fail(ZERO_EINVAL, "unit calls are for stage 3");
    const int32_t U = (int32_t)c->unit_S.size();
    if (n_units < 1 || first_unit < 0 || first_unit > U - n_units)
        return fail(ZERO_EINVAL, "units [%d, %d) outside [0, %d)", first_unit,
                    first_unit + n_units, U);
    if ((int64_t)n_units * c->world > zgb::kMaxRows)
        return fail(ZERO_EINVAL, "a group gather places at most %d shards (%d units x %d ranks)",
                    zgb::kMaxRows, n_units, c->world);
    if (n_shards != n_units * c->world)
        return fail(ZERO_EINVAL, "shards: %d pointers given, the group needs %d", n_shards,
                    n_units * c->world);
    if (!shards || !unit_fulls) return fail(ZERO_EINVAL, "null pointer array");
    const int es = zgb::elem_size(c->pdt);
    zgb::GatherRowsArgs a;
    memset(&a, 0, sizeof a);
    a.es = es;
    for (int32_t ul = 0; ul < n_units; ++ul) {
        const int64_t Su = c->unit_S[first_unit + ul];
        char *full = static_cast<char *>(unit_fulls[ul]);
        if (!full && Su > 0) return fail(ZERO_EINVAL, "unit_fulls[%d] is null", ul);
        if (!aligned(full, es)) return fail(ZERO_EALIGN, "unit_fulls[%d] not aligned to %d bytes", ul, es);
        for (int32_t k = 0; k < c->world; ++k) {
            const int32_t y = ul * c->world + k;
            if (shards[y] && !aligned(shards[y], es))
                return fail(ZERO_EALIGN, "shards[%d] is not aligned to its %d-byte elements", y, es);
            a.src[y] = Su > 0 ? shards[y] : nullptr;
            a.dst[y] = full + (int64_t)k * Su * es;
            a.bytes[y] = Su * es;
        }
    }
    a.n = n_units * c->world;
    // like every gather, this one leaves the flag word alone and does not
    // become the stream zero_step_status waits on
    const cudaError_t e = (c->gather_mode == ZERO_GATHER_LEAN && zgb::lean_gather_rows_eligible(a))
                              ? zgb::launch_gather_rows_lean(a, c->sms, (cudaStream_t)stream)
                              : zgb::launch_gather_rows(a, c->sms, (cudaStream_t)stream);
    return e == cudaSuccess ? ZERO_OK : cuda_fail(e, "group gather kernel");
}

int zero3_step_group(zero_ctx *c, int32_t first_unit, int32_t n_units, const void *const *grads,
                     int32_t n_grads, double lr, double b1, double b2, double eps, int64_t t,
                     void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if ((rc = check_unit(c, first_unit))) return rc;
    if ((rc = check_hyper(lr, b1, b2, eps, t))) return rc;
    if ((rc = check_stage3_pass(c))) return rc;
    Range r;
    if ((rc = group_range(c, first_unit, n_units, &r))) return rc;
    rc = check_ptr_array(grads, n_grads, c->world, zgb::elem_size(c->gdt), r.n > 0, "grads");
    if (rc) return rc;
    return stage3_fused(c, r, grads, lr, b1, b2, eps, t, (cudaStream_t)stream);
}

int zero3_reduce_group(zero_ctx *c, int32_t first_unit, int32_t n_units,
                       const void *const *grads, int32_t n_grads, float loss_scale, void *stream)
{
    int rc = check_ready(c);
    if (rc || (rc = check_scale(loss_scale))) return rc;
    if ((rc = check_unit(c, first_unit))) return rc;
    if (c->cur) return fail(ZERO_ESTATE, kTwoSetsStage3);
    if (!c->g) return fail(ZERO_ESTATE, "the two-pass step needs g_scratch (zero_bind)");
    Range r;
    if ((rc = group_range(c, first_unit, n_units, &r))) return rc;
    rc = check_ptr_array(grads, n_grads, c->world, zgb::elem_size(c->gdt), r.n > 0, "grads");
    if (rc) return rc;
    if (c->hyper) {
        if ((loss_scale > 0.0f) != c->step_scaled)
            return fail(ZERO_EINVAL, "loss scaling differs from the prepared step");
    } else if (loss_scale > 0.0f) {
        c->step_scaled = true;
    }
    return do_reduce(c, r, grads, loss_scale, (cudaStream_t)stream);
}

}  // extern "C"

// ------------------------------------------------- step without allocation
//
// zero_step_noalloc: the two-pass step with its fp32 scratch in a fixed
// array compiled into this library instead of a caller buffer.  The array is
// a device-side object; host code cannot use its name as an address, so the
// address is looked up once per device (cudaGetSymbolAddress, with that
// device current) and handed to the kernels.
namespace {

constexpr int64_t kNoAllocScratchFloats = (int64_t)1 << 22;   // 16 MiB per device

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

std::mutex g_noalloc_mu;
std::vector<std::pair<int, float *>> g_noalloc_addr;   // (device, scratch address)

int noalloc_scratch_address(float **out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    for (const auto &p : g_noalloc_addr)
        if (p.first == dev) {
            *out = p.second;
            return ZERO_OK;
        }
    void *addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the built-in scratch");
    g_noalloc_addr.push_back({dev, static_cast<float *>(addr)});
    *out = static_cast<float *>(addr);
    return ZERO_OK;
}

}  // namespace

extern "C" int zero_step_noalloc(zero_ctx *c, const void *const *grads, int32_t n_grads,
                                 double lr, double b1, double b2, double eps, int64_t t,
                                 float loss_scale, void *stream)
{
    int rc = check_ready(c);
    if (rc) return rc;
    if ((rc = check_hyper(lr, b1, b2, eps, t)) || (rc = check_scale(loss_scale))) return rc;
    if (c->stage == 3) return fail(ZERO_EINVAL, "zero_step_noalloc covers stages 1 and 2");
    if (c->bucket_open) return fail(ZERO_ESTATE, "a bucketed step is open (zero_bucket_end)");
    const Range r = vector_range(c);
    if (r.n > kNoAllocScratchFloats)
        return fail(ZERO_EINVAL,
                    "zero_step_noalloc: this rank's range has %lld elements but the built-in "
                    "scratch holds %lld floats (16 MiB); bind a g_scratch and use zero_step",
                    (long long)r.n, (long long)kNoAllocScratchFloats);
    rc = check_ptr_array(grads, n_grads, c->world, zgb::elem_size(c->gdt), r.n_valid > 0, "grads");
    if (rc) return rc;
    float *scratch = nullptr;
    if ((rc = noalloc_scratch_address(&scratch))) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    if ((rc = begin_step(c, loss_scale > 0.0f))) return rc;
    if (r.n == 0) return ZERO_OK;
    if ((rc = load_slot_if_stale(c, s))) return rc;

    StepArgs a = make_args(c, r, grads);
    a.g = scratch;    // every element of the range is written by the reduce pass first
    // the same predicate as every other launch, over the arguments as they
    // now stand (a second state set, when bound, still counts)
    a.vec_ok = zgb::step_vector_path_ok(a) ? 1 : 0;
    a.av = average_scalars(c->world, loss_scale);
    a.step_id = c->step_id;
    rc = finish_launch(c, zgb::launch_reduce(c->gdt, a, c->sms, c->step_per_sm, s),
                       "reduce kernel", s);
    if (rc) return rc;
    a.ad = adam_scalars(lr, b1, b2, eps, t, c->weight_decay);
    a.step_id = c->step_scaled ? c->step_id : ~0ull;
    return finish_launch(c, zgb::launch_apply(c->pdt, a, c->sms, c->step_per_sm, s),
                         "apply kernel", s);
}
