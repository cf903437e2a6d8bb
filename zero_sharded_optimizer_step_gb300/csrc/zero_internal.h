// Internal interface between the C ABI (zero_abi.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace zgb {

constexpr int kMaxRanks = 256;   // == ZERO_MAX_RANKS
constexpr int kThreads = 256;    // threads per block of every streaming kernel
constexpr int kVec = 8;          // elements per thread per iteration

enum DType : int32_t { F32 = 0, BF16 = 1, F16 = 2 };

inline int elem_size(int32_t dt) { return dt == F32 ? 4 : 2; }

// fp32 scalars of one Adam step, each rounded once from a double.
struct AdamScalars {
    float lr, b1, b2, c1, c2, bc1, bc2, eps;
    float decay;        // 1 - lr * weight_decay (AdamW), used when decoupled != 0
    int32_t decoupled;
};

// How the rank sum becomes the gradient: g = acc / world, then / loss_scale.
// Division by a power of two equals multiplication by its reciprocal (both
// round the same exact value once), so those cases multiply.
struct AverageScalars {
    float world_f, inv_world;
    float scale, inv_scale;
    int32_t world_pow2, scaled, scale_pow2, pad_;
};

// Per-step scalars in device memory, for steps captured in a CUDA graph: the
// kernels read them at run time instead of taking them as launch arguments.
struct DeviceHyper {
    AdamScalars ad;
    AverageScalars av;
    unsigned long long flag_id;   // id a pass records a non-finite grad under
    unsigned long long skip_id;   // id apply/finalize treat as "skip" (~0 = never)
};

// The device-resident step state of steps whose scalars advance on the
// device (zero_bind_advance): what the host's loss-scale policy keeps, for
// the step the device block currently describes.
struct AdvanceState {
    int64_t t;                 // the step count of the described step
    float scale;               // its loss scale (as prepared; 0 = unscaled)
    int32_t status;            // 0, or 1 once the bias table ran out
    int64_t good_steps;        // clean steps since the scale last changed
    int64_t growth_interval;   // doubling period (<= 0: never)
};
static_assert(sizeof(AdvanceState) == 32, "AdvanceState is 32 bytes");

// Arguments of the per-element step kernels over one contiguous range of
// `n` elements of the state.  Every pointer is already offset to the
// range's first element.
struct StepArgs {
    const void *grads[kMaxRanks];  // rank k's grads for this range
    int32_t world;
    int32_t vec_ok;                // the vector path may run (step_vector_path_ok)
    int32_t grad_align;            // 16 or 8: how the vector path loads the rank grads
    int32_t param_align;           // byte alignment of `params` (2..16)
    int32_t avg_align;             // byte alignment of `grad_avg`
    int64_t n;                     // elements in the range
    int64_t n_valid;               // leading elements with real grads (rest = pad)
    float *master, *m, *v;
    void *params;                  // low-precision output
    void *grad_avg;                // stage-1 all-reduce output (grad type) or null
    float *g;                      // two-pass scratch
    // second state set (null when not bound) and the word naming the
    // current set: bit 0 clear = master/m/v, set = xb/mb/vb
    float *xb, *mb, *vb;
    unsigned long long *cur;
    unsigned long long *flag;      // id of the latest step with a non-finite grad
    unsigned long long step_id;
    const DeviceHyper *hyper;      // when set, ad/av/step_id come from constant slot `slot`,
    int32_t slot;                  // a copy of this block made at the step's first launch
    AverageScalars av;
    AdamScalars ad;
};

// The common byte alignment of the rank grads, as the vector path reads
// them: 16 (one 16-byte load per 16 bytes), 8 (two 8-byte loads: a rank's
// slices of flat vectors whose shard length is 4 mod 8 elements start on an
// 8-byte boundary) or 0 (the per-element path).
inline int32_t step_grad_align(const StepArgs &a)
{
    uintptr_t bits = 0;
    for (int32_t k = 0; k < a.world && k < kMaxRanks; ++k) bits |= (uintptr_t)a.grads[k];
    return (bits & 15) == 0 ? 16 : (bits & 7) == 0 ? 8 : 0;
}

// Whether the step kernels may take their vector path over a range: every
// fp32 buffer they read or write with 16-byte accesses -- master/m/v, the
// fp32 scratch and, with a second state set bound, that set too -- starts
// on a 16-byte boundary (null pointers are not accessed), and the rank
// grads on an 8-byte one (step_grad_align).  The params and the stage-1
// output are stored at their own alignment (param_align, avg_align) and
// take no part.  Computed from the finished arguments, so that no launch
// can leave one of the buffers out.
inline bool step_vector_path_ok(const StepArgs &a)
{
    auto al16 = [](const void *p) { return ((uintptr_t)p & 15) == 0; };
    bool ok = al16(a.master) && al16(a.m) && al16(a.v) && al16(a.g);
    if (a.cur) ok = ok && al16(a.xb) && al16(a.mb) && al16(a.vb);
    return ok && step_grad_align(a) >= 8;
}

struct GatherArgs {
    const void *src[kMaxRanks];    // shard k (null = skip)
    char *dst;                     // shard k lands at dst + k * shard_bytes
    int64_t shard_bytes;
    int32_t n;
    int32_t es;                    // element size in bytes
};

// A ZeRO-3 backward visit in one launch: the fused pass over one unit's
// range (`step`, blocks [0, step_blocks)) and the placement of another
// unit's shards (`gather`, row_blocks blocks per shard after them).
struct StepGatherArgs {
    StepArgs step;
    GatherArgs gather;
    int32_t step_blocks;
    int32_t row_blocks;
    int32_t step_short;            // the step part takes the 4-wide body
};

// A ZeRO-3 backward visit of up to two units in one launch: the fused pass
// over each of up to kVisitSteps unit ranges (step s owns blocks
// [step_first_block[s], step_first_block[s + 1])), then the placement of up
// to kVisitRows shards (row y owns the blocks [row_first_block[y],
// row_first_block[y + 1]) after the steps' blocks).
constexpr int kVisitSteps = 2;
constexpr int kVisitRows = 64;
struct VisitArgs {
    StepArgs step[kVisitSteps];
    int32_t step_first_block[kVisitSteps + 1];
    int32_t step_short[kVisitSteps];   // the step takes the 4-wide body
    int32_t n_steps;
    const void *src[kVisitRows];       // null = skip the row
    char *dst[kVisitRows];
    int64_t bytes[kVisitRows];
    int32_t row_first_block[kVisitRows + 1];
    int32_t n_rows;
    int32_t es;
};

// A placement of independent rows in one launch: row y copies bytes[y]
// bytes from src[y] to dst[y] (a group of units, one row per unit and shard).
// The launcher fills first_block: row y owns blocks [first_block[y],
// first_block[y + 1]) of the one-dimensional grid, as many as its length
// needs.
constexpr int kMaxRows = 512;
struct GatherRowsArgs {
    const void *src[kMaxRows];     // null = skip the row
    char *dst[kMaxRows];
    int64_t bytes[kMaxRows];       // multiple of es
    int32_t first_block[kMaxRows + 1];
    int32_t n;                     // rows
    int32_t es;
};

// Constant-memory slots holding the device scalar blocks of the contexts in
// the graph form (one slot per bound block and device): the step kernels read
// their scalars there as constant-bank operands, as eager launches read their
// parameters.  load_hyper_slot copies a block into its slot on `s`.
constexpr int kHyperSlots = 8;
cudaError_t load_hyper_slot(int slot, const DeviceHyper *block, cudaStream_t s);
// Device address of a slot (a caller may copy its block straight there).
cudaError_t hyper_slot_address(int slot, void **addr);

// Blocks of `threads` threads of `kernel` that fit on one SM of the current
// device (cached per kernel and device; at least 1).
int resident_blocks_per_sm(const void *kernel, int threads);

// Programmatic dependent launch.  A kernel launched by launch_dependent may
// be scheduled while the kernel before it in the stream is still finishing:
// its blocks become resident as that kernel's blocks retire, so the launch
// latency and the ramp-up overlap the previous kernel's tail.  Every such
// kernel calls pdl_wait() before its first access to global memory, which
// returns once the previous kernel has completed and its writes are visible,
// so the stream's ordering is unchanged.  pdl_launch_dependents() lets the
// next kernel be scheduled the same way (without it, that happens when every
// block has exited).  Other work in the stream (copies, event waits) keeps
// its full ordering.
#ifdef __CUDACC__
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}
#endif

// Launchers: return a cudaError_t.  `sms` is the device's SM count;
// cap_per_sm > 0 sizes the grid for at most that many blocks per SM (fewer
// than fit), leaving the rest of every SM to kernels that run beside it.
cudaError_t launch_fused_step(int32_t gdt, int32_t pdt, const StepArgs &a, int sms,
                              int cap_per_sm, cudaStream_t s);
cudaError_t launch_reduce(int32_t gdt, const StepArgs &a, int sms, int cap_per_sm,
                          cudaStream_t s);
cudaError_t launch_apply(int32_t pdt, const StepArgs &a, int sms, int cap_per_sm,
                         cudaStream_t s);
// After a single-pass step on two state sets: make the written set current,
// or, when the step overflowed, keep the old set and rewrite the params
// from it.
cudaError_t launch_finalize(int32_t pdt, const StepArgs &a, int sms, int cap_per_sm,
                            cudaStream_t s);
cudaError_t launch_gather(const GatherArgs &a, int sms, cudaStream_t s);
// The visit kernel: the fused pass of launch_fused_step over `step` (eager
// scalars, no stage-1 output) and the placement of launch_gather over
// `gather`, in one launch; the launcher sizes both parts of the grid.
cudaError_t launch_step_gather(int32_t gdt, int32_t pdt, const StepArgs &step,
                               const GatherArgs &gather, int sms, int cap_per_sm,
                               cudaStream_t s);
// A visit of up to two units (VisitArgs): the launcher fills a copy's block
// tables (each step range the grid launch_fused_step would give it, each
// row the blocks launch_gather would) and launches once.
cudaError_t launch_visit(int32_t gdt, int32_t pdt, const VisitArgs &a, int sms, int cap_per_sm,
                         cudaStream_t s);
// Fills a copy's first_block table and launches; `a` itself is not changed.
cudaError_t launch_gather_rows(const GatherRowsArgs &a, int sms, cudaStream_t s);
// The bulk-copy (TMA) placement for 16-byte aligned shards: one warp per SM,
// for gathers that run beside other kernels.  cudaErrorInvalidValue when the
// shards are not eligible (lean_gather_eligible).
bool lean_gather_eligible(const GatherArgs &a);
cudaError_t launch_gather_lean(const GatherArgs &a, int sms, cudaStream_t s);
// The same for rows of any lengths (a group gather): every row 16-byte
// aligned at both ends, lengths multiples of 16 bytes.
bool lean_gather_rows_eligible(const GatherRowsArgs &a);
cudaError_t launch_gather_rows_lean(const GatherRowsArgs &a, int sms, cudaStream_t s);
// After a step: read its verdict, advance *st by the loss-scale policy and
// rewrite *hyper for the next step (bias corrections from table: 2 floats per
// t = 1..t_max).  One thread.
cudaError_t launch_advance(DeviceHyper *hyper, const unsigned long long *flag, AdvanceState *st,
                           const float *table, int64_t t_max, cudaStream_t s);
// Waits of the lean gather that ran out (cumulative, this process).
cudaError_t lean_gather_timeouts(unsigned int *count);
cudaError_t set_lean_first_wait_polls(long long polls);

}  // namespace zgb
