// Streaming kernels of the ZeRO step on sm_103a.
//
//   fused_step  reduce-scatter sum over N rank buffers (rank order) -> average
//               -> unscale -> Adam on fp32 master/m/v -> cast -> param store,
//               one read-modify-write pass ("ZeRO 与 FSDP…", 从零实现 ZeRO 的
//               Adam: reduce_scatter_tensor, g /= world, the Adam update and
//               all_gather_into_tensor, here fused into a single pass because
//               every rank's buffers are on this GPU).
//   reduce      first pass of the loss-scaled step: the same sum, average and
//               unscale, written to an fp32 scratch, with the overflow flag.
//   apply       second pass: Adam + cast from the scratch, or nothing at all
//               when the flag names this step ("PaddlePaddle ZeRO优化",
//               混合精度才是最佳拍档: the step is skipped on inf/nan).
//   finalize    with two state sets bound, the loss-scaled step is a single
//               pass: fused_step reads the current set and writes the other
//               one; finalize then makes the written set current, or, if the
//               step overflowed, leaves the old set current and rewrites the
//               params from it -- the skip without a second pass.
//
// The work is a few flops per byte, so HBM bandwidth bounds every kernel;
// no tensor cores are involved.  Each thread handles kVec = 8 consecutive
// elements per iteration with 16-byte loads (one per 16-bit gradient
// buffer): the ranks' loads in chunks of 4, each chunk issued before its
// adds, then the state loads, and walks a grid sized to fill every SM
// (grid-stride loop, 64-bit indices).  Elements past the last full vector, padding
// positions and buffers that are not 16-byte aligned take a per-element path
// that performs the same operations in the same order.
//
// Numerics follow the header's definition operation by operation; explicit
// __fadd_rn/__fmul_rn/__fdiv_rn/__fsqrt_rn keep the compiler from fusing or
// reordering anything, and the library is built without fast-math or FTZ.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "zero_internal.h"
#include "zero_row_copy.cuh"

namespace zgb {
namespace {

// ------------------------------------------------------------ memory ops

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ float4 ld_state(const float *p)
{
    return __ldcs(reinterpret_cast<const float4 *>(p));
}

__device__ __forceinline__ void st_state(float *p, float4 v)
{
    __stcs(reinterpret_cast<float4 *>(p), v);
}

// Store 16 bytes at an address aligned to `align` (16, 8, 4 or 2) bytes.
__device__ __forceinline__ void st16(void *p, uint4 v, int align)
{
    if (align >= 16) {
        __stcs(reinterpret_cast<uint4 *>(p), v);
    } else if (align == 8) {
        uint2 *q = reinterpret_cast<uint2 *>(p);
        __stcs(q, make_uint2(v.x, v.y));
        __stcs(q + 1, make_uint2(v.z, v.w));
    } else if (align == 4) {
        unsigned *q = reinterpret_cast<unsigned *>(p);
        q[0] = v.x; q[1] = v.y; q[2] = v.z; q[3] = v.w;
    } else {
        unsigned short *q = reinterpret_cast<unsigned short *>(p);
        const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            q[2 * i] = (unsigned short)(w[i] & 0xffffu);
            q[2 * i + 1] = (unsigned short)(w[i] >> 16);
        }
    }
}

// ------------------------------------------------------- element types

template <int DT> struct Ty;

template <> struct Ty<F32> {
    static constexpr int kLoads = 2;   // 16-byte loads per 8 elements
    __device__ static float load1(const void *p, int64_t i) { return static_cast<const float *>(p)[i]; }
    __device__ static void store1(void *p, int64_t i, float x) { static_cast<float *>(p)[i] = x; }
    __device__ static void widen(const uint4 *r, float (&o)[kVec])
    {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            o[4 * h + 0] = __uint_as_float(r[h].x);
            o[4 * h + 1] = __uint_as_float(r[h].y);
            o[4 * h + 2] = __uint_as_float(r[h].z);
            o[4 * h + 3] = __uint_as_float(r[h].w);
        }
    }
    __device__ static void narrow(const float (&x)[kVec], uint4 *r)
    {
#pragma unroll
        for (int h = 0; h < 2; ++h)
            r[h] = make_uint4(__float_as_uint(x[4 * h]), __float_as_uint(x[4 * h + 1]),
                              __float_as_uint(x[4 * h + 2]), __float_as_uint(x[4 * h + 3]));
    }
};

template <> struct Ty<BF16> {
    static constexpr int kLoads = 1;
    __device__ static float load1(const void *p, int64_t i)
    {
        return __uint_as_float((unsigned)static_cast<const unsigned short *>(p)[i] << 16);
    }
    __device__ static void store1(void *p, int64_t i, float x)
    {
        static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(x);
    }
    // bf16 -> fp32 is exact: the 16 bits become the top half of the word.
    __device__ static void widen(const uint4 *r, float (&o)[kVec])
    {
        const unsigned w[4] = {r[0].x, r[0].y, r[0].z, r[0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            o[2 * i] = __uint_as_float(w[i] << 16);
            o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static void narrow(const float (&x)[kVec], uint4 *r)
    {
        unsigned w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
            w[i] = *reinterpret_cast<unsigned *>(&h);
        }
        r[0] = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <> struct Ty<F16> {
    static constexpr int kLoads = 1;
    __device__ static float load1(const void *p, int64_t i)
    {
        return __half2float(static_cast<const __half *>(p)[i]);
    }
    __device__ static void store1(void *p, int64_t i, float x)
    {
        static_cast<__half *>(p)[i] = __float2half_rn(x);
    }
    __device__ static void widen(const uint4 *r, float (&o)[kVec])
    {
        const unsigned w[4] = {r[0].x, r[0].y, r[0].z, r[0].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
            float2 f = __half22float2(h);
            o[2 * i] = f.x;
            o[2 * i + 1] = f.y;
        }
    }
    __device__ static void narrow(const float (&x)[kVec], uint4 *r)
    {
        unsigned w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __half2 h = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
            w[i] = *reinterpret_cast<unsigned *>(&h);
        }
        r[0] = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// ------------------------------------------------------------ arithmetic

__device__ __forceinline__ bool nonfinite(float x)
{
    return (__float_as_uint(x) & 0x7f800000u) == 0x7f800000u;
}

// acc -> g: divide by N, then by the loss scale.
__device__ __forceinline__ float average(float acc, const AverageScalars &s)
{
    float g = s.world_pow2 ? __fmul_rn(acc, s.inv_world) : __fdiv_rn(acc, s.world_f);
    if (s.scaled) g = s.scale_pow2 ? __fmul_rn(g, s.inv_scale) : __fdiv_rn(g, s.scale);
    return g;
}

// One element of Adam with bias correction, eps outside the root; with
// decoupled weight decay (AdamW) the weight is scaled before the step is
// subtracted.
__device__ __forceinline__ void adam1(float g, float &x, float &m, float &v, const AdamScalars &s)
{
    const float mj = __fadd_rn(__fmul_rn(m, s.b1), __fmul_rn(s.c1, g));
    const float vj = __fadd_rn(__fmul_rn(v, s.b2), __fmul_rn(s.c2, __fmul_rn(g, g)));
    const float mh = __fdiv_rn(mj, s.bc1);
    const float vh = __fdiv_rn(vj, s.bc2);
    const float den = __fadd_rn(__fsqrt_rn(vh), s.eps);
    const float upd = __fdiv_rn(__fmul_rn(s.lr, mh), den);
    m = mj;
    v = vj;
    const float xd = s.decoupled ? __fmul_rn(x, s.decay) : x;
    x = __fsub_rn(xd, upd);
}

// 16 bytes from an address on an 8-byte boundary, as two 8-byte loads.
__device__ __forceinline__ uint4 ld_stream_halves(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2+8];" : "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Rank-order sum of 8 consecutive elements at vector index k of every rank
// buffer, chunk by chunk: a chunk's loads (4 ranks) are all issued before
// any of them is added, and within the chunk the adds go in rank order.
// Four ranks per chunk keeps the registers low enough for four resident
// blocks per SM; the bytes in flight come from occupancy.  Rank grads on a
// 16-byte boundary are read 16 bytes per load, those on an 8-byte boundary
// (grad_align, the same for the whole launch) 8 bytes per load.
template <int GT>
__device__ __forceinline__ void rank_sum8(const StepArgs &a, int64_t i, float (&acc)[kVec])
{
    constexpr int L = Ty<GT>::kLoads;
    constexpr int kChunk = 4;
    const int64_t byte_off = i * (GT == F32 ? 4 : 2);
    const bool halves = a.grad_align < 16;
    for (int c = 0; c < a.world; c += kChunk) {
        uint4 raw[kChunk][L];
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
            if (c + u < a.world) {
                const char *p = static_cast<const char *>(a.grads[c + u]) + byte_off;
#pragma unroll
                for (int l = 0; l < L; ++l)
                    raw[u][l] = halves ? ld_stream_halves(p + 16 * l) : ld_stream(p + 16 * l);
            }
        }
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
            if (c + u < a.world) {
                float f[kVec];
                Ty<GT>::widen(raw[u], f);
                if (c + u == 0) {
#pragma unroll
                    for (int e = 0; e < kVec; ++e) acc[e] = f[e];
                } else {
#pragma unroll
                    for (int e = 0; e < kVec; ++e) acc[e] = __fadd_rn(acc[e], f[e]);
                }
            }
        }
    }
}

template <int GT>
__device__ __forceinline__ float rank_sum1(const StepArgs &a, int64_t i)
{
    if (i >= a.n_valid) return 0.0f;
    float acc = Ty<GT>::load1(a.grads[0], i);
    for (int r = 1; r < a.world; ++r) acc = __fadd_rn(acc, Ty<GT>::load1(a.grads[r], i));
    return acc;
}

template <int PT>
__device__ __forceinline__ void store_params8(void *base, int64_t i, const float (&x)[kVec],
                                              int align)
{
    constexpr int L = Ty<PT>::kLoads;
    uint4 r[L];
    Ty<PT>::narrow(x, r);
    char *p = static_cast<char *>(base) + i * (PT == F32 ? 4 : 2);
#pragma unroll
    for (int l = 0; l < L; ++l) st16(p + 16 * l, r[l], align);
}

__device__ __forceinline__ void load_state8(const float *p, int64_t i, float (&o)[kVec])
{
    const float4 a = ld_state(p + i), b = ld_state(p + i + 4);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

__device__ __forceinline__ void store_state8(float *p, int64_t i, const float (&o)[kVec])
{
    st_state(p + i, make_float4(o[0], o[1], o[2], o[3]));
    st_state(p + i + 4, make_float4(o[4], o[5], o[6], o[7]));
}

// One block-wide OR of the per-thread overflow bits, then at most one atomic
// per block.  Every thread of the block reaches this point.
__device__ __forceinline__ void publish_flag(const StepArgs &a, bool bad, unsigned long long id)
{
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicMax(a.flag, id);
}

// The step's scalars.  An eager launch reads them straight from the kernel's
// parameters (constant-bank operands: no registers held across the loop).  A
// step in the graph form (HYPER) reads them from the context's constant
// slot, into which the step's first launch copied the device block.  The
// choice is a template argument, so the eager kernels carry neither a branch
// nor a copy of the scalars.
__constant__ DeviceHyper c_hyper_slots[kHyperSlots];
template <bool HYPER>
struct ScalarRefs {
    const AdamScalars &ad;
    const AverageScalars &av;
    unsigned long long id;
};

template <bool HYPER>
__device__ __forceinline__ ScalarRefs<HYPER> step_scalars(const StepArgs &a, bool publishing)
{
    if constexpr (HYPER) {
        const DeviceHyper &h = c_hyper_slots[a.slot];
        return ScalarRefs<HYPER>{h.ad, h.av, publishing ? h.flag_id : h.skip_id};
    } else
        return ScalarRefs<HYPER>{a.ad, a.av, a.step_id};
}

// Where a pass reads and writes the state.  One set: in place.  Two sets:
// read the current one; `fresh` passes (fused_step) write the other one,
// in-place passes (apply) write the current one.
struct StatePtrs {
    const float *sx, *sm, *sv;
    float *dx, *dm, *dv;
};

__device__ __forceinline__ StatePtrs select_state(const StepArgs &a, bool fresh)
{
    StatePtrs p{a.master, a.m, a.v, a.master, a.m, a.v};
    if (a.cur) {
        const bool b = (*reinterpret_cast<volatile unsigned long long *>(a.cur) & 1ull) != 0;
        float *cx = b ? a.xb : a.master, *cm = b ? a.mb : a.m, *cv = b ? a.vb : a.v;
        float *ox = b ? a.master : a.xb, *om = b ? a.m : a.mb, *ov = b ? a.v : a.vb;
        p.sx = cx; p.sm = cm; p.sv = cv;
        p.dx = fresh ? ox : cx; p.dm = fresh ? om : cm; p.dv = fresh ? ov : cv;
    }
    return p;
}

// Resident blocks per SM the step kernels are compiled for: four with 16-bit
// grads (measured fastest on GB300: more warps in flight beat a deeper
// per-thread chunk); two with fp32 grads, whose eight-element vectors need
// twice the load registers.
template <int GT> struct MinBlocks { static constexpr int value = GT == F32 ? 2 : 4; };


// ---------------------------------------------------------------- kernels

// The fused pass over the range, as block `block` of the `nblocks` blocks
// that share it (grid-stride over the aligned vectors, then the tail).
template <int GT, int PT, bool AVG, bool HYPER>
__device__ __forceinline__ void fused_step_body(const StepArgs &a, int64_t block, int64_t nblocks)
{
    const int64_t stride = nblocks * blockDim.x;
    const int64_t tid = block * blockDim.x + threadIdx.x;
    const int64_t nvec = a.vec_ok ? a.n_valid / kVec : 0;
    const StatePtrs st = select_state(a, true);
    const ScalarRefs<HYPER> sc = step_scalars<HYPER>(a, true);
    const AverageScalars &av = sc.av;
    const AdamScalars &ad = sc.ad;
    bool bad = false;
    for (int64_t k = tid; k < nvec; k += stride) {
        const int64_t i = k * kVec;
        float x[kVec], m[kVec], v[kVec], acc[kVec];
        // the ranks' grads first, then the state: the state's 24 registers
        // are not held through the rank sum, so the kernel fits 64 registers
        // (four blocks per SM) without spilling
        rank_sum8<GT>(a, i, acc);
        load_state8(st.sx, i, x);
        load_state8(st.sm, i, m);
        load_state8(st.sv, i, v);
        float g[kVec];
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            if (AVG) {
                // the all-reduce mean itself, before unscaling
                acc[e] = av.world_pow2 ? __fmul_rn(acc[e], av.inv_world)
                                       : __fdiv_rn(acc[e], av.world_f);
                g[e] = !av.scaled ? acc[e]
                       : (av.scale_pow2 ? __fmul_rn(acc[e], av.inv_scale)
                                        : __fdiv_rn(acc[e], av.scale));
            } else {
                g[e] = average(acc[e], av);
            }
            bad |= nonfinite(g[e]);
            adam1(g[e], x[e], m[e], v[e], ad);
        }
        store_state8(st.dx, i, x);
        store_state8(st.dm, i, m);
        store_state8(st.dv, i, v);
        store_params8<PT>(a.params, i, x, a.param_align);
        if (AVG) store_params8<GT>(a.grad_avg, i, acc, a.avg_align);
    }
    // per-element path: ragged tail, padding, unaligned buffers
    for (int64_t i = nvec * kVec + tid; i < a.n; i += stride) {
        float acc = rank_sum1<GT>(a, i);
        float mean = av.world_pow2 ? __fmul_rn(acc, av.inv_world) : __fdiv_rn(acc, av.world_f);
        float g = !av.scaled ? mean
                  : (av.scale_pow2 ? __fmul_rn(mean, av.inv_scale) : __fdiv_rn(mean, av.scale));
        bad |= nonfinite(g);
        float x = st.sx[i], m = st.sm[i], v = st.sv[i];
        adam1(g, x, m, v, ad);
        st.dx[i] = x;
        st.dm[i] = m;
        st.dv[i] = v;
        Ty<PT>::store1(a.params, i, x);
        if (AVG) Ty<GT>::store1(a.grad_avg, i, mean);
    }
    publish_flag(a, bad, sc.id);
}

template <int GT, int PT, bool AVG, bool HYPER>
__global__ void __launch_bounds__(kThreads, MinBlocks<GT>::value)
fused_step_kernel(const __grid_constant__ StepArgs a)
{
    pdl_wait();                 // the previous kernel in the stream is done
    pdl_launch_dependents();
    fused_step_body<GT, PT, AVG, HYPER>(a, blockIdx.x, gridDim.x);
}

// ------------------------------------------------ the 4-wide fused pass

__device__ __forceinline__ uint2 ld_stream8(const void *p)
{
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// Store 8 bytes at an address aligned to `align` (8, 4 or 2) bytes.
__device__ __forceinline__ void st8(void *p, uint2 v, int align)
{
    if (align >= 8) {
        __stcs(reinterpret_cast<uint2 *>(p), v);
    } else if (align == 4) {
        unsigned *q = reinterpret_cast<unsigned *>(p);
        q[0] = v.x;
        q[1] = v.y;
    } else {
        unsigned short *q = reinterpret_cast<unsigned short *>(p);
        q[0] = (unsigned short)(v.x & 0xffffu);
        q[1] = (unsigned short)(v.x >> 16);
        q[2] = (unsigned short)(v.y & 0xffffu);
        q[3] = (unsigned short)(v.y >> 16);
    }
}

// Four 16-bit values (8 bytes) widened to fp32, exactly.
template <int GT>
__device__ __forceinline__ void widen4(uint2 r, float (&o)[4])
{
    if constexpr (GT == BF16) {
        o[0] = __uint_as_float(r.x << 16);
        o[1] = __uint_as_float(r.x & 0xffff0000u);
        o[2] = __uint_as_float(r.y << 16);
        o[3] = __uint_as_float(r.y & 0xffff0000u);
    } else {
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&r.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&r.y));
        o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
    }
}

// Four params cast (RNE) and stored at element i of `base`, whose byte
// alignment is `align`.
template <int PT>
__device__ __forceinline__ void store_params4(void *base, int64_t i, const float (&x)[4],
                                              int align)
{
    if constexpr (PT == F32) {
        st16(static_cast<char *>(base) + i * 4,
             make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                        __float_as_uint(x[3])), align);
    } else {
        unsigned w[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if constexpr (PT == BF16) {
                __nv_bfloat162 v = __floats2bfloat162_rn(x[2 * h], x[2 * h + 1]);
                w[h] = *reinterpret_cast<unsigned *>(&v);
            } else {
                __half2 v = __floats2half2_rn(x[2 * h], x[2 * h + 1]);
                w[h] = *reinterpret_cast<unsigned *>(&v);
            }
        }
        st8(static_cast<char *>(base) + i * 2, make_uint2(w[0], w[1]), align < 8 ? align : 8);
    }
}

// The fused pass with 4 elements per thread and every load of an iteration
// issued before its arithmetic: the state first, then the ranks 8 at a time
// -- one memory round trip for up to 8 ranks, where fused_step_body makes
// three (two rank chunks, then the state, which it loads last to stay at 64
// registers).  For ranges that give a thread one iteration of the 8-wide
// layout at most (a small unit's step inside a visit), where those round
// trips are the launch's latency.  16-bit grads; the same operations in the
// same order as fused_step_body, element by element.
template <int GT, int PT>
__device__ __forceinline__ void fused_step_body4(const StepArgs &a, int64_t block, int64_t nblocks)
{
    static_assert(GT != F32, "16-bit grads only");
    constexpr int kChunk = 8;
    const int64_t stride = nblocks * blockDim.x;
    const int64_t tid = block * blockDim.x + threadIdx.x;
    const int64_t nvec = a.vec_ok ? a.n_valid / 4 : 0;
    const StatePtrs st = select_state(a, true);
    const AverageScalars &av = a.av;
    const AdamScalars &ad = a.ad;
    bool bad = false;
    for (int64_t k = tid; k < nvec; k += stride) {
        const int64_t i = k * 4;
        const float4 xs = ld_state(st.sx + i), ms = ld_state(st.sm + i), vs = ld_state(st.sv + i);
        float acc[4];
        for (int c = 0; c < a.world; c += kChunk) {
            uint2 raw[kChunk];
#pragma unroll
            for (int u = 0; u < kChunk; ++u)
                if (c + u < a.world)
                    raw[u] = ld_stream8(static_cast<const char *>(a.grads[c + u]) + i * 2);
#pragma unroll
            for (int u = 0; u < kChunk; ++u) {
                if (c + u < a.world) {
                    float f[4];
                    widen4<GT>(raw[u], f);
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[e] = c + u == 0 ? f[e] : __fadd_rn(acc[e], f[e]);
                }
            }
        }
        float x[4] = {xs.x, xs.y, xs.z, xs.w}, m[4] = {ms.x, ms.y, ms.z, ms.w};
        float v[4] = {vs.x, vs.y, vs.z, vs.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float g = average(acc[e], av);
            bad |= nonfinite(g);
            adam1(g, x[e], m[e], v[e], ad);
        }
        st_state(st.dx + i, make_float4(x[0], x[1], x[2], x[3]));
        st_state(st.dm + i, make_float4(m[0], m[1], m[2], m[3]));
        st_state(st.dv + i, make_float4(v[0], v[1], v[2], v[3]));
        store_params4<PT>(a.params, i, x, a.param_align);
    }
    // per-element path: ragged tail, padding, unaligned buffers
    for (int64_t i = nvec * 4 + tid; i < a.n; i += stride) {
        const float g = average(rank_sum1<GT>(a, i), av);
        bad |= nonfinite(g);
        float x = st.sx[i], m = st.sm[i], v = st.sv[i];
        adam1(g, x, m, v, ad);
        st.dx[i] = x;
        st.dm[i] = m;
        st.dv[i] = v;
        Ty<PT>::store1(a.params, i, x);
    }
    publish_flag(a, bad, a.step_id);
}

// A ZeRO-3 backward visit in one launch: blocks [0, step_blocks) run the
// fused pass over one unit (as fused_step_kernel), the rest place the next
// unit's shards (as gather_kernel, row_blocks blocks per shard).  The two
// touch disjoint memory (the host checks it), so neither waits for the
// other; one launch pays one ramp-up and one drain instead of two.
template <int GT, int PT>
__global__ void __launch_bounds__(kThreads, MinBlocks<GT>::value)
step_gather_kernel(const __grid_constant__ StepGatherArgs a)
{
    pdl_wait();                 // the previous kernel in the stream is done
    pdl_launch_dependents();
    const int b = (int)blockIdx.x;
    if (b < a.step_blocks) {
        if constexpr (GT != F32) {
            if (a.step_short) {
                fused_step_body4<GT, PT>(a.step, b, a.step_blocks);
                return;
            }
        }
        fused_step_body<GT, PT, false, false>(a.step, b, a.step_blocks);
        return;
    }
    const int gb = b - a.step_blocks;
    const int k = gb / a.row_blocks;
    const char *src = static_cast<const char *>(a.gather.src[k]);
    if (src == nullptr) return;
    rowcopy::gather_row(src, a.gather.dst + (int64_t)k * a.gather.shard_bytes,
                        a.gather.shard_bytes, a.gather.es, gb % a.row_blocks, a.row_blocks);
}

// A backward visit of up to two units in one launch (launch_visit): the
// blocks of step range s run the fused pass over it (the 4-wide body when
// its range gives a thread one 8-wide iteration at most), the blocks after
// all steps place the rows.  The parts touch disjoint memory (the host
// checks it), so none waits for another.  The two step ranges are selected
// with constant indices, so each reads its arguments at fixed offsets.
template <int GT, int PT>
__device__ __forceinline__ void visit_step(const StepArgs &st, int short_body, int32_t block,
                                           int32_t nblocks)
{
    if constexpr (GT != F32) {
        if (short_body) {
            fused_step_body4<GT, PT>(st, block, nblocks);
            return;
        }
    }
    fused_step_body<GT, PT, false, false>(st, block, nblocks);
}

template <int GT, int PT>
__global__ void __launch_bounds__(kThreads, MinBlocks<GT>::value)
visit_kernel(const __grid_constant__ VisitArgs a)
{
    pdl_wait();                 // the previous kernel in the stream is done
    pdl_launch_dependents();
    const int32_t b = (int32_t)blockIdx.x;
    if (a.n_steps > 0 && b < a.step_first_block[1]) {
        visit_step<GT, PT>(a.step[0], a.step_short[0], b, a.step_first_block[1]);
        return;
    }
    if (a.n_steps > 1 && b < a.step_first_block[2]) {
        visit_step<GT, PT>(a.step[1], a.step_short[1], b - a.step_first_block[1],
                           a.step_first_block[2] - a.step_first_block[1]);
        return;
    }
    if (a.n_rows <= 0) return;
    // the row this block belongs to: the last y with row_first_block[y] <= gb
    const int32_t gb = b - a.step_first_block[a.n_steps];
    int lo = 0, hi = a.n_rows - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.row_first_block[mid] <= gb) lo = mid; else hi = mid - 1;
    }
    const char *src = static_cast<const char *>(a.src[lo]);
    if (src == nullptr || a.bytes[lo] <= 0) return;
    rowcopy::gather_row(src, a.dst[lo], a.bytes[lo], a.es, gb - a.row_first_block[lo],
                        a.row_first_block[lo + 1] - a.row_first_block[lo]);
}

template <int GT, bool AVG, bool HYPER>
__global__ void __launch_bounds__(kThreads, MinBlocks<GT>::value)
reduce_kernel(const __grid_constant__ StepArgs a)
{
    pdl_wait();                 // the previous kernel in the stream is done
    pdl_launch_dependents();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nvec = a.vec_ok ? a.n_valid / kVec : 0;
    const ScalarRefs<HYPER> sc = step_scalars<HYPER>(a, true);
    bool bad = false;
    for (int64_t k = tid; k < nvec; k += stride) {
        const int64_t i = k * kVec;
        float acc[kVec], g[kVec];
        rank_sum8<GT>(a, i, acc);
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            acc[e] = sc.av.world_pow2 ? __fmul_rn(acc[e], sc.av.inv_world)
                                     : __fdiv_rn(acc[e], sc.av.world_f);
            g[e] = !sc.av.scaled ? acc[e]
                   : (sc.av.scale_pow2 ? __fmul_rn(acc[e], sc.av.inv_scale)
                                      : __fdiv_rn(acc[e], sc.av.scale));
            bad |= nonfinite(g[e]);
        }
        store_state8(a.g, i, g);
        if (AVG) store_params8<GT>(a.grad_avg, i, acc, a.avg_align);
    }
    for (int64_t i = nvec * kVec + tid; i < a.n; i += stride) {
        float acc = rank_sum1<GT>(a, i);
        float mean = sc.av.world_pow2 ? __fmul_rn(acc, sc.av.inv_world) : __fdiv_rn(acc, sc.av.world_f);
        float g = !sc.av.scaled ? mean
                  : (sc.av.scale_pow2 ? __fmul_rn(mean, sc.av.inv_scale) : __fdiv_rn(mean, sc.av.scale));
        bad |= nonfinite(g);
        a.g[i] = g;
        if (AVG) Ty<GT>::store1(a.grad_avg, i, mean);
    }
    publish_flag(a, bad, sc.id);
}

// The second pass of the two-pass step: Adam from the fp32 scratch, 4
// elements per thread per iteration (each iteration's 4 loads issued before
// its arithmetic, its 4 stores after), four resident blocks per SM.  The
// division and square root per element make this pass twice as heavy in
// arithmetic per byte as the fused pass; with 8 elements per thread (the
// fused pass's layout) it reached 0.89 of the measured copy rate, with 4
// per thread 0.96 (GPT-2 XL, 16 fp16 ranks: 7.76 against 7.14 ms).
template <int PT, bool HYPER>
__global__ void __launch_bounds__(kThreads, 4)
apply_kernel(const __grid_constant__ StepArgs a)
{
    pdl_wait();                 // the previous kernel in the stream is done
    pdl_launch_dependents();
    // The verdict of the whole step is known: a skipped step writes nothing.
    const ScalarRefs<HYPER> sc = step_scalars<HYPER>(a, false);
    if (*reinterpret_cast<volatile unsigned long long *>(a.flag) == sc.id) return;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nvec = a.vec_ok ? a.n / 4 : 0;
    const StatePtrs st = select_state(a, false);
    for (int64_t k = tid; k < nvec; k += stride) {
        const int64_t i = k * 4;
        const float4 gs = ld_state(a.g + i), xs = ld_state(st.sx + i), ms = ld_state(st.sm + i),
                     vs = ld_state(st.sv + i);
        float g[4] = {gs.x, gs.y, gs.z, gs.w}, x[4] = {xs.x, xs.y, xs.z, xs.w};
        float m[4] = {ms.x, ms.y, ms.z, ms.w}, v[4] = {vs.x, vs.y, vs.z, vs.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) adam1(g[e], x[e], m[e], v[e], sc.ad);
        st_state(st.dx + i, make_float4(x[0], x[1], x[2], x[3]));
        st_state(st.dm + i, make_float4(m[0], m[1], m[2], m[3]));
        st_state(st.dv + i, make_float4(v[0], v[1], v[2], v[3]));
        store_params4<PT>(a.params, i, x, a.param_align);
    }
    for (int64_t i = nvec * 4 + tid; i < a.n; i += stride) {
        float x = st.sx[i], m = st.sm[i], v = st.sv[i];
        adam1(a.g[i], x, m, v, sc.ad);
        st.dx[i] = x;
        st.dm[i] = m;
        st.dv[i] = v;
        Ty<PT>::store1(a.params, i, x);
    }
}

template <int PT>
__global__ void __launch_bounds__(kThreads)
finalize_kernel(const __grid_constant__ StepArgs a)
{
    pdl_wait();                 // the previous kernel in the stream is done
    pdl_launch_dependents();
    const unsigned long long skip_id = a.hyper ? c_hyper_slots[a.slot].skip_id : a.step_id;
    const bool overflowed =
        *reinterpret_cast<volatile unsigned long long *>(a.flag) == skip_id;
    if (!overflowed) {
        // the set the step wrote becomes current; no block reads the word here
        if (blockIdx.x == 0 && threadIdx.x == 0) *a.cur ^= 1ull;
        return;
    }
    // skipped step: the old set stays current; the params were written from
    // the discarded update, so cast them again from the kept master
    const bool b = (*reinterpret_cast<volatile unsigned long long *>(a.cur) & 1ull) != 0;
    const float *x = b ? a.xb : a.master;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nvec = a.vec_ok ? a.n / kVec : 0;
    for (int64_t k = tid; k < nvec; k += stride) {
        float v[kVec];
        load_state8(x, k * kVec, v);
        store_params8<PT>(a.params, k * kVec, v, a.param_align);
    }
    for (int64_t i = nvec * kVec + tid; i < a.n; i += stride) Ty<PT>::store1(a.params, i, x[i]);
}

// ------------------------------------------------------------- launching

}  // namespace

cudaError_t hyper_slot_address(int slot, void **addr)
{
    if (slot < 0 || slot >= kHyperSlots) return cudaErrorInvalidValue;
    void *base = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&base, c_hyper_slots);
    if (e != cudaSuccess) return e;
    *addr = static_cast<char *>(base) + (size_t)slot * sizeof(DeviceHyper);
    return cudaSuccess;
}

cudaError_t load_hyper_slot(int slot, const DeviceHyper *block, cudaStream_t s)
{
    if (slot < 0 || slot >= kHyperSlots) return cudaErrorInvalidValue;
    return cudaMemcpyToSymbolAsync(c_hyper_slots, block, sizeof(DeviceHyper),
                                   (size_t)slot * sizeof(DeviceHyper), cudaMemcpyDeviceToDevice,
                                   s);
}

namespace {

template <typename K>
cudaError_t launch(K kernel, const StepArgs &a, int64_t work_items, int sms, int cap_per_sm, cudaStream_t s)
{
    int per_sm = resident_blocks_per_sm(reinterpret_cast<const void *>(kernel), kThreads);
    if (cap_per_sm > 0 && per_sm > cap_per_sm) per_sm = cap_per_sm;   // room for other kernels
    int64_t want = (work_items + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)sms * per_sm;
    int64_t blocks = want < cap ? want : cap;
    if (blocks < 1) blocks = 1;
    return launch_dependent(kernel, dim3((unsigned)blocks), dim3(kThreads), 0, s, a);
}

int64_t items(const StepArgs &a, int64_t nvec_src)
{
    // threads needed: one per vector of the aligned part, plus the tail
    const int64_t nvec = a.vec_ok ? nvec_src / kVec : 0;
    const int64_t tail = a.n - nvec * kVec;
    return nvec > tail ? nvec : tail;
}

template <int GT, int PT, bool HYPER>
cudaError_t fused_h(const StepArgs &a, int sms, int cap_per_sm, cudaStream_t s)
{
    const int64_t w = items(a, a.n_valid);
    return a.grad_avg ? launch(fused_step_kernel<GT, PT, true, HYPER>, a, w, sms, cap_per_sm, s)
                      : launch(fused_step_kernel<GT, PT, false, HYPER>, a, w, sms, cap_per_sm, s);
}

template <int GT, int PT>
cudaError_t fused_pt(const StepArgs &a, int sms, int cap_per_sm, cudaStream_t s)
{
    return a.hyper ? fused_h<GT, PT, true>(a, sms, cap_per_sm, s) : fused_h<GT, PT, false>(a, sms, cap_per_sm, s);
}

template <int GT>
cudaError_t fused_gt(int32_t pdt, const StepArgs &a, int sms, int cap_per_sm, cudaStream_t s)
{
    switch (pdt) {
    case F32: return fused_pt<GT, F32>(a, sms, cap_per_sm, s);
    case BF16: return fused_pt<GT, BF16>(a, sms, cap_per_sm, s);
    case F16: return fused_pt<GT, F16>(a, sms, cap_per_sm, s);
    }
    return cudaErrorInvalidValue;
}

template <int GT, bool HYPER>
cudaError_t reduce_h(const StepArgs &a, int sms, int cap_per_sm, cudaStream_t s)
{
    const int64_t w = items(a, a.n_valid);
    return a.grad_avg ? launch(reduce_kernel<GT, true, HYPER>, a, w, sms, cap_per_sm, s)
                      : launch(reduce_kernel<GT, false, HYPER>, a, w, sms, cap_per_sm, s);
}

template <int GT>
cudaError_t reduce_gt(const StepArgs &a, int sms, int cap_per_sm, cudaStream_t s)
{
    return a.hyper ? reduce_h<GT, true>(a, sms, cap_per_sm, s) : reduce_h<GT, false>(a, sms, cap_per_sm, s);
}

template <int PT>
cudaError_t apply_pt(const StepArgs &a, int sms, int cap_per_sm, cudaStream_t s)
{
    // threads needed: one per 4-element vector, or per element of the tail
    const int64_t nvec = a.vec_ok ? a.n / 4 : 0, tail = a.n - nvec * 4;
    const int64_t w = nvec > tail ? nvec : tail;
    return a.hyper ? launch(apply_kernel<PT, true>, a, w, sms, cap_per_sm, s)
                   : launch(apply_kernel<PT, false>, a, w, sms, cap_per_sm, s);
}

}  // namespace

cudaError_t launch_fused_step(int32_t gdt, int32_t pdt, const StepArgs &a, int sms,
                              int cap_per_sm, cudaStream_t s)
{
    switch (gdt) {
    case F32: return fused_gt<F32>(pdt, a, sms, cap_per_sm, s);
    case BF16: return fused_gt<BF16>(pdt, a, sms, cap_per_sm, s);
    case F16: return fused_gt<F16>(pdt, a, sms, cap_per_sm, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_reduce(int32_t gdt, const StepArgs &a, int sms, int cap_per_sm, cudaStream_t s)
{
    switch (gdt) {
    case F32: return reduce_gt<F32>(a, sms, cap_per_sm, s);
    case BF16: return reduce_gt<BF16>(a, sms, cap_per_sm, s);
    case F16: return reduce_gt<F16>(a, sms, cap_per_sm, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_finalize(int32_t pdt, const StepArgs &a, int sms, int cap_per_sm, cudaStream_t s)
{
    const int64_t w = items(a, a.n);
    switch (pdt) {
    case F32: return launch(finalize_kernel<F32>, a, w, sms, cap_per_sm, s);
    case BF16: return launch(finalize_kernel<BF16>, a, w, sms, cap_per_sm, s);
    case F16: return launch(finalize_kernel<F16>, a, w, sms, cap_per_sm, s);
    }
    return cudaErrorInvalidValue;
}

namespace {

template <int GT, int PT>
cudaError_t step_gather_pt(const StepArgs &st, const GatherArgs &g, int sms, int cap_per_sm,
                           cudaStream_t s)
{
    auto kernel = step_gather_kernel<GT, PT>;
    int per_sm = resident_blocks_per_sm(reinterpret_cast<const void *>(kernel), kThreads);
    const int resident = sms * per_sm;
    if (cap_per_sm > 0 && per_sm > cap_per_sm) per_sm = cap_per_sm;
    const int64_t cap = (int64_t)sms * per_sm;
    // a short step range (one 8-wide iteration per thread at most) of 16-bit
    // grads takes the 4-wide body, which issues an iteration's loads at once
    const bool step_short = GT != F32 && st.vec_ok && st.n_valid <= cap * kThreads * kVec;
    int64_t work = items(st, st.n_valid);
    if (step_short) {
        const int64_t nvec4 = st.n_valid / 4, tail = st.n - nvec4 * 4;
        work = nvec4 > tail ? nvec4 : tail;
    }
    // the step part: the grid fused_step_kernel would get for that work
    const int64_t want = (work + kThreads - 1) / kThreads;
    int64_t step_blocks = st.n > 0 ? (want < cap ? want : cap) : 0;
    if (st.n > 0 && step_blocks < 1) step_blocks = 1;
    // the gather part: the rows gather_kernel would get
    StepGatherArgs a;
    a.step = st;
    a.gather = g;
    const int64_t row_blocks =
        g.shard_bytes > 0 ? rowcopy::row_blocks(g.shard_bytes, kThreads, resident) : 0;
    a.step_blocks = (int32_t)step_blocks;
    a.row_blocks = (int32_t)row_blocks;
    a.step_short = step_short ? 1 : 0;
    const int64_t blocks = step_blocks + row_blocks * (g.shard_bytes > 0 ? g.n : 0);
    if (blocks == 0) return cudaSuccess;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    return launch_dependent(kernel, dim3((unsigned)blocks), dim3(kThreads), 0, s, a);
}

template <int GT>
cudaError_t step_gather_gt(int32_t pdt, const StepArgs &st, const GatherArgs &g, int sms,
                           int cap_per_sm, cudaStream_t s)
{
    switch (pdt) {
    case F32: return step_gather_pt<GT, F32>(st, g, sms, cap_per_sm, s);
    case BF16: return step_gather_pt<GT, BF16>(st, g, sms, cap_per_sm, s);
    case F16: return step_gather_pt<GT, F16>(st, g, sms, cap_per_sm, s);
    }
    return cudaErrorInvalidValue;
}

template <int GT, int PT>
cudaError_t visit_pt(const VisitArgs &in, int sms, int cap_per_sm, cudaStream_t s)
{
    auto kernel = visit_kernel<GT, PT>;
    int per_sm = resident_blocks_per_sm(reinterpret_cast<const void *>(kernel), kThreads);
    const int resident = sms * per_sm;
    if (cap_per_sm > 0 && per_sm > cap_per_sm) per_sm = cap_per_sm;
    const int64_t cap = (int64_t)sms * per_sm;
    if (in.n_steps < 0 || in.n_steps > kVisitSteps || in.n_rows < 0 || in.n_rows > kVisitRows)
        return cudaErrorInvalidValue;
    VisitArgs a = in;
    int64_t total = 0;
    for (int i = 0; i < a.n_steps; ++i) {
        // each step range gets the grid step_gather_pt gives one
        const StepArgs &st = a.step[i];
        const bool step_short = GT != F32 && st.vec_ok && st.n_valid <= cap * kThreads * kVec;
        int64_t work = items(st, st.n_valid);
        if (step_short) {
            const int64_t nvec4 = st.n_valid / 4, tail = st.n - nvec4 * 4;
            work = nvec4 > tail ? nvec4 : tail;
        }
        const int64_t want = (work + kThreads - 1) / kThreads;
        int64_t blocks = st.n > 0 ? (want < cap ? want : cap) : 0;
        if (st.n > 0 && blocks < 1) blocks = 1;
        a.step_first_block[i] = (int32_t)total;
        a.step_short[i] = step_short ? 1 : 0;
        total += blocks;
    }
    a.step_first_block[a.n_steps] = (int32_t)total;
    int64_t rows = 0;
    for (int32_t y = 0; y < a.n_rows; ++y) {
        a.row_first_block[y] = (int32_t)rows;
        if (a.src[y] && a.bytes[y] > 0)
            rows += rowcopy::row_blocks(a.bytes[y], kThreads, resident);
        if (total + rows > 0x7fffffff) return cudaErrorInvalidValue;
    }
    a.row_first_block[a.n_rows] = (int32_t)rows;
    const int64_t blocks = total + rows;
    if (blocks == 0) return cudaSuccess;
    return launch_dependent(kernel, dim3((unsigned)blocks), dim3(kThreads), 0, s, a);
}

template <int GT>
cudaError_t visit_gt(int32_t pdt, const VisitArgs &a, int sms, int cap_per_sm, cudaStream_t s)
{
    switch (pdt) {
    case F32: return visit_pt<GT, F32>(a, sms, cap_per_sm, s);
    case BF16: return visit_pt<GT, BF16>(a, sms, cap_per_sm, s);
    case F16: return visit_pt<GT, F16>(a, sms, cap_per_sm, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_visit(int32_t gdt, int32_t pdt, const VisitArgs &a, int sms, int cap_per_sm,
                         cudaStream_t s)
{
    for (int i = 0; i < a.n_steps && i < kVisitSteps; ++i)
        if (a.step[i].hyper || a.step[i].grad_avg) return cudaErrorInvalidValue;   // eager only
    switch (gdt) {
    case F32: return visit_gt<F32>(pdt, a, sms, cap_per_sm, s);
    case BF16: return visit_gt<BF16>(pdt, a, sms, cap_per_sm, s);
    case F16: return visit_gt<F16>(pdt, a, sms, cap_per_sm, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_step_gather(int32_t gdt, int32_t pdt, const StepArgs &st,
                               const GatherArgs &g, int sms, int cap_per_sm, cudaStream_t s)
{
    if (st.hyper || st.grad_avg) return cudaErrorInvalidValue;   // eager unit steps only
    switch (gdt) {
    case F32: return step_gather_gt<F32>(pdt, st, g, sms, cap_per_sm, s);
    case BF16: return step_gather_gt<BF16>(pdt, st, g, sms, cap_per_sm, s);
    case F16: return step_gather_gt<F16>(pdt, st, g, sms, cap_per_sm, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_apply(int32_t pdt, const StepArgs &a, int sms, int cap_per_sm, cudaStream_t s)
{
    switch (pdt) {
    case F32: return apply_pt<F32>(a, sms, cap_per_sm, s);
    case BF16: return apply_pt<BF16>(a, sms, cap_per_sm, s);
    case F16: return apply_pt<F16>(a, sms, cap_per_sm, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace zgb
