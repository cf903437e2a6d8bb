// Steps whose scalars advance on the device.
//
// A step captured in a CUDA graph, or launched without waiting for the last
// verdict, takes its per-step scalars from a device block (DeviceHyper).
// advance_kernel, launched after a step's kernels, does on the device what
// the host otherwise does between steps: read the step's overflow verdict
// from the flag word, apply the loss-scale policy ("PaddlePaddle ZeRO优化",
// 混合精度才是最佳拍档: a skipped step halves the scale and does not count;
// after growth_interval clean steps the scale doubles, never to infinity),
// advance t on applied steps, and rewrite the block for the next step: the
// bias corrections 1 - beta^t from a table the host computed (so they are
// the host's values bit for bit), the unscale factor from the new scale, and
// the next step id.  One thread; a few hundred bytes move.
#include <cstdint>

#include "zero_internal.h"

namespace zgb {
namespace {

// A power of two whose reciprocal is a normal number (division by it is
// then exactly multiplication by the reciprocal).
__device__ __forceinline__ bool pow2_normal_inverse(float x)
{
    const uint32_t u = __float_as_uint(x);
    const uint32_t exp = (u >> 23) & 0xffu, man = u & 0x7fffffu;
    return (u >> 31) == 0 && man == 0 && exp >= 1 && exp <= 253;
}

__global__ void __launch_bounds__(32)
advance_kernel(DeviceHyper *hyper, const unsigned long long *flag, AdvanceState *st,
               const float *table, int64_t t_max)
{
    pdl_wait();                 // the step's kernels are done
    pdl_launch_dependents();
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    const DeviceHyper cur = *hyper;
    AdvanceState s = *st;
    if (s.status != 0) return;  // the table ran out before: nothing advances
    const bool scaled = cur.av.scaled != 0;
    const bool skipped =
        scaled && *reinterpret_cast<const volatile unsigned long long *>(flag) == cur.skip_id;
    int64_t t = s.t;
    float scale = s.scale;
    int64_t good = s.good_steps;
    if (scaled) {
        if (skipped) {
            good = 0;
            scale = __fmul_rn(scale, 0.5f);
        } else {
            t += 1;
            good += 1;
            if (s.growth_interval > 0 && good >= s.growth_interval) {
                good = 0;
                const float grown = __fmul_rn(scale, 2.0f);
                if (isfinite(grown)) scale = grown;
            }
        }
    } else {
        t += 1;
    }
    if (t > t_max) {            // no bias corrections for step t: stop here
        st->status = 1;
        return;
    }
    DeviceHyper next = cur;
    next.ad.bc1 = table[2 * (t - 1)];
    next.ad.bc2 = table[2 * (t - 1) + 1];
    if (scaled) {
        // as the host derives them from a loss scale (a scale of 0 is no scaling)
        const bool on = scale > 0.0f;
        next.av.scaled = on ? 1 : 0;
        next.av.scale = on ? scale : 1.0f;
        next.av.scale_pow2 = (on && pow2_normal_inverse(scale)) ? 1 : 0;
        next.av.inv_scale = __fdiv_rn(1.0f, next.av.scale);
    }
    const unsigned long long id = cur.flag_id + 1;
    next.flag_id = id;
    next.skip_id = next.av.scaled ? id : ~0ull;
    *hyper = next;
    s.t = t;
    s.scale = scale;
    s.good_steps = good;
    *st = s;
}

}  // namespace

cudaError_t launch_advance(DeviceHyper *hyper, const unsigned long long *flag, AdvanceState *st,
                           const float *table, int64_t t_max, cudaStream_t s)
{
    return launch_dependent(advance_kernel, dim3(1), dim3(32), 0, s, hyper, flag, st, table,
                            t_max);
}

}  // namespace zgb
