// Stand-in for a model unit's forward/backward compute in the ZeRO-3
// overlap measurement (not part of the method): `iters` dependent FMAs per
// thread on registers, one store per thread so the work is kept.  It
// occupies `blocks` blocks of 128 threads, leaving room on the SMs for a
// concurrent gather.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {
__global__ void busy_kernel(float *sink, int64_t iters)
{
    float a = 1.0f + threadIdx.x * 1e-7f, b = 0.999999f, c = 1e-7f;
    for (int64_t i = 0; i < iters; ++i) a = fmaf(a, b, c);
    sink[(int64_t)blockIdx.x * blockDim.x + threadIdx.x] = a;
}
}  // namespace

// The stand-in asks for the largest shared-memory carveout (it uses none), so
// a lean gather's shared-memory ring can be resident beside it.
extern "C" int standin_busy(float *sink, int blocks, int64_t iters, void *stream)
{
    if (blocks <= 0 || iters < 0 || !sink) return (int)cudaErrorInvalidValue;
    static bool carveout_set = false;
    if (!carveout_set) {
        cudaFuncSetAttribute(busy_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        carveout_set = true;
    }
    busy_kernel<<<blocks, 128, 0, (cudaStream_t)stream>>>(sink, iters);
    return (int)cudaGetLastError();
}
