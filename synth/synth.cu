// Seeded synthetic inputs for the ZeRO step: gradients and initial master
// weights with an approximately normal distribution N(0, sigma^2).
//
// This module holds no arithmetic of the method.  It is the one piece of code
// both sides of the parity tests use: the CPU oracle receives arrays produced
// by synth_fill_host(), the CUDA library receives buffers filled on the
// device by synth_fill_device(), and a GPU test checks that the two fills are
// bit-identical.
//
// Definition (counter-based, so any element can be drawn on its own):
//   mix64(z)     = the splitmix64 output function (Steele, Lea and Flood,
//                  "Fast splittable pseudorandom number generators", OOPSLA
//                  2014; constants as in Vigna's public-domain splitmix64.c):
//                  z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27;
//                  z *= 0x94D049BB133111EB; z ^= z>>31
//   key          = mix64(mix64(tag) ^ seed),
//                  tag = step<<36 | rank<<20 | unit<<4 | kind
//   word(i)      = mix64(key + (i+1) * 0x9E3779B97F4A7C15)   (mod 2^64): the
//                  (i+1)-th splitmix64 output from state `key`
//   c(i)         = sum of the four 16-bit fields of word(i) - 131070, an
//                  integer in [-131070, 131070] (Irwin-Hall of 4 discrete
//                  uniforms, variance (65536^2-1)/3)
//   value(i)     = float(c(i)) * scale, scale = float(sigma/sqrt((65536^2-1)/3))
//                  (one binary32 multiply, round to nearest even)
//   stored value = value(i) rounded to nearest even in the buffer's type.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <string.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__host__ __device__ inline uint64_t mix64(uint64_t z)
{
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z;
}

__host__ __device__ inline int32_t centered(uint64_t w)
{
    int32_t s = (int32_t)(w & 0xffff) + (int32_t)((w >> 16) & 0xffff) +
                (int32_t)((w >> 32) & 0xffff) + (int32_t)((w >> 48) & 0xffff);
    return s - 131070;
}

__host__ __device__ inline uint64_t word_at(uint64_t key, int64_t i)
{
    return mix64(key + (uint64_t)(i + 1) * kGolden);
}

// Host-side binary32 -> 16-bit conversions, round to nearest even.
inline uint16_t host_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t hi = u >> 16, lo = u & 0xffffu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) ++hi;
    return (uint16_t)hi;
}

inline uint16_t host_f16(float f)
{
    _Float16 h = (_Float16)f;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

inline void host_store(void *out, int dtype, int64_t j, float x)
{
    if (dtype == 0) ((float *)out)[j] = x;
    else if (dtype == 1) ((uint16_t *)out)[j] = host_bf16(x);
    else ((uint16_t *)out)[j] = host_f16(x);
}

__global__ void fill_kernel(void *out, int dtype, int64_t n, int64_t index0,
                            const int64_t *indices, uint64_t key, float scale)
{
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
        int64_t i = indices ? indices[j] : index0 + j;
        float x = __fmul_rn((float)centered(word_at(key, i)), scale);
        if (dtype == 0) ((float *)out)[j] = x;
        else if (dtype == 1) ((__nv_bfloat16 *)out)[j] = __float2bfloat16_rn(x);
        else ((__half *)out)[j] = __float2half_rn(x);
    }
}

}  // namespace

extern "C" {

uint64_t synth_tag(int64_t kind, int64_t step, int64_t rank, int64_t unit)
{
    return ((uint64_t)step << 36) | (((uint64_t)rank & 0xffff) << 20) |
           (((uint64_t)unit & 0xffff) << 4) | ((uint64_t)kind & 0xf);
}

uint64_t synth_key(uint64_t seed, uint64_t tag) { return mix64(mix64(tag) ^ seed); }

uint64_t synth_word(uint64_t key, int64_t i) { return word_at(key, i); }

// A seed-chosen index in [0, n): word 0 of the stream, reduced mod n.
int64_t synth_pick_index(uint64_t key, int64_t n)
{
    return n > 0 ? (int64_t)(word_at(key, -1) % (uint64_t)n) : -1;
}

// out[j] = value(index0 + j), or value(indices[j]) when indices != NULL.
void synth_fill_host(void *out, int dtype, int64_t n, int64_t index0,
                     const int64_t *indices, uint64_t key, float scale)
{
    for (int64_t j = 0; j < n; ++j) {
        int64_t i = indices ? indices[j] : index0 + j;
        float x = (float)centered(word_at(key, i)) * scale;
        host_store(out, dtype, j, x);
    }
}

// The same on the device, asynchronously on `stream`.  `indices`, when not
// NULL, is a device array of n int64.  Returns a cudaError_t value.
int synth_fill_device(void *out, int dtype, int64_t n, int64_t index0,
                      const int64_t *indices, uint64_t key, float scale, void *stream)
{
    if (n <= 0) return 0;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 152 * 32) blocks = 152 * 32;
    fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(out, dtype, n, index0,
                                                                    indices, key, scale);
    return (int)cudaGetLastError();
}

}  // extern "C"
