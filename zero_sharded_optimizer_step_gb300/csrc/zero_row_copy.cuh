// One row of an all-gather placement as device code: `nb` bytes from `src`
// to `dst` spread over the `nblk` blocks of a row, 16 bytes per access.
// Shared by the placement kernels (zero_gather.cu) and the ZeRO-3 visit
// kernel that steps one unit and places the next one's shards in the same
// launch (zero_step_kernels.cu).
//
// A destination k*S elements into a full buffer is, for an odd S and 16-bit
// elements, only 2-byte aligned.  The row therefore peels the bytes before
// the source's first 16-byte boundary, copies the body with 16-byte loads,
// and writes each 16 bytes with the widest store the destination's alignment
// allows (one 16-byte store, or two of 8, four of 4, eight of 2); the last
// partial 16 bytes go element by element.
#pragma once

#include <cstdint>

namespace zgb {
namespace rowcopy {

constexpr int kItems = 4;   // 16-byte chunks in flight per thread

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ void st_any(char *p, uint4 v, int align)
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

__device__ __forceinline__ void copy_elem(char *d, const char *s, int es)
{
    if (es == 4) *reinterpret_cast<unsigned *>(d) = *reinterpret_cast<const unsigned *>(s);
    else *reinterpret_cast<unsigned short *>(d) = *reinterpret_cast<const unsigned short *>(s);
}

// This block (number blk of the row's nblk) copies its part of the row.
// Block 0 of the row also copies the ragged head (up to the source's next
// 16-byte boundary) and tail element by element.
__device__ __forceinline__ void gather_row(const char *src, char *dst, int64_t nb, int es,
                                           int64_t blk, int64_t nblk)
{
    int64_t head = (int64_t)((16 - ((uintptr_t)src & 15)) & 15);
    if (head > nb) head = nb;
    const int64_t nchunks = (nb - head) >> 4;
    const int64_t tail = head + (nchunks << 4);
    const uintptr_t d0 = (uintptr_t)(dst + head);
    const int align = (d0 & 15) == 0 ? 16 : (d0 & 7) == 0 ? 8 : (d0 & 3) == 0 ? 4 : 2;

    if (blk == 0) {
        for (int64_t b = (int64_t)threadIdx.x * es; b < head; b += (int64_t)blockDim.x * es)
            copy_elem(dst + b, src + b, es);
        for (int64_t b = tail + (int64_t)threadIdx.x * es; b < nb; b += (int64_t)blockDim.x * es)
            copy_elem(dst + b, src + b, es);
    }

    const char *s = src + head;
    char *d = dst + head;
    const int64_t T = nblk * blockDim.x;
    int64_t c = blk * blockDim.x + threadIdx.x;
    // kItems chunks per thread per round, each T apart so a warp's accesses
    // stay contiguous
    for (; c + (kItems - 1) * T < nchunks; c += kItems * T) {
        uint4 v[kItems];
#pragma unroll
        for (int u = 0; u < kItems; ++u) v[u] = ld_stream(s + ((c + u * T) << 4));
#pragma unroll
        for (int u = 0; u < kItems; ++u) st_any(d + ((c + u * T) << 4), v[u], align);
    }
    for (; c < nchunks; c += T) st_any(d + (c << 4), ld_stream(s + (c << 4)), align);
}

// Blocks per row of a placement of rows of `row_bytes`: enough for one
// round of kItems chunks per thread, at most twice the resident blocks, so
// that the rows are dispatched one after another and only one or two are in
// flight (measured on GB300 for 63 shards of 234 MB: 6.9 TB/s, against 5.4
// TB/s with ~32 shards in flight and 4.1 TB/s when every block streamed its
// own contiguous slice).
inline int64_t row_blocks(int64_t row_bytes, int threads, int64_t resident)
{
    const int64_t chunks = (row_bytes + 15) / 16;
    int64_t want = (chunks + (int64_t)threads * kItems - 1) / ((int64_t)threads * kItems);
    int64_t bx = 2 * resident < want ? 2 * resident : want;
    return bx < 1 ? 1 : bx;
}

}  // namespace rowcopy
}  // namespace zgb
