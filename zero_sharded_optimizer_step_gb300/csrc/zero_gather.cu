// All-gather placement on one GPU: shard k (S elements) is copied to
// full + k*S ("ZeRO 与 FSDP…", all_gather_into_tensor; for stage 3 the same
// placement per unit before its forward and backward, section ZeRO-3 与
// FSDP).  A pure copy, bound by HBM bandwidth: 2 bytes moved per byte placed.
//
// One grid row (blockIdx.y) per shard, each with more blocks than the GPU
// holds at once (see launch_gather); the row copy itself (peeled head,
// 16-byte body, widest store the destination allows) is in zero_row_copy.cuh.
#include <cstring>

#include "zero_internal.h"
#include "zero_row_copy.cuh"

namespace zgb {
namespace {

using rowcopy::gather_row;

__global__ void __launch_bounds__(kThreads)
gather_kernel(const __grid_constant__ GatherArgs a)
{
    pdl_wait();                 // the previous kernel in the stream is done
    pdl_launch_dependents();
    const int k = blockIdx.y;
    const char *src = static_cast<const char *>(a.src[k]);
    if (src == nullptr) return;
    gather_row(src, a.dst + (int64_t)k * a.shard_bytes, a.shard_bytes, a.es, blockIdx.x,
               gridDim.x);
}

__global__ void __launch_bounds__(kThreads)
gather_rows_kernel(const __grid_constant__ GatherRowsArgs a)
{
    pdl_wait();                 // the previous kernel in the stream is done
    pdl_launch_dependents();
    // the row this block belongs to: the last y with first_block[y] <= b
    const int32_t b = (int32_t)blockIdx.x;
    int lo = 0, hi = a.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.first_block[mid] <= b) lo = mid; else hi = mid - 1;
    }
    const int y = lo;
    const char *src = static_cast<const char *>(a.src[y]);
    if (src == nullptr || a.bytes[y] <= 0) return;
    gather_row(src, a.dst[y], a.bytes[y], a.es, b - a.first_block[y],
               a.first_block[y + 1] - a.first_block[y]);
}


// ------------------------------------------------------------ lean gather
//
// The same placement driven by the SM's bulk-copy (TMA) unit: one warp per
// CTA, one CTA per SM, 1-D cp.async.bulk copies of up to 32 KB global ->
// shared -> global through a 4-stage ring (128 KB of shared memory), with
// completion of each load signalled on an mbarrier.  Lane 0 issues
// everything; the CTA holds 32 threads and few registers, so kernels running
// concurrently (the next unit's compute during a ZeRO-3 prefetch) keep
// almost all of every SM.  Tiles are numbered row-major over all placed
// shards and dealt round-robin to the CTAs, so the GPU sweeps one compact
// window of one shard at a time.  Needs 16-byte aligned sources and
// destinations and a shard length that is a multiple of 16 bytes.
//
// Every wait is bounded: a load that has not completed after kWaitPolls
// polls counts a timeout in g_gather_timeouts, stops issuing, drains what is
// in flight (again with bounded waits) and returns.

constexpr int kTmaTile = 32768;
constexpr int kTmaStages = 4;
constexpr long long kWaitPolls = 1ll << 22;

__device__ unsigned int g_gather_timeouts;
// Polls of the first wait on each tile's load (the drain after a timeout
// always takes kWaitPolls).  Lowered only to exercise the timeout path.
__device__ long long g_first_wait_polls = kWaitPolls;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, long long polls)
{
    for (long long i = 0; i < polls; ++i) {
        uint32_t done;
        asm volatile("{\n .reg .pred p;\n"
                     " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                     " selp.u32 %0, 1, 0, p;\n}"
                     : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ void tma_load(uint32_t dst_smem, const char *src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(bar), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%0], [%1], %2, [%3];"
                 :: "r"(dst_smem), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void tma_store(char *dst, uint32_t src_smem, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(dst), "r"(src_smem), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

struct LeanArgs {
    const char *src[kMaxRows];    // active rows only
    char *dst[kMaxRows];
    int64_t bytes[kMaxRows];      // multiple of 16
    int64_t first_tile[kMaxRows + 1];   // row r owns tiles [first_tile[r], first_tile[r+1])
    int32_t rows;
};

__global__ void __launch_bounds__(32)
lean_gather_kernel(const __grid_constant__ LeanArgs a)
{
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t bars[kTmaStages];
    if (threadIdx.x != 0) return;
    const uint32_t ring0 = smem_addr(ring);
    for (int s = 0; s < kTmaStages; ++s)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(smem_addr(&bars[s])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");

    const int64_t total = a.first_tile[a.rows];
    const int64_t G = gridDim.x;
    const long long first_polls = g_first_wait_polls;
    auto tile_of = [&](int64_t m, const char *&src, char *&dst, uint32_t &bytes) -> bool {
        const int64_t t = blockIdx.x + m * G;
        if (t >= total) return false;
        // the row holding tile t: the last r with first_tile[r] <= t
        int lo = 0, hi = a.rows - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.first_tile[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int64_t off = (t - a.first_tile[lo]) * kTmaTile;
        const int64_t left = a.bytes[lo] - off;
        bytes = (uint32_t)(left < kTmaTile ? left : kTmaTile);
        src = a.src[lo] + off;
        dst = a.dst[lo] + off;
        return true;
    };

    int64_t issued = 0;   // loads issued (tiles m = 0 .. issued-1)
    for (; issued < kTmaStages; ++issued) {
        const char *src; char *dst; uint32_t bytes;
        if (!tile_of(issued, src, dst, bytes)) break;
        tma_load(ring0 + (uint32_t)(issued * kTmaTile), src, bytes,
                 smem_addr(&bars[issued % kTmaStages]));
    }
    bool ok = true;
    int64_t m = 0;
    for (; m < issued; ++m) {
        const int s = (int)(m % kTmaStages);
        const uint32_t parity = (uint32_t)((m / kTmaStages) & 1);
        if (!mbar_wait(smem_addr(&bars[s]), parity, first_polls)) { ok = false; break; }
        const char *src; char *dst; uint32_t bytes;
        tile_of(m, src, dst, bytes);
        tma_store(dst, ring0 + (uint32_t)(s * kTmaTile), bytes);
        // the buffer may take the next load once this store has read it
        const char *nsrc; char *ndst; uint32_t nbytes;
        if (tile_of(issued, nsrc, ndst, nbytes)) {
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            tma_load(ring0 + (uint32_t)(s * kTmaTile), nsrc, nbytes, smem_addr(&bars[s]));
            ++issued;
        }
    }
    if (!ok) {
        atomicAdd(&g_gather_timeouts, 1u);
        // drain: every load still in flight must land before the ring goes away
        for (int64_t k = m; k < issued; ++k) {     // tile m's own load included
            const int s = (int)(k % kTmaStages);
            if (!mbar_wait(smem_addr(&bars[s]), (uint32_t)((k / kTmaStages) & 1), kWaitPolls))
                atomicAdd(&g_gather_timeouts, 1u);
        }
    }
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
}  // namespace

cudaError_t launch_gather(const GatherArgs &a, int sms, cudaStream_t s)
{
    if (a.n <= 0 || a.shard_bytes <= 0) return cudaSuccess;
    const int per_sm = resident_blocks_per_sm(reinterpret_cast<const void *>(gather_kernel), kThreads);
    // each row (shard) gets up to twice as many blocks as fit on the GPU at
    // once, so one or two shards are in flight at any time
    const int64_t bx = rowcopy::row_blocks(a.shard_bytes, kThreads, (int64_t)sms * per_sm);
    dim3 grid((unsigned)bx, (unsigned)a.n);
    return launch_dependent(gather_kernel, grid, dim3(kThreads), 0, s, a);
}

cudaError_t launch_gather_rows(const GatherRowsArgs &a, int sms, cudaStream_t s)
{
    if (a.n <= 0) return cudaSuccess;
    if (a.n > kMaxRows) return cudaErrorInvalidValue;
    const int per_sm = resident_blocks_per_sm(reinterpret_cast<const void *>(gather_rows_kernel),
                                              kThreads);
    // each row gets the blocks its length needs, at most twice the resident
    // blocks (as launch_gather); rows are laid out one after another in the
    // grid, so they are dispatched in order and one or two are in flight
    const int64_t cap = 2 * (int64_t)sms * per_sm;
    GatherRowsArgs r = a;
    int64_t total = 0;
    for (int32_t y = 0; y < a.n; ++y) {
        r.first_block[y] = (int32_t)total;
        int64_t want = 0;
        if (a.src[y] && a.bytes[y] > 0) want = rowcopy::row_blocks(a.bytes[y], kThreads, cap / 2);
        total += want;
        if (total > 0x7fffffff) return cudaErrorInvalidValue;
    }
    r.first_block[a.n] = (int32_t)total;
    if (total == 0) return cudaSuccess;
    return launch_dependent(gather_rows_kernel, dim3((unsigned)total), dim3(kThreads), 0, s, r);
}

bool lean_gather_eligible(const GatherArgs &a)
{
    if (a.shard_bytes % 16) return false;
    for (int32_t k = 0; k < a.n; ++k) {
        if (!a.src[k]) continue;
        if (((uintptr_t)a.src[k] & 15) || ((uintptr_t)(a.dst + (int64_t)k * a.shard_bytes) & 15))
            return false;
    }
    return true;
}

namespace {

// Rows in the lean form: every active row 16-byte aligned at both ends with a
// length that is a multiple of 16 bytes.  Returns false when some row is not.
bool lean_rows(const void *const *src, char *const *dst, const int64_t *bytes, int32_t n,
               LeanArgs &l)
{
    memset(&l, 0, sizeof l);
    int64_t tiles = 0;
    for (int32_t y = 0; y < n; ++y) {
        if (!src[y] || bytes[y] <= 0) continue;
        if (bytes[y] % 16 || ((uintptr_t)src[y] & 15) || ((uintptr_t)dst[y] & 15)) return false;
        l.src[l.rows] = static_cast<const char *>(src[y]);
        l.dst[l.rows] = dst[y];
        l.bytes[l.rows] = bytes[y];
        l.first_tile[l.rows] = tiles;
        tiles += (bytes[y] + kTmaTile - 1) / kTmaTile;
        ++l.rows;
    }
    l.first_tile[l.rows] = tiles;
    return true;
}

cudaError_t launch_lean(const LeanArgs &l, int sms, cudaStream_t s)
{
    const int64_t total = l.first_tile[l.rows];
    if (l.rows == 0 || total == 0) return cudaSuccess;
    const int smem = kTmaStages * kTmaTile;
    static int attr_device = -1;   // the attribute is per device
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(lean_gather_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_device = dev;
    }
    const int blocks = (int)(total < sms ? total : sms);
    lean_gather_kernel<<<blocks, 32, smem, s>>>(l);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gather_lean(const GatherArgs &a, int sms, cudaStream_t s)
{
    if (a.n <= 0 || a.shard_bytes <= 0) return cudaSuccess;
    const void *src[kMaxRanks];
    char *dst[kMaxRanks];
    int64_t bytes[kMaxRanks];
    for (int32_t k = 0; k < a.n; ++k) {
        src[k] = a.src[k];
        dst[k] = a.dst + (int64_t)k * a.shard_bytes;
        bytes[k] = a.shard_bytes;
    }
    LeanArgs l;
    if (!lean_rows(src, dst, bytes, a.n, l)) return cudaErrorInvalidValue;
    return launch_lean(l, sms, s);
}

bool lean_gather_rows_eligible(const GatherRowsArgs &a)
{
    LeanArgs l;
    return a.n <= kMaxRows && lean_rows(a.src, a.dst, a.bytes, a.n, l);
}

cudaError_t launch_gather_rows_lean(const GatherRowsArgs &a, int sms, cudaStream_t s)
{
    if (a.n <= 0) return cudaSuccess;
    if (a.n > kMaxRows) return cudaErrorInvalidValue;
    LeanArgs l;
    if (!lean_rows(a.src, a.dst, a.bytes, a.n, l)) return cudaErrorInvalidValue;
    return launch_lean(l, sms, s);
}

cudaError_t lean_gather_timeouts(unsigned int *count)
{
    return cudaMemcpyFromSymbol(count, g_gather_timeouts, sizeof(unsigned int));
}

cudaError_t set_lean_first_wait_polls(long long polls)
{
    const long long v = polls < 0 ? kWaitPolls : polls;
    return cudaMemcpyToSymbol(g_first_wait_polls, &v, sizeof v);
}

}  // namespace zgb
