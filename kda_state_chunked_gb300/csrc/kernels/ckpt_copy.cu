// Object -> object copy through two page lists (checkpoint snapshot and restore).
//
// A checkpoint is read-only: a hit is copied into the request's private state, and a new
// checkpoint is written to fresh pages ("Cache de préfixe hybride KDA–MLA", §Les checkpoints
// sont en lecture seule).  Both directions are this one bandwidth-bound copy.
//
// The logical object [0, object_bytes) is cut at page boundaries: page p of the object is
// one contiguous run in the source pool page and one in the destination page, so a block
// copies a run with plain 128-bit loads and stores and no per-vector translation.
#include "common.cuh"

namespace kda {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int64_t kSliceBytes = 65536;   // bytes of one page run handled by one block

__global__ void __launch_bounds__(kCopyThreads) copy_objects_kernel(CopyArgs a, int slices) {
    const int P = a.pool.pages_per_object;
    const int obj = blockIdx.x / P;
    const int p = blockIdx.x % P;
    if (obj >= a.n) return;
    const int64_t run0 = (int64_t)p * a.pool.page_bytes;
    if (run0 >= a.object_bytes) return;
    const int64_t run = min(a.pool.page_bytes, a.object_bytes - run0);
    const int32_t sid = a.src_pages[(int64_t)obj * P + p];
    const int32_t did = a.dst_pages[(int64_t)obj * P + p];
    if ((uint32_t)sid >= (uint32_t)a.pool.num_pages || (uint32_t)did >= (uint32_t)a.pool.num_pages) {
        if (threadIdx.x == 0 && blockIdx.y == 0) flag_status(a.status, KDA_DEV_BAD_PAGE);
        return;
    }
    const int4 *src = reinterpret_cast<const int4 *>(a.pool.base + (int64_t)sid * a.pool.page_bytes);
    int4 *dst = reinterpret_cast<int4 *>(a.pool.base + (int64_t)did * a.pool.page_bytes);
    const int64_t nvec = run / 16;
    const int64_t per_slice = (nvec + slices - 1) / slices;
    const int64_t v0 = (int64_t)blockIdx.y * per_slice;
    const int64_t v1 = min(nvec, v0 + per_slice);
    const int64_t step = (int64_t)kCopyThreads * kCopyUnroll;
    for (int64_t base = v0; base < v1; base += step) {
        int4 r[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t v = base + threadIdx.x + (int64_t)u * kCopyThreads;
            if (v < v1) r[u] = __ldcs(src + v);
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t v = base + threadIdx.x + (int64_t)u * kCopyThreads;
            if (v < v1) __stcs(dst + v, r[u]);
        }
    }
}

// Page runs between the pool and a linear host buffer (write-back offload of checkpoints that
// leave the GPU, and prefetch before their reuse: "Infrastructure pour le RL à un million de
// jetons", §La solution : découpler la rétention de la résidence GPU).  The host buffer is
// pinned and mapped into the device address space, so the copy runs over the CPU-GPU link as
// plain 128-bit loads and stores.
__global__ void __launch_bounds__(kCopyThreads) host_copy_kernel(HostCopyArgs a, int slices) {
    const int P = a.pool.pages_per_object;
    const int obj = blockIdx.x / P;
    const int p = blockIdx.x % P;
    if (obj >= a.n) return;
    const int64_t run0 = (int64_t)p * a.pool.page_bytes;
    if (run0 >= a.object_bytes) return;
    const int64_t run = min(a.pool.page_bytes, a.object_bytes - run0);
    const int32_t id = a.pages[(int64_t)obj * P + p];
    if ((uint32_t)id >= (uint32_t)a.pool.num_pages) {
        if (threadIdx.x == 0 && blockIdx.y == 0) flag_status(a.status, KDA_DEV_BAD_PAGE);
        return;
    }
    int4 *pg = reinterpret_cast<int4 *>(a.pool.base + (int64_t)id * a.pool.page_bytes);
    int4 *hs = reinterpret_cast<int4 *>(a.host + (int64_t)obj * a.object_bytes + run0);
    const int4 *src = a.to_host ? pg : hs;
    int4 *dst = a.to_host ? hs : pg;
    const int64_t nvec = run / 16;
    const int64_t per_slice = (nvec + slices - 1) / slices;
    const int64_t v0 = (int64_t)blockIdx.y * per_slice;
    const int64_t v1 = min(nvec, v0 + per_slice);
    const int64_t step = (int64_t)kCopyThreads * kCopyUnroll;
    for (int64_t base = v0; base < v1; base += step) {
        int4 r[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t v = base + threadIdx.x + (int64_t)u * kCopyThreads;
            if (v < v1) r[u] = __ldcs(src + v);
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
            const int64_t v = base + threadIdx.x + (int64_t)u * kCopyThreads;
            if (v < v1) __stcs(dst + v, r[u]);
        }
    }
}

}  // namespace

cudaError_t launch_host_copy(const HostCopyArgs &a, cudaStream_t s) {
    if (a.n <= 0) return cudaSuccess;
    const int slices = (int)((a.pool.page_bytes + kSliceBytes - 1) / kSliceBytes);
    dim3 grid((unsigned)(a.n * a.pool.pages_per_object), (unsigned)slices);
    host_copy_kernel<<<grid, kCopyThreads, 0, s>>>(a, slices);
    return cudaGetLastError();
}

cudaError_t launch_copy_objects(const CopyArgs &a, cudaStream_t s) {
    if (a.n <= 0) return cudaSuccess;
    const int slices = (int)((a.pool.page_bytes + kSliceBytes - 1) / kSliceBytes);
    dim3 grid((unsigned)(a.n * a.pool.pages_per_object), (unsigned)slices);
    copy_objects_kernel<<<grid, kCopyThreads, 0, s>>>(a, slices);
    return cudaGetLastError();
}

}  // namespace kda
